// prefill.cu -- launcher for the tensor-core prefill kernel.
#include <climits>
#include <cmath>

#include "../../include/attn.h"
#include "internal.h"
#include "prefill_kernel.cuh"

namespace {
__device__ unsigned int g_prefill_status;

template <int D>
int launch_d(const attn_host::PrefillArgs &a, unsigned int *status) {
  using C = attn_dev::PrefillCfg<D>;
  CUtensorMap tq, tk, tv, to;
  const uint64_t bhq = (uint64_t)a.B * a.Hq, bhk = (uint64_t)a.B * a.Hkv;
  if (!attn_host::encode_tmap_3d_bf16(&tq, a.q, D, a.Tq, bhq, C::CHUNK, C::BM, C::SPAN) ||
      !attn_host::encode_tmap_3d_bf16(&tk, a.k, D, a.Tk, bhk, C::CHUNK, C::BN, C::SPAN) ||
      !attn_host::encode_tmap_3d_bf16(&tv, a.v, D, a.Tk, bhk, C::CHUNK, C::BN, C::SPAN) ||
      !attn_host::encode_tmap_3d_bf16(&to, a.o, D, a.Tq, bhq, C::CHUNK, C::BM, C::SPAN))
    return ATTN_ERR_CUDA;
  attn_dev::PrefillParams p;
  p.lse = a.lse;
  p.status = status;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.group = a.Hq / a.Hkv;
  p.Tq = a.Tq;
  p.Tk = a.Tk;
  p.n_qt = (a.Tq + C::NQ * C::BM - 1) / (C::NQ * C::BM);
  p.causal = a.causal;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.wait_ns = a.wait_ns;
  p.inject = a.inject;
  const uint64_t grid = bhq * (uint64_t)p.n_qt;
  if (grid > (uint64_t)INT_MAX) return ATTN_ERR_INVALID_ARG;
  auto kern = attn_dev::prefill_fwd_kernel<D>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)C::SMEM_BYTES) != cudaSuccess)
    return ATTN_ERR_CUDA;
  kern<<<(unsigned)grid, C::THREADS, C::SMEM_BYTES, a.stream>>>(tq, tk, tv, to, p);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}
}  // namespace

namespace attn_host {

int prefill_launch(const PrefillArgs &a) {
  unsigned int *status = nullptr;
  if (cudaGetSymbolAddress(reinterpret_cast<void **>(&status), g_prefill_status) !=
      cudaSuccess)
    return ATTN_ERR_CUDA;
  switch (a.d) {
    case 32: return launch_d<32>(a, status);
    case 64: return launch_d<64>(a, status);
    case 128: return launch_d<128>(a, status);
    default: return ATTN_ERR_UNSUPPORTED;
  }
}

int prefill_take_status(cudaStream_t s, unsigned int *out) {
  const unsigned int zero = 0;
  if (cudaMemcpyFromSymbolAsync(out, g_prefill_status, sizeof(unsigned int), 0,
                                cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess ||
      cudaMemcpyToSymbolAsync(g_prefill_status, &zero, sizeof zero, 0,
                              cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return ATTN_OK;
}

}  // namespace attn_host
