// backward.cu -- launcher for the attention backward kernels.
#include <cmath>
#include <type_traits>

#include "../../include/attn.h"
#include "backward_kernel.cuh"
#include "internal.h"

namespace {
__device__ unsigned int g_bwd_status;

// Launch the key-tile kernel with its tensor maps: K, V (128-key boxes), Q
// and dO (C::BM-query boxes), and, for the 128-query kernel, the fp32 dQ
// accumulator it reduces into by TMA.
template <int D, typename C, typename Kern>
int launch_main(const attn_host::BwdArgs &a, Kern kern, const attn_dev::BwdParams &p,
                float *dq_acc, uint64_t bhq, uint64_t bhk, bool dq_map) {
  CUtensorMap tq, tk, tv, tdo, tdq;
  if (!attn_host::encode_tmap_3d_bf16(&tq, a.q, D, a.Tq, bhq, C::CHUNK, C::BM, 1, C::SPAN) ||
      !attn_host::encode_tmap_3d_bf16(&tdo, a.dout, D, a.Tq, bhq, C::CHUNK, C::BM, 1, C::SPAN) ||
      !attn_host::encode_tmap_3d_bf16(&tk, a.k, D, a.Tk, bhk, C::CHUNK, C::BN, 1, C::SPAN) ||
      !attn_host::encode_tmap_3d_bf16(&tv, a.v, D, a.Tk, bhk, C::CHUNK, C::BN, 1, C::SPAN) ||
      (dq_map && !attn_host::encode_tmap_3d_f32(&tdq, dq_acc, D, a.Tq, bhq, 32, C::BM, 1)))
    return ATTN_ERR_CUDA;
  if (attn_host::ensure_smem_limit((const void *)kern, (int)C::SMEM_BYTES) != ATTN_OK)
    return ATTN_ERR_CUDA;
  const int n_kt = (a.Tk + C::BN - 1) / C::BN;
  const dim3 grid(n_kt, (unsigned)bhk);
  if constexpr (std::is_same<C, attn_dev::BwdBm128Cfg<D>>::value) {
    // dK and dV leave by TMA stores of the same boxes as K and V
    CUtensorMap tdk, tdv;
    if (!attn_host::encode_tmap_3d_bf16(&tdk, a.dk, D, a.Tk, bhk, C::CHUNK, C::BN, 1, C::SPAN) ||
        !attn_host::encode_tmap_3d_bf16(&tdv, a.dv, D, a.Tk, bhk, C::CHUNK, C::BN, 1, C::SPAN))
      return ATTN_ERR_CUDA;
    kern<<<grid, C::THREADS, C::SMEM_BYTES, a.stream>>>(tq, tk, tv, tdo, tdk, tdv, p);
  } else
    kern<<<grid, C::THREADS, C::SMEM_BYTES, a.stream>>>(tq, tk, tv, tdo, tdq, p);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

template <int D>
int launch_bwd(const attn_host::BwdArgs &a, unsigned int *status) {
  constexpr int kRowPad = 128;  // query rows are padded to whole 128-row tiles
  const int Tq_pad = (a.Tq + kRowPad - 1) / kRowPad * kRowPad;
  const uint64_t bhq = (uint64_t)a.B * a.Hq, bhk = (uint64_t)a.B * a.Hkv;
  if (bhk > 65535) return ATTN_ERR_INVALID_ARG;
  float *dq_acc = static_cast<float *>(a.workspace);
  // per 64-query block, 16 bf16 per row: the aux operand that folds L and D
  // into S^T and dP^T
  uint8_t *aux = reinterpret_cast<uint8_t *>(dq_acc + bhq * (uint64_t)a.Tq * D);

  // 1. the aux rows (L and D = rowsum(dO o O)); zero the dQ accumulator
  {
    const uint64_t warps = bhq * (uint64_t)Tq_pad;
    const uint64_t blocks = (warps * 32 + 255) / 256;
    if (blocks > 0x7fffffffull) return ATTN_ERR_INVALID_ARG;
    attn_dev::attn_bwd_prep_kernel<D><<<(unsigned)blocks, 256, 0, a.stream>>>(
        static_cast<const __nv_bfloat16 *>(a.o), static_cast<const __nv_bfloat16 *>(a.dout),
        a.lse, dq_acc, aux, 1.f / a.scale, (int)bhq, a.Tq, Tq_pad);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
  }
  // 2. dK, dV per key tile; dQ accumulated
  attn_dev::BwdParams p{};
  p.dk = static_cast<__nv_bfloat16 *>(a.dk);
  p.dv = static_cast<__nv_bfloat16 *>(a.dv);
  p.aux = aux;
  p.dq_acc = dq_acc;
  p.status = status;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.group = a.Hq / a.Hkv;
  p.Tq = a.Tq;
  p.Tk = a.Tk;
  p.Tq_pad = Tq_pad;
  p.n_qt = Tq_pad / 128;
  p.causal = a.causal;
  p.window = a.window;
  p.scale = a.scale;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.wait_ns = a.wait_ns;
  p.inject = a.inject;
  int rc;
  if constexpr (D >= 64)
    rc = launch_main<D, attn_dev::BwdBm128Cfg<D>>(a, attn_dev::attn_bwd_bm128_kernel<D>, p,
                                                 dq_acc, bhq, bhk, false);
  else
    rc = launch_main<D, attn_dev::BwdCfg<D>>(a, attn_dev::attn_bwd_kernel<D>, p, dq_acc, bhq,
                                             bhk, true);
  if (rc != ATTN_OK) return rc;
  // 3. dQ = scale * accumulator in bf16
  {
    const size_t n4 = bhq * (size_t)a.Tq * D / 4;
    const size_t blocks = (n4 + 255) / 256 < 152 * 16 ? (n4 + 255) / 256 : 152 * 16;
    attn_dev::attn_bwd_dq_kernel<<<(unsigned)blocks, 256, 0, a.stream>>>(
        reinterpret_cast<const float4 *>(dq_acc), static_cast<uint2 *>(a.dq), n4, a.scale);
  }
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}
}  // namespace

namespace attn_host {

size_t bwd_workspace_bytes_for(int B, int Hq, int Tq, int d) {
  const size_t tq_pad = ((size_t)Tq + 127) / 128 * 128;
  const size_t rows = (size_t)B * Hq;
  // fp32 dQ accumulator, then 32 bytes of aux operand per padded query row
  return rows * (size_t)Tq * d * sizeof(float) + rows * tq_pad * 32;
}

int bwd_launch(const BwdArgs &a) {
  int rc = check_device_sm103(nullptr);
  if (rc != ATTN_OK) return rc;
  unsigned int *status = nullptr;
  if (symbol_address((const void *)&g_bwd_status, reinterpret_cast<void **>(&status)) !=
      ATTN_OK)
    return ATTN_ERR_CUDA;
  switch (a.d) {
    case 32: return launch_bwd<32>(a, status);
    case 64: return launch_bwd<64>(a, status);
    case 128: return launch_bwd<128>(a, status);
    default: return ATTN_ERR_UNSUPPORTED;
  }
}

int bwd_take_status(cudaStream_t s, unsigned int *out) {
  const unsigned int zero = 0;
  if (cudaMemcpyFromSymbolAsync(out, g_bwd_status, sizeof(unsigned int), 0,
                                cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess ||
      cudaMemcpyToSymbolAsync(g_bwd_status, &zero, sizeof zero, 0, cudaMemcpyHostToDevice,
                              s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return ATTN_OK;
}

}  // namespace attn_host
