// prefill.cu -- launcher for the tensor-core prefill kernel.
#include <atomic>
#include <climits>
#include <cmath>

#include "../../include/attn.h"
#include "internal.h"
#include "prefill_kernel.cuh"

namespace {
__device__ unsigned int g_prefill_status;

// Work counters of the persistent prefill kernel: one {next item, finished
// CTAs} pair per launch slot.  A launch takes the next slot in turn, finds it
// zero and leaves it zero (its last CTA resets it), so up to kWorkSlots
// launches may be in flight at once on different streams.
constexpr int kWorkSlots = 64;
__device__ unsigned int g_prefill_work[2 * kWorkSlots];
std::atomic<unsigned int> g_launch_seq{0};

template <int D, bool kWindow>
int launch_d(const attn_host::PrefillArgs &a, unsigned int *status, unsigned int *work,
             int sms) {
  using C = attn_dev::PrefillCfg<D>;
  CUtensorMap tq, tk, tv;
  const uint64_t bhq = (uint64_t)a.B * a.Hq, bhk = (uint64_t)a.B * a.Hkv;
  if (!attn_host::encode_tmap_3d_bf16(&tq, a.q, D, a.Tq, bhq, C::CHUNK, C::BM, C::SPAN) ||
      !attn_host::encode_tmap_3d_bf16(&tk, a.k, D, a.Tk, bhk, C::CHUNK, C::BN, C::SPAN) ||
      !attn_host::encode_tmap_3d_bf16(&tv, a.v, D, a.Tk, bhk, C::CHUNK, C::BN, C::SPAN))
    return ATTN_ERR_CUDA;
  attn_dev::PrefillParams p;
  p.o = static_cast<__nv_bfloat16 *>(a.o);
  p.lse = a.lse;
  p.status = status;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.group = a.Hq / a.Hkv;
  p.Tq = a.Tq;
  p.Tk = a.Tk;
  p.n_qt = (a.Tq + C::NQ * C::BM - 1) / (C::NQ * C::BM);
  p.n_bh = (int)bhq;
  {
    // Heads per scheduling group: as many as keep the group's K and V
    // (about 48 MiB) resident in L2 while its CTAs run.
    const uint64_t kv_bytes = 2ull * (uint64_t)a.Tk * D * 2;
    const uint64_t budget = 48ull << 20;
    uint64_t g = (budget / kv_bytes) * (uint64_t)(a.Hq / a.Hkv);
    if (g < 1) g = 1;
    if (g > bhq) g = bhq;
    p.head_group = (int)g;
  }
  p.causal = a.causal;
  p.window = a.window;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.wait_ns = a.wait_ns;
  p.inject = a.inject;
  const uint64_t items = bhq * (uint64_t)p.n_qt;
  if (items > (uint64_t)INT_MAX) return ATTN_ERR_INVALID_ARG;
  p.n_items = (int)items;
  p.work = work + 2 * (g_launch_seq.fetch_add(1) % kWorkSlots);
  // Persistent: one CTA per SM (each holds all of an SM's tensor memory);
  // CTAs take work items from the slot's counter until the list is done.
  const uint64_t grid = items < (uint64_t)sms ? items : (uint64_t)sms;
  auto kern = attn_dev::prefill_fwd_kernel<D, kWindow>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)C::SMEM_BYTES) != cudaSuccess)
    return ATTN_ERR_CUDA;
  kern<<<(unsigned)grid, C::THREADS, C::SMEM_BYTES, a.stream>>>(tq, tk, tv, p);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}
}  // namespace

namespace attn_host {

int prefill_launch(const PrefillArgs &a) {
  int sms = 0;
  const int rc = check_device_sm103(&sms);
  if (rc != ATTN_OK) return rc;
  unsigned int *status = nullptr, *work = nullptr;
  if (cudaGetSymbolAddress(reinterpret_cast<void **>(&status), g_prefill_status) !=
          cudaSuccess ||
      cudaGetSymbolAddress(reinterpret_cast<void **>(&work), g_prefill_work) != cudaSuccess)
    return ATTN_ERR_CUDA;
  const bool win = a.window > 0;
  switch (a.d) {
    case 32: return win ? launch_d<32, true>(a, status, work, sms)
                        : launch_d<32, false>(a, status, work, sms);
    case 64: return win ? launch_d<64, true>(a, status, work, sms)
                        : launch_d<64, false>(a, status, work, sms);
    case 128: return win ? launch_d<128, true>(a, status, work, sms)
                         : launch_d<128, false>(a, status, work, sms);
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
