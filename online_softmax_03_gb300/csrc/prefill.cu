// prefill.cu -- launcher for the tensor-core prefill kernel.
#include <atomic>
#include <climits>
#include <cmath>

#include "../../include/attn.h"
#include "internal.h"
#include "prefill_kernel.cuh"

namespace {
__device__ unsigned int g_prefill_status;

// Work counters of the persistent prefill kernel: per slot two 64-bit words
// {items taken, CTAs finished}, each (tag << 32) | count.  A launch made
// outside graph capture gets a fresh tag e and uses slot e % kWorkSlots of
// the first pool; its first fetch finds an older tag there and restarts the
// count, so nothing needs resetting afterwards.  A launch captured into a
// CUDA graph replays with the same tag, so it uses the second pool, and its
// last CTA frees the slot (tag 0) for the next replay.  A launch whose slot
// was taken over by a newer one (more than kWorkSlots launches of a pool in
// flight at once) stops and reports ATTN_ERR_IN_FLIGHT_LIMIT instead of
// sharing the count.
constexpr int kWorkSlots = ATTN_FWD_MAX_IN_FLIGHT;
__device__ unsigned long long g_prefill_work[2 * 2 * kWorkSlots];
std::atomic<unsigned int> g_launch_seq{0};
std::atomic<unsigned int> g_graph_seq{0};

// Tag of the next launch of a pool (never 0: 0 marks a free slot).
unsigned int next_epoch(std::atomic<unsigned int> &seq) {
  unsigned int e = seq.fetch_add(1) + 1;
  if (e == 0) e = seq.fetch_add(1) + 1;
  return e;
}

// Picks the pool, tag and slot of a launch (graph: captured into a CUDA
// graph).
void take_slot(bool graph, unsigned long long *work, attn_dev::PrefillParams &p) {
  p.graph_mode = graph ? 1 : 0;
  p.epoch = next_epoch(graph ? g_graph_seq : g_launch_seq);
  const int slot = (graph ? kWorkSlots : 0) + (int)(p.epoch % kWorkSlots);
  p.work = work + 2 * slot;
}

template <int D, bool kWindow>
int launch_d(const attn_host::PrefillArgs &a, unsigned int *status, unsigned long long *work,
             int sms) {
  using C = attn_dev::PrefillCfg<D>;
  CUtensorMap tq, tk, tv;
  const uint64_t bhq = (uint64_t)a.B * a.Hq, bhk = (uint64_t)a.B * a.Hkv;
  if (!attn_host::encode_tmap_3d_bf16(&tq, a.q, D, a.Tq, bhq, C::CHUNK, C::BM, 1, C::SPAN) ||
      !attn_host::encode_tmap_3d_bf16(&tk, a.k, D, a.Tk, bhk, C::CHUNK, C::BN, 1, C::SPAN) ||
      !attn_host::encode_tmap_3d_bf16(&tv, a.v, D, a.Tk, bhk, C::CHUNK, C::BN, 1, C::SPAN))
    return ATTN_ERR_CUDA;
  attn_dev::PrefillParams p{};
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
  {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(a.stream, &cs) != cudaSuccess) return ATTN_ERR_CUDA;
    take_slot(cs == cudaStreamCaptureStatusActive, work, p);
  }
  // Persistent: one CTA per SM (each holds all of an SM's tensor memory);
  // CTAs take work items from the slot's counter until the list is done.
  const uint64_t grid = items < (uint64_t)sms ? items : (uint64_t)sms;
  auto kern = attn_dev::prefill_fwd_kernel<D, kWindow, false>;
  if (attn_host::ensure_smem_limit((const void *)kern, (int)C::SMEM_BYTES) != ATTN_OK)
    return ATTN_ERR_CUDA;
  kern<<<(unsigned)grid, C::THREADS, C::SMEM_BYTES, a.stream>>>(tq, tk, tv, p);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}
// Packed batches: list every (sequence, query-tile pair) heaviest first, as
// {entries, 0, (b, pair) x entries}.  The weight of a pair is the number of
// K/V tiles its two query tiles visit; a counting sort over weight classes
// (pairs of more than kPlanBins - 1 tiles share the top class) orders the
// list.  The order of equal weights varies from run to run, which changes
// nothing in the results: every entry owns its output rows.  Offsets that
// break the documented rules leave the list empty and record
// ATTN_ERR_INVALID_ARG.
constexpr int kPlanThreads = 1024;
constexpr int kPlanBins = 8192;
constexpr int kBinsPerThread = kPlanBins / kPlanThreads;

__device__ __forceinline__ int pair_weight(int nq, int nk, int pair, int causal, int window) {
  const int n_kt = (nk + 127) / 128;
  if (!causal) return n_kt;
  const int last = min(pair * 256 + 255, nq - 1);
  const int hi = min(n_kt, (last + nk - nq) / 128 + 1);
  if (window <= 0) return hi;
  // under a window the pair's first row starts the tiles it visits
  return hi - max(0, pair * 256 + nk - nq - window + 1) / 128;
}

__global__ void __launch_bounds__(kPlanThreads)
    varlen_plan_kernel(const int *__restrict__ cu_q, const int *__restrict__ cu_k, int B,
                       int total_q, int total_k, int max_q, int max_k, int causal,
                       int window, int *__restrict__ list, long long capacity,
                       unsigned int *__restrict__ status) {
  __shared__ int hist[kPlanBins];
  __shared__ int part[kPlanThreads];
  __shared__ int bad;
  const int tid = threadIdx.x;
  if (tid == 0) bad = (cu_q[0] != 0 || cu_k[0] != 0);
  for (int i = tid; i < kPlanBins; i += kPlanThreads) hist[i] = 0;
  __syncthreads();
  for (int b = tid; b < B; b += kPlanThreads) {
    const long long q1 = cu_q[b + 1], k1 = cu_k[b + 1];
    const long long nq = q1 - cu_q[b], nk = k1 - cu_k[b];
    if (nq < 0 || nk < 0 || q1 > total_q || k1 > total_k || nq > max_q || nk > max_k ||
        (nq > 0 && nk < 1) || (causal && nq > nk))
      bad = 1;
  }
  __syncthreads();
  if (bad) {
    if (tid == 0) {
      list[0] = 0;
      list[1] = 0;
      atomicMax(status, 1u);  // ATTN_ERR_INVALID_ARG
    }
    return;
  }
  // Offsets are valid from here on: 0 <= cu[b] <= cu[b+1] <= total.
  for (int b = tid; b < B; b += kPlanThreads) {
    const int nq = cu_q[b + 1] - cu_q[b], nk = cu_k[b + 1] - cu_k[b];
    for (int pr = 0; (long long)pr * 256 < nq; ++pr) {
      const int w = min(pair_weight(nq, nk, pr, causal, window), kPlanBins - 1);
      atomicAdd(&hist[kPlanBins - 1 - w], 1);  // heaviest class first
    }
  }
  __syncthreads();
  // Exclusive prefix sum over the classes: per-thread runs, then a scan of
  // the run totals.
  int run = 0;
#pragma unroll
  for (int i = 0; i < kBinsPerThread; ++i) run += hist[tid * kBinsPerThread + i];
  part[tid] = run;
  __syncthreads();
  for (int off = 1; off < kPlanThreads; off <<= 1) {
    const int add = tid >= off ? part[tid - off] : 0;
    __syncthreads();
    part[tid] += add;
    __syncthreads();
  }
  const int total = part[kPlanThreads - 1];
  int start = part[tid] - run;
#pragma unroll
  for (int i = 0; i < kBinsPerThread; ++i) {
    const int c = hist[tid * kBinsPerThread + i];
    hist[tid * kBinsPerThread + i] = start;
    start += c;
  }
  __syncthreads();
  for (int b = tid; b < B; b += kPlanThreads) {
    const int nq = cu_q[b + 1] - cu_q[b], nk = cu_k[b + 1] - cu_k[b];
    for (int pr = 0; (long long)pr * 256 < nq; ++pr) {
      const int w = min(pair_weight(nq, nk, pr, causal, window), kPlanBins - 1);
      const int pos = atomicAdd(&hist[kPlanBins - 1 - w], 1);
      if (pos < capacity) {
        list[2 + 2 * pos] = b;
        list[3 + 2 * pos] = pr;
      }
    }
  }
  if (tid == 0) {
    if (total > capacity) {  // cannot happen for offsets within the documented rules
      list[0] = 0;
      atomicMax(status, 1u);
    } else {
      list[0] = total;
    }
    list[1] = 0;
  }
}

template <int D>
int launch_varlen(const attn_host::PrefillArgs &a, unsigned int *status,
                  unsigned long long *work, int sms) {
  using C = attn_dev::PrefillCfg<D>;
  const long long capacity = attn_host::varlen_list_capacity(a.B, a.total_q, a.Tq);
  if (capacity < 1 || capacity * a.Hq > (long long)INT_MAX) return ATTN_ERR_INVALID_ARG;
  // (D, heads, tokens) views of the token-major tensors: a box is 128
  // consecutive tokens of one head.
  CUtensorMap tq, tk, tv;
  if (!attn_host::encode_tmap_3d_bf16(&tq, a.q, D, a.Hq, a.total_q, C::CHUNK, 1, C::BM,
                                      C::SPAN) ||
      !attn_host::encode_tmap_3d_bf16(&tk, a.k, D, a.Hkv, a.total_k, C::CHUNK, 1, C::BN,
                                      C::SPAN) ||
      !attn_host::encode_tmap_3d_bf16(&tv, a.v, D, a.Hkv, a.total_k, C::CHUNK, 1, C::BN,
                                      C::SPAN))
    return ATTN_ERR_CUDA;
  attn_dev::PrefillParams p{};
  p.o = static_cast<__nv_bfloat16 *>(a.o);
  p.lse = a.lse;
  p.status = status;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.group = a.Hq / a.Hkv;
  p.Tq = a.Tq;
  p.Tk = a.Tk;
  p.n_bh = a.Hq;
  {
    // Heads per scheduling group: as many as keep the group's K and V
    // (about 48 MiB over all sequences) resident in L2.
    const uint64_t kv_bytes = 2ull * (uint64_t)a.total_k * D * 2;
    uint64_t g = ((48ull << 20) / kv_bytes) * (uint64_t)(a.Hq / a.Hkv);
    if (g < 1) g = 1;
    if (g > (uint64_t)a.Hq) g = a.Hq;
    p.head_group = (int)g;
  }
  p.causal = a.causal;
  p.window = a.window;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.wait_ns = a.wait_ns;
  p.inject = a.inject;
  p.cu_q = a.cu_q;
  p.cu_k = a.cu_k;
  p.vl_list = static_cast<const int *>(a.workspace);
  p.total_q = a.total_q;
  {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(a.stream, &cs) != cudaSuccess) return ATTN_ERR_CUDA;
    take_slot(cs == cudaStreamCaptureStatusActive, work, p);
  }
  varlen_plan_kernel<<<1, kPlanThreads, 0, a.stream>>>(
      a.cu_q, a.cu_k, a.B, a.total_q, a.total_k, a.Tq, a.Tk, a.causal, a.window,
      static_cast<int *>(a.workspace), capacity, status);
  if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
  const long long items = capacity * a.Hq;  // upper bound; the list holds the count
  const long long grid = items < sms ? items : sms;
  // the sliding window inside each sequence compiles a variant of its own
  auto kern = a.window > 0 ? attn_dev::prefill_fwd_kernel<D, true, true>
                           : attn_dev::prefill_fwd_kernel<D, false, true>;
  if (attn_host::ensure_smem_limit((const void *)kern, (int)C::SMEM_BYTES) != ATTN_OK)
    return ATTN_ERR_CUDA;
  kern<<<(unsigned)grid, C::THREADS, C::SMEM_BYTES, a.stream>>>(tq, tk, tv, p);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}
}  // namespace

namespace attn_host {

long long varlen_list_capacity(int B, int total_q, int max_seqlen_q) {
  if (B < 1 || total_q < 1 || max_seqlen_q < 1) return 0;
  const long long by_max = (long long)B * ((max_seqlen_q + 255) / 256);
  const long long by_total = (long long)(total_q + 255) / 256 + B;
  return by_max < by_total ? by_max : by_total;
}

size_t varlen_workspace_bytes_for(int B, int total_q, int max_seqlen_q) {
  const long long cap = varlen_list_capacity(B, total_q, max_seqlen_q);
  if (cap < 1) return 0;
  return ((size_t)(2 + 2 * cap) * sizeof(int) + 15) / 16 * 16;
}

int prefill_launch(const PrefillArgs &a) {
  int sms = 0;
  const int rc = check_device_sm103(&sms);
  if (rc != ATTN_OK) return rc;
  unsigned int *status = nullptr;
  unsigned long long *work = nullptr;
  if (symbol_address((const void *)&g_prefill_status, reinterpret_cast<void **>(&status)) !=
          ATTN_OK ||
      symbol_address((const void *)&g_prefill_work, reinterpret_cast<void **>(&work)) !=
          ATTN_OK)
    return ATTN_ERR_CUDA;
  if (a.varlen) {
    switch (a.d) {
      case 32: return launch_varlen<32>(a, status, work, sms);
      case 64: return launch_varlen<64>(a, status, work, sms);
      case 128: return launch_varlen<128>(a, status, work, sms);
      default: return ATTN_ERR_UNSUPPORTED;
    }
  }
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
