// decode.cu -- launchers for the split-KV decode kernels.
#include <algorithm>
#include <atomic>
#include <climits>

#include "../../include/attn.h"
#include "decode_kernel.cuh"
#include "internal.h"

namespace {
__device__ unsigned int g_decode_status;

template <int D, int GP, bool kPaged>
int launch_split(const attn_dev::DecodeParams &p, dim3 grid, cudaStream_t st) {
  using C = attn_dev::DecodeCfg<D, GP>;
  auto kern = attn_dev::decode_split_kernel<D, GP, kPaged>;
  if (attn_host::ensure_smem_limit((const void *)kern, (int)C::SMEM_BYTES) != ATTN_OK)
    return ATTN_ERR_CUDA;
  kern<<<grid, C::THREADS, C::SMEM_BYTES, st>>>(p);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

// Resident split CTAs per SM, queried once per device.
template <int D, int GP>
int resident_ctas(int *out) {
  using C = attn_dev::DecodeCfg<D, GP>;
  constexpr int kMaxDevices = 64;
  static std::atomic<int> cached[kMaxDevices];  // 0 = not queried yet
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return ATTN_ERR_CUDA;
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    auto kern = attn_dev::decode_split_kernel<D, GP, false>;
    if (attn_host::ensure_smem_limit((const void *)kern, (int)C::SMEM_BYTES) != ATTN_OK ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, C::THREADS, C::SMEM_BYTES) !=
            cudaSuccess)
      return ATTN_ERR_CUDA;
    if (n < 1) n = 1;
    cached[dev].store(n, std::memory_order_relaxed);
  }
  *out = n;
  return ATTN_OK;
}

template <int D>
int dispatch_split(int gp, bool paged, const attn_dev::DecodeParams &p, dim3 grid,
                   cudaStream_t st) {
  if (paged)
    return gp == 4 ? launch_split<D, 4, true>(p, grid, st) : launch_split<D, 8, true>(p, grid, st);
  return gp == 4 ? launch_split<D, 4, false>(p, grid, st) : launch_split<D, 8, false>(p, grid, st);
}

template <int D>
int dispatch_resident(int gp, int *out) {
  return gp == 4 ? resident_ctas<D, 4>(out) : resident_ctas<D, 8>(out);
}

// Choose the number of KV splits: model each CTA's time as proportional to
// its chunk plus a fixed start-up cost, run them in waves of `slots`
// resident CTAs, and take the split count with the smallest total.
int plan_splits(int pairs, int slots, int Tk, int max_splits) {
  constexpr long long kStartupKeys = 64;
  long long best_cost = LLONG_MAX;
  int best = 1;
  for (int ns = 1; ns <= max_splits; ++ns) {
    const long long chunk = ((long long)(Tk + ns - 1) / ns + 31) / 32 * 32;
    const long long eff = (Tk + chunk - 1) / chunk;
    if (eff != ns) continue;
    const long long waves = ((long long)pairs * ns + slots - 1) / slots;
    const long long cost = waves * (chunk + kStartupKeys);
    if (cost < best_cost) {
      best_cost = cost;
      best = ns;
    }
  }
  return best;
}
}  // namespace

namespace attn_host {

int decode_max_splits(int Tk) { return std::max(1, std::min(64, (Tk + 255) / 256)); }

size_t decode_workspace_bytes_for(int B, int Hq, int Tk, int d) {
  const size_t rows = (size_t)B * Hq * decode_max_splits(Tk);
  return rows * (size_t)d * sizeof(float) + rows * 2 * sizeof(float);
}

int decode_launch(const DecodeArgs &a) {
  int sms = 0;
  int rc = check_device_sm103(&sms);
  if (rc != ATTN_OK) return rc;
  unsigned int *status = nullptr;
  if (symbol_address((const void *)&g_decode_status, reinterpret_cast<void **>(&status)) !=
      ATTN_OK)
    return ATTN_ERR_CUDA;
  const int group = a.Hq / a.Hkv;
  const int gp = group <= 4 ? 4 : 8;
  const int n_hc = (group + gp - 1) / gp;
  if ((long long)a.Hkv * n_hc > 65535 || a.B > 65535) return ATTN_ERR_INVALID_ARG;
  int per_sm = 0;
  switch (a.d) {
    case 32: rc = dispatch_resident<32>(gp, &per_sm); break;
    case 64: rc = dispatch_resident<64>(gp, &per_sm); break;
    case 128: rc = dispatch_resident<128>(gp, &per_sm); break;
    default: return ATTN_ERR_UNSUPPORTED;
  }
  if (rc != ATTN_OK) return rc;
  const int max_s = decode_max_splits(a.Tk);
  const int pairs = a.B * a.Hkv * n_hc;
  const int nsplit = plan_splits(pairs, std::max(1, sms * std::max(1, per_sm)), a.Tk, max_s);
  const int chunk = ((a.Tk + nsplit - 1) / nsplit + 31) / 32 * 32;
  const size_t rows = (size_t)a.B * a.Hq;
  const size_t need = rows * nsplit * (size_t)a.d * sizeof(float) + rows * nsplit * 2 * sizeof(float);
  if (need > a.workspace_bytes) return ATTN_ERR_WORKSPACE;

  attn_dev::DecodeParams p;
  p.q = static_cast<const __nv_bfloat16 *>(a.q);
  p.k = static_cast<const __nv_bfloat16 *>(a.k);
  p.v = static_cast<const __nv_bfloat16 *>(a.v);
  p.part_acc = static_cast<float *>(a.workspace);
  p.part_ml = p.part_acc + rows * nsplit * a.d;
  p.status = status;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.group = group;
  p.Tk = a.Tk;
  p.nsplit = nsplit;
  p.chunk = chunk;
  p.n_hc = n_hc;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.wait_ns = a.wait_ns;
  p.inject = a.inject;
  p.block_table = a.block_table;
  p.seq_lens = a.seq_lens;
  p.page_shift = 0;
  while (a.paged && (1 << p.page_shift) < a.page_size) ++p.page_shift;
  p.max_pages = a.max_pages;
  p.num_pages = a.num_pages;
  const dim3 grid(nsplit, a.Hkv * n_hc, a.B);
  switch (a.d) {
    case 32: rc = dispatch_split<32>(gp, a.paged, p, grid, a.stream); break;
    case 64: rc = dispatch_split<64>(gp, a.paged, p, grid, a.stream); break;
    default: rc = dispatch_split<128>(gp, a.paged, p, grid, a.stream); break;
  }
  if (rc != ATTN_OK) return rc;
  const unsigned cblocks = (unsigned)((rows + 3) / 4);
  auto *o = static_cast<__nv_bfloat16 *>(a.o);
  switch (a.d) {
    case 32:
      attn_dev::decode_combine_kernel<32><<<cblocks, 128, 0, a.stream>>>(
          p.part_acc, p.part_ml, o, a.lse, (int)rows, nsplit);
      break;
    case 64:
      attn_dev::decode_combine_kernel<64><<<cblocks, 128, 0, a.stream>>>(
          p.part_acc, p.part_ml, o, a.lse, (int)rows, nsplit);
      break;
    default:
      attn_dev::decode_combine_kernel<128><<<cblocks, 128, 0, a.stream>>>(
          p.part_acc, p.part_ml, o, a.lse, (int)rows, nsplit);
      break;
  }
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int decode_take_status(cudaStream_t s, unsigned int *out) {
  const unsigned int zero = 0;
  if (cudaMemcpyFromSymbolAsync(out, g_decode_status, sizeof(unsigned int), 0,
                                cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess ||
      cudaMemcpyToSymbolAsync(g_decode_status, &zero, sizeof zero, 0,
                              cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return ATTN_OK;
}

}  // namespace attn_host
