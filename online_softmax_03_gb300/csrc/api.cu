// api.cu -- the C ABI: argument validation (before any CUDA call), device
// checks, TMA descriptor encoding, and dispatch to the kernel launchers.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/attn.h"
#include "internal.h"

#define ATTN_API extern "C" __attribute__((visibility("default")))

namespace {

constexpr unsigned long long kDefaultWaitNs = 1000000000ull;  // 1 s
std::atomic<unsigned long long> g_wait_ns{kDefaultWaitNs};
std::atomic<int> g_inject{0};

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *,
                                   const cuuint32_t *, const cuuint32_t *,
                                   CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Shared argument checks of attn_fwd / attn_decode.  No CUDA call.
int validate(const void *q, const void *k, const void *v, const void *o,
             const float *lse, int B, int Hq, int Hkv, int Tq, int Tk, int d,
             int causal, float scale, float *scale_out) {
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || Hq < 1 || Hkv < 1 || Tq < 1 || Tk < 1) return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (causal && Tq > Tk) return ATTN_ERR_INVALID_ARG;
  if (!(std::isfinite(scale) && scale >= 0.f)) return ATTN_ERR_INVALID_ARG;
  if (d != 32 && d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(lse, 4))
    return ATTN_ERR_MISALIGNED;
  *scale_out = (scale == 0.f) ? 1.f / std::sqrt((float)d) : scale;
  return ATTN_OK;
}

}  // namespace

namespace attn_host {

// Per-device facts and lookups made once, on the first call that runs on a
// device, so that a call's host work is validation, tensor-map encoding and
// the launch.
namespace {
constexpr int kMaxDevices = 64;
constexpr int kMaxCached = 64;  // symbols or kernels remembered per device

struct DeviceFacts {
  int state = 0;  // 0 = not queried, 1 = sm_103, 2 = another GPU
  int sms = 0;
};

std::mutex g_cache_mu;
DeviceFacts g_facts[kMaxDevices];
struct CachedPtr {
  const void *key;
  void *value;
};
CachedPtr g_symbols[kMaxDevices][kMaxCached];
int g_n_symbols[kMaxDevices];
const void *g_smem_set[kMaxDevices][kMaxCached];
int g_smem_bytes[kMaxDevices][kMaxCached];
int g_n_smem[kMaxDevices];

int current_device(int *dev) {
  if (cudaGetDevice(dev) != cudaSuccess) return ATTN_ERR_CUDA;
  if (*dev < 0 || *dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED;
  return ATTN_OK;
}
}  // namespace

int check_device_sm103(int *num_sms) {
  int dev = 0;
  int rc = current_device(&dev);
  if (rc != ATTN_OK) return rc;
  std::lock_guard<std::mutex> lock(g_cache_mu);
  DeviceFacts &f = g_facts[dev];
  if (f.state == 0) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return ATTN_ERR_CUDA;
    f.state = (major == 10 && minor == 3) ? 1 : 2;
    f.sms = sms;
  }
  if (f.state != 1) return ATTN_ERR_UNSUPPORTED;
  if (num_sms) *num_sms = f.sms;
  return ATTN_OK;
}

int symbol_address(const void *symbol, void **out) {
  int dev = 0;
  int rc = current_device(&dev);
  if (rc != ATTN_OK) return rc;
  std::lock_guard<std::mutex> lock(g_cache_mu);
  for (int i = 0; i < g_n_symbols[dev]; ++i)
    if (g_symbols[dev][i].key == symbol) {
      *out = g_symbols[dev][i].value;
      return ATTN_OK;
    }
  void *ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, symbol) != cudaSuccess || !ptr) return ATTN_ERR_CUDA;
  if (g_n_symbols[dev] < kMaxCached) g_symbols[dev][g_n_symbols[dev]++] = {symbol, ptr};
  *out = ptr;
  return ATTN_OK;
}

int ensure_smem_limit(const void *kern, int bytes) {
  int dev = 0;
  int rc = current_device(&dev);
  if (rc != ATTN_OK) return rc;
  std::lock_guard<std::mutex> lock(g_cache_mu);
  for (int i = 0; i < g_n_smem[dev]; ++i)
    if (g_smem_set[dev][i] == kern && g_smem_bytes[dev][i] >= bytes) return ATTN_OK;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
      cudaSuccess)
    return ATTN_ERR_CUDA;
  if (g_n_smem[dev] < kMaxCached) {
    g_smem_set[dev][g_n_smem[dev]] = kern;
    g_smem_bytes[dev][g_n_smem[dev]++] = bytes;
  }
  return ATTN_OK;
}

unsigned long long wait_limit_ns() { return g_wait_ns.load(); }
int inject_hook() { return g_inject.load(); }

bool encode_tmap_3d_bf16(CUtensorMap *map, const void *base, uint64_t inner,
                         uint64_t rows, uint64_t planes, uint32_t box_inner,
                         uint32_t box_rows, uint32_t box_planes, int swizzle_bytes) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {inner, rows, planes};
  const cuuint64_t strides[2] = {inner * 2, inner * rows * 2};
  const cuuint32_t box[3] = {box_inner, box_rows, box_planes};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapSwizzle sw =
      swizzle_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
            strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tmap_3d_f32(CUtensorMap *map, const void *base, uint64_t inner, uint64_t rows,
                        uint64_t planes, uint32_t box_inner, uint32_t box_rows,
                        uint32_t box_planes) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {inner, rows, planes};
  const cuuint64_t strides[2] = {inner * 4, inner * rows * 4};
  const cuuint32_t box[3] = {box_inner, box_rows, box_planes};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void *>(base), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Argument checks of attn_decode (Tq = 1, no mask), for entry points that
// supply their own scratch.  No CUDA call.
int validate_decode_args(const void *q, const void *k, const void *v, const void *o,
                         const float *lse, int B, int Hq, int Hkv, int Tk, int d,
                         float scale, float *scale_out) {
  return validate(q, k, v, o, lse, B, Hq, Hkv, 1, Tk, d, 0, scale, scale_out);
}

}  // namespace attn_host

namespace {
int fwd_common(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq,
               int Hkv, int Tq, int Tk, int d, int causal, int window, float scale,
               void *stream) {
  float sc = 0.f;
  int rc = validate(q, k, v, o, lse, B, Hq, Hkv, Tq, Tk, d, causal, scale, &sc);
  if (rc != ATTN_OK) return rc;
  rc = attn_host::check_device_sm103(nullptr);
  if (rc != ATTN_OK) return rc;
  attn_host::PrefillArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.Tq = Tq;
  a.Tk = Tk;
  a.d = d;
  a.causal = causal;
  a.window = window;
  a.scale = sc;
  a.stream = static_cast<cudaStream_t>(stream);
  a.wait_ns = g_wait_ns.load();
  a.inject = g_inject.load();
  return attn_host::prefill_launch(a);
}
}  // namespace

ATTN_API int attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                      int B, int Hq, int Hkv, int Tq, int Tk, int d, int causal,
                      float scale, void *stream) {
  return fwd_common(q, k, v, o, lse, B, Hq, Hkv, Tq, Tk, d, causal, 0, scale, stream);
}

ATTN_API int attn_fwd_window(const void *q, const void *k, const void *v, void *o,
                             float *lse, int B, int Hq, int Hkv, int Tq, int Tk, int d,
                             int window, float scale, void *stream) {
  if (window < 1) return ATTN_ERR_INVALID_ARG;
  // a window of Tk keys or more leaves every key at or before a query's
  // position visible: plain causal attention, computed by that path
  return fwd_common(q, k, v, o, lse, B, Hq, Hkv, Tq, Tk, d, 1, window >= Tk ? 0 : window, scale,
                    stream);
}

ATTN_API size_t attn_fwd_varlen_workspace_bytes(int B, int total_q, int max_seqlen_q) {
  return attn_host::varlen_workspace_bytes_for(B, total_q, max_seqlen_q);
}

namespace {
int varlen_common(const void *q, const void *k, const void *v, void *o, float *lse,
                  const int *cu_seqlens_q, const int *cu_seqlens_k, int B, int Hq, int Hkv,
                  int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int d,
                  int causal, int window, float scale, void *workspace,
                  size_t workspace_bytes, void *stream) {
  float sc = 0.f;
  // the shared checks, with the longest sequences standing in for Tq and Tk
  int rc = validate(q, k, v, o, lse, B, Hq, Hkv, max_seqlen_q, max_seqlen_k, d, 0, scale, &sc);
  if (rc != ATTN_OK) return rc;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (!cu_seqlens_q || !cu_seqlens_k || total_q < 1 || total_k < 1)
    return ATTN_ERR_INVALID_ARG;
  if (!aligned(cu_seqlens_q, 4) || !aligned(cu_seqlens_k, 4)) return ATTN_ERR_MISALIGNED;
  const long long cap = attn_host::varlen_list_capacity(B, total_q, max_seqlen_q);
  if (cap < 1 || cap * Hq > 0x7fffffffLL) return ATTN_ERR_INVALID_ARG;
  if (!workspace || !aligned(workspace, 16) ||
      workspace_bytes < attn_host::varlen_workspace_bytes_for(B, total_q, max_seqlen_q))
    return ATTN_ERR_WORKSPACE;
  rc = attn_host::check_device_sm103(nullptr);
  if (rc != ATTN_OK) return rc;
  attn_host::PrefillArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.Tq = max_seqlen_q;
  a.Tk = max_seqlen_k;
  a.d = d;
  a.causal = causal;
  a.window = window;
  a.scale = sc;
  a.stream = static_cast<cudaStream_t>(stream);
  a.wait_ns = g_wait_ns.load();
  a.inject = g_inject.load();
  a.varlen = true;
  a.cu_q = cu_seqlens_q;
  a.cu_k = cu_seqlens_k;
  a.total_q = total_q;
  a.total_k = total_k;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  return attn_host::prefill_launch(a);
}
}  // namespace

ATTN_API int attn_fwd_varlen(const void *q, const void *k, const void *v, void *o, float *lse,
                             const int *cu_seqlens_q, const int *cu_seqlens_k, int B, int Hq,
                             int Hkv, int total_q, int total_k, int max_seqlen_q,
                             int max_seqlen_k, int d, int causal, float scale, void *workspace,
                             size_t workspace_bytes, void *stream) {
  return varlen_common(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, B, Hq, Hkv, total_q,
                       total_k, max_seqlen_q, max_seqlen_k, d, causal, 0, scale, workspace,
                       workspace_bytes, stream);
}

ATTN_API int attn_fwd_varlen_window(const void *q, const void *k, const void *v, void *o,
                                    float *lse, const int *cu_seqlens_q,
                                    const int *cu_seqlens_k, int B, int Hq, int Hkv,
                                    int total_q, int total_k, int max_seqlen_q,
                                    int max_seqlen_k, int d, int window, float scale,
                                    void *workspace, size_t workspace_bytes, void *stream) {
  if (window < 1) return ATTN_ERR_INVALID_ARG;
  return varlen_common(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, B, Hq, Hkv, total_q,
                       total_k, max_seqlen_q, max_seqlen_k, d, 1, window, scale, workspace,
                       workspace_bytes, stream);
}

ATTN_API size_t attn_decode_workspace_bytes(int B, int Hq, int Hkv, int Tk, int d) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Tk < 1 || Hq % Hkv != 0) return 0;
  if (d != 32 && d != 64 && d != 128) return 0;
  return attn_host::decode_workspace_bytes_for(B, Hq, Tk, d);
}

ATTN_API int attn_decode(const void *q, const void *k_cache, const void *v_cache, void *o,
                         float *lse, int B, int Hq, int Hkv, int Tk, int d, float scale,
                         void *workspace, size_t workspace_bytes, void *stream) {
  float sc = 0.f;
  int rc = validate(q, k_cache, v_cache, o, lse, B, Hq, Hkv, 1, Tk, d, 0, scale, &sc);
  if (rc != ATTN_OK) return rc;
  if (!workspace || !aligned(workspace, 16) ||
      workspace_bytes < attn_decode_workspace_bytes(B, Hq, Hkv, Tk, d))
    return ATTN_ERR_WORKSPACE;
  attn_host::DecodeArgs a;
  a.q = q;
  a.k = k_cache;
  a.v = v_cache;
  a.o = o;
  a.lse = lse;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.Tk = Tk;
  a.d = d;
  a.scale = sc;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  a.stream = static_cast<cudaStream_t>(stream);
  a.wait_ns = g_wait_ns.load();
  a.inject = g_inject.load();
  return attn_host::decode_launch(a);
}

ATTN_API int attn_decode_paged(const void *q, const void *k_pages, const void *v_pages,
                               const int *block_table, const int *seq_lens, void *o,
                               float *lse, int B, int Hq, int Hkv, int d, int page_size,
                               int num_pages, int max_pages_per_seq, int max_seq_len,
                               float scale, void *workspace, size_t workspace_bytes,
                               void *stream) {
  float sc = 0.f;
  int rc = validate(q, k_pages, v_pages, o, lse, B, Hq, Hkv, 1, max_seq_len, d, 0, scale, &sc);
  if (rc != ATTN_OK) return rc;
  if (!block_table || !seq_lens) return ATTN_ERR_INVALID_ARG;
  if (!aligned(block_table, 4) || !aligned(seq_lens, 4)) return ATTN_ERR_MISALIGNED;
  if (page_size < 1 || page_size > 4096 || (page_size & (page_size - 1)) != 0)
    return ATTN_ERR_INVALID_ARG;
  if (num_pages < 1 || max_pages_per_seq < 1 ||
      (long long)max_seq_len > (long long)max_pages_per_seq * page_size)
    return ATTN_ERR_INVALID_ARG;
  if (!workspace || !aligned(workspace, 16) ||
      workspace_bytes < attn_decode_workspace_bytes(B, Hq, Hkv, max_seq_len, d))
    return ATTN_ERR_WORKSPACE;
  attn_host::DecodeArgs a;
  a.q = q;
  a.k = k_pages;
  a.v = v_pages;
  a.o = o;
  a.lse = lse;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.Tk = max_seq_len;
  a.d = d;
  a.scale = sc;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  a.stream = static_cast<cudaStream_t>(stream);
  a.wait_ns = g_wait_ns.load();
  a.inject = g_inject.load();
  a.paged = true;
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.page_size = page_size;
  a.num_pages = num_pages;
  a.max_pages = max_pages_per_seq;
  return attn_host::decode_launch(a);
}

ATTN_API size_t attn_bwd_workspace_bytes(int B, int Hq, int Tq, int d) {
  if (B < 1 || Hq < 1 || Tq < 1 || (d != 32 && d != 64 && d != 128)) return 0;
  return attn_host::bwd_workspace_bytes_for(B, Hq, Tq, d);
}

namespace {
int bwd_common(const void *q, const void *k, const void *v, const void *o, const float *lse,
               const void *dout, void *dq, void *dk, void *dv, int B, int Hq, int Hkv, int Tq,
               int Tk, int d, int causal, int window, float scale, void *workspace,
               size_t workspace_bytes, void *stream) {
  float sc = 0.f;
  // q/k/v/o/lse as for attn_fwd, then the gradient tensors
  int rc = validate(q, k, v, o, lse, B, Hq, Hkv, Tq, Tk, d, causal, scale, &sc);
  if (rc != ATTN_OK) return rc;
  if (!dout || !dq || !dk || !dv) return ATTN_ERR_INVALID_ARG;
  if (!aligned(dout, 16) || !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16))
    return ATTN_ERR_MISALIGNED;
  if (!workspace || !aligned(workspace, 16) ||
      workspace_bytes < attn_bwd_workspace_bytes(B, Hq, Tq, d))
    return ATTN_ERR_WORKSPACE;
  attn_host::BwdArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.dout = dout;
  a.lse = lse;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.Tq = Tq;
  a.Tk = Tk;
  a.d = d;
  a.causal = causal;
  a.window = window;
  a.scale = sc;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  a.stream = static_cast<cudaStream_t>(stream);
  a.wait_ns = g_wait_ns.load();
  a.inject = g_inject.load();
  return attn_host::bwd_launch(a);
}
}  // namespace

ATTN_API int attn_bwd(const void *q, const void *k, const void *v, const void *o,
                      const float *lse, const void *dout, void *dq, void *dk, void *dv, int B,
                      int Hq, int Hkv, int Tq, int Tk, int d, int causal, float scale,
                      void *workspace, size_t workspace_bytes, void *stream) {
  return bwd_common(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, Tq, Tk, d, causal, 0, scale,
                    workspace, workspace_bytes, stream);
}

ATTN_API int attn_bwd_window(const void *q, const void *k, const void *v, const void *o,
                             const float *lse, const void *dout, void *dq, void *dk, void *dv,
                             int B, int Hq, int Hkv, int Tq, int Tk, int d, int window,
                             float scale, void *workspace, size_t workspace_bytes,
                             void *stream) {
  if (window < 1) return ATTN_ERR_INVALID_ARG;
  return bwd_common(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, Tq, Tk, d, 1, window, scale,
                    workspace, workspace_bytes, stream);
}

ATTN_API const char *attn_status_string(int status) {
  switch (status) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG: invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED: unsupported head dim or GPU";
    case ATTN_ERR_MISALIGNED: return "ATTN_ERR_MISALIGNED: pointer alignment";
    case ATTN_ERR_WORKSPACE: return "ATTN_ERR_WORKSPACE: workspace missing or too small";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA: CUDA call failed";
    case ATTN_ERR_DEVICE_TIMEOUT: return "ATTN_ERR_DEVICE_TIMEOUT: kernel wait expired";
    case ATTN_ERR_IN_FLIGHT_LIMIT:
      return "ATTN_ERR_IN_FLIGHT_LIMIT: too many forward launches in flight";
    default: return "ATTN_ERR_UNKNOWN";
  }
}

ATTN_API int attn_device_status(void *stream, int *status) {
  if (!status) return ATTN_ERR_INVALID_ARG;
  unsigned int a = 0, b = 0, c = 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (attn_host::prefill_take_status(st, &a) != ATTN_OK ||
      attn_host::decode_take_status(st, &b) != ATTN_OK ||
      attn_host::bwd_take_status(st, &c) != ATTN_OK)
    return ATTN_ERR_CUDA;
  unsigned int m = a > b ? a : b;
  *status = (int)(m > c ? m : c);
  return ATTN_OK;
}

ATTN_API void attn_debug_set(unsigned long long wait_limit_ns, int inject) {
  g_wait_ns.store(wait_limit_ns ? wait_limit_ns : kDefaultWaitNs);
  g_inject.store(inject);
}
