// decode_noalloc.cu -- attn_decode without a caller-supplied workspace.
//
// attn_decode needs scratch for the per-split partial results, and asks the
// caller to provide it.  Some callers cannot allocate device memory at the
// point where they decode: code that runs under a host framework which owns
// every device allocation and gives kernels no allocator, latency-critical
// serving loops that must not pay cudaMalloc's implicit device
// synchronisation, or fixed-budget deployments whose memory plan is frozen
// at start-up.  For them this file keeps the scratch in a statically sized
// device array that is part of the library image itself.
//
// Costs and limits:
//  * every GPU on which the library is loaded holds kNoAllocScratchBytes
//    (16 MiB) for this array until the process exits;
//  * problems whose split plan needs more partial storage than that are
//    rejected with ATTN_ERR_WORKSPACE (see attn_decode_noalloc in attn.h);
//  * all calls share the one array, so calls that overlap on the GPU (on
//    different streams, or from different host threads without ordering)
//    race on it; the array keeps whatever the last call left there, and
//    nothing needs it zeroed because every partial is written before it is
//    read within a call.
#include <mutex>

#include "../../include/attn.h"
#include "internal.h"

#define ATTN_API extern "C" __attribute__((visibility("default")))

namespace {

constexpr size_t kNoAllocScratchBytes = ATTN_DECODE_NOALLOC_MAX_BYTES;
constexpr int kMaxDevices = 64;

// In host code this name is only a host-side stand-in for the device
// array; its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device (the first call on a device does this).
int scratch_for_current_device(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_decode_scratch) != cudaSuccess || !ptr)
      return ATTN_ERR_CUDA;
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return ATTN_OK;
}

}  // namespace

ATTN_API int attn_decode_noalloc(const void *q, const void *k_cache, const void *v_cache,
                                 void *o, float *lse, int B, int Hq, int Hkv, int Tk, int d,
                                 float scale, void *stream) {
  float sc = 0.f;
  int rc = attn_host::validate_decode_args(q, k_cache, v_cache, o, lse, B, Hq, Hkv, Tk, d,
                                           scale, &sc);
  if (rc != ATTN_OK) return rc;
  rc = attn_host::check_device_sm103(nullptr);
  if (rc != ATTN_OK) return rc;
  void *scratch = nullptr;
  rc = scratch_for_current_device(&scratch);
  if (rc != ATTN_OK) return rc;
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
  a.workspace = scratch;
  a.workspace_bytes = kNoAllocScratchBytes;  // plans needing more are rejected
  a.stream = static_cast<cudaStream_t>(stream);
  a.wait_ns = attn_host::wait_limit_ns();
  a.inject = attn_host::inject_hook();
  return attn_host::decode_launch(a);
}
