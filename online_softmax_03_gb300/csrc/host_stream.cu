// host_stream.cu -- attention from and to host memory: the inputs are copied
// to the device, the kernels run, and the outputs are copied back, with the
// three stages overlapped across slices of the batch.
//
// A call splits the problem into chunks of whole (batch, K/V head) slices --
// a slice's Q, K, V, O and LSE rows are contiguous in the [B, H, T, d]
// layout -- and runs three streams joined by events: the host-to-device
// copies of chunk c+1 and the device-to-host copies of chunk c-1 proceed
// while the kernels work on chunk c.  Every chunk is computed by the same
// entry point as a device call (attn_fwd / attn_decode on the chunk's part
// of the device workspace).  The forward's rows come out bit-identical to a
// single attn_fwd call; attn_decode picks its key splits from the number of
// sequences it is given, so the decode's agree to rounding.
//
// The host link of this part moves about 210 GB/s in each direction
// (measured with copy engines on one to eight streams and with kernels
// reading page-locked memory alike), so the copies set the pace and the
// overlap hides the kernels and the copies out behind the copies in.
#include <cstdint>

#include "../../include/attn.h"
#include "internal.h"

#define ATTN_API extern "C" __attribute__((visibility("default")))

namespace {

constexpr int kMaxChunks = 16;
constexpr size_t kChunkTargetBytes = 16ull << 20;  // smaller problems use fewer chunks

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// Byte offsets of the device copies inside the workspace.
struct Layout {
  size_t q, k, v, o, lse, scratch, total;
};

Layout make_layout(int B, int Hq, int Hkv, int Tq, int Tk, int d, size_t scratch_bytes) {
  const size_t qb = (size_t)B * Hq * Tq * d * 2, kb = (size_t)B * Hkv * Tk * d * 2;
  const size_t lb = (size_t)B * Hq * Tq * 4;
  Layout L;
  L.q = 0;
  L.k = L.q + round256(qb);
  L.v = L.k + round256(kb);
  L.o = L.v + round256(kb);
  L.lse = L.o + round256(qb);
  L.scratch = L.lse + round256(lb);
  L.total = L.scratch + round256(scratch_bytes);
  return L;
}

// One chunk: batches [b0, b0 + nb) and, within them, K/V heads [g0, g0 + ng)
// (ng < Hkv only when nb == 1).
struct Chunk {
  int b0, nb, g0, ng;
};

// Chunks of whole batches when there are at least as many batches as
// chunks, else each batch split into runs of K/V heads.
int plan_chunks(int B, int Hkv, size_t total_bytes, Chunk *out) {
  size_t want = total_bytes / kChunkTargetBytes;
  int nc = want < 1 ? 1 : want > (size_t)kMaxChunks ? kMaxChunks : (int)want;
  int n = 0;
  if (B >= nc) {
    const int bpc = (B + nc - 1) / nc;
    for (int b = 0; b < B; b += bpc) out[n++] = {b, b + bpc <= B ? bpc : B - b, 0, Hkv};
  } else {
    int parts = (nc + B - 1) / B;
    if (parts > Hkv) parts = Hkv;
    const int hpc = (Hkv + parts - 1) / parts;
    for (int b = 0; b < B; ++b)
      for (int g = 0; g < Hkv; g += hpc) out[n++] = {b, 1, g, g + hpc <= Hkv ? hpc : Hkv - g};
  }
  return n;  // <= kMaxChunks + B - 1 <= 2 * kMaxChunks
}

// The auxiliary streams and events of one call.  Destroying them while work
// is pending is allowed: CUDA releases them once that work completes.
struct Pipeline {
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, in_done = nullptr, comp_done = nullptr, out_done = nullptr;
  bool ok = false;
  Pipeline() {
    ok = cudaStreamCreateWithFlags(&in, cudaStreamNonBlocking) == cudaSuccess &&
         cudaStreamCreateWithFlags(&out, cudaStreamNonBlocking) == cudaSuccess &&
         cudaEventCreateWithFlags(&start, cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&in_done, cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&comp_done, cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&out_done, cudaEventDisableTiming) == cudaSuccess;
  }
  ~Pipeline() {
    for (cudaEvent_t e : {start, in_done, comp_done, out_done})
      if (e) cudaEventDestroy(e);
    for (cudaStream_t s : {in, out})
      if (s) cudaStreamDestroy(s);
  }
};

bool h2d(void *dst, const void *src, size_t bytes, cudaStream_t s) {
  return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, s) == cudaSuccess;
}
bool d2h(void *dst, const void *src, size_t bytes, cudaStream_t s) {
  return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToHost, s) == cudaSuccess;
}

// Host-side checks shared by both entry points.  No CUDA call.
int check_common(const void *q, const void *k, const void *v, const void *o, const float *lse,
                 int B, int Hq, int Hkv, int Tq, int Tk, int d, void *workspace) {
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || Hq < 1 || Hkv < 1 || Tq < 1 || Tk < 1 || Hq % Hkv != 0)
    return ATTN_ERR_INVALID_ARG;
  if (d != 32 && d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
    return ATTN_ERR_WORKSPACE;
  return ATTN_OK;
}

// Runs the chunks: copies in on p.in, compute(chunk, device pointers) on
// `stream`, copies out on p.out; `stream` ends after the last copy out.
template <typename Compute>
int run_pipeline(const uint8_t *qh, const uint8_t *kh, const uint8_t *vh, uint8_t *oh,
                 uint8_t *lh, uint8_t *ws, const Layout &L, int B, int Hq, int Hkv, int Tq,
                 int Tk, int d, cudaStream_t stream, Compute compute) {
  const int G = Hq / Hkv;
  const size_t q_row = (size_t)Tq * d * 2, k_row = (size_t)Tk * d * 2, l_row = (size_t)Tq * 4;
  Chunk chunks[2 * kMaxChunks];
  const size_t total = L.scratch;
  const int n = plan_chunks(B, Hkv, total, chunks);
  Pipeline p;
  if (!p.ok) return ATTN_ERR_CUDA;
  // the copies in wait for the work already queued on the caller's stream
  if (cudaEventRecord(p.start, stream) != cudaSuccess ||
      cudaStreamWaitEvent(p.in, p.start, 0) != cudaSuccess)
    return ATTN_ERR_CUDA;
  for (int c = 0; c < n; ++c) {
    const Chunk &ch = chunks[c];
    // first query head row and first K/V head row of the chunk
    const size_t qh0 = (size_t)ch.b0 * Hq + (size_t)ch.g0 * G;
    const size_t kh0 = (size_t)ch.b0 * Hkv + ch.g0;
    const size_t nq = (size_t)ch.nb * ch.ng * G, nk = (size_t)ch.nb * ch.ng;
    if (!h2d(ws + L.q + qh0 * q_row, qh + qh0 * q_row, nq * q_row, p.in) ||
        !h2d(ws + L.k + kh0 * k_row, kh + kh0 * k_row, nk * k_row, p.in) ||
        !h2d(ws + L.v + kh0 * k_row, vh + kh0 * k_row, nk * k_row, p.in) ||
        cudaEventRecord(p.in_done, p.in) != cudaSuccess ||
        cudaStreamWaitEvent(stream, p.in_done, 0) != cudaSuccess)
      return ATTN_ERR_CUDA;
    const int rc = compute(ws + L.q + qh0 * q_row, ws + L.k + kh0 * k_row,
                           ws + L.v + kh0 * k_row, ws + L.o + qh0 * q_row,
                           reinterpret_cast<float *>(ws + L.lse + qh0 * l_row), ch.nb,
                           ch.ng * G, ch.ng);
    if (rc != ATTN_OK) return rc;
    if (cudaEventRecord(p.comp_done, stream) != cudaSuccess ||
        cudaStreamWaitEvent(p.out, p.comp_done, 0) != cudaSuccess ||
        !d2h(oh + qh0 * q_row, ws + L.o + qh0 * q_row, nq * q_row, p.out) ||
        !d2h(lh + qh0 * l_row, ws + L.lse + qh0 * l_row, nq * l_row, p.out))
      return ATTN_ERR_CUDA;
  }
  if (cudaEventRecord(p.out_done, p.out) != cudaSuccess ||
      cudaStreamWaitEvent(stream, p.out_done, 0) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return ATTN_OK;
}

}  // namespace

ATTN_API size_t attn_fwd_host_workspace_bytes(int B, int Hq, int Hkv, int Tq, int Tk, int d) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Tq < 1 || Tk < 1 || Hq % Hkv != 0) return 0;
  if (d != 32 && d != 64 && d != 128) return 0;
  return make_layout(B, Hq, Hkv, Tq, Tk, d, 0).total;
}

ATTN_API int attn_fwd_host(const void *q, const void *k, const void *v, void *o, float *lse,
                           int B, int Hq, int Hkv, int Tq, int Tk, int d, int causal,
                           float scale, void *workspace, size_t workspace_bytes,
                           void *stream) {
  int rc = check_common(q, k, v, o, lse, B, Hq, Hkv, Tq, Tk, d, workspace);
  if (rc != ATTN_OK) return rc;
  // the remaining argument rules (causal, scale, ...) before any CUDA call
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (causal && Tq > Tk) return ATTN_ERR_INVALID_ARG;
  if (!(scale >= 0.f && scale <= 3.4e38f)) return ATTN_ERR_INVALID_ARG;
  const Layout L = make_layout(B, Hq, Hkv, Tq, Tk, d, 0);
  if (workspace_bytes < L.total) return ATTN_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return run_pipeline(
      static_cast<const uint8_t *>(q), static_cast<const uint8_t *>(k),
      static_cast<const uint8_t *>(v), static_cast<uint8_t *>(o),
      reinterpret_cast<uint8_t *>(lse), static_cast<uint8_t *>(workspace), L, B, Hq, Hkv, Tq,
      Tk, d, s,
      [&](const void *dq, const void *dk, const void *dv, void *dout, float *dlse, int nb,
          int hq, int hkv) {
        return attn_fwd(dq, dk, dv, dout, dlse, nb, hq, hkv, Tq, Tk, d, causal, scale, stream);
      });
}

ATTN_API size_t attn_decode_host_workspace_bytes(int B, int Hq, int Hkv, int Tk, int d) {
  const size_t part = attn_decode_workspace_bytes(B, Hq, Hkv, Tk, d);
  if (part == 0) return 0;
  return make_layout(B, Hq, Hkv, 1, Tk, d, part).total;
}

ATTN_API int attn_decode_host(const void *q, const void *k_cache, const void *v_cache, void *o,
                              float *lse, int B, int Hq, int Hkv, int Tk, int d, float scale,
                              void *workspace, size_t workspace_bytes, void *stream) {
  int rc = check_common(q, k_cache, v_cache, o, lse, B, Hq, Hkv, 1, Tk, d, workspace);
  if (rc != ATTN_OK) return rc;
  if (!(scale >= 0.f && scale <= 3.4e38f)) return ATTN_ERR_INVALID_ARG;
  const size_t part = attn_decode_workspace_bytes(B, Hq, Hkv, Tk, d);
  const Layout L = make_layout(B, Hq, Hkv, 1, Tk, d, part);
  if (workspace_bytes < L.total) return ATTN_ERR_WORKSPACE;
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The chunks run one after another on `stream`, so they share the split
  // partials' scratch, sized for the whole problem.
  return run_pipeline(
      static_cast<const uint8_t *>(q), static_cast<const uint8_t *>(k_cache),
      static_cast<const uint8_t *>(v_cache), static_cast<uint8_t *>(o),
      reinterpret_cast<uint8_t *>(lse), ws, L, B, Hq, Hkv, 1, Tk, d, s,
      [&](const void *dq, const void *dk, const void *dv, void *dout, float *dlse, int nb,
          int hq, int hkv) {
        return attn_decode(dq, dk, dv, dout, dlse, nb, hq, hkv, Tk, d, scale, ws + L.scratch,
                           part, stream);
      });
}
