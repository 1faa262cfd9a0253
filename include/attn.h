/*
 * attn.h -- C ABI of the GB300 (sm_103a) exact attention forward library.
 *
 * The operation is exact scaled-dot-product attention with the row
 * log-sum-exp, O = softmax(scale * Q K^T [+ causal mask]) V, computed with the
 * online softmax: K/V tiles stream past a resident Q tile while a running
 * row max m, running sum l and unnormalised accumulator acc are kept and
 * rescaled by exp(m - m') whenever the max grows; O = acc / l and
 * LSE = m + ln l.  Sources: "Efficient attention & KV cache", sections 2.1
 * (online softmax, boxed recurrence) and 3 (blockwise forward with lse and
 * the causal kv_end stop); "4.2 FlashAttention I: IO-Awareness & The Online
 * Softmax", section "FlashAttention forward: tiling + online softmax fused
 * into one pass" (the -inf guards, LSE = m + log l).  The argument list
 * follows the fused attention signature quoted in "SDPA and
 * FlashAttention's tiling" (query, key, value, is_causal, scale,
 * enable_gqa) in the (batch, heads, seq, head_dim) layout.
 *
 * Conventions shared by every entry point
 * --------------------------------------
 *  - All tensor pointers are DEVICE pointers owned by the caller, except the
 *    host buffers of attn_fwd_host / attn_decode_host.  The library never
 *    allocates, frees or retains memory (those two create and release
 *    their own streams and events).
 *  - bf16 tensors are dense and row-major:
 *        q [B, Hq, Tq, d]      k, v [B, Hkv, Tk, d]      o [B, Hq, Tq, d]
 *    lse is fp32 [B, Hq, Tq] and holds the natural-log log-sum-exp of the
 *    scaled, masked scores of each row.
 *  - q, k, v and o must be 16-byte aligned, lse 4-byte aligned.
 *  - d (head_dim) must be 32, 64 or 128.
 *  - Grouped-query attention: Hq % Hkv == 0 and query head h reads K/V
 *    head h / (Hq / Hkv).
 *  - Causal masking is aligned to the bottom-right corner: query row i sits
 *    at key position i + (Tk - Tq) and sees keys j <= i + (Tk - Tq).  With
 *    Tq == Tk this is the usual lower-triangular mask; causal with Tq > Tk
 *    is rejected.
 *  - scale must be finite and > 0; 0.0f selects 1/sqrt(d).
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *    default stream) and return after enqueueing.  Argument errors are
 *    detected on the host before any CUDA call and leave every buffer
 *    untouched.  Launch failures return ATTN_ERR_CUDA.  Faults inside a
 *    kernel surface at the caller's next synchronisation; a kernel that
 *    gives up on a bounded wait records ATTN_ERR_DEVICE_TIMEOUT in a device
 *    status word read by attn_device_status().
 *  - The entry points keep no per-call state and may be called from several
 *    host threads.  The first call on a device looks up, once, the device's
 *    SM count and the addresses of the library's device words, and raises
 *    each kernel's shared-memory limit; make that first call before any
 *    stream capture begins.
 *  - The forward kernels (attn_fwd, attn_fwd_window, attn_fwd_varlen,
 *    attn_fwd_varlen_window) take their work items from ATTN_FWD_MAX_IN_FLIGHT
 *    work counters per device, used in turn, and from as many more for
 *    launches captured into CUDA graphs.  At most that many forward launches
 *    (of each kind) may be in flight on one device at once, across all
 *    streams and threads.  If a launch's counter is taken over by a newer
 *    launch before it finishes, the older launch stops (its outputs are then
 *    incomplete) and attn_device_status reports ATTN_ERR_IN_FLIGHT_LIMIT;
 *    counts are never shared silently.  A captured launch may be replayed
 *    any number of times, one replay at a time.
 */
#ifndef ATTN_GB300_H
#define ATTN_GB300_H

#include <stddef.h>

/* Forward launches that may be in flight at once on one device. */
#define ATTN_FWD_MAX_IN_FLIGHT 64

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,    /* null pointer, bad size, bad scale, ...      */
  ATTN_ERR_UNSUPPORTED = 2,    /* d not in {32,64,128}, or not an sm_103 GPU  */
  ATTN_ERR_MISALIGNED = 3,     /* a pointer breaks the alignment rule         */
  ATTN_ERR_WORKSPACE = 4,      /* decode workspace missing or too small       */
  ATTN_ERR_CUDA = 5,           /* a CUDA runtime/driver call failed           */
  ATTN_ERR_DEVICE_TIMEOUT = 6, /* a kernel gave up waiting (see below)        */
  ATTN_ERR_IN_FLIGHT_LIMIT = 7 /* more forward launches in flight than slots  */
} attn_status;

/*
 * attn_fwd -- prefill / general forward pass.
 *
 *   q, k, v   inputs as described above (device, bf16, read only)
 *   o         output [B, Hq, Tq, d] bf16 (device, written)
 *   lse       output [B, Hq, Tq] fp32 (device, written)
 *   B, Hq, Hkv, Tq, Tk, d   sizes (all >= 1)
 *   causal    0 = full attention, 1 = bottom-right causal mask
 *   scale     softmax scale (0.0f = 1/sqrt(d))
 *   stream    cudaStream_t to enqueue on
 *
 * The kernel keeps per query tile of 128 rows the running (m, l, acc) in
 * fp32 (acc in tensor memory), computes both products on the tensor cores
 * from bf16 operands with fp32 accumulation, and never writes a score or
 * probability to global memory.  Under causal masking, K/V tiles wholly
 * above the diagonal are not visited.
 *
 * Returns ATTN_OK or an attn_status code.
 */
int attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
             int B, int Hq, int Hkv, int Tq, int Tk, int d, int causal,
             float scale, void *stream);

/*
 * attn_fwd_window -- causal sliding-window forward pass.
 *
 * As attn_fwd with the causal mask, and each query additionally sees only the
 * `window` most recent keys: query row i (at key position p = i + Tk - Tq)
 * attends to keys j with p - window < j <= p ("4.2 FlashAttention I",
 * Exercise 4: i - W < j <= i; "Efficient attention & KV cache", exercise 2).
 * K/V tiles that lie wholly outside every row's window are never loaded.
 *   window    number of keys each query sees (>= 1; window >= Tk is plain
 *             causal attention)
 * Other arguments, layouts and errors are those of attn_fwd; Tq > Tk and
 * window < 1 return ATTN_ERR_INVALID_ARG.
 */
int attn_fwd_window(const void *q, const void *k, const void *v, void *o, float *lse,
                    int B, int Hq, int Hkv, int Tq, int Tk, int d, int window,
                    float scale, void *stream);

/*
 * attn_fwd_varlen_workspace_bytes -- scratch needed by attn_fwd_varlen.
 *
 * Depends only on the sizes; returns 0 for invalid sizes.
 */
size_t attn_fwd_varlen_workspace_bytes(int B, int total_q, int max_seqlen_q);

/*
 * attn_fwd_varlen -- forward pass over a packed batch of variable-length
 * sequences.
 *
 * The B sequences are concatenated without padding and located by
 * cumulative offsets, and no score between two sequences is ever formed
 * ("SDPA and FlashAttention's tiling": the packed flash_attn_varlen_func
 * call with int32 cu_seqlens of length B+1).  Each sequence is attention as
 * in attn_fwd on its own (causal: bottom-right aligned inside the sequence).
 *
 *   q, o          [total_q, Hq, d] bf16, token-major (device)
 *   k, v          [total_k, Hkv, d] bf16, token-major (device)
 *   lse           [Hq, total_q] fp32 (device, written)
 *   cu_seqlens_q  [B+1] int32 (device): sequence b owns query rows
 *                 cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1
 *   cu_seqlens_k  [B+1] int32 (device): likewise for key/value rows
 *   max_seqlen_q, max_seqlen_k   host-side upper bounds of the lengths
 *   d, causal, scale             as for attn_fwd
 *   workspace     device scratch of attn_fwd_varlen_workspace_bytes(B,
 *                 total_q, max_seqlen_q) bytes, 16-byte aligned, caller-
 *                 owned (contents ignored; it holds the launch's work list)
 *
 * Offsets must start at 0, never decrease and end at most at total_q /
 * total_k; every length must be within its max_seqlen; a sequence with
 * queries needs at least one key, and causal needs no more queries than
 * keys.  Empty sequences are allowed.  The offsets live on the device and
 * are checked there: if they break these rules nothing is computed, rows
 * of o and lse stay as they were, and attn_device_status reports
 * ATTN_ERR_INVALID_ARG.  Rows of o and lse outside every sequence are never
 * written.  Host-visible errors return before any launch, as for attn_fwd.
 * Inputs must be finite: a key tile that runs past its sequence holds the
 * next sequence's rows, which are masked out of the softmax (their value
 * rows are multiplied by zero).
 */
int attn_fwd_varlen(const void *q, const void *k, const void *v, void *o, float *lse,
                    const int *cu_seqlens_q, const int *cu_seqlens_k, int B, int Hq,
                    int Hkv, int total_q, int total_k, int max_seqlen_q, int max_seqlen_k,
                    int d, int causal, float scale, void *workspace, size_t workspace_bytes,
                    void *stream);

/*
 * attn_fwd_varlen_window -- packed variable-length forward with a causal
 * sliding window inside each sequence.
 *
 * As attn_fwd_varlen with the causal mask, and each query of a sequence sees
 * only that sequence's `window` most recent keys (p - window < j <= p with
 * p = i + nk - nq inside the sequence; "4.2 FlashAttention I", Exercise 4).
 * K/V tiles wholly outside every row's window are never loaded.
 *   window    number of keys each query sees (>= 1)
 * Other arguments, layouts, workspace and errors are those of
 * attn_fwd_varlen; window < 1 returns ATTN_ERR_INVALID_ARG.
 */
int attn_fwd_varlen_window(const void *q, const void *k, const void *v, void *o, float *lse,
                           const int *cu_seqlens_q, const int *cu_seqlens_k, int B, int Hq,
                           int Hkv, int total_q, int total_k, int max_seqlen_q,
                           int max_seqlen_k, int d, int window, float scale, void *workspace,
                           size_t workspace_bytes, void *stream);

/*
 * attn_decode_workspace_bytes -- scratch needed by attn_decode.
 *
 * Depends only on the sizes (not on the GPU), so it may be called before any
 * device exists.  Returns 0 for invalid sizes.
 */
size_t attn_decode_workspace_bytes(int B, int Hq, int Hkv, int Tk, int d);

/*
 * attn_decode -- one query token per sequence against a KV cache (Tq = 1).
 *
 *   q         [B, Hq, 1, d] bf16      k_cache, v_cache [B, Hkv, Tk, d] bf16
 *   o         [B, Hq, 1, d] bf16      lse [B, Hq, 1] fp32
 *   scale     as for attn_fwd
 *   workspace device scratch of at least attn_decode_workspace_bytes(...)
 *             bytes, 16-byte aligned, owned by the caller; its contents on
 *             entry do not matter and are overwritten.
 *
 * The cache is split along Tk into chunks processed in parallel; each chunk
 * produces a partial (m, l, acc) per query head, and a second kernel merges
 * the partials with the same rescaling the online softmax uses
 * (m* = max m_s, l = sum e^(m_s - m*) l_s, O = sum e^(m_s - m*) acc_s / l).
 * The merge rule follows from the associativity of the recurrence
 * ("Efficient attention & KV cache", section 2.1: any running max gives the
 * same final ratio); the pages show only sequential blocks.  Every query
 * token sees the whole cache (the causal reading above with Tq = 1).
 *
 * Returns ATTN_OK or an attn_status code (ATTN_ERR_WORKSPACE if the
 * workspace is NULL, misaligned or too small).
 */
int attn_decode(const void *q, const void *k_cache, const void *v_cache,
                void *o, float *lse, int B, int Hq, int Hkv, int Tk, int d,
                float scale, void *workspace, size_t workspace_bytes,
                void *stream);

/*
 * attn_decode_noalloc -- attn_decode for callers that cannot allocate.
 *
 * The pages have no counterpart: this is a deployment variant of
 * attn_decode.  It exists for callers that cannot call cudaMalloc where they
 * decode -- code running inside a host framework that owns every device
 * allocation, serving loops that cannot afford cudaMalloc's implicit device
 * synchronisation, or deployments whose memory plan is fixed at start-up.
 * Instead of a caller workspace it uses a scratch array that is part of the
 * library image: ATTN_DECODE_NOALLOC_MAX_BYTES (16 MiB) of device memory on
 * every GPU where the library is loaded, held until the process exits.
 *
 * Arguments, layouts and results are those of attn_decode, without the
 * workspace.  The call allocates nothing (no cudaMalloc, cudaFree or
 * allocating library routine).
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress) for that device, so make that first call before
 *    any stream capture begins.
 *  - Problems whose split plan needs more than ATTN_DECODE_NOALLOC_MAX_BYTES
 *    of partial results (B * Hq * splits * (d + 2) * 4 bytes) are rejected
 *    with ATTN_ERR_WORKSPACE before anything is launched.
 *  - Every call uses the same array.  Calls that overlap on the GPU (other
 *    streams, other host threads) race on it and must be ordered by the
 *    caller.  The array keeps the last call's contents; no call depends on
 *    them, since every partial is written before it is read, including the
 *    empty partial a split writes when it gives up on a bounded wait.
 *  - The wait limit and test hooks of attn_debug_set apply as for
 *    attn_decode; after ATTN_ERR_DEVICE_TIMEOUT, o and lse are unspecified.
 */
#define ATTN_DECODE_NOALLOC_MAX_BYTES ((size_t)16 << 20)
int attn_decode_noalloc(const void *q, const void *k_cache, const void *v_cache,
                        void *o, float *lse, int B, int Hq, int Hkv, int Tk, int d,
                        float scale, void *stream);

/*
 * attn_decode_paged -- decode (Tq = 1) against a paged KV cache.
 *
 * The cache lives in fixed-size pages of `page_size` tokens held in two
 * pools, and each sequence lists its pages in a block table; the kernel
 * fetches each page from wherever it sits instead of reading one
 * contiguous cache ("Efficient attention & KV cache", section 2.5 "Paged
 * and shared caches", and the same page's answer on what PagedAttention
 * changes in the attention kernel).  Sequences may have different lengths
 * and may share pages (a common prefix).
 *
 *   q            [B, Hq, 1, d] bf16 (device)
 *   k_pages      [num_pages, Hkv, page_size, d] bf16 (device): page p holds,
 *   v_pages      for every K/V head, page_size consecutive token rows
 *   block_table  [B, max_pages_per_seq] int32 (device): entry [b][i] is the
 *                physical page holding tokens i*page_size .. (i+1)*page_size-1
 *                of sequence b; entries past a sequence's last page are
 *                never read
 *   seq_lens     [B] int32 (device): tokens in sequence b's cache,
 *                1 <= seq_lens[b] <= max_seq_len
 *   o, lse       [B, Hq, 1, d] bf16 and [B, Hq, 1] fp32 (device, written)
 *   page_size    a power of two, 1 .. 4096
 *   num_pages    pages in each pool (bounds the table entries)
 *   max_seq_len  host-side upper bound of seq_lens, used to plan the split
 *                along the keys; max_seq_len <= max_pages_per_seq*page_size
 *   scale        as for attn_fwd
 *   workspace    device scratch of at least
 *                attn_decode_workspace_bytes(B, Hq, Hkv, max_seq_len, d)
 *                bytes, 16-byte aligned, caller-owned (contents ignored)
 *
 * Query head h reads K/V head h / (Hq/Hkv), and every query token sees its
 * whole cache, as in attn_decode.  Host-visible errors (sizes, alignment,
 * page_size, workspace) return before anything is launched.  The lengths
 * and table entries live on the device and are checked there: a length
 * outside 1..max_seq_len or a page outside 0..num_pages-1 is never used to
 * address memory (the sequence is skipped, or page 0 is read in its place),
 * the affected rows are unspecified, and attn_device_status then reports
 * ATTN_ERR_INVALID_ARG.
 */
int attn_decode_paged(const void *q, const void *k_pages, const void *v_pages,
                      const int *block_table, const int *seq_lens, void *o, float *lse,
                      int B, int Hq, int Hkv, int d, int page_size, int num_pages,
                      int max_pages_per_seq, int max_seq_len, float scale,
                      void *workspace, size_t workspace_bytes, void *stream);

/*
 * attn_bwd_workspace_bytes -- scratch needed by attn_bwd.
 *
 * B*Hq*Tq*d fp32 for the dQ accumulator plus, per query row padded to a
 * multiple of 128, 32 bytes of derived operands (the row's LSE and
 * D = dout . o).
 * Depends only on the sizes; returns 0 for invalid sizes.
 */
size_t attn_bwd_workspace_bytes(int B, int Hq, int Tq, int d);

/*
 * attn_bwd -- gradients of attn_fwd with recomputation.
 *
 * Given the forward's inputs, its outputs o and lse, and the upstream
 * gradient dout = dL/dO, computes dq, dk, dv without storing anything of
 * size Tq x Tk: every probability tile is rebuilt from the saved
 * log-sum-exp as P = e^(S - lse) ("4.2 FlashAttention I", section "The
 * backward pass: recomputation instead of storage"; "Efficient attention &
 * KV cache", section 2.2):
 *   D_i = dout_i . o_i,  dV = P^T dout,  dS = P o (dout V^T - D),
 *   dQ = scale dS K,  dK = scale dS^T Q.
 *
 *   q, k, v, causal, scale, sizes   exactly as passed to attn_fwd
 *   o, lse        attn_fwd's outputs for those inputs (device, read only)
 *   dout          [B, Hq, Tq, d] bf16 (device, read only)
 *   dq            [B, Hq, Tq, d] bf16 (device, written)
 *   dk, dv        [B, Hkv, Tk, d] bf16 (device, written); under grouped-query
 *                 attention a K/V head's gradient sums over its query heads
 *   workspace     device scratch of attn_bwd_workspace_bytes(B, Hq, Tq, d)
 *                 bytes, 16-byte aligned, caller-owned (contents ignored)
 *
 * dQ is accumulated in fp32 across key tiles by atomic reductions into the
 * workspace (coalesced global reductions at d >= 64, TMA tensor reductions
 * at d = 32), so its last bits may differ from run to run (the page's note
 * on the nondeterminism of the atomic backward); dK and dV are
 * deterministic.
 * Errors are those of attn_fwd, plus ATTN_ERR_INVALID_ARG for a NULL
 * gradient pointer, ATTN_ERR_MISALIGNED for one not 16-byte aligned, and
 * ATTN_ERR_WORKSPACE.
 */
int attn_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse,
             const void *dout, void *dq, void *dk, void *dv, int B, int Hq, int Hkv, int Tq,
             int Tk, int d, int causal, float scale, void *workspace, size_t workspace_bytes,
             void *stream);

/*
 * attn_bwd_window -- gradients of attn_fwd_window.
 *
 * As attn_bwd with the causal mask, and each query's probabilities confined
 * to its `window` most recent keys (p - window < j <= p, p = i + Tk - Tq;
 * "4.2 FlashAttention I", Exercise 4): masked entries have P = 0 and carry
 * no gradient, so every K/V tile only visits the query tiles whose window
 * reaches it.  o and lse must be attn_fwd_window's outputs for the same
 * window.  Keys that no query sees get zero dk and dv.
 *   window    number of keys each query sees (>= 1)
 * Other arguments, layouts, workspace and errors are those of attn_bwd;
 * window < 1 or Tq > Tk return ATTN_ERR_INVALID_ARG.
 */
int attn_bwd_window(const void *q, const void *k, const void *v, const void *o,
                    const float *lse, const void *dout, void *dq, void *dk, void *dv, int B,
                    int Hq, int Hkv, int Tq, int Tk, int d, int window, float scale,
                    void *workspace, size_t workspace_bytes, void *stream);

/*
 * attn_fwd_host / attn_decode_host -- the same operations on HOST buffers.
 *
 * The exception to the device-pointer rule above: q, k, v (k_cache,
 * v_cache) are read from, and o, lse written to, HOST memory in the layouts
 * given above.  The buffers should be page-locked (cudaHostAlloc or
 * cudaHostRegister); pageable memory works but its copies do not overlap.
 * They must stay valid and unmodified until `stream` has completed the call.
 *
 *   workspace        DEVICE scratch of attn_fwd_host_workspace_bytes(...)
 *                    (attn_decode_host_workspace_bytes(...)) bytes,
 *                    256-byte aligned, caller-owned; it receives the device
 *                    copies of every input and output (and, for decode, the
 *                    split partials of attn_decode)
 *   other arguments  as for attn_fwd (attn_decode)
 *
 * The call splits the problem into up to 16 chunks of whole (batch, K/V
 * head) slices and overlaps, through two auxiliary streams and events that
 * it creates and releases itself, the host-to-device copies of one chunk,
 * the kernels of the previous one (attn_fwd / attn_decode on the chunk's
 * part of the workspace) and the device-to-host copies of the one before.
 * attn_fwd_host's results are bit-identical to copying the whole problem in
 * and calling attn_fwd once (every query row is computed the same way
 * whatever else the launch holds); attn_decode_host's agree with
 * attn_decode to rounding, since attn_decode chooses its number of key
 * splits from the number of sequences in a launch.  `stream` waits for its earlier work before
 * the first copy and completes only after the last copy out, so
 * synchronising `stream` makes o and lse valid in host memory.
 *
 * Errors: those of attn_fwd (attn_decode) checked on the host before any
 * CUDA call, ATTN_ERR_WORKSPACE for a missing, misaligned or short
 * workspace, ATTN_ERR_CUDA if a copy, a stream or an event cannot be set
 * up.  A failure part-way leaves o and lse partly written.
 */
size_t attn_fwd_host_workspace_bytes(int B, int Hq, int Hkv, int Tq, int Tk, int d);
int attn_fwd_host(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                  int Hq, int Hkv, int Tq, int Tk, int d, int causal, float scale,
                  void *workspace, size_t workspace_bytes, void *stream);
size_t attn_decode_host_workspace_bytes(int B, int Hq, int Hkv, int Tk, int d);
int attn_decode_host(const void *q, const void *k_cache, const void *v_cache, void *o,
                     float *lse, int B, int Hq, int Hkv, int Tk, int d, float scale,
                     void *workspace, size_t workspace_bytes, void *stream);

/* Human-readable name of a status code (never NULL). */
const char *attn_status_string(int status);

/*
 * attn_device_status -- read and clear the device-side status word of the
 * current device.
 *
 * Every wait inside the kernels is bounded in time.  A kernel that gives up
 * stops its work, drains its own copies and tensor-core operations, frees
 * its tensor memory, records ATTN_ERR_DEVICE_TIMEOUT here and returns, so
 * the CUDA context stays usable.  attn_decode_paged and attn_fwd_varlen
 * also record ATTN_ERR_INVALID_ARG here for device-side lengths, offsets or
 * page indices they could not use.  This call synchronises `stream`, copies
 * the word to *status (ATTN_OK when nothing was recorded) and resets it.
 * Returns ATTN_OK, or ATTN_ERR_CUDA if the copy fails.
 */
int attn_device_status(void *stream, int *status);

/*
 * attn_debug_set -- test hooks (process-wide; not for production use).
 *
 *   wait_limit_ns  time a kernel waits on one barrier before giving up
 *                  (0 restores the default of 1 s)
 *   inject         0 = none; otherwise one load is withheld so that a
 *                  bounded wait must expire and report
 *                  ATTN_ERR_DEVICE_TIMEOUT:
 *                    1 = the forward kernel's first V tile,
 *                    2 = the first K/V tile of the decode kernels' first
 *                        CTA (attn_decode, attn_decode_paged,
 *                        attn_decode_noalloc),
 *                    3 = the first dO tile of the backward kernel's first
 *                        CTA (attn_bwd, attn_bwd_window)
 *                  The outputs of a call that timed out are unspecified.
 */
void attn_debug_set(unsigned long long wait_limit_ns, int inject);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_H */
