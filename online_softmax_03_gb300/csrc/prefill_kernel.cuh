// prefill_kernel.cuh -- exact attention forward on sm_103a tensor cores.
//
// A work item is two tiles of 128 query rows (256 consecutive rows) of one
// (batch, head); the K/V tiles of its K/V head stream past them: the
// outer-Q / inner-KV loop order of "4.2 FlashAttention I: IO-Awareness & The
// Online Softmax", section "FlashAttention forward: tiling + online softmax
// fused into one pass", and of "Efficient attention & KV cache", section 3.
// Per query row the running max m, running sum l and the unnormalised
// accumulator acc are kept in fp32 and updated with the recurrence of
// "Efficient attention & KV cache", section 2.1:
//
//   m' = max(m, rowmax S_j),  l' = e^(m-m') l + rowsum e^(S_j-m'),
//   acc' = e^(m-m') acc + e^(S_j-m') V_j,  O = acc / l,  LSE = m + ln l.
//
// GB300 mapping: a persistent kernel, one CTA of 320 threads per SM.  The
// producer thread takes work items from a launch-wide atomic counter (so
// faster CTAs take more of the unequal causal items) and publishes each one
// to the other roles through a two-entry shared-memory ring.
// Every role runs ahead into the next item, so one item's tail (last PV,
// epilogue) overlaps the next item's loads and first products.
//   warps 0-3, 4-7  two softmax warpgroups, one per query tile t.  Thread r
//              of group t owns row r of tile t = TMEM lane r.  It reads its
//              row of S_t from tensor memory, masks, updates (m, l), rescales
//              its row of O_t when needed, and writes P as bf16 back into the
//              first 64 columns of S_t.  At the end of an item it reads O_t,
//              normalises it and passes its row of O through a per-warp
//              shared-memory staging area, so that the warp's global stores
//              write whole 128-byte lines; LSE is stored directly.
//   warp 8     TMA producer: Q tiles (as soon as the previous item's last
//              S_t no longer needs them) and K and V tiles into a ring of
//              STAGES shared-memory slots (swizzled boxes), across items.
//   warp 9     MMA issuer (the warp runs converged; one elected lane issues),
//              tcgen05.mma kind::f16, bf16 operands,
//              fp32 accumulation in tensor memory:
//                S_t = Q_t K_j^T    A and B from shared memory,
//                O_t += P_t V_j     A = P_t from tensor memory, B = V_j.
//              The two tiles ping-pong: while group 0 turns S_0 into P_0 the
//              tensor core runs PV_1 and S_1 of the next K tile, and the other
//              way round, so exponentials and MMAs overlap.
//
// Tensor memory (512 columns): S_0 [0,128), S_1 [128,256), O_0 [256,256+D),
// O_1 [256+D, 256+2D).  P_t aliases S_t.  The MMAs of one thread execute in
// issue order, so S_t(j+1) (issued after PV_t(j)) overwrites P_t(j) only after
// PV_t(j) has read it, and the commit that signals S_t(j+1) also covers
// PV_t(j), so a softmax group that sees S_t(j+1) may rescale O_t.  Across
// items, a softmax group reads O_t of item i before it publishes any P_t of
// item i+1, and the first PV_t of item i+1 (which overwrites O_t) waits for
// that P_t.
//
// Exponentials run in base 2 on scores pre-multiplied by scale*log2(e); m is
// kept in those units and LSE is converted back to natural log.  The
// accumulator is rescaled lazily: the reference max a row uses moves only
// when the tile max exceeds it by more than kRescaleLog2, since any
// reference value gives the same final ratio acc / l ("any m gives the same
// final ratio", section 2.1) while e^(s - m) stays in range (<= 2^8 here).
//
// Causal masking is bottom-right aligned (query i sees keys j <= i + Tk - Tq);
// with a sliding window of W keys it also sees only j > i + Tk - Tq - W
// ("4.2 FlashAttention I", Exercise 4; "Efficient attention & KV cache",
// exercise 2).  K/V tiles wholly outside every row's visible range are never
// loaded, and only tiles that cross an edge of it or the ragged end of K are
// masked element by element.
// Work items are ordered by groups of heads whose K/V fit in L2, heaviest
// query tiles first within a group.
//
// Packed variable-length batches (kVarlen; "SDPA and FlashAttention's
// tiling", flash_attn_varlen_func): sequences are concatenated without
// padding in token-major tensors q [total_q, Hq, D], k/v [total_k, Hkv, D]
// and located by offsets cu_q / cu_k.  A small planning kernel lists every
// (sequence, query-tile pair) heaviest first; an item is one list entry for
// one head, and the producer publishes its geometry (offsets and lengths)
// with the item.  The tensor maps view each tensor as (D, heads, tokens), so
// a box is 128 consecutive tokens of one head, laid out in shared memory
// exactly like a box of the [B, H, T, D] layout.  A tile that runs past its
// sequence reads the next sequence's rows (or zero fill at the end): their
// keys are masked like a ragged K tail and their query rows are not stored.
//
// Every barrier wait is bounded in time; on expiry the kernel records
// ATTN_ERR_DEVICE_TIMEOUT, stops issuing work, drains its own copies and
// MMAs, frees tensor memory and returns.
#pragma once

#include <cuda_bf16.h>

#include "ptx.cuh"

namespace attn_dev {

constexpr unsigned int kStatusTimeout = 6;  // ATTN_ERR_DEVICE_TIMEOUT
constexpr unsigned int kStatusSlotLost = 7;  // ATTN_ERR_IN_FLIGHT_LIMIT
constexpr float kRescaleLog2 = 8.0f;
constexpr float kLn2 = 0.6931471805599453f;

struct PrefillParams {
  __nv_bfloat16 *o;        // [B, Hq, Tq, D]
  float *lse;              // [B, Hq, Tq]
  unsigned int *status;   // device status word
  int Hq, Hkv, group;     // group = Hq / Hkv
  int Tq, Tk;
  int n_qt;               // ceil(Tq / 256): query-tile pairs per head
  int n_bh;               // B * Hq
  int head_group;         // heads per scheduling group (K/V working set in L2)
  int n_items;            // n_bh * n_qt
  unsigned long long *work;  // work slot: {items taken, CTAs finished}, each (tag << 32) | n
  unsigned int epoch;        // this launch's tag (never 0)
  int graph_mode;            // 1: captured into a CUDA graph (the last CTA frees the slot)
  int causal;
  int window;             // > 0: causal sliding window of this many keys
  float scale_log2;       // scale * log2(e)
  unsigned long long wait_ns;
  int inject;             // test hook: 1 = withhold the first V tile
  // packed variable-length batches only
  const int *cu_q, *cu_k;  // [B+1] token offsets of each sequence
  const int *vl_list;      // {entries, 0, (b, pair) x entries}, heaviest first
  int total_q;             // tokens in q (row stride of lse [Hq, total_q])
};

template <int D>
struct PrefillCfg {
  static constexpr int BM = 128;                      // query rows per tile
  static constexpr int NQ = 2;                        // query tiles per item
  static constexpr int BN = 128;                      // keys per K/V tile
  static constexpr int SPAN = (D >= 64) ? 128 : 64;   // swizzle span, bytes
  static constexpr int CHUNK = SPAN / 2;              // bf16 columns per box
  static constexpr int NCHUNK = D / CHUNK;
  static constexpr uint32_t LAYOUT = (SPAN == 128) ? kLayoutSW128 : kLayoutSW64;
  static constexpr int STAGES = (D == 128) ? 2 : 4;
  static constexpr uint32_t Q_BYTES = BM * D * 2;     // one query tile
  static constexpr uint32_t KV_BYTES = BN * D * 2;
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = OFF_Q + NQ * Q_BYTES;
  static constexpr uint32_t OFF_V = OFF_K + STAGES * KV_BYTES;
  // Epilogue staging: each softmax warp turns its 32 rows of O around in its
  // own area, EPI_ROW bytes of every row per pass (EPI_UNITS 16-byte units).
  static constexpr int EPI_ROW = (2 * D < 128) ? 2 * D : 128;
  static constexpr int EPI_UNITS = EPI_ROW / 16;
  static constexpr int EPI_PASSES = 2 * D / EPI_ROW;
  static constexpr uint32_t EPI_WARP_BYTES = 32 * EPI_ROW;
  static constexpr uint32_t OFF_EPI = OFF_V + STAGES * KV_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_EPI + 8 * EPI_WARP_BYTES;
  // drain, q_full[2], q_empty[2], s_full[2], p_full[2], o_done[2],
  // item_full[2], item_empty[2], then per stage k_full, v_full, k_empty, v_empty
  // At D <= 64 tensor memory has room for P beside S: P_t gets a region of
  // its own, so S_t of the next K/V tile may be written while P_t is formed.
  static constexpr bool SEP_P = D <= 64;
  // ..., then s_free[2] and pv_done[2] (SEP_P)
  static constexpr int NBAR = 19 + 4 * STAGES;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  // tmem slot, abort flag, then the two-entry item ring of kRingInts ints each
  static constexpr uint32_t SMEM_USED = OFF_MISC + 128 + 1024;  // + align slack
  // At least ~116 KB so that only one CTA (which holds all 512 TMEM
  // columns) is resident per SM.
  static constexpr uint32_t SMEM_BYTES = SMEM_USED > 118784u ? SMEM_USED : 118784u;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr int THREADS = 320;
  static constexpr int PRODUCER_WARP = 8;
  static constexpr int MMA_WARP = 9;
  __host__ __device__ static constexpr uint32_t tm_s(int t) { return t * 128; }
  __host__ __device__ static constexpr uint32_t tm_o(int t) { return 256 + t * D; }
  // P_t: 64 columns of bf16 pairs (128 keys), after both O regions
  __host__ __device__ static constexpr uint32_t tm_p(int t) {
    return SEP_P ? 384 + t * 64 : tm_s(t);
  }
  static_assert(D % CHUNK == 0, "head dim must be a whole number of boxes");
  static_assert(Q_BYTES % 1024 == 0 && KV_BYTES % 1024 == 0, "1 KiB regions");
  static_assert(256 + 2 * D <= 512, "tensor memory budget");
  static_assert(!SEP_P || 256 + 2 * D <= 384, "P regions after the O regions");
  static_assert(SMEM_BYTES <= 232448u, "shared memory budget");
  static_assert(EPI_UNITS == 8 || EPI_UNITS == 4, "epilogue swizzle");
  // The 16-byte unit u of staged row r sits at unit epi_swz(u, r) of the row,
  // so the eight lanes of a shared-memory phase hit eight different banks
  // both when a lane writes its own row and when eight lanes read one row
  // (four and two rows at EPI_UNITS = 4).
  __device__ __forceinline__ static int epi_swz(int u, int r) {
    return EPI_UNITS == 8 ? (u ^ (r & 7)) : (u ^ ((r >> 1) & 3));
  }
};

// Geometry of one work item, computed identically by every role: query tile
// t visits the K/V tiles [lo_t, hi_t) (empty if equal); the item walks the
// union of the two ranges, which is contiguous.
struct PrefillItem {
  int bh, bh_kv, q0;
  int lo0, hi0, lo1, hi1;
  __device__ __forceinline__ int lo(int t) const { return t == 0 ? lo0 : lo1; }
  __device__ __forceinline__ int hi(int t) const { return t == 0 ? hi0 : hi1; }
  __device__ __forceinline__ bool has(int t) const { return lo(t) < hi(t); }
  __device__ __forceinline__ int jbeg() const {
    return !(lo1 < hi1) ? lo0 : !(lo0 < hi0) ? lo1 : min(lo0, lo1);
  }
  __device__ __forceinline__ int jend() const { return max(hi0, hi1); }
};

// Ints per item-ring entry: the item index, its geometry (bh, bh_kv, q0,
// lo0, hi0, lo1, hi1), then (packed batches) the sequence's query offset and
// length and key offset and length.  The producer computes the geometry once
// (integer divisions by launch parameters) so that the MMA and softmax roles
// start the next item without that latency on their critical path.
constexpr int kRingInts = 12;
// the ring sits at byte 16 of the 128-byte misc area
static_assert(16 + 2 * kRingInts * 4 <= 128, "item ring size");

// Tile ranges of the two query tiles of the pair starting at row q0 of a
// sequence with Tq queries and Tk keys.
template <bool kWindow>
__device__ __forceinline__ void prefill_ranges(PrefillItem &it, int Tq, int Tk, int causal,
                                               int window) {
  const int delta = Tk - Tq;
  const int n_kv_all = (Tk + 127) / 128;
  int lo[2], hi[2];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int row0 = it.q0 + t * 128;
    if (row0 >= Tq) {
      lo[t] = hi[t] = 0;
    } else {
      const int last_row = min(row0 + 127, Tq - 1);
      hi[t] = causal ? min(n_kv_all, (last_row + delta) / 128 + 1) : n_kv_all;
      // the window's left edge for the tile's first row: keys below it are
      // outside every row's window
      lo[t] = kWindow ? max(0, row0 + delta - window + 1) / 128 : 0;
    }
  }
  it.lo0 = lo[0];
  it.hi0 = hi[0];
  it.lo1 = lo[1];
  it.hi1 = hi[1];
}

// Packed batches: entry e of the planned list for head h.
struct VarlenItem {
  int h, pair, q_base, Tq, k_base, Tk;
};

__device__ __forceinline__ VarlenItem varlen_item(const PrefillParams &p, int idx,
                                                  int entries) {
  // Heads in groups of head_group (K/V of a group stay in L2); inside a
  // group the list's order (heaviest first), each entry for every head of
  // the group in turn.
  const int per_full = p.head_group * entries;
  const int n_full = p.Hq / p.head_group;
  int g0, gsize, r;
  if (idx < n_full * per_full) {
    g0 = (idx / per_full) * p.head_group;
    gsize = p.head_group;
    r = idx % per_full;
  } else {
    g0 = n_full * p.head_group;
    gsize = p.Hq - g0;
    r = idx - n_full * per_full;
  }
  const int e = r / gsize;
  VarlenItem v;
  v.h = g0 + r % gsize;
  const int b = p.vl_list[2 + 2 * e];
  v.pair = p.vl_list[3 + 2 * e];
  v.q_base = p.cu_q[b];
  v.Tq = p.cu_q[b + 1] - v.q_base;
  v.k_base = p.cu_k[b];
  v.Tk = p.cu_k[b + 1] - v.k_base;
  return v;
}

template <bool kWindow>
__device__ __forceinline__ PrefillItem varlen_prefill_item(const PrefillParams &p,
                                                           const VarlenItem &v) {
  PrefillItem it;
  it.bh = v.h;
  it.bh_kv = v.h / p.group;
  it.q0 = v.pair * 256;
  prefill_ranges<kWindow>(it, v.Tq, v.Tk, p.causal, p.window);
  return it;
}

template <bool kWindow>
__device__ __forceinline__ PrefillItem prefill_item(const PrefillParams &p, int idx) {
  // Heads are taken in groups of head_group; inside a group the heaviest
  // query-tile pairs of every head come first, so the items in flight share
  // the K/V of one group in L2 and the light items that end a group fill in.
  const int per_full = p.head_group * p.n_qt;
  const int n_full = p.n_bh / p.head_group;
  int g0, gsize, r;
  if (idx < n_full * per_full) {
    g0 = (idx / per_full) * p.head_group;
    gsize = p.head_group;
    r = idx % per_full;
  } else {
    g0 = n_full * p.head_group;
    gsize = p.n_bh - g0;
    r = idx - n_full * per_full;
  }
  PrefillItem it;
  const int qt = p.n_qt - 1 - r / gsize;
  it.bh = g0 + r % gsize;
  const int b = it.bh / p.Hq;
  const int h = it.bh - b * p.Hq;
  it.bh_kv = b * p.Hkv + h / p.group;
  it.q0 = qt * 256;
  prefill_ranges<kWindow>(it, p.Tq, p.Tk, p.causal, p.window);
  return it;
}

// Work slot of a launch: two words, each (tag << 32) | count, counting the
// items taken and the CTAs that have finished.  Tag 0 marks a free word; the
// launch's first increment of a word that is free or carries an older tag
// claims it (compare-and-swap) and restarts the count.  Every other
// increment is one atomicAdd: an add that lands on an unclaimed word only
// moves that word's stale count and is retried after the claim.  Every
// launch made outside graph capture has a tag of its own, so it leaves its
// words as they are; a launch captured into a CUDA graph keeps its tag for
// every replay, so its last CTA frees the words again (those launches use
// slots of their own).  Returns false if a newer launch owns the word (more
// launches in flight than there are slots), or if the claim keeps losing
// for an implausible number of rounds.
__device__ __forceinline__ bool tagged_increment(unsigned long long *word, unsigned int tag,
                                                 unsigned int *before) {
  const unsigned long long mine = (unsigned long long)tag << 32;
  for (int round = 0; round < 4096; ++round) {
    const unsigned long long old = atomicAdd(word, 1ull);
    const unsigned int t = (unsigned int)(old >> 32);
    if (t == tag) {
      *before = (unsigned int)old;
      return true;
    }
    if (t != 0 && (int)(t - tag) > 0) return false;  // a newer launch owns it
    // free or older: claim it, unless another CTA of this launch already has
    unsigned long long cur = old + 1ull;
    for (int c = 0; c < 4096; ++c) {
      const unsigned long long prev = atomicCAS(word, cur, mine | 1ull);
      if (prev == cur) {
        *before = 0;
        return true;
      }
      const unsigned int pt = (unsigned int)(prev >> 32);
      if (pt == tag) break;  // claimed by another CTA: add again
      if (pt != 0 && (int)(pt - tag) > 0) return false;
      cur = prev;
    }
  }
  return false;
}

// Frees the word if the launch with this tag still owns it.
__device__ __forceinline__ void tagged_release(unsigned long long *word, unsigned int tag) {
  unsigned long long w = atomicAdd(word, 0ull);
  for (int round = 0; round < (1 << 20); ++round) {
    if ((unsigned int)(w >> 32) != tag) return;
    const unsigned long long prev = atomicCAS(word, w, 0ull);
    if (prev == w) return;
    w = prev;
  }
}

template <int D, bool kWindow, bool kVarlen>
__global__ void __launch_bounds__(320, 1)
    prefill_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const PrefillParams p) {
  using C = PrefillCfg<D>;
  constexpr int ST = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
  uint64_t *drain = bars + 0;
  uint64_t *q_full = bars + 1, *q_empty = bars + 3, *s_full = bars + 5;
  uint64_t *p_full = bars + 7, *o_done = bars + 9;
  uint64_t *item_full = bars + 11, *item_empty = bars + 13;
  uint64_t *k_full = bars + 15, *v_full = k_full + ST;
  uint64_t *k_empty = v_full + ST, *v_empty = k_empty + ST;
  // SEP_P: S_t has been loaded (its region may be rewritten); P_t V done
  uint64_t *s_free = v_empty + ST, *pv_done = s_free + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);
  volatile int *item_ring =
      reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 16);  // [2][kRingInts]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t wait_ns = p.wait_ns;

  if (threadIdx.x == 0) {
    mbar_init(drain, 1);
    for (int t = 0; t < C::NQ; ++t) {
      mbar_init(&q_full[t], 1);
      mbar_init(&q_empty[t], 1);
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], C::BM);
      mbar_init(&o_done[t], 1);
      mbar_init(&s_free[t], C::BM);
      mbar_init(&pv_done[t], 1);
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(&item_full[k], 1);
      mbar_init(&item_empty[k], 9);  // 8 softmax warps + the MMA thread
    }
    for (int s = 0; s < ST; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  auto fail = [&]() {
    atomicExch(p.status, kStatusTimeout);
    *abort_flag = 1;
  };
  // Consumers read the next work item index from the producer's ring
  // (-1 ends the walk).  Returns false if the wait expired.
  // Packed batches: the geometry published with the item.
  auto take_item = [&](int &fetch, int &idx, PrefillItem &it, VarlenItem &vi) -> bool {
    const int k = fetch & 1;
    if (!mbar_wait(&item_full[k], (fetch >> 1) & 1, wait_ns)) return false;
    const volatile int *e = item_ring + k * kRingInts;
    idx = e[0];
    it.bh = e[1];
    it.bh_kv = e[2];
    it.q0 = e[3];
    it.lo0 = e[4];
    it.hi0 = e[5];
    it.lo1 = e[6];
    it.hi1 = e[7];
    if constexpr (kVarlen) {
      vi.q_base = e[8];
      vi.Tq = e[9];
      vi.k_base = e[10];
      vi.Tk = e[11];
    }
    ++fetch;
    return true;
  };

  if (warp == C::PRODUCER_WARP) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      bool ok = true;
      int last_k[ST], last_v[ST];
      for (int s = 0; s < ST; ++s) last_k[s] = last_v[s] = -1;
      int q_cnt[C::NQ] = {0, 0};
      int kv = 0;  // K/V tiles issued so far (all items)
      bool first = true;
      int n_items = p.n_items;
      if constexpr (kVarlen) n_items = p.vl_list[0] * p.Hq;  // written by the planner
      for (int fetch = 0; ok; ++fetch) {
        // Take the next work item from the launch-wide counter and publish
        // it to the other roles through a two-entry ring.
        const int k = fetch & 1;
        if (fetch >= 2 && !mbar_wait(&item_empty[k], ((fetch >> 1) - 1) & 1, wait_ns)) {
          ok = false;
          break;
        }
        // The first item of every CTA is its block index (the heaviest items
        // come first); later ones come from the launch's counter.
        int idx = -1;
        if (fetch == 0) {
          idx = (int)blockIdx.x < n_items ? (int)blockIdx.x : -1;
        } else {
          unsigned int taken = 0;
          if (!tagged_increment(&p.work[0], p.epoch, &taken))
            atomicMax(p.status, kStatusSlotLost);
          else if ((long long)taken + gridDim.x < (long long)n_items)
            idx = (int)(taken + gridDim.x);
        }
        volatile int *ring = item_ring + k * kRingInts;
        ring[0] = idx;
        VarlenItem vi{};
        PrefillItem it{};
        if (idx >= 0) {
          if constexpr (kVarlen) {
            vi = varlen_item(p, idx, n_items / p.Hq);
            it = varlen_prefill_item<kWindow>(p, vi);
            ring[8] = vi.q_base;
            ring[9] = vi.Tq;
            ring[10] = vi.k_base;
            ring[11] = vi.Tk;
          } else {
            it = prefill_item<kWindow>(p, idx);
          }
          ring[1] = it.bh;
          ring[2] = it.bh_kv;
          ring[3] = it.q0;
          ring[4] = it.lo0;
          ring[5] = it.hi0;
          ring[6] = it.lo1;
          ring[7] = it.hi1;
        }
        mbar_arrive(&item_full[k]);
        if (idx < 0) break;
        for (int t = 0; t < C::NQ && ok; ++t) {
          if (!it.has(t)) continue;
          // Q_t is free once the previous item's last S_t has completed.
          if (q_cnt[t] > 0 && !mbar_wait(&q_empty[t], (q_cnt[t] - 1) & 1, wait_ns)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&q_full[t], C::Q_BYTES);
          for (int c = 0; c < C::NCHUNK; ++c) {
            uint8_t *dst = smem + C::OFF_Q + t * C::Q_BYTES + c * (C::BM * C::SPAN);
            if constexpr (kVarlen)
              tma_load_3d(dst, &tm_q, &q_full[t], c * C::CHUNK, it.bh,
                          vi.q_base + it.q0 + t * C::BM);
            else
              tma_load_3d(dst, &tm_q, &q_full[t], c * C::CHUNK, it.q0 + t * C::BM, it.bh);
          }
          ++q_cnt[t];
        }
        const int jb = kWindow ? it.jbeg() : 0, je = it.jend();
        for (int j = jb; ok && j < je; ++j, ++kv) {
          const int s = kv % ST, u = kv / ST;
          if (*abort_flag) { ok = false; break; }
          if (kv >= ST && !mbar_wait(&k_empty[s], (u - 1) & 1, wait_ns)) { ok = false; break; }
          // K/V row j*BN of the item's K/V head: (column, row, plane) in the
          // [B*Hkv, Tk, D] view, (column, head, token) in the packed view
          const int ky = kVarlen ? it.bh_kv : j * C::BN;
          const int kz = kVarlen ? vi.k_base + j * C::BN : it.bh_kv;
          mbar_arrive_expect_tx(&k_full[s], C::KV_BYTES);
          for (int c = 0; c < C::NCHUNK; ++c)
            tma_load_3d(smem + C::OFF_K + s * C::KV_BYTES + c * (C::BN * C::SPAN),
                        &tm_k, &k_full[s], c * C::CHUNK, ky, kz);
          last_k[s] = kv;
          if (kv >= ST && !mbar_wait(&v_empty[s], (u - 1) & 1, wait_ns)) { ok = false; break; }
          if (!(p.inject == 1 && first && j == jb)) {
            mbar_arrive_expect_tx(&v_full[s], C::KV_BYTES);
            for (int c = 0; c < C::NCHUNK; ++c)
              tma_load_3d(smem + C::OFF_V + s * C::KV_BYTES + c * (C::BN * C::SPAN),
                          &tm_v, &v_full[s], c * C::CHUNK, ky, kz);
            last_v[s] = kv;
          }
        }
        first = false;
      }
      if (!ok) fail();
      // Drain: every copy this thread issued has landed before the CTA's
      // shared memory can be released.
      for (int t = 0; t < C::NQ; ++t)
        if (q_cnt[t] > 0) mbar_wait(&q_full[t], (q_cnt[t] - 1) & 1, wait_ns);
      for (int s = 0; s < ST; ++s) {
        if (last_k[s] >= 0) mbar_wait(&k_full[s], (last_k[s] / ST) & 1, wait_ns);
        if (last_v[s] >= 0) mbar_wait(&v_full[s], (last_v[s] / ST) & 1, wait_ns);
      }
    }
    __syncwarp();
  } else if (warp == C::MMA_WARP) {
    // ------------------------------------------------------- MMA issuer
    // The tensor core's instruction queue is short, so every instruction the
    // issuer runs between MMAs can leave it idle.  The whole warp runs this
    // loop converged and one elected lane issues each MMA and commit: the
    // descriptors (built once, advanced by compile-time byte offsets; the
    // start address sits in the low bits in 16-byte units) then stay in
    // uniform registers, which keeps the issue stream short even while the
    // softmax warps on the same sub-partition compete for issue slots.  Every
    // wait is a warp vote so the lanes cannot diverge.  Only waits on barriers
    // that other threads' tensor-memory writes complete are followed by a
    // tcgen05 fence.
    {
      auto wait_all = [&](uint64_t *bar, uint32_t parity) -> bool {
        return __all_sync(0xffffffffu, mbar_wait(bar, parity, wait_ns));
      };
      auto aborted = [&]() -> bool { return __any_sync(0xffffffffu, *abort_flag != 0); };
      constexpr uint32_t IDESC_QK = make_idesc_bf16(C::BM, C::BN, false);
      constexpr uint32_t IDESC_PV = make_idesc_bf16(C::BM, D, true);
      const uint64_t q_desc = make_smem_desc(sbase + C::OFF_Q, 16, 8 * C::SPAN, C::LAYOUT);
      const uint64_t k_desc = make_smem_desc(sbase + C::OFF_K, 16, 8 * C::SPAN, C::LAYOUT);
      // V as B of P V: MN-major, LBO = next CHUNK head-dim columns, SBO = next 8 keys
      const uint64_t v_desc =
          make_smem_desc(sbase + C::OFF_V, C::BN * C::SPAN, 8 * C::SPAN, C::LAYOUT);
      auto adv = [](uint64_t desc, uint32_t bytes) { return desc + (uint64_t)(bytes >> 4); };
      auto issue_s = [&](const int t, const int s) {
        const uint64_t kd = adv(k_desc, s * C::KV_BYTES);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk * 16) / C::CHUNK) * (C::BM * C::SPAN) + ((kk * 16) % C::CHUNK) * 2;
          mma_bf16_ss_elect(tmem + C::tm_s(t), adv(q_desc, t * C::Q_BYTES + off), adv(kd, off),
                      IDESC_QK, kk > 0 ? 1u : 0u);
        }
      };
      auto issue_pv = [&](const int t, const int s, const bool acc) {
        const uint64_t vd = adv(v_desc, s * C::KV_BYTES);
#pragma unroll
        for (int kk = 0; kk < C::BN / 16; ++kk)  // 16 keys = 8 TMEM columns of P
          mma_bf16_ts_elect(tmem + C::tm_o(t), tmem + C::tm_p(t) + kk * 8, adv(vd, kk * 16 * C::SPAN),
                      IDESC_PV, (acc || kk > 0) ? 1u : 0u);
      };
      bool ok = true;
      int q_cnt0 = 0, q_cnt1 = 0;  // Q_t tiles consumed
      int p_cnt0 = 0, p_cnt1 = 0;  // P_t tiles consumed
      int f_cnt0 = 0, f_cnt1 = 0;  // S_t loads signalled (SEP_P)
      int kv = 0;                  // K/V tiles consumed (all items)
      for (int fetch = 0; ok;) {
        int idx = -1;
        VarlenItem vi;
        PrefillItem it;
        if (!__all_sync(0xffffffffu, take_item(fetch, idx, it, vi))) { ok = false; break; }
        if (lane == 0) mbar_arrive(&item_empty[(fetch - 1) & 1]);
        if (idx < 0) break;
        const int jb = kWindow ? it.jbeg() : 0, je = it.jend();
        // S_t of K/V tile jj in stage sj, the first S of tile t's range.
        auto start_tile = [&](const int t, int &q_cnt, const int sj, const int jj) -> bool {
          if (!wait_all(&q_full[t], q_cnt & 1)) return false;
          ++q_cnt;
          issue_s(t, sj);
          mma_commit_elect(&s_full[t]);
          if (jj + 1 == it.hi(t)) mma_commit_elect(&q_empty[t]);  // its only S
          return true;
        };
        {
          // First S of the tiles whose range starts at the item's first tile.
          const int s0 = kv % ST;
          if (aborted() || !wait_all(&k_full[s0], (kv / ST) & 1)) { ok = false; break; }
          if (it.has(0) && it.lo0 == jb && !start_tile(0, q_cnt0, s0, jb)) { ok = false; break; }
          if (it.has(1) && it.lo1 == jb && !start_tile(1, q_cnt1, s0, jb)) { ok = false; break; }
          mma_commit_elect(&k_empty[s0]);
        }
        for (int j = jb; j < je; ++j) {
          const int c = kv + (j - jb);  // ring position of K/V tile j
          const int s = c % ST, u = c / ST;
          const int s1 = (c + 1) % ST, u1 = (c + 1) / ST;
          bool v_ready = false, k_ready = false;
          auto need_k = [&]() -> bool {
            if (k_ready) return true;
            if (!wait_all(&k_full[s1], u1 & 1)) return false;
            k_ready = true;
            return true;
          };
          // One query tile: P_t V_j and S_t of the next K/V tile, or the first
          // S_t if the tile's range starts with the next K/V tile.
          auto tile_step = [&](const int t, int &p_cnt, int &q_cnt) -> bool {
            // Without a window every range starts at 0 and this reduces to
            // "j < hi": the issuing warp is the kernel's bottleneck, so the
            // plain case carries none of the range logic.
            const int lo = kWindow ? it.lo(t) : 0, hi = it.hi(t);
            if ((!kWindow || lo <= j) && j < hi) {
              if (!wait_all(&p_full[t], p_cnt & 1)) return false;
              ++p_cnt;
              if (!v_ready) {
                if (!wait_all(&v_full[s], u & 1)) return false;
                v_ready = true;
              }
              tc_fence_after();  // P_t was written to tensor memory by the softmax threads
              issue_pv(t, s, j > lo);
              if (j + 1 < hi) {
                if (!need_k()) return false;
                issue_s(t, s1);
                mma_commit_elect(&s_full[t]);
                if (j + 2 == hi) mma_commit_elect(&q_empty[t]);  // last S_t of the item
              } else {
                mma_commit_elect(&o_done[t]);
              }
            } else if (kWindow && j + 1 == lo && lo < hi) {
              if (!need_k() || !start_tile(t, q_cnt, s1, j + 1)) return false;
            }
            return true;
          };
          if constexpr (C::SEP_P) {
            // S_t of the next K/V tile as soon as the group has loaded S_t(j)
            // (P_t has a region of its own), then P_t V_j once P_t is ready.
            auto next_s = [&](const int t, int &f_cnt, int &q_cnt) -> bool {
              const int lo = kWindow ? it.lo(t) : 0, hi = it.hi(t);
              if ((!kWindow || lo <= j) && j + 1 < hi) {
                if (!wait_all(&s_free[t], f_cnt & 1)) return false;
                ++f_cnt;
                if (!need_k()) return false;
                tc_fence_after();  // the group's loads of S_t(j) completed before its arrive
                issue_s(t, s1);
                mma_commit_elect(&s_full[t]);
                if (j + 2 == hi) mma_commit_elect(&q_empty[t]);  // last S_t of the item
              } else if (kWindow && j + 1 == lo && lo < hi) {
                if (!need_k() || !start_tile(t, q_cnt, s1, j + 1)) return false;
              }
              return true;
            };
            auto pv = [&](const int t, int &p_cnt) -> bool {
              const int lo = kWindow ? it.lo(t) : 0, hi = it.hi(t);
              if ((!kWindow || lo <= j) && j < hi) {
                if (!wait_all(&p_full[t], p_cnt & 1)) return false;
                ++p_cnt;
                if (!v_ready) {
                  if (!wait_all(&v_full[s], u & 1)) return false;
                  v_ready = true;
                }
                tc_fence_after();  // P_t was written to tensor memory by the softmax threads
                issue_pv(t, s, j > lo);
                mma_commit_elect(j + 1 < hi ? &pv_done[t] : &o_done[t]);
              }
              return true;
            };
            if (aborted() || !next_s(0, f_cnt0, q_cnt0) || !next_s(1, f_cnt1, q_cnt1) ||
                !pv(0, p_cnt0) || !pv(1, p_cnt1)) {
              ok = false;
              break;
            }
          } else if (aborted() || !tile_step(0, p_cnt0, q_cnt0) ||
                     !tile_step(1, p_cnt1, q_cnt1)) {
            ok = false;
            break;
          }
          mma_commit_elect(&v_empty[s]);
          if (k_ready) mma_commit_elect(&k_empty[s1]);
        }
        kv += je - jb;
      }
      if (!ok) fail();
      // Drain: all MMAs issued by this warp have completed before tensor
      // memory is freed.
      mma_commit_elect(drain);
      wait_all(drain, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------- softmax + epilogue rows
    const int t = warp >> 2;                      // query tile of this group
    const int r = threadIdx.x & 127;              // row in tile == TMEM lane
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t t_s = tmem + lane_base + C::tm_s(t);
    const uint32_t t_o = tmem + lane_base + C::tm_o(t);
    const uint32_t t_p = tmem + lane_base + C::tm_p(t);
    const float sl2 = p.scale_log2;
    int s_cnt = 0;  // S_t tiles consumed (all items)
    int o_cnt = 0;  // O_t tiles finished (all items)
    int v_cnt = 0;  // P_t V products waited for (SEP_P)
    bool ok = true;

    for (int fetch = 0; ok;) {
      int idx = -1;
      VarlenItem vi;
      PrefillItem it;
      ok = __all_sync(0xffffffffu, take_item(fetch, idx, it, vi));
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(&item_empty[(fetch - 1) & 1]);
      if (idx < 0) break;
      if (!it.has(t)) continue;
      const int Tq = kVarlen ? vi.Tq : p.Tq;
      const int Tk = kVarlen ? vi.Tk : p.Tk;
      const int delta = Tk - Tq;
      const int jlo = kWindow ? it.lo(t) : 0, jhi = it.hi(t);
      const int row0 = it.q0 + t * C::BM;
      const int row_g = row0 + r;
      const int lim = p.causal ? row_g + delta : 0x7fffffff;                 // last visible key
      const int lim_lo = kWindow ? row_g + delta - p.window + 1 : -1;   // first visible key
      // the largest first-visible key of the tile's rows
      const int tile_lo = kWindow ? min(row0 + C::BM - 1, Tq - 1) + delta - p.window + 1 : -1;
      float m_used = -INFINITY;  // reference max, log2 units
      float l_sum = 0.f;

      for (int j = jlo; j < jhi; ++j) {
        ok = __all_sync(0xffffffffu, mbar_wait(&s_full[t], s_cnt & 1, wait_ns) && !*abort_flag);
        if (!ok) break;
        ++s_cnt;
        tc_fence_after();
        float s[C::BN];
        tmem_ld128_wait(t_s, s);
        if constexpr (C::SEP_P) {
          // S_t(j) is in registers: the next S_t may overwrite its region
          if (j + 1 < jhi) {
            tc_fence_before();
            mbar_arrive(&s_free[t]);
          }
        }

        const int kbase = j * C::BN;
        const bool need_mask = (kbase + C::BN > Tk) ||
                               (p.causal && kbase + C::BN - 1 > row0 + delta) ||
                               (kWindow && kbase < tile_lo);
        if (need_mask) {
          // the row sees the columns [lo, lo + cnt) of this tile: keys from
          // max(lim_lo, 0) to min(lim, Tk - 1)
          const int lo = max((kWindow ? max(lim_lo, 0) : 0) - kbase, 0);
          const int hi = min(min(lim, Tk - 1) - kbase, C::BN - 1);
          const unsigned cnt = (unsigned)max(hi - lo + 1, 0);
#pragma unroll
          for (int c = 0; c < C::BN; ++c)
            if ((unsigned)(c - lo) >= cnt) s[c] = -INFINITY;
        }
        float mx[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[i] = s[i];
#pragma unroll
        for (int c = 8; c < C::BN; c += 8)
#pragma unroll
          for (int i = 0; i < 8; ++i) mx[i] = fmaxf(mx[i], s[c + i]);
        const float mxa = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
        const float m_tile = mxa * sl2;  // scale > 0, so the max commutes
        const float m_new = fmaxf(m_used, m_tile);
        const bool resc = m_new > m_used + kRescaleLog2;
        float alpha = 1.f;
        if (resc) {
          alpha = ex2_approx(m_used - m_new);  // 0 while nothing was seen
          m_used = m_new;
        }
        // Rescaling O_t by alpha: chunks of 16 columns keep the registers this
        // rare path needs small next to the S row.
        auto rescale_o = [&]() {
          const float2 al2 = make_float2(alpha, alpha);
#pragma unroll 1
          for (int cb = 0; cb < D / 16; ++cb) {
            float o[16];
            tmem_ld16_wait(t_o + cb * 16, o);
            uint32_t ow[16];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float2 y = __fmul2_rn(make_float2(o[2 * i], o[2 * i + 1]), al2);
              ow[2 * i] = __float_as_uint(y.x);
              ow[2 * i + 1] = __float_as_uint(y.y);
            }
            tmem_st16(t_o + cb * 16, ow);
          }
          tmem_st_wait();
        };
        if constexpr (C::SEP_P) {
          // P_t V_(j-1) has read P_t and updated O_t before either is touched
          if (j > jlo) {
            ok = __all_sync(0xffffffffu,
                            mbar_wait(&pv_done[t], v_cnt & 1, wait_ns) && !*abort_flag);
            if (!ok) break;
            ++v_cnt;
            tc_fence_after();
          }
        }
        // O_t is stable here (PV_t(j-1) completed before S_t(j) was signalled,
        // or, with a P region of its own, was waited for above): rescale it
        // before any of P_t(j) is published.
        if (j > jlo && __any_sync(0xffffffffu, resc)) rescale_o();
        const float m_ref = (m_used == -INFINITY) ? 0.f : m_used;
        const float2 c2 = make_float2(sl2, sl2);
        const float2 b2 = make_float2(-m_ref, -m_ref);
        float2 acc2[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) acc2[i] = make_float2(0.f, 0.f);
        // P_t as bf16 pairs into the first 64 columns of S_t (whose scores
        // are all in registers already), stored 16 columns (32 keys) at a
        // time as they are produced so the packed row never lives whole.
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint32_t pw[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const int cc = q4 * 16 + c;
            const float2 x = __ffma2_rn(make_float2(s[2 * cc], s[2 * cc + 1]), c2, b2);
            const float2 e = make_float2(ex2_approx(x.x), ex2_approx(x.y));
            acc2[c & 3] = __fadd2_rn(acc2[c & 3], e);
            pw[c] = pack_bf16x2(e.x, e.y);
          }
          tmem_st16(t_p + q4 * 16, pw);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&p_full[t]);
        const float2 a01 = __fadd2_rn(acc2[0], acc2[1]);
        const float2 a23 = __fadd2_rn(acc2[2], acc2[3]);
        const float2 a = __fadd2_rn(a01, a23);
        l_sum = fmaf(l_sum, alpha, a.x + a.y);
      }
      if (!ok) break;

      // ---------------------------------------------------------- epilogue
      ok = __all_sync(0xffffffffu, mbar_wait(&o_done[t], o_cnt & 1, wait_ns));
      if (!ok) break;
      ++o_cnt;
      tc_fence_after();
      const float inv_l = (l_sum > 0.f) ? 1.f / l_sum : 0.f;
      // O leaves through this warp's staging area: each thread writes its
      // own row there, then each global store instruction writes whole
      // 128-byte lines of 32 / EPI_UNITS rows (a thread storing its own row
      // touches 32 lines per instruction, and those partial-line stores held
      // up the next item's TMA loads).  The lane index is read here, not
      // hoisted out of the item loop, so the staging addresses derived from
      // it do not stay live across the loop.
      uint32_t el;
      asm volatile("mov.u32 %0, %%laneid;" : "=r"(el));
      const int elane = (int)el;
      uint8_t *stage = smem + C::OFF_EPI + warp * C::EPI_WARP_BYTES;
      constexpr int EPI_COLS = C::EPI_ROW / 2;   // bf16 columns per pass
      constexpr int ROWS_PER_ST = 32 / C::EPI_UNITS;
      const int un = elane % C::EPI_UNITS;        // 16-byte unit this lane stores
      // the first row this lane stores, and the rows after it ROWS_PER_ST apart:
      // [B, Hq, Tq, D] rows, or token-major [total_q, Hq, D] rows when packed
      const int g0 = row0 + (warp & 3) * 32 + elane / C::EPI_UNITS;
      const size_t row_step = kVarlen ? (size_t)p.Hq * D : (size_t)D;
      __nv_bfloat16 *optr = p.o + (kVarlen ? (size_t)(vi.q_base + g0) * p.Hq + it.bh
                                           : (size_t)it.bh * Tq + g0) * D + un * 8;
      // the whole row of O_t in one tensor-memory load (one wait)
      float o[D];
      if constexpr (D == 128)
        tmem_ld128_wait(t_o, o);
      else if constexpr (D == 64)
        tmem_ld64_wait(t_o, o);
      else
        tmem_ld32_wait(t_o, o);
#pragma unroll
      for (int ps = 0; ps < C::EPI_PASSES; ++ps) {
#pragma unroll
        for (int u = 0; u < C::EPI_UNITS; ++u) {
          const float *x = o + ps * EPI_COLS + u * 8;
          uint4 w;
          w.x = pack_bf16x2(x[0] * inv_l, x[1] * inv_l);
          w.y = pack_bf16x2(x[2] * inv_l, x[3] * inv_l);
          w.z = pack_bf16x2(x[4] * inv_l, x[5] * inv_l);
          w.w = pack_bf16x2(x[6] * inv_l, x[7] * inv_l);
          *reinterpret_cast<uint4 *>(stage + elane * C::EPI_ROW + (C::epi_swz(u, elane) << 4)) = w;
        }
        __syncwarp();
#pragma unroll
        for (int i = 0; i < C::EPI_UNITS; ++i) {
          const int rr = i * ROWS_PER_ST + elane / C::EPI_UNITS;  // row in this warp
          const uint4 w = *reinterpret_cast<const uint4 *>(stage + rr * C::EPI_ROW +
                                                           (C::epi_swz(un, rr) << 4));
          if (g0 + i * ROWS_PER_ST < Tq)
            *reinterpret_cast<uint4 *>(optr + i * ROWS_PER_ST * row_step + ps * EPI_COLS) = w;
        }
        __syncwarp();
      }
      // O_t has been read: the next item's first PV_t may overwrite it (it
      // waits for this group's next P_t, published after this fence).
      tc_fence_before();
      if (row_g < Tq) {
        const size_t lse_idx = kVarlen ? (size_t)it.bh * p.total_q + vi.q_base + row_g
                                       : (size_t)it.bh * Tq + row_g;
        float lse;
        if (l_sum > 0.f)
          lse = (m_used + log2f(l_sum)) * kLn2;
        else
          lse = (m_used == -INFINITY) ? 0.f : m_used * kLn2;
        p.lse[lse_idx] = lse;
      }
    }
    if (!ok) fail();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
  if (p.graph_mode && threadIdx.x == 0) {
    // Every producer of this launch has stopped fetching once all its CTAs
    // have arrived here, so the last one frees the slot for the next replay.
    __threadfence();
    unsigned int done = 0;
    if (tagged_increment(&p.work[1], p.epoch, &done) && done + 1 == gridDim.x) {
      tagged_release(&p.work[0], p.epoch);
      tagged_release(&p.work[1], p.epoch);
      __threadfence();
    }
  }
}

}  // namespace attn_dev
