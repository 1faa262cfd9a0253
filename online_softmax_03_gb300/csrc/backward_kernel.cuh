// backward_kernel.cuh -- attention backward on sm_103a tensor cores.
//
// Gradients with recomputation ("4.2 FlashAttention I: IO-Awareness & The
// Online Softmax", section "The backward pass: recomputation instead of
// storage"; "Efficient attention & KV cache", section 2.2): nothing of size
// T x T is stored; each probability tile is rebuilt from the saved row
// log-sum-exp, P = e^(S - L), and
//
//   dV = P^T dO,  dP = dO V^T,  dS = P o (dP - D)  with D_i = dO_i . O_i,
//   dQ = scale dS K,  dK = scale dS^T Q.
//
// Loop order: keys outer, as the page describes for FlashAttention-1's
// backward, so a CTA finishes dK and dV of its key tile in tensor memory
// and only dQ is accumulated across CTAs.  The rest of this comment
// describes attn_bwd_kernel<D> (d = 32); d = 64 and d = 128 run
// attn_bwd_bm128_kernel, described at its definition.  One CTA (320 threads, one per SM)
// owns 128 keys of one K/V head and walks every query tile of every query
// head of that head's group (grouped-query attention); under causal masking
// it starts at the first query tile that sees its keys, and under a sliding
// window of W keys ("4.2 FlashAttention I", Exercise 4) it also stops after
// the last query tile whose window reaches them, masking the steps that
// cross either edge.  Per step of 128 queries:
//
//   warp 8     producer: K and V of the key tile once, then per step the Q
//              and dO tiles (TMA) and the step's aux rows (bulk copy).
//   warp 9     MMA issuer (converged warp, one elected lane issues), tcgen05.mma
//              kind::f16, fp32 accumulate:
//                S^T  = K Q^T     (A = K, B = Q, both from shared memory)
//                dP^T = V dO^T    (A = V, B = dO)
//                dV  += P^T dO    (A = P^T from tensor memory, B = dO)
//                dK  += dS^T Q    (A = dS^T from tensor memory, B = Q)
//                dQ   = dS K      (A = dS from shared memory, B = K)
//   warps 0-3  one thread per key (TMEM lane): P^T = e^(scale (S^T - L/scale)) with
//              the causal mask, dS^T = P^T o (dP^T - D), written as bf16 into
//              tensor memory (for dV and dK) and into shared memory (for dQ);
//              at the end dK (times scale) and dV are stored as bf16.
//   warps 4-7  one thread per query: dQ of the step from tensor memory into
//              a swizzled shared-memory tile, added into an fp32 buffer in
//              global memory by TMA reduce-add (the page's "dQ is
//              accumulated with atomics"; the order of the additions, and so
//              the last bits of dQ, vary from run to run).
//
// The row statistics enter through the products: one more K-step multiplies
// a constant key-side operand ([1, 1, 0, ...] for S^T, [0, 0, 1, 1, 0, ...]
// for dP^T) by per-query aux rows [-L/scale, -D] (each split into a bf16
// high and low part), so S^T arrives as S - L/scale and dP^T as dP - D and
// the P/dS threads read no per-query values.
//
// Shared memory: K and V of the tile, two stages of (Q, dO, aux), and the
// dS tile, which also stages dQ for the reduction once the dQ MMA has read
// dS (the next step's dS waits for that reduction to have read it).
//
// Tensor memory (512 columns): S^T [0,128) with P^T (bf16) over its first
// 64 columns; dP^T [128,256) with dS^T (bf16) over its first 64 columns and
// dQ over [128,128+D) once dK has read dS^T; dV [256,256+D); dK
// [256+D,256+2D).  MMAs of one thread run in issue order, so a later MMA
// overwrites a region only after the earlier ones have read it.
//
// Every barrier wait is bounded; on expiry the kernel records
// ATTN_ERR_DEVICE_TIMEOUT, stops, drains its own copies and MMAs, frees
// tensor memory and returns.
#pragma once

#include <cuda_bf16.h>

#include "ptx.cuh"

namespace attn_dev {

// The two bf16 halves of a pack_bf16x2 word as fp32 (exact).
__device__ __forceinline__ float2 unpack_bf16x2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

constexpr unsigned int kBwdStatusTimeout = 6;     // ATTN_ERR_DEVICE_TIMEOUT
constexpr unsigned int kBwdStatusMisaligned = 3;  // ATTN_ERR_MISALIGNED

struct BwdParams {
  __nv_bfloat16 *dk, *dv;  // [B, Hkv, Tk, D]
  // per 64-query block of a (batch, head), 2 KB: 16 bf16 per query row,
  // [-L/scale (hi, lo), -D (hi, lo), 0 x 12] with D = rowsum(dO o O), laid out
  // as 8-row x 16-byte core matrices; padding rows carry -1e30 and 0
  const uint8_t *aux;
  float *dq_acc;           // [B*Hq, Tq, D] fp32 dQ accumulator (d = 128 kernel)
  unsigned int *status;
  int Hq, Hkv, group;
  int Tq, Tk, Tq_pad;
  int n_qt;                // ceil(Tq / 128)
  int causal;
  int window;              // > 0: causal sliding window of this many keys
  float scale, scale_log2;
  unsigned long long wait_ns;
  int inject;              // test hook: 3 = CTA (0, 0) withholds its first dO tile
};

template <int D>
struct BwdCfg {
  static constexpr int BM = 128;                      // queries per step
  static constexpr int BN = 128;                      // keys per CTA
  static constexpr int SPAN = (D >= 64) ? 128 : 64;   // swizzle span of Q/K/V/dO rows
  static constexpr int CHUNK = SPAN / 2;
  static constexpr int NCHUNK = D / CHUNK;
  static constexpr uint32_t LAYOUT = (SPAN == 128) ? kLayoutSW128 : kLayoutSW64;
  static constexpr int STAGES = 2;
  static constexpr uint32_t KV_BYTES = BN * D * 2;
  static constexpr uint32_t QT_BYTES = BM * D * 2;
  static constexpr uint32_t AUX_BYTES = BM * 32;  // 16 bf16 per query (see BwdParams::aux)
  static constexpr uint32_t STAGE_BYTES = 2 * QT_BYTES + AUX_BYTES;  // Q | dO | aux
  static constexpr uint32_t OFF_K = 0;
  static constexpr uint32_t OFF_V = OFF_K + KV_BYTES;
  static constexpr uint32_t OFF_STAGE = OFF_V + KV_BYTES;
  static constexpr uint32_t OFF_DS = OFF_STAGE + STAGES * STAGE_BYTES;  // dS^T, bf16
  static constexpr uint32_t DS_HALF = BN * 128;  // 64 queries x 128 keys, 128-byte rows
  // dQ is staged, in two 128 x 32 fp32 chunks (128-byte swizzled rows),
  // in the dS region once the step's dQ MMA has read dS.
  static constexpr uint32_t DQ_CHUNK = BM * 128;
  static_assert(2 * DQ_CHUNK <= 2 * DS_HALF, "dQ staging fits the dS region");
  // constant key-side aux operands: [1, 1, 0, ...] (S^T) and [0, 0, 1, 1, 0, ...] (dP^T)
  static constexpr uint32_t OFF_KAUX = OFF_DS + 2 * DS_HALF;
  static constexpr uint32_t OFF_VAUX = OFF_KAUX + BN * 32;
  static constexpr uint32_t OFF_BAR = OFF_VAUX + BN * 32;
  // kv_full, s_full, p_full, dq_full, dq_empty, dkdv_full, drain, ds_free,
  // q_full[ST], q_empty[ST]
  static constexpr int NBAR = 8 + 2 * STAGES;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  // The dynamic shared-memory window starts 1024-byte aligned (the kernel
  // checks this), so no alignment slack is added.
  static constexpr uint32_t SMEM_USED = OFF_MISC + 16;
  // At least ~116 KB so that only one CTA (which holds all 512 tensor-memory
  // columns) is resident per SM.
  static constexpr uint32_t SMEM_BYTES = SMEM_USED > 118784u ? SMEM_USED : 118784u;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t TM_S = 0, TM_DP = 128, TM_DQ = 128;
  static constexpr uint32_t TM_DV = 256, TM_DK = 256 + D;
  static constexpr int THREADS = 320;
  static_assert(D % CHUNK == 0 && D % 32 == 0, "head dim");
  static_assert(TM_DK + D <= TMEM_COLS, "tensor memory budget");
  static_assert(STAGE_BYTES % 1024 == 0 && KV_BYTES % 1024 == 0, "1 KiB regions");
  static_assert(SMEM_USED <= 232448, "shared memory budget");
};

template <int D>
__global__ void __launch_bounds__(320, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_dq,
                    const BwdParams p) {
  using C = BwdCfg<D>;
  constexpr int ST = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw;
  const uint32_t sbase = smem_u32(smem);
  if (sbase & 1023u) {  // the swizzled tiles need 1024-byte alignment
    if (threadIdx.x == 0) atomicExch(p.status, kBwdStatusMisaligned);
    return;
  }
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
  uint64_t *kv_full = bars + 0, *s_full = bars + 1, *p_full = bars + 2;
  uint64_t *dq_full = bars + 3, *dq_empty = bars + 4, *dkdv_full = bars + 5;
  uint64_t *drain = bars + 6, *ds_free = bars + 7;
  uint64_t *q_full = bars + 8, *q_empty = q_full + ST;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t wait_ns = p.wait_ns;

  const int kt = blockIdx.x;               // key tile
  const int bkv = blockIdx.y;              // b * Hkv + K/V head
  const int b = bkv / p.Hkv;
  const int g = bkv - b * p.Hkv;
  const int delta = p.Tk - p.Tq;           // bottom-right causal alignment
  // Query tiles that see any key of this tile: under causal masking query i
  // sees key j iff j <= i + delta.
  const int qt_lo = p.causal ? max(0, kt * C::BN - delta) / C::BM : 0;
  // Under a sliding window query i also needs j > i + delta - window: the
  // tile's last key is seen by queries up to kt*BN + BN - 2 - delta + window.
  const int q_last = kt * C::BN + C::BN - 2 - delta + p.window;
  const int qt_end = p.window > 0 ? (q_last < 0 ? 0 : min(p.n_qt, q_last / C::BM + 1)) : p.n_qt;
  const int n_q = qt_end - qt_lo;
  const int n_steps = n_q > 0 ? p.group * n_q : 0;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    mbar_init(s_full, 1);
    mbar_init(p_full, 128);
    mbar_init(dq_full, 1);
    mbar_init(dq_empty, 128);
    mbar_init(dkdv_full, 1);
    mbar_init(drain, 1);
    mbar_init(ds_free, 1);
    for (int s = 0; s < ST; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    prefetch_tmap(&tm_do);
    prefetch_tmap(&tm_dq);
  }
  if (threadIdx.x < C::BN) {
    // row r of the key-side aux operands, in 8-row x 16-byte core matrices
    // (bf16 1.0 is 0x3f80)
    const int r = threadIdx.x;
    const uint32_t off = (r >> 3) * 256 + (r & 7) * 16;
    *reinterpret_cast<uint4 *>(smem + C::OFF_KAUX + off) = make_uint4(0x3f803f80u, 0u, 0u, 0u);
    *reinterpret_cast<uint4 *>(smem + C::OFF_KAUX + off + 128) = make_uint4(0u, 0u, 0u, 0u);
    *reinterpret_cast<uint4 *>(smem + C::OFF_VAUX + off) = make_uint4(0u, 0x3f803f80u, 0u, 0u);
    *reinterpret_cast<uint4 *>(smem + C::OFF_VAUX + off + 128) = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
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
    atomicExch(p.status, kBwdStatusTimeout);
    *abort_flag = 1;
  };
  // step s -> query head and query tile
  auto step_head = [&](int s) { return g * p.group + s / n_q; };
  auto step_qt = [&](int s) { return qt_lo + s % n_q; };

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      bool ok = true;
      int last[ST];
      for (int s = 0; s < ST; ++s) last[s] = -1;
      mbar_arrive_expect_tx(kv_full, 2 * C::KV_BYTES);
      for (int c = 0; c < C::NCHUNK; ++c) {
        tma_load_3d(smem + C::OFF_K + c * (C::BN * C::SPAN), &tm_k, kv_full, c * C::CHUNK,
                    kt * C::BN, bkv);
        tma_load_3d(smem + C::OFF_V + c * (C::BN * C::SPAN), &tm_v, kv_full, c * C::CHUNK,
                    kt * C::BN, bkv);
      }
      for (int s = 0; s < n_steps && ok; ++s) {
        const int st = s % ST, u = s / ST;
        if (*abort_flag) { ok = false; break; }
        if (s >= ST && !mbar_wait(&q_empty[st], (u - 1) & 1, wait_ns)) { ok = false; break; }
        const int bh = b * p.Hq + step_head(s);
        const int q0 = step_qt(s) * C::BM;
        uint8_t *stage = smem + C::OFF_STAGE + st * C::STAGE_BYTES;
        mbar_arrive_expect_tx(&q_full[st], 2 * C::QT_BYTES + C::AUX_BYTES);
        // test hook: the first dO tile of CTA (0, 0) is never loaded, so the
        // wait for it must expire
        const bool withhold = p.inject == 3 && s == 0 && blockIdx.x == 0 && blockIdx.y == 0;
        for (int c = 0; c < C::NCHUNK; ++c) {
          tma_load_3d(stage + c * (C::BM * C::SPAN), &tm_q, &q_full[st], c * C::CHUNK, q0, bh);
          if (!withhold)
            tma_load_3d(stage + C::QT_BYTES + c * (C::BM * C::SPAN), &tm_do, &q_full[st],
                        c * C::CHUNK, q0, bh);
        }
        // the aux rows of the step's 128 queries: two consecutive 64-row blocks
        const size_t aoff = ((size_t)bh * (p.Tq_pad / 64) + q0 / 64) * 2048;
        bulk_load(stage + 2 * C::QT_BYTES, p.aux + aoff, C::AUX_BYTES, &q_full[st]);
        last[st] = s;
      }
      if (!ok) fail();
      // Drain: every copy issued has landed before shared memory is released.
      mbar_wait(kv_full, 0, wait_ns);
      for (int s = 0; s < ST; ++s)
        if (last[s] >= 0) mbar_wait(&q_full[s], (last[s] / ST) & 1, wait_ns);
    }
    __syncwarp();
  } else if (warp == 9) {
    // ---------------------------------------------------------- MMA issuer
    // The warp runs converged and one elected lane issues each MMA and commit
    // (descriptors stay in uniform registers); every wait is a warp vote.
    {
      auto wait_all = [&](uint64_t *bar, uint32_t parity) -> bool {
        return __all_sync(0xffffffffu, mbar_wait(bar, parity, wait_ns));
      };
      constexpr uint32_t I_S = make_idesc_bf16(C::BN, C::BM, false);   // S^T, dP^T
      constexpr uint32_t I_ACC = make_idesc_bf16(C::BN, D, true);      // dV, dK
      constexpr uint32_t I_DQ = make_idesc_bf16_ab(C::BM, D, true, true);
      // K-major operands (rows of D, chunks of CHUNK columns)
      const uint64_t k_kd = make_smem_desc(sbase + C::OFF_K, 16, 8 * C::SPAN, C::LAYOUT);
      const uint64_t v_kd = make_smem_desc(sbase + C::OFF_V, 16, 8 * C::SPAN, C::LAYOUT);
      // MN-major views of the same tiles: LBO = next CHUNK columns, SBO = next 8 rows
      const uint64_t k_md =
          make_smem_desc(sbase + C::OFF_K, C::BN * C::SPAN, 8 * C::SPAN, C::LAYOUT);
      // dS as the MN-major A of dQ: rows = keys (128 bytes = 64 queries per half)
      const uint64_t ds_md = make_smem_desc(sbase + C::OFF_DS, C::DS_HALF, 8 * 128, kLayoutSW128);
      auto adv = [](uint64_t desc, uint32_t bytes) { return desc + (uint64_t)(bytes >> 4); };
      // aux K-step: S^T gains -L/scale per query column, dP^T gains -D
      const uint64_t kaux_d = make_smem_desc(sbase + C::OFF_KAUX, 128, 256, kLayoutNone);
      const uint64_t vaux_d = make_smem_desc(sbase + C::OFF_VAUX, 128, 256, kLayoutNone);
      bool ok = wait_all(kv_full, 0);
      for (int s = 0; s < n_steps && ok; ++s) {
        const int st = s % ST, u = s / ST;
        if (__any_sync(0xffffffffu, *abort_flag != 0) || !wait_all(&q_full[st], u & 1)) {
          ok = false;
          break;
        }
        const uint32_t stage = sbase + C::OFF_STAGE + st * C::STAGE_BYTES;
        const uint64_t q_kd = make_smem_desc(stage, 16, 8 * C::SPAN, C::LAYOUT);
        const uint64_t do_kd = make_smem_desc(stage + C::QT_BYTES, 16, 8 * C::SPAN, C::LAYOUT);
        const uint64_t q_md = make_smem_desc(stage, C::BM * C::SPAN, 8 * C::SPAN, C::LAYOUT);
        const uint64_t qaux_d = make_smem_desc(stage + 2 * C::QT_BYTES, 128, 256, kLayoutNone);
        const uint64_t do_md =
            make_smem_desc(stage + C::QT_BYTES, C::BM * C::SPAN, 8 * C::SPAN, C::LAYOUT);
        // S^T = K Q^T
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk * 16) / C::CHUNK) * (C::BN * C::SPAN) + ((kk * 16) % C::CHUNK) * 2;
          mma_bf16_ss_elect(tmem + C::TM_S, adv(k_kd, off), adv(q_kd, off), I_S, kk > 0 ? 1u : 0u);
        }
        mma_bf16_ss_elect(tmem + C::TM_S, kaux_d, qaux_d, I_S, 1u);
        // dP^T overwrites the previous step's dQ: wait until it has been read.
        if (s > 0 && !wait_all(dq_empty, (s - 1) & 1)) { ok = false; break; }
        // dP^T = V dO^T
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk * 16) / C::CHUNK) * (C::BN * C::SPAN) + ((kk * 16) % C::CHUNK) * 2;
          mma_bf16_ss_elect(tmem + C::TM_DP, adv(v_kd, off), adv(do_kd, off), I_S, kk > 0 ? 1u : 0u);
        }
        mma_bf16_ss_elect(tmem + C::TM_DP, vaux_d, qaux_d, I_S, 1u);
        mma_commit_elect(s_full);
        if (!wait_all(p_full, s & 1)) { ok = false; break; }
        tc_fence_after();  // P^T and dS^T were written to tensor memory by other threads
        // dV += P^T dO,  dK += dS^T Q   (16 queries = 8 columns of packed bf16)
#pragma unroll
        for (int kk = 0; kk < C::BM / 16; ++kk)
          mma_bf16_ts_elect(tmem + C::TM_DV, tmem + C::TM_S + kk * 8, adv(do_md, kk * 16 * C::SPAN),
                      I_ACC, (s > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < C::BM / 16; ++kk)
          mma_bf16_ts_elect(tmem + C::TM_DK, tmem + C::TM_DP + kk * 8, adv(q_md, kk * 16 * C::SPAN),
                      I_ACC, (s > 0 || kk > 0) ? 1u : 0u);
        mma_commit_elect(&q_empty[st]);  // Q, dO and aux of this stage are no longer read
        // dQ = dS K   (16 keys per MMA)
#pragma unroll
        for (int kk = 0; kk < C::BN / 16; ++kk)
          mma_bf16_ss_elect(tmem + C::TM_DQ, adv(ds_md, kk * 16 * 128), adv(k_md, kk * 16 * C::SPAN),
                      I_DQ, kk > 0 ? 1u : 0u);
        mma_commit_elect(dq_full);
      }
      if (!ok) fail();
      mma_commit_elect(dkdv_full);
      mma_commit_elect(drain);
      wait_all(drain, 0);
    }
    __syncwarp();
  } else if (warp < 4) {
    // ------------------------------------------- P and dS, one key per thread
    const int r = threadIdx.x;  // key row of the tile == TMEM lane
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const int key = kt * C::BN + r;
    const bool key_ok = key < p.Tk;
    // keys a query sees after its first one (the whole rest without a window)
    const unsigned span = p.window > 0 ? (unsigned)p.window : 0x7fffffffu;
    const float sl2 = p.scale_log2;
    uint8_t *ds_row = smem + C::OFF_DS + r * 128;
    bool ok = true;
    for (int s = 0; s < n_steps; ++s) {
      ok = __all_sync(0xffffffffu, mbar_wait(s_full, s & 1, wait_ns) && !*abort_flag);
      if (!ok) break;
      tc_fence_after();
      const int q0 = step_qt(s) * C::BM;
      // keys above the diagonal of some query of the tile, or (window)
      // left of some query's window, need the mask
      const bool need_mask =
          (p.causal && (kt * C::BN + C::BN - 1 > q0 + delta)) ||
          (p.window > 0 && q0 + C::BM - 1 >= kt * C::BN - delta + p.window);
      // query q (in tile) sees the key iff lim <= q < lim + span
      const int lim = key - delta - q0;
#pragma unroll 1
      for (int c = 0; c < C::BM / 32; ++c) {
        float sv[32], dp[32];
        tmem_ld32_wait(tmem + lane_base + C::TM_S + c * 32, sv);
        tmem_ld32_wait(tmem + lane_base + C::TM_DP + c * 32, dp);
        uint32_t pw[16], dw[16];
        // S^T already holds S - L/scale and dP^T holds dP - D (the aux K-step)
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const int q = c * 32 + i;
          const float2 x = __fmul2_rn(make_float2(sv[i], sv[i + 1]), make_float2(sl2, sl2));
          float p0 = ex2_approx(x.x);
          float p1 = ex2_approx(x.y);
          if (need_mask) {
            if ((unsigned)(q - lim) >= span) p0 = 0.f;
            if ((unsigned)(q + 1 - lim) >= span) p1 = 0.f;
          }
          if (!key_ok) p0 = p1 = 0.f;
          const float2 d = __fmul2_rn(make_float2(p0, p1), make_float2(dp[i], dp[i + 1]));
          pw[i / 2] = pack_bf16x2(p0, p1);
          dw[i / 2] = pack_bf16x2(d.x, d.y);
        }
        // P^T over S^T's columns [16c, 16c+16) and dS^T over dP^T's: those
        // scores were loaded in this or an earlier chunk.
        tmem_st16(tmem + lane_base + C::TM_S + c * 16, pw);
        tmem_st16(tmem + lane_base + C::TM_DP + c * 16, dw);
        // The dS region held the previous step's dQ staging: wait until the
        // reduction has read it.
        if (c == 0 && s > 0) {
          ok = __all_sync(0xffffffffu, mbar_wait(ds_free, (s - 1) & 1, wait_ns));
          if (!ok) break;
        }
        // dS^T row into shared memory: queries [32c, 32c+32) are 16-byte
        // units 4(c%2) .. 4(c%2)+3 of half c/2, swizzled by the row.
        uint8_t *half = ds_row + (c >> 1) * C::DS_HALF;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int unit = (c & 1) * 4 + j;
          *reinterpret_cast<uint4 *>(half + ((unit ^ (r & 7)) << 4)) =
              make_uint4(dw[4 * j], dw[4 * j + 1], dw[4 * j + 2], dw[4 * j + 3]);
        }
      }
      if (!ok) break;
      tmem_st_wait();
      fence_proxy_async_smem();  // dS in shared memory, for the tensor core
      tc_fence_before();
      mbar_arrive(p_full);
    }
    tmem_st_wait();  // no store to tensor memory is in flight past this point
    if (!ok) fail();
    // ---- dK (times scale) and dV of this key tile, bf16
    if (n_steps > 0 && ok) {
      ok = __all_sync(0xffffffffu, mbar_wait(dkdv_full, 0, wait_ns));
      if (!ok) fail();
    }
    if (ok) {
      tc_fence_after();
      const size_t row = ((size_t)bkv * p.Tk + key) * D;
#pragma unroll 1
      for (int which = 0; which < 2; ++which) {
        const uint32_t col = which == 0 ? C::TM_DV : C::TM_DK;
        const float mul = which == 0 ? 1.f : p.scale;
        __nv_bfloat16 *dst = (which == 0 ? p.dv : p.dk) + row;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          float v[32];
          if (n_steps > 0) {
            tmem_ld32_wait(tmem + lane_base + col + c * 32, v);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0.f;
          }
          if (key_ok) {
            uint4 *o = reinterpret_cast<uint4 *>(dst + c * 32);
#pragma unroll
            for (int u = 0; u < 4; ++u)
              o[u] = make_uint4(pack_bf16x2(v[8 * u] * mul, v[8 * u + 1] * mul),
                                pack_bf16x2(v[8 * u + 2] * mul, v[8 * u + 3] * mul),
                                pack_bf16x2(v[8 * u + 4] * mul, v[8 * u + 5] * mul),
                                pack_bf16x2(v[8 * u + 6] * mul, v[8 * u + 7] * mul));
          }
        }
      }
    }
  } else {
    // ------------------------------------ dQ of each step, one query per thread
    const int r = threadIdx.x - 128;  // query row of the step == TMEM lane
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const bool elected = (r == 0);
    bool ok = true;
    int n = 0;  // dQ chunks staged so far
    for (int s = 0; s < n_steps; ++s) {
      // The four warps meet at named barriers below, so they take one
      // decision on whether to go on.
      const bool w_ok =
          __all_sync(0xffffffffu, mbar_wait(dq_full, s & 1, wait_ns) && !*abort_flag);
      ok = named_barrier_and(1, 128, w_ok);
      if (!ok) break;
      tc_fence_after();
      const int bh = b * p.Hq + step_head(s);
      const int q0 = step_qt(s) * C::BM;
      // Read the whole row first so that tensor memory is released (and the
      // next dP^T may start) before the shared-memory staging.
      float vall[D];
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        float v[32];
        tmem_ld32_wait(tmem + lane_base + C::TM_DQ + c * 32, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) vall[c * 32 + i] = v[i];
      }
      tc_fence_before();
      mbar_arrive(dq_empty);  // the step's dQ has left tensor memory
#pragma unroll
      for (int c = 0; c < D / 32; ++c, ++n) {
        const float *v = vall + c * 32;
        uint8_t *buf = smem + C::OFF_DS + (n & 1) * C::DQ_CHUNK;
        // the reduce that last read this buffer (two chunks ago) is done
        if (elected && n >= 2) bulk_wait_group_read1();
        named_barrier_sync(1, 128);
        uint8_t *row = buf + r * 128;
#pragma unroll
        for (int u = 0; u < 8; ++u)
          *reinterpret_cast<float4 *>(row + ((u ^ (r & 7)) << 4)) =
              make_float4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
        fence_proxy_async_smem();
        named_barrier_sync(1, 128);
        if (elected) {
          tma_reduce_add_3d(&tm_dq, buf, c * 32, q0, bh);
          bulk_commit_group();
        }
      }
      // the next step's dS may overwrite the staging once it has been read
      if (elected) {
        bulk_wait_group_read0();
        mbar_arrive(ds_free);
      }
    }
    if (!ok) fail();
    if (elected) bulk_wait_group0();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// d = 64 and 128, 128-query steps: S^T, dP^T and dQ^T are M = 128, N = 128
// MMAs (an N = 64 product costs about 50 cycles of the tensor pipe for 32
// cycles of work, N = 128 costs its 64), dV and dK have N = d.  Tensor memory
// holds one step: region A [0,128) S^T, then the bf16 P^T packed in place;
// region B [128,256) dP^T, then the packed dS^T, then dQ^T (128 head-dim
// rows; at d = 64 rows 64..127 come from zero rows of K^T and are never
// read); dV [256, 256+d); dK [256+d, 256+2d).  Per step the
// tensor pipe runs, in issue order,
//     dP(s)  dV(s)  S(s+1)  dK(s)  dQ^T(s)
// dP(s) goes first (once dQ^T(s-1) has left region B), so the P/dS threads
// form dS(s) right after P(s); S(s+1) runs while they do.  Q (with its aux
// rows) is double-buffered, dO single-buffered.
//
// The fp32 reductions of dQ bound this kernel: every (key tile, 128-query
// step) pair adds 64 KB into the accumulator, and the GPU's L2 completes
// fp32 reductions at about 3.3 TB/s whatever the instruction width, so the
// additions alone take about as long as the whole step.
//
// Warps 0-7: P and dS, one key per thread, warpgroup c owning queries
// [64c, 64c+64); warps 8-15: dQ^T drain, warp w owning TMEM lanes
// 32(w%4).. (head-dim columns; at d = 64 only lanes below 64 have any) for
// queries [64h, 64h+64), h = (w-8)/4; warp 16: TMA producer; warp 17: MMA
// issuer (converged, elected lane).
template <int D_>
struct BwdBm128Cfg {
  static constexpr int D = D_;
  static constexpr int BM = 128;                      // queries per step
  static constexpr int BN = 128;                      // keys per CTA
  static constexpr int SPAN = 128;
  static constexpr int CHUNK = 64;
  static constexpr int NCHUNK = D / CHUNK;
  static constexpr uint32_t KV_BYTES = BN * D * 2;    // 32 KB at d = 128
  static constexpr uint32_t QT_BYTES = BM * D * 2;    // 32 KB at d = 128
  // K^T is the M = 128 A operand of dQ^T whatever d is: at d = 64 the K tile
  // is followed by 16 KB of zeros standing for head-dim rows 64..127
  static constexpr uint32_t KREG_BYTES = BN * 128 * 2;
  static constexpr uint32_t AUX_BYTES = BM * 32;      // 4 KB: 16 bf16 per query
  static constexpr uint32_t QBUF_BYTES = QT_BYTES + AUX_BYTES;  // Q | aux, 36 KB
  static constexpr uint32_t OFF_K = 0;
  static constexpr uint32_t OFF_V = OFF_K + KREG_BYTES;
  static constexpr uint32_t OFF_Q = OFF_V + KV_BYTES;               // 2 buffers
  static constexpr uint32_t OFF_DO = OFF_Q + 2 * QBUF_BYTES;        // 1 buffer
  static constexpr uint32_t OFF_DS = OFF_DO + QT_BYTES;             // dS^T, 2 x 16 KB
  static constexpr uint32_t DS_CHUNK = BN * 128;                    // 64 queries x 128 keys
  static constexpr uint32_t OFF_KAUX = OFF_DS + 2 * DS_CHUNK;
  static constexpr uint32_t OFF_VAUX = OFF_KAUX + BN * 32;
  static constexpr uint32_t OFF_BAR = OFF_VAUX + BN * 32;
  // kv_full, do_full, do_empty, s_full, p_full, dp_full, ds_full, dq_full,
  // dq_empty, ds_free, dkdv_full, drain, q_full[2], q_empty[2]
  static constexpr int NBAR = 16;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 1024;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t TM_A = 0, TM_B = 128, TM_DV = 256, TM_DK = 256 + D;
  static constexpr int THREADS = 576;
  // column of the packed bf16 queries [16kk, 16kk+16) within region A / B
  __host__ __device__ static constexpr uint32_t packed_col(int kk) {
    return (kk / 4) * 64 + (kk % 4) * 8;
  }
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  static_assert(OFF_Q % 1024 == 0 && QBUF_BYTES % 1024 == 0 && OFF_DO % 1024 == 0 &&
                    OFF_DS % 1024 == 0,
                "1 KiB aligned swizzled tiles");
  static_assert(2 * NCHUNK * BN * SPAN <= 2 * QBUF_BYTES, "dK/dV staging fits the Q buffers");
  static_assert(D == 64 || D == 128, "head dim");
};

template <int D_>
__global__ void __launch_bounds__(576, 1)
    attn_bwd_bm128_kernel(const __grid_constant__ CUtensorMap tm_q,
                          const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v,
                          const __grid_constant__ CUtensorMap tm_do,
                          const __grid_constant__ CUtensorMap tm_dk,
                          const __grid_constant__ CUtensorMap tm_dv,
                          const BwdParams p) {
  using C = BwdBm128Cfg<D_>;
  constexpr int D = C::D;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
  uint64_t *kv_full = bars + 0, *do_full = bars + 1, *do_empty = bars + 2;
  uint64_t *s_full = bars + 3, *p_full = bars + 4, *dp_full = bars + 5, *ds_full = bars + 6;
  uint64_t *dq_full = bars + 7, *dq_empty = bars + 8, *ds_free = bars + 9;
  uint64_t *dkdv_full = bars + 10, *drain = bars + 11;
  uint64_t *q_full = bars + 12, *q_empty = bars + 14;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t wait_ns = p.wait_ns;

  const int kt = blockIdx.x;
  const int bkv = blockIdx.y;
  const int b = bkv / p.Hkv;
  const int g = bkv - b * p.Hkv;
  const int delta = p.Tk - p.Tq;
  const int n_qt = p.Tq_pad / C::BM;  // 128-query tiles
  const int qt_lo = p.causal ? max(0, kt * C::BN - delta) / C::BM : 0;
  // Under a sliding window query i also needs j > i + delta - window: the
  // tile's last key is seen by queries up to kt*BN + BN - 2 - delta + window.
  const int q_last = kt * C::BN + C::BN - 2 - delta + p.window;
  const int qt_end = p.window > 0 ? (q_last < 0 ? 0 : min(n_qt, q_last / C::BM + 1)) : n_qt;
  const int n_q = qt_end - qt_lo;
  const int n_steps = n_q > 0 ? p.group * n_q : 0;

  if (threadIdx.x == 0) {
    // p_full and ds_full: all 256 P/dS threads; dq_empty: all 256 dQ threads
    for (int i = 0; i < C::NBAR; ++i)
      mbar_init(&bars[i], (i == 4 || i == 6) ? 2 * C::BN : i == 8 ? 2 * D : 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    prefetch_tmap(&tm_do);
  }
  if (threadIdx.x < C::BN) {
    // row r of the key-side aux operands, in 8-row x 16-byte core matrices
    // (core matrix (r / 8, k-half) at (r / 8) * 256 + k-half * 128, row r % 8
    // at + (r % 8) * 16); bf16 1.0 is 0x3f80
    const int r = threadIdx.x;
    const uint32_t off = (r >> 3) * 256 + (r & 7) * 16;
    *reinterpret_cast<uint4 *>(smem + C::OFF_KAUX + off) = make_uint4(0x3f803f80u, 0u, 0u, 0u);
    *reinterpret_cast<uint4 *>(smem + C::OFF_KAUX + off + 128) = make_uint4(0u, 0u, 0u, 0u);
    *reinterpret_cast<uint4 *>(smem + C::OFF_VAUX + off) = make_uint4(0u, 0x3f803f80u, 0u, 0u);
    *reinterpret_cast<uint4 *>(smem + C::OFF_VAUX + off + 128) = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
  }
  if constexpr (D < 128) {
    // the zero head-dim rows 64..127 of K^T (read by the dQ^T products)
    for (uint32_t o = threadIdx.x * 16; o < C::KREG_BYTES - C::KV_BYTES; o += C::THREADS * 16)
      *reinterpret_cast<uint4 *>(smem + C::OFF_K + C::KV_BYTES + o) = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
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
    atomicExch(p.status, kBwdStatusTimeout);
    *abort_flag = 1;
  };
  auto step_head = [&](int s) { return g * p.group + s / n_q; };
  auto step_qt = [&](int s) { return qt_lo + s % n_q; };

  if (warp == 16) {
    // ------------------------------------------------------------ producer
    // Loads in the order the tensor pipe frees their buffers: Q(s) once
    // dK(s-2) has read Q(s-2), dO(s) once dV(s-1) and dP(s-1) have read dO(s-1).
    if (lane == 0) {
      bool ok = true;
      int last_q[2] = {-1, -1};
      mbar_arrive_expect_tx(kv_full, 2 * C::KV_BYTES);
      for (int c = 0; c < C::NCHUNK; ++c) {
        tma_load_3d(smem + C::OFF_K + c * (C::BN * C::SPAN), &tm_k, kv_full, c * C::CHUNK,
                    kt * C::BN, bkv);
        tma_load_3d(smem + C::OFF_V + c * (C::BN * C::SPAN), &tm_v, kv_full, c * C::CHUNK,
                    kt * C::BN, bkv);
      }
      for (int s = 0; s < n_steps && ok; ++s) {
        if (*abort_flag) { ok = false; break; }
        const int bh = b * p.Hq + step_head(s);
        const int q0 = step_qt(s) * C::BM;
        const int qb = s & 1;
        if (s >= 2 && !mbar_wait(&q_empty[qb], ((s >> 1) - 1) & 1, wait_ns)) { ok = false; break; }
        uint8_t *qbuf = smem + C::OFF_Q + qb * C::QBUF_BYTES;
        mbar_arrive_expect_tx(&q_full[qb], C::QT_BYTES + C::AUX_BYTES);
        for (int c = 0; c < C::NCHUNK; ++c)
          tma_load_3d(qbuf + c * (C::BM * C::SPAN), &tm_q, &q_full[qb], c * C::CHUNK, q0, bh);
        // aux rows of 64-row blocks are 2 KB each and contiguous
        const size_t aoff = ((size_t)bh * (p.Tq_pad / 64) + q0 / 64) * 2048;
        bulk_load(qbuf + C::QT_BYTES, p.aux + aoff, C::AUX_BYTES, &q_full[qb]);
        last_q[qb] = s;
        if (s >= 1 && !mbar_wait(do_empty, (s - 1) & 1, wait_ns)) { ok = false; break; }
        mbar_arrive_expect_tx(do_full, C::QT_BYTES);
        // test hook: the first dO tile of CTA (0, 0) is never loaded, so the
        // wait for it must expire
        if (!(p.inject == 3 && s == 0 && blockIdx.x == 0 && blockIdx.y == 0))
          for (int c = 0; c < C::NCHUNK; ++c)
            tma_load_3d(smem + C::OFF_DO + c * (C::BM * C::SPAN), &tm_do, do_full,
                        c * C::CHUNK, q0, bh);
      }
      if (!ok) fail();
      // Drain: every copy issued has landed before shared memory is released.
      mbar_wait(kv_full, 0, wait_ns);
      for (int qb = 0; qb < 2; ++qb)
        if (last_q[qb] >= 0) mbar_wait(&q_full[qb], (last_q[qb] >> 1) & 1, wait_ns);
      if (n_steps > 0) mbar_wait(do_full, (n_steps - 1) & 1, wait_ns);
    }
    __syncwarp();
  } else if (warp == 17) {
    // ------------------------------------- MMA issuer (converged, elected lane)
    auto wait_all = [&](uint64_t *bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, wait_ns));
    };
    constexpr uint32_t I_S = make_idesc_bf16(C::BN, C::BM, false);       // S^T, dP^T
    constexpr uint32_t I_ACC = make_idesc_bf16(C::BN, D, true);          // dV, dK
    // dQ^T: M = 128 head-dim rows (zero rows past d)
    constexpr uint32_t I_DQ = make_idesc_bf16_ab(128, C::BM, true, true);
    const uint64_t k_kd = make_smem_desc(sbase + C::OFF_K, 16, 8 * C::SPAN, kLayoutSW128);
    const uint64_t v_kd = make_smem_desc(sbase + C::OFF_V, 16, 8 * C::SPAN, kLayoutSW128);
    // K^T as the MN-major A of dQ^T: M = head dim (next 64 columns at +BN*SPAN)
    const uint64_t k_md =
        make_smem_desc(sbase + C::OFF_K, C::BN * C::SPAN, 8 * C::SPAN, kLayoutSW128);
    const uint64_t do_kd = make_smem_desc(sbase + C::OFF_DO, 16, 8 * C::SPAN, kLayoutSW128);
    const uint64_t do_md =
        make_smem_desc(sbase + C::OFF_DO, C::BM * C::SPAN, 8 * C::SPAN, kLayoutSW128);
    // dS^T as the MN-major B of dQ^T: N = queries (next 64 at +DS_CHUNK)
    const uint64_t ds_md =
        make_smem_desc(sbase + C::OFF_DS, C::DS_CHUNK, 8 * 128, kLayoutSW128);
    auto adv = [](uint64_t desc, uint32_t bytes) { return desc + (uint64_t)(bytes >> 4); };
    // aux K-step: S^T gains -L/scale per query column, dP^T gains -D
    const uint64_t kaux_d = make_smem_desc(sbase + C::OFF_KAUX, 128, 256, kLayoutNone);
    const uint64_t vaux_d = make_smem_desc(sbase + C::OFF_VAUX, 128, 256, kLayoutNone);
    auto qbuf = [&](int s) { return sbase + C::OFF_Q + (s & 1) * C::QBUF_BYTES; };
    auto k_off = [](int kk, uint32_t rows) {
      return ((kk * 16) / C::CHUNK) * (rows * C::SPAN) + ((kk * 16) % C::CHUNK) * 2;
    };
    // S^T(s) into region A; dP^T(s) into region B (both with the aux K-step)
    auto issue_s = [&](int s) {
      const uint64_t q_kd = make_smem_desc(qbuf(s), 16, 8 * C::SPAN, kLayoutSW128);
      const uint64_t qaux_d = make_smem_desc(qbuf(s) + C::QT_BYTES, 128, 256, kLayoutNone);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        mma_bf16_ss_elect(tmem + C::TM_A, adv(k_kd, k_off(kk, C::BN)),
                          adv(q_kd, k_off(kk, C::BM)), I_S, kk > 0 ? 1u : 0u);
      mma_bf16_ss_elect(tmem + C::TM_A, kaux_d, qaux_d, I_S, 1u);
      mma_commit_elect(s_full);
    };
    auto issue_dp = [&](int s) {
      const uint64_t qaux_d = make_smem_desc(qbuf(s) + C::QT_BYTES, 128, 256, kLayoutNone);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        mma_bf16_ss_elect(tmem + C::TM_B, adv(v_kd, k_off(kk, C::BN)),
                          adv(do_kd, k_off(kk, C::BM)), I_S, kk > 0 ? 1u : 0u);
      mma_bf16_ss_elect(tmem + C::TM_B, vaux_d, qaux_d, I_S, 1u);
      mma_commit_elect(dp_full);
    };
    bool ok = wait_all(kv_full, 0);
    if (ok && n_steps > 0) {
      ok = wait_all(&q_full[0], 0) && wait_all(do_full, 0);
      if (ok) {
        issue_s(0);
        issue_dp(0);
      }
    }
    for (int s = 0; s < n_steps && ok; ++s) {
      if (__any_sync(0xffffffffu, *abort_flag != 0)) { ok = false; break; }
      // ---- dV(s) += P^T(s) dO(s)  (dP^T(s) was issued before P(s) was formed)
      if (!wait_all(p_full, s & 1)) { ok = false; break; }
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < C::BM / 16; ++kk)
        mma_bf16_ts_elect(tmem + C::TM_DV, tmem + C::TM_A + C::packed_col(kk),
                          adv(do_md, kk * 16 * C::SPAN), I_ACC, (s > 0 || kk > 0) ? 1u : 0u);
      mma_commit_elect(do_empty);  // dO(s) has been read by dP^T(s) and dV(s)
      // ---- S^T(s+1): region A is free once dV(s) has read P^T(s)
      if (s + 1 < n_steps) {
        if (!wait_all(&q_full[(s + 1) & 1], ((s + 1) >> 1) & 1)) { ok = false; break; }
        issue_s(s + 1);
      }
      // ---- dK(s) += dS^T(s) Q(s), then dQ^T(s) = K^T dS^T(s) into region B
      if (!wait_all(ds_full, s & 1)) { ok = false; break; }
      tc_fence_after();
      const uint64_t q_md = make_smem_desc(qbuf(s), C::BM * C::SPAN, 8 * C::SPAN, kLayoutSW128);
#pragma unroll
      for (int kk = 0; kk < C::BM / 16; ++kk)
        mma_bf16_ts_elect(tmem + C::TM_DK, tmem + C::TM_B + C::packed_col(kk),
                          adv(q_md, kk * 16 * C::SPAN), I_ACC, (s > 0 || kk > 0) ? 1u : 0u);
      mma_commit_elect(&q_empty[s & 1]);  // Q(s) and its aux rows have been read
#pragma unroll
      for (int kk = 0; kk < C::BN / 16; ++kk)
        mma_bf16_ss_elect(tmem + C::TM_B, adv(k_md, kk * 16 * C::SPAN),
                          adv(ds_md, kk * 16 * 128), I_DQ, kk > 0 ? 1u : 0u);
      mma_commit_elect(dq_full);
      mma_commit_elect(ds_free);
      // ---- dP^T(s+1) into region B once dQ^T(s) has left it, so that dS(s+1)
      // can follow P(s+1) without waiting for dV(s+1)
      if (s + 1 < n_steps) {
        if (!wait_all(do_full, (s + 1) & 1) || !wait_all(dq_empty, s & 1)) { ok = false; break; }
        tc_fence_after();
        issue_dp(s + 1);
      }
    }
    if (!ok) fail();
    mma_commit_elect(dkdv_full);
    mma_commit_elect(drain);
    wait_all(drain, 0);
    __syncwarp();
  } else if (warp < 8) {
    // ------------------------------------------- P and dS, one key per thread
    // Warpgroup c owns queries [64c, 64c+64) of each step, in two 32-query
    // halves; each half's bf16 pairs go to the 16 columns at 64c + 16h, inside
    // the 64 columns this warpgroup read, so neither warpgroup overwrites
    // columns the other still reads.  P is kept packed for dS = P (dP - D).
    const int r = threadIdx.x & (C::BN - 1);
    const int c = warp >> 2;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const int key = kt * C::BN + r;
    const bool key_ok = key < p.Tk;
    // keys a query sees after its first one (the whole rest without a window)
    const unsigned span = p.window > 0 ? (unsigned)p.window : 0x7fffffffu;
    const float sl2 = p.scale_log2;
    // dS^T row r of this warpgroup's 64 queries: 128 bytes in chunk c
    uint8_t *ds_row = smem + C::OFF_DS + c * C::DS_CHUNK + r * 128;
    bool ok = true;
    for (int s = 0; s < n_steps; ++s) {
      ok = __all_sync(0xffffffffu, mbar_wait(s_full, s & 1, wait_ns) && !*abort_flag);
      if (!ok) break;
      tc_fence_after();
      const int q0 = step_qt(s) * C::BM;
      const bool need_mask =
          (p.causal && (kt * C::BN + C::BN - 1 > q0 + delta)) ||
          (p.window > 0 && q0 + C::BM - 1 >= kt * C::BN - delta + p.window);
      // query q (in tile) sees the key iff lim <= q < lim + span
      const int lim = key - delta - q0;
      uint32_t pk[32];                   // P of the 64 queries, bf16 pairs
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float sv[32];
        tmem_ld32_wait(tmem + lane_base + C::TM_A + 64 * c + 32 * h, sv);
        // S^T already holds S - L/scale (the aux K-step)
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const int q = 64 * c + 32 * h + i;
          const float2 x = __fmul2_rn(make_float2(sv[i], sv[i + 1]), make_float2(sl2, sl2));
          float p0 = ex2_approx(x.x);
          float p1 = ex2_approx(x.y);
          if (need_mask) {
            if ((unsigned)(q - lim) >= span) p0 = 0.f;
            if ((unsigned)(q + 1 - lim) >= span) p1 = 0.f;
          }
          if (!key_ok) p0 = p1 = 0.f;
          pk[16 * h + i / 2] = pack_bf16x2(p0, p1);
        }
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) w[i] = pk[16 * h + i];
        tmem_st16(tmem + lane_base + C::TM_A + 64 * c + 16 * h, w);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(p_full);
      // ---- dS = P (dP - D); dP^T already holds dP - D (the aux K-step)
      ok = __all_sync(0xffffffffu, mbar_wait(dp_full, s & 1, wait_ns) && !*abort_flag);
      if (!ok) break;
      tc_fence_after();
      // the dS^T tile is free once dQ^T(s-1) has read it
      if (s >= 1) {
        ok = __all_sync(0xffffffffu, mbar_wait(ds_free, (s - 1) & 1, wait_ns));
        if (!ok) break;
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float dp[32];
        tmem_ld32_wait(tmem + lane_base + C::TM_B + 64 * c + 32 * h, dp);
        uint32_t dw[16];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float2 pp = unpack_bf16x2(pk[16 * h + i / 2]);
          const float2 d = __fmul2_rn(pp, make_float2(dp[i], dp[i + 1]));
          dw[i / 2] = pack_bf16x2(d.x, d.y);
        }
        tmem_st16(tmem + lane_base + C::TM_B + 64 * c + 16 * h, dw);
        // queries [32h, 32h+32) of this warpgroup are 16-byte units 4h .. 4h+3
        // of the 128-byte row, swizzled by the row
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int unit = 4 * h + j;
          *reinterpret_cast<uint4 *>(ds_row + ((unit ^ (r & 7)) << 4)) =
              make_uint4(dw[4 * j], dw[4 * j + 1], dw[4 * j + 2], dw[4 * j + 3]);
        }
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(ds_full);
    }
    tmem_st_wait();
    if (!ok) fail();
    if (n_steps > 0 && ok) {
      ok = __all_sync(0xffffffffu, mbar_wait(dkdv_full, 0, wait_ns));
      if (!ok) fail();
    }
    // Both warpgroups meet at a named barrier before the stores below, so
    // they take one decision: a group that gave up on a wait stops both.
    ok = named_barrier_and(1, 2 * C::BN, ok);
    if (ok) {
      // All MMAs have completed (dkdv_full), so the Q buffers are free: dV
      // (warpgroup 0) and dK times scale (warpgroup 1) go there as bf16 in the
      // 128-byte-swizzled layout of the K/V tiles (per tile two 64-column
      // chunks of 128 rows x 128 B) and leave by TMA stores, which also drop
      // rows past the sequence end.
      tc_fence_after();
      uint8_t *out = smem + C::OFF_Q;  // dV chunks, then dK chunks
      const uint32_t col = c == 0 ? C::TM_DV : C::TM_DK;
      const float mul = c == 0 ? 1.f : p.scale;
#pragma unroll 1
      for (int cg = 0; cg < D / 32; ++cg) {
        float v[32];
        if (n_steps > 0) {
          tmem_ld32_wait(tmem + lane_base + col + cg * 32, v);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0.f;
        }
        // columns [32cg, 32cg+32) are 16-byte units 4(cg%2) .. 4(cg%2)+3 of
        // row r in chunk cg/2, swizzled by the row
        uint8_t *row = out + (c * C::NCHUNK + cg / 2) * (C::BN * C::SPAN) + r * C::SPAN;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int unit = (cg & 1) * 4 + u;
          *reinterpret_cast<uint4 *>(row + ((unit ^ (r & 7)) << 4)) =
              make_uint4(pack_bf16x2(v[8 * u] * mul, v[8 * u + 1] * mul),
                         pack_bf16x2(v[8 * u + 2] * mul, v[8 * u + 3] * mul),
                         pack_bf16x2(v[8 * u + 4] * mul, v[8 * u + 5] * mul),
                         pack_bf16x2(v[8 * u + 6] * mul, v[8 * u + 7] * mul));
        }
      }
      fence_proxy_async_smem();
      named_barrier_sync(1, 2 * C::BN);
      if (threadIdx.x == 0) {
        for (int cc = 0; cc < C::NCHUNK; ++cc) {
          tma_store_3d(&tm_dv, out + cc * (C::BN * C::SPAN), cc * C::CHUNK, kt * C::BN, bkv);
          tma_store_3d(&tm_dk, out + (C::NCHUNK + cc) * (C::BN * C::SPAN), cc * C::CHUNK,
                       kt * C::BN, bkv);
        }
        bulk_commit_group();
        bulk_wait_group0();
      }
    }
  } else {
    // --------------------------- dQ^T of each step, one head-dim column per thread
    // Warp w drains head-dim columns 32(w%4) .. +31 (its TMEM lanes) for the
    // queries [64h, 64h+64) of the step and adds each into the fp32
    // accumulator: one coalesced 128-byte reduction per warp instruction.
    const int cdim = (warp & 3) * 32 + lane;  // head-dim column == TMEM lane
    const int h = (warp - 8) >> 2;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    bool ok = true;
    // at d = 64 only the warps of TMEM lanes 0..63 have head-dim columns
    const int my_steps = cdim < D ? n_steps : 0;
    for (int s = 0; s < my_steps; ++s) {
      ok = __all_sync(0xffffffffu, mbar_wait(dq_full, s & 1, wait_ns) && !*abort_flag);
      if (!ok) break;
      tc_fence_after();
      float v[64];
      tmem_ld64_wait(tmem + lane_base + C::TM_B + 64 * h, v);
      tc_fence_before();
      mbar_arrive(dq_empty);  // this part of dQ^T(s) has left tensor memory
      const int bh = b * p.Hq + step_head(s);
      const int q0 = step_qt(s) * C::BM + 64 * h;
      const int nq = min(64, p.Tq - q0);
      float *dst = p.dq_acc + ((size_t)bh * p.Tq + q0) * D + cdim;
      if (nq == 64) {
#pragma unroll
        for (int q = 0; q < 64; ++q) atomicAdd(dst + (size_t)q * D, v[q]);
      } else {
#pragma unroll
        for (int q = 0; q < 64; ++q)
          if (q < nq) atomicAdd(dst + (size_t)q * D, v[q]);
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
}

// Per query row D_i = dO_i . O_i and the aux row [-L_i/scale, -D_i] (each as
// a bf16 high and low part) that the backward kernels fold into S^T and dP^T;
// padding rows (to a multiple of 128) get -1e30 and 0, so their
// probabilities vanish.  Also zeroes the fp32 dQ accumulator.  One warp per
// row.
template <int D>
__global__ void __launch_bounds__(256)
    attn_bwd_prep_kernel(const __nv_bfloat16 *__restrict__ o,
                         const __nv_bfloat16 *__restrict__ dout,
                         const float *__restrict__ lse, float *__restrict__ dq_acc,
                         uint8_t *__restrict__ aux, float inv_scale, int rows_bh, int Tq,
                         int Tq_pad) {
  constexpr int VEC = D / 32;
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= rows_bh * Tq_pad) return;
  const int bh = warp / Tq_pad;
  const int i = warp - bh * Tq_pad;
  // aux row i of its 64-row block: core matrix (r / 8, k-half 0) holds
  // [-L/scale hi, lo, -D hi, lo, 0 x 4]; k-half 1 is zero
  auto write_aux = [&](float a, float dd) {
    const int r = i & 63;
    uint8_t *blk = aux + ((size_t)bh * (Tq_pad / 64) + i / 64) * 2048 + (r >> 3) * 256 + (r & 7) * 16;
    const __nv_bfloat16 ah = __float2bfloat16_rn(a);
    const __nv_bfloat16 al = __float2bfloat16_rn(a - __bfloat162float(ah));
    const __nv_bfloat16 dh = __float2bfloat16_rn(dd);
    const __nv_bfloat16 dl = __float2bfloat16_rn(dd - __bfloat162float(dh));
    const uint32_t w0 = (uint32_t)__bfloat16_as_ushort(ah) | ((uint32_t)__bfloat16_as_ushort(al) << 16);
    const uint32_t w1 = (uint32_t)__bfloat16_as_ushort(dh) | ((uint32_t)__bfloat16_as_ushort(dl) << 16);
    *reinterpret_cast<uint4 *>(blk) = make_uint4(w0, w1, 0u, 0u);
    *reinterpret_cast<uint4 *>(blk + 128) = make_uint4(0u, 0u, 0u, 0u);
  };
  if (i >= Tq) {
    if (lane == 0) write_aux(-1e30f, 0.f);  // a probability of exactly 0, finite products
    return;
  }
  const size_t row = (size_t)bh * Tq + i;
  const __nv_bfloat16 *orow = o + row * D + lane * VEC;
  const __nv_bfloat16 *drow = dout + row * D + lane * VEC;
  float acc = 0.f;
#pragma unroll
  for (int e = 0; e < VEC; ++e)
    acc = fmaf(__bfloat162float(orow[e]), __bfloat162float(drow[e]), acc);
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  float *qrow = dq_acc + row * D + lane * VEC;
#pragma unroll
  for (int e = 0; e < VEC; ++e) qrow[e] = 0.f;
  if (lane == 0) write_aux(-lse[row] * inv_scale, -acc);
}

// dQ = scale * accumulator, rounded to bf16.
__global__ void __launch_bounds__(256)
    attn_bwd_dq_kernel(const float4 *__restrict__ acc, uint2 *__restrict__ dq, size_t n4,
                       float scale) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4;
       i += (size_t)gridDim.x * blockDim.x) {
    const float4 a = acc[i];
    dq[i] = make_uint2(pack_bf16x2(a.x * scale, a.y * scale), pack_bf16x2(a.z * scale, a.w * scale));
  }
}

}  // namespace attn_dev
