// prefill_kernel.cuh -- exact attention forward on sm_103a tensor cores.
//
// One CTA owns two tiles of 128 query rows (256 consecutive rows) of one
// (batch, head) and streams the K/V tiles of its K/V head past them: the
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
// GB300 mapping (warp-specialised, 320 threads, one CTA per SM):
//   warps 0-3, 4-7  two softmax warpgroups, one per query tile t.  Thread r
//              of group t owns row r of tile t = TMEM lane r.  It reads its
//              row of S_t from tensor memory, masks, updates (m, l), writes P
//              as bf16 back into the first 64 columns of S_t's tensor memory,
//              rescales its row of the O_t accumulator when needed, and at the
//              end writes O_t (through shared memory and a TMA store) and LSE.
//   warp 8     TMA producer: both Q tiles once, then K and V tiles into a
//              ring of STAGES shared-memory slots (swizzled boxes).
//   warp 9     MMA issuer (one thread), tcgen05.mma kind::f16, bf16 operands,
//              fp32 accumulation in tensor memory:
//                S_t = Q_t K_j^T    A and B from shared memory,
//                O_t += P_t V_j     A = P_t from tensor memory, B = V_j.
//              The two tiles ping-pong: while group 0 turns S_0 into P_0 the
//              tensor core runs PV_1 and S_1 of the next K tile, and the
//              other way round, so exponentials and MMAs overlap.
//
// Tensor memory (512 columns): S_0 [0,128), S_1 [128,256), O_0 [256,256+D),
// O_1 [256+D, 256+2D).  P_t aliases S_t: the MMAs of one thread execute in
// issue order, so S_t(j+1) (issued after PV_t(j)) overwrites P_t(j) only
// after PV_t(j) has read it, and the commit that signals S_t(j+1) also
// covers PV_t(j), so a softmax group that sees S_t(j+1) may rescale O_t.
//
// Exponentials run in base 2 on scores pre-multiplied by scale*log2(e); m is
// kept in those units and LSE is converted back to natural log.  The
// accumulator is rescaled lazily: the reference max a row uses moves only
// when the tile max exceeds it by more than kRescaleLog2, since any
// reference value gives the same final ratio acc / l ("any m gives the same
// final ratio", section 2.1) while e^(s - m) stays in range (<= 2^8 here).
//
// Causal masking is bottom-right aligned (query i sees keys j <= i + Tk - Tq);
// K/V tiles wholly above the diagonal are never loaded, and only tiles that
// cross the diagonal or the ragged end of K are masked element by element.
//
// Every barrier wait is bounded in time; on expiry the kernel records
// ATTN_ERR_DEVICE_TIMEOUT, stops issuing work, drains its own copies and
// MMAs, frees tensor memory and returns.
#pragma once

#include <cuda_bf16.h>

#include "ptx.cuh"

namespace attn_dev {

constexpr unsigned int kStatusTimeout = 6;  // ATTN_ERR_DEVICE_TIMEOUT
constexpr float kRescaleLog2 = 8.0f;
constexpr float kLn2 = 0.6931471805599453f;

struct PrefillParams {
  float *lse;              // [B, Hq, Tq]
  unsigned int *status;   // device status word
  int Hq, Hkv, group;     // group = Hq / Hkv
  int Tq, Tk;
  int n_qt;               // ceil(Tq / 256): query-tile pairs per head
  int causal;
  float scale_log2;       // scale * log2(e)
  unsigned long long wait_ns;
  int inject;             // test hook: 1 = withhold the first V tile
};

template <int D>
struct PrefillCfg {
  static constexpr int BM = 128;                      // query rows per tile
  static constexpr int NQ = 2;                        // query tiles per CTA
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
  static constexpr uint32_t OFF_BAR = OFF_V + STAGES * KV_BYTES;
  // q_full, drain, s_full[2], p_full[2], o_done[2], then per stage
  // k_full, v_full, k_empty, v_empty
  static constexpr int NBAR = 8 + 4 * STAGES;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t SMEM_USED = OFF_MISC + 16 + 1024;  // + align slack
  // At least ~116 KB so that only one CTA (which holds all 512 TMEM
  // columns) is resident per SM.
  static constexpr uint32_t SMEM_BYTES = SMEM_USED > 118784u ? SMEM_USED : 118784u;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr int THREADS = 320;
  static constexpr int PRODUCER_WARP = 8;
  static constexpr int MMA_WARP = 9;
  __host__ __device__ static constexpr uint32_t tm_s(int t) { return t * 128; }
  __host__ __device__ static constexpr uint32_t tm_o(int t) { return 256 + t * D; }
  static_assert(D % CHUNK == 0, "head dim must be a whole number of boxes");
  static_assert(Q_BYTES % 1024 == 0 && KV_BYTES % 1024 == 0, "1 KiB regions");
  static_assert(256 + 2 * D <= 512, "tensor memory budget");
};

template <int D>
__global__ void __launch_bounds__(320, 1)
    prefill_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_o,
                       const PrefillParams p) {
  using C = PrefillCfg<D>;
  constexpr int ST = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
  uint64_t *q_full = bars + 0, *drain = bars + 1;
  uint64_t *s_full = bars + 2, *p_full = bars + 4, *o_done = bars + 6;
  uint64_t *k_full = bars + 8, *v_full = k_full + ST;
  uint64_t *k_empty = v_full + ST, *v_empty = k_empty + ST;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t wait_ns = p.wait_ns;

  // Work item: the heaviest query-tile pairs of a head first, heads in
  // order, so the CTAs resident at one time share a few heads' K/V in L2.
  const int bh = blockIdx.x / p.n_qt;
  const int qt = p.n_qt - 1 - (int)(blockIdx.x % p.n_qt);
  const int q0 = qt * (C::NQ * C::BM);
  const int b = bh / p.Hq;
  const int h = bh - b * p.Hq;
  const int bh_kv = b * p.Hkv + h / p.group;
  const int delta = p.Tk - p.Tq;
  const int n_kv_all = (p.Tk + C::BN - 1) / C::BN;
  int n_t[C::NQ];
#pragma unroll
  for (int t = 0; t < C::NQ; ++t) {
    const int row0 = q0 + t * C::BM;
    if (row0 >= p.Tq) {
      n_t[t] = 0;
    } else {
      const int last_row = min(row0 + C::BM - 1, p.Tq - 1);
      n_t[t] = p.causal ? min(n_kv_all, (last_row + delta) / C::BN + 1) : n_kv_all;
    }
  }
  const int n_max = max(n_t[0], n_t[1]);

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(drain, 1);
    for (int t = 0; t < C::NQ; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], C::BM);
      mbar_init(&o_done[t], 1);
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
    prefetch_tmap(&tm_o);
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

  if (warp == C::PRODUCER_WARP) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      bool ok = true;
      int last_k[ST], last_v[ST];
      for (int s = 0; s < ST; ++s) last_k[s] = last_v[s] = -1;
      mbar_arrive_expect_tx(q_full, C::NQ * C::Q_BYTES);
      for (int t = 0; t < C::NQ; ++t)
        for (int c = 0; c < C::NCHUNK; ++c)
          tma_load_3d(smem + C::OFF_Q + t * C::Q_BYTES + c * (C::BM * C::SPAN), &tm_q,
                      q_full, c * C::CHUNK, q0 + t * C::BM, bh);
      for (int j = 0; j < n_max; ++j) {
        const int s = j % ST, u = j / ST;
        if (*abort_flag) { ok = false; break; }
        if (j >= ST && !mbar_wait(&k_empty[s], (u - 1) & 1, wait_ns)) { ok = false; break; }
        mbar_arrive_expect_tx(&k_full[s], C::KV_BYTES);
        for (int c = 0; c < C::NCHUNK; ++c)
          tma_load_3d(smem + C::OFF_K + s * C::KV_BYTES + c * (C::BN * C::SPAN),
                      &tm_k, &k_full[s], c * C::CHUNK, j * C::BN, bh_kv);
        last_k[s] = j;
        if (j >= ST && !mbar_wait(&v_empty[s], (u - 1) & 1, wait_ns)) { ok = false; break; }
        if (!(p.inject == 1 && j == 0)) {
          mbar_arrive_expect_tx(&v_full[s], C::KV_BYTES);
          for (int c = 0; c < C::NCHUNK; ++c)
            tma_load_3d(smem + C::OFF_V + s * C::KV_BYTES + c * (C::BN * C::SPAN),
                        &tm_v, &v_full[s], c * C::CHUNK, j * C::BN, bh_kv);
          last_v[s] = j;
        }
      }
      if (!ok) fail();
      // Drain: every copy this thread issued has landed before the CTA's
      // shared memory can be released.
      mbar_wait(q_full, 0, wait_ns);
      for (int s = 0; s < ST; ++s) {
        if (last_k[s] >= 0) mbar_wait(&k_full[s], (last_k[s] / ST) & 1, wait_ns);
        if (last_v[s] >= 0) mbar_wait(&v_full[s], (last_v[s] / ST) & 1, wait_ns);
      }
    }
    __syncwarp();
  } else if (warp == C::MMA_WARP) {
    // ------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC_QK = make_idesc_bf16(C::BM, C::BN, false);
      constexpr uint32_t IDESC_PV = make_idesc_bf16(C::BM, D, true);
      auto issue_s = [&](int t, int s) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const int c = (kk * 16) / C::CHUNK;
          const int inner = ((kk * 16) % C::CHUNK) * 2;
          const uint64_t ad = make_smem_desc(
              sbase + C::OFF_Q + t * C::Q_BYTES + c * (C::BM * C::SPAN) + inner, 16,
              8 * C::SPAN, C::LAYOUT);
          const uint64_t bd = make_smem_desc(
              sbase + C::OFF_K + s * C::KV_BYTES + c * (C::BN * C::SPAN) + inner, 16,
              8 * C::SPAN, C::LAYOUT);
          mma_bf16_ss(tmem + C::tm_s(t), ad, bd, IDESC_QK, kk > 0 ? 1u : 0u);
        }
      };
      auto issue_pv = [&](int t, int s, bool acc) {
#pragma unroll
        for (int kk = 0; kk < C::BN / 16; ++kk) {
          // A = P_t in tensor memory: 16 keys = 8 columns of bf16 pairs.
          // B = V tile, MN-major (d contiguous): 16 keys = 16 rows per step,
          // LBO = next group of CHUNK head-dim columns, SBO = next 8 keys.
          const uint64_t bd = make_smem_desc(
              sbase + C::OFF_V + s * C::KV_BYTES + kk * 16 * C::SPAN, C::BN * C::SPAN,
              8 * C::SPAN, C::LAYOUT);
          mma_bf16_ts(tmem + C::tm_o(t), tmem + C::tm_s(t) + kk * 8, bd, IDESC_PV,
                      (acc || kk > 0) ? 1u : 0u);
        }
      };
      bool ok = mbar_wait(q_full, 0, wait_ns) && mbar_wait(&k_full[0], 0, wait_ns);
      if (ok && n_max > 0) {
        tc_fence_after();
        for (int t = 0; t < C::NQ; ++t) {
          if (n_t[t] > 0) {
            issue_s(t, 0);
            mma_commit(&s_full[t]);
          }
        }
        mma_commit(&k_empty[0]);
      }
      for (int j = 0; ok && j < n_max; ++j) {
        const int s = j % ST, u = j / ST;
        const int s1 = (j + 1) % ST, u1 = (j + 1) / ST;
        if (*abort_flag) { ok = false; break; }
        bool v_ready = false, k_ready = false;
        for (int t = 0; t < C::NQ && ok; ++t) {
          if (j >= n_t[t]) continue;
          if (!mbar_wait(&p_full[t], j & 1, wait_ns)) { ok = false; break; }
          if (!v_ready) {
            if (!mbar_wait(&v_full[s], u & 1, wait_ns)) { ok = false; break; }
            v_ready = true;
          }
          tc_fence_after();
          issue_pv(t, s, j > 0);
          if (j + 1 < n_t[t]) {
            if (!k_ready) {
              if (!mbar_wait(&k_full[s1], u1 & 1, wait_ns)) { ok = false; break; }
              k_ready = true;
              tc_fence_after();
            }
            issue_s(t, s1);
            mma_commit(&s_full[t]);
          } else {
            mma_commit(&o_done[t]);
          }
        }
        if (!ok) break;
        mma_commit(&v_empty[s]);
        if (k_ready) mma_commit(&k_empty[s1]);
      }
      if (!ok) fail();
      // Drain: all MMAs issued by this thread have completed before tensor
      // memory is freed.
      mma_commit(drain);
      mbar_wait(drain, 0, wait_ns);
    }
    __syncwarp();
  } else {
    // ------------------------------------------- softmax + epilogue rows
    const int t = warp >> 2;                      // query tile of this group
    const int r = threadIdx.x & 127;              // row in tile == TMEM lane
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t t_s = tmem + lane_base + C::tm_s(t);
    const uint32_t t_o = tmem + lane_base + C::tm_o(t);
    const int row0 = q0 + t * C::BM;
    const int row_g = row0 + r;
    const int lim = p.causal ? row_g + delta : 0x7fffffff;
    const float sl2 = p.scale_log2;
    const int n = n_t[t];
    float m_used = -INFINITY;  // reference max, log2 units
    float l_sum = 0.f;
    bool ok = true;

    for (int j = 0; j < n; ++j) {
      ok = __all_sync(0xffffffffu, mbar_wait(&s_full[t], j & 1, wait_ns) && !*abort_flag);
      if (!ok) break;
      tc_fence_after();
      float s[C::BN];
      tmem_ld128_wait(t_s, s);

      const int kbase = j * C::BN;
      const bool need_mask =
          (kbase + C::BN > p.Tk) || (p.causal && kbase + C::BN - 1 > row0 + delta);
      if (need_mask) {
#pragma unroll
        for (int c = 0; c < C::BN; ++c) {
          const int key = kbase + c;
          if (key > lim || key >= p.Tk) s[c] = -INFINITY;
        }
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
      const float m_ref = (m_used == -INFINITY) ? 0.f : m_used;
      const float2 c2 = make_float2(sl2, sl2);
      const float2 b2 = make_float2(-m_ref, -m_ref);
      float2 acc2[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) acc2[i] = make_float2(0.f, 0.f);
      uint32_t pw[C::BN / 2];
#pragma unroll
      for (int c = 0; c < C::BN / 2; ++c) {
        const float2 x = __ffma2_rn(make_float2(s[2 * c], s[2 * c + 1]), c2, b2);
        const float2 e = make_float2(ex2_approx(x.x), ex2_approx(x.y));
        acc2[c & 3] = __fadd2_rn(acc2[c & 3], e);
        pw[c] = pack_bf16x2(e.x, e.y);
      }
      const float2 a01 = __fadd2_rn(acc2[0], acc2[1]);
      const float2 a23 = __fadd2_rn(acc2[2], acc2[3]);
      const float2 a = __fadd2_rn(a01, a23);
      l_sum = fmaf(l_sum, alpha, a.x + a.y);

      // O_t is stable here (PV_t(j-1) completed before S_t(j) was signalled).
      if (j > 0 && __any_sync(0xffffffffu, resc)) {
        const float2 al2 = make_float2(alpha, alpha);
#pragma unroll
        for (int cb = 0; cb < D / 32; ++cb) {
          float o[32];
          tmem_ld32_wait(t_o + cb * 32, o);
          uint32_t ow[32];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float2 y = __fmul2_rn(make_float2(o[2 * i], o[2 * i + 1]), al2);
            ow[2 * i] = __float_as_uint(y.x);
            ow[2 * i + 1] = __float_as_uint(y.y);
          }
          tmem_st32(t_o + cb * 32, ow);
        }
      }
      // P_t (bf16 pairs) into the first 64 columns of S_t.
      {
        uint32_t w0[32], w1[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          w0[i] = pw[i];
          w1[i] = pw[32 + i];
        }
        tmem_st32(t_s, w0);
        tmem_st32(t_s + 32, w1);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&p_full[t]);
    }

    // ------------------------------------------------------------ epilogue
    uint8_t *stage = smem + C::OFF_Q + t * C::Q_BYTES;  // Q_t is no longer read
    if (n > 0) {
      if (ok)
        ok = __all_sync(0xffffffffu, mbar_wait(&o_done[t], 0, wait_ns));
      if (ok) {
        tc_fence_after();
        const float inv_l = (l_sum > 0.f) ? 1.f / l_sum : 0.f;
#pragma unroll
        for (int cb = 0; cb < D / 32; ++cb) {
          float o[32];
          tmem_ld32_wait(t_o + cb * 32, o);
#pragma unroll
          for (int u4 = 0; u4 < 4; ++u4) {
            uint4 w;
            w.x = pack_bf16x2(o[u4 * 8 + 0] * inv_l, o[u4 * 8 + 1] * inv_l);
            w.y = pack_bf16x2(o[u4 * 8 + 2] * inv_l, o[u4 * 8 + 3] * inv_l);
            w.z = pack_bf16x2(o[u4 * 8 + 4] * inv_l, o[u4 * 8 + 5] * inv_l);
            w.w = pack_bf16x2(o[u4 * 8 + 6] * inv_l, o[u4 * 8 + 7] * inv_l);
            const int col = cb * 32 + u4 * 8;
            const int c = col / C::CHUNK;
            const uint32_t off = c * (C::BM * C::SPAN) +
                                 swizzle_off(r * C::SPAN + (col % C::CHUNK) * 2, C::SPAN);
            *reinterpret_cast<uint4 *>(stage + off) = w;
          }
        }
        if (row_g < p.Tq) {
          float lse;
          if (l_sum > 0.f)
            lse = (m_used + log2f(l_sum)) * kLn2;
          else
            lse = (m_used == -INFINITY) ? 0.f : m_used * kLn2;
          p.lse[(size_t)bh * p.Tq + row_g] = lse;
        }
      } else {
        fail();
      }
      fence_proxy_async_smem();
      named_barrier_sync(1 + t, C::BM);
      if (r == 0 && !*abort_flag) {
        for (int c = 0; c < C::NCHUNK; ++c)
          tma_store_3d(&tm_o, stage + c * (C::BM * C::SPAN), c * C::CHUNK, row0, bh);
        bulk_commit_group();
        bulk_wait_group_read0();
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace attn_dev
