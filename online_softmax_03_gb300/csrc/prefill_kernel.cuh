// prefill_kernel.cuh -- exact attention forward on sm_103a tensor cores.
//
// One CTA owns one tile of 128 query rows of one (batch, head) and streams
// the K/V tiles of its K/V head past it (the outer-Q / inner-KV loop order of
// "4.2 FlashAttention I: IO-Awareness & The Online Softmax", section
// "FlashAttention forward: tiling + online softmax fused into one pass", and
// of "Efficient attention & KV cache", section 3).  Per query row the
// running max m, running sum l and the unnormalised accumulator acc are kept
// in fp32 and updated with the recurrence of "Efficient attention & KV
// cache", section 2.1:
//
//   m' = max(m, rowmax S_j),  l' = e^(m-m') l + rowsum e^(S_j-m'),
//   acc' = e^(m-m') acc + e^(S_j-m') V_j,  O = acc / l,  LSE = m + ln l.
//
// GB300 mapping (warp-specialised, 192 threads):
//   warps 0-3  softmax: thread r owns query row r = TMEM lane r.  It reads
//              its row of S from tensor memory, masks, updates (m, l),
//              writes P as bf16 into shared memory, rescales its row of the
//              O accumulator in tensor memory when needed, and finally
//              writes O (via a TMA store) and LSE.
//   warp 4     TMA producer: Q once, then K and V tiles into a ring of
//              STAGES shared-memory slots (128-byte swizzled boxes).
//   warp 5     MMA issuer (one thread): S = Q K^T into TMEM columns [0,128),
//              O (+)= P V into TMEM columns [128, 128+D), tcgen05.mma
//              kind::f16 with bf16 operands and fp32 accumulation.
//
// The exponentials run in base 2 on scores pre-multiplied by scale*log2(e);
// m is kept in the same units and LSE is converted back to natural log.
// The accumulator is rescaled lazily: the reference max a row uses moves only
// when the tile max exceeds it by more than kRescaleLog2, since any reference
// value gives the same final ratio acc / l ("any m gives the same final
// ratio", section 2.1) as long as e^(s - m) stays in range (<= 2^8 here).
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
  int n_qt;               // ceil(Tq / 128)
  int causal;
  float scale_log2;       // scale * log2(e)
  unsigned long long wait_ns;
  int inject;             // test hook: 1 = withhold the first V tile
};

template <int D>
struct PrefillCfg {
  static constexpr int BM = 128;                      // query rows per CTA
  static constexpr int BN = 128;                      // keys per K/V tile
  static constexpr int SPAN = (D >= 64) ? 128 : 64;   // swizzle span, bytes
  static constexpr int CHUNK = SPAN / 2;              // bf16 columns per box
  static constexpr int NCHUNK = D / CHUNK;
  static constexpr uint32_t LAYOUT = (SPAN == 128) ? kLayoutSW128 : kLayoutSW64;
  static constexpr int STAGES = (D == 128) ? 2 : 4;
  static constexpr uint32_t Q_BYTES = BM * D * 2;
  static constexpr uint32_t KV_BYTES = BN * D * 2;
  static constexpr uint32_t P_BYTES = BM * BN * 2;
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_P = OFF_Q + Q_BYTES;
  static constexpr uint32_t OFF_K = OFF_P + P_BYTES;
  static constexpr uint32_t OFF_V = OFF_K + STAGES * KV_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_V + STAGES * KV_BYTES;
  // q_full, s_full, s_free, p_full, o_done, drain, then per stage
  // k_full, v_full, k_empty, v_empty
  static constexpr int NBAR = 6 + 4 * STAGES;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 1024;  // + align slack
  static constexpr uint32_t TMEM_COLS = 256;
  static constexpr uint32_t TM_S = 0;
  static constexpr uint32_t TM_O = 128;
  static constexpr int THREADS = 192;
  static_assert(D % CHUNK == 0, "head dim must be a whole number of boxes");
  static_assert(Q_BYTES % 1024 == 0 && KV_BYTES % 1024 == 0, "1 KiB regions");
};

template <int D>
__global__ void __launch_bounds__(192, 1)
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
  uint64_t *q_full = bars + 0, *s_full = bars + 1, *s_free = bars + 2;
  uint64_t *p_full = bars + 3, *o_done = bars + 4, *drain = bars + 5;
  uint64_t *k_full = bars + 6, *v_full = k_full + ST;
  uint64_t *k_empty = v_full + ST, *v_empty = k_empty + ST;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t wait_ns = p.wait_ns;

  // Work item: heaviest query tiles of a head first, heads in order, so the
  // CTAs resident at one time share the K/V of a few heads through L2.
  const int bh = blockIdx.x / p.n_qt;
  const int qt = p.n_qt - 1 - (int)(blockIdx.x % p.n_qt);
  const int q0 = qt * C::BM;
  const int b = bh / p.Hq;
  const int h = bh - b * p.Hq;
  const int bh_kv = b * p.Hkv + h / p.group;
  const int delta = p.Tk - p.Tq;
  const int last_row = min(q0 + C::BM - 1, p.Tq - 1);
  const int n_kv_all = (p.Tk + C::BN - 1) / C::BN;
  const int n_kv = p.causal ? min(n_kv_all, (last_row + delta) / C::BN + 1) : n_kv_all;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(s_full, 1);
    mbar_init(s_free, C::BM);
    mbar_init(p_full, C::BM);
    mbar_init(o_done, 1);
    mbar_init(drain, 1);
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

  if (warp == 4) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      bool ok = true;
      int last_k[ST], last_v[ST];
      for (int s = 0; s < ST; ++s) last_k[s] = last_v[s] = -1;
      mbar_arrive_expect_tx(q_full, C::Q_BYTES);
      for (int c = 0; c < C::NCHUNK; ++c)
        tma_load_3d(smem + C::OFF_Q + c * (C::BM * C::SPAN), &tm_q, q_full,
                    c * C::CHUNK, q0, bh);
      for (int j = 0; j < n_kv; ++j) {
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
  } else if (warp == 5) {
    // ------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC_QK = make_idesc_bf16(C::BM, C::BN, false);
      constexpr uint32_t IDESC_PV = make_idesc_bf16(C::BM, D, true);
      auto issue_pv = [&](int jj) -> bool {
        const int s = jj % ST, u = jj / ST;
        if (!mbar_wait(p_full, jj & 1, wait_ns)) return false;
        if (!mbar_wait(&v_full[s], u & 1, wait_ns)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < C::BN / 16; ++kk) {
          // A = P, K-major over keys, 128-byte swizzle, 64 keys per region.
          const uint64_t ad = make_smem_desc(
              sbase + C::OFF_P + (kk / 4) * (C::BM * 128) + (kk % 4) * 32, 16,
              1024, kLayoutSW128);
          // B = V tile, MN-major (d contiguous): 16 keys = 16 rows per step,
          // LBO = next group of CHUNK head-dim columns, SBO = next 8 keys.
          const uint64_t bd = make_smem_desc(
              sbase + C::OFF_V + s * C::KV_BYTES + kk * 16 * C::SPAN,
              C::BN * C::SPAN, 8 * C::SPAN, C::LAYOUT);
          mma_bf16_ss(tmem + C::TM_O, ad, bd, IDESC_PV, (jj > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(o_done);
        mma_commit(&v_empty[s]);
        return true;
      };
      bool ok = mbar_wait(q_full, 0, wait_ns);
      for (int j = 0; ok && j < n_kv; ++j) {
        const int s = j % ST, u = j / ST;
        if (*abort_flag) { ok = false; break; }
        if (!mbar_wait(&k_full[s], u & 1, wait_ns)) { ok = false; break; }
        if (j > 0 && !mbar_wait(s_free, (j - 1) & 1, wait_ns)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const int c = (kk * 16) / C::CHUNK;
          const int inner = ((kk * 16) % C::CHUNK) * 2;
          const uint64_t ad = make_smem_desc(
              sbase + C::OFF_Q + c * (C::BM * C::SPAN) + inner, 16, 8 * C::SPAN, C::LAYOUT);
          const uint64_t bd = make_smem_desc(
              sbase + C::OFF_K + s * C::KV_BYTES + c * (C::BN * C::SPAN) + inner, 16,
              8 * C::SPAN, C::LAYOUT);
          mma_bf16_ss(tmem + C::TM_S, ad, bd, IDESC_QK, kk > 0 ? 1u : 0u);
        }
        mma_commit(s_full);
        mma_commit(&k_empty[s]);
        if (j > 0 && !issue_pv(j - 1)) { ok = false; break; }
      }
      if (ok) ok = issue_pv(n_kv - 1);
      if (!ok) fail();
      // Drain: all MMAs issued by this thread have completed before tensor
      // memory is freed.
      mma_commit(drain);
      mbar_wait(drain, 0, wait_ns);
    }
    __syncwarp();
  } else {
    // ------------------------------------------- softmax + epilogue rows
    const int r = threadIdx.x;                 // row in tile == TMEM lane
    const uint32_t t_row = tmem + ((uint32_t)(warp * 32) << 16);
    const int row_g = q0 + r;
    const int lim = p.causal ? row_g + delta : 0x7fffffff;
    const float sl2 = p.scale_log2;
    float m_used = -INFINITY;  // reference max, log2 units
    float l_sum = 0.f;
    bool ok = true;

    for (int j = 0; j < n_kv; ++j) {
      ok = __all_sync(0xffffffffu, mbar_wait(s_full, j & 1, wait_ns) && !*abort_flag);
      if (!ok) break;
      tc_fence_after();
      float s[C::BN];
#pragma unroll
      for (int cb = 0; cb < C::BN / 32; ++cb)
        tmem_ld32_wait(t_row + C::TM_S + cb * 32,
                       *reinterpret_cast<float(*)[32]>(&s[cb * 32]));
      tc_fence_before();
      mbar_arrive(s_free);

      const int kbase = j * C::BN;
      const bool need_mask =
          (kbase + C::BN > p.Tk) || (p.causal && kbase + C::BN - 1 > q0 + delta);
      if (need_mask) {
#pragma unroll
        for (int c = 0; c < C::BN; ++c) {
          const int key = kbase + c;
          if (key > lim || key >= p.Tk) s[c] = -INFINITY;
        }
      }
      float mx = s[0];
#pragma unroll
      for (int c = 1; c < C::BN; ++c) mx = fmaxf(mx, s[c]);
      const float m_tile = mx * sl2;  // scale > 0, so the max commutes
      const float m_new = fmaxf(m_used, m_tile);
      const bool resc = m_new > m_used + kRescaleLog2;
      float alpha = 1.f;
      if (resc) {
        alpha = ex2_approx(m_used - m_new);  // 0 while nothing was seen
        m_used = m_new;
      }
      const float m_ref = (m_used == -INFINITY) ? 0.f : m_used;
      float rowsum = 0.f;
#pragma unroll
      for (int c = 0; c < C::BN; ++c) {
        s[c] = ex2_approx(fmaf(s[c], sl2, -m_ref));
        rowsum += s[c];
      }
      l_sum = fmaf(l_sum, alpha, rowsum);

      if (j > 0) {
        // PV of the previous tile must be finished before O is rescaled and
        // before P is overwritten.
        ok = __all_sync(0xffffffffu, mbar_wait(o_done, (j - 1) & 1, wait_ns));
        if (!ok) break;
        tc_fence_after();
        if (__any_sync(0xffffffffu, resc)) {
#pragma unroll
          for (int cb = 0; cb < D / 32; ++cb) {
            float o[32];
            tmem_ld32_wait(t_row + C::TM_O + cb * 32, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= alpha;
            tmem_st32_wait(t_row + C::TM_O + cb * 32, o);
          }
        }
      }
      // P row -> shared memory, bf16, K-major 128-byte swizzle (two regions
      // of 64 keys), 16 bytes (8 keys) per store.
#pragma unroll
      for (int u = 0; u < C::BN / 8; ++u) {
        uint4 w;
        __nv_bfloat162 t0 = __floats2bfloat162_rn(s[u * 8 + 0], s[u * 8 + 1]);
        __nv_bfloat162 t1 = __floats2bfloat162_rn(s[u * 8 + 2], s[u * 8 + 3]);
        __nv_bfloat162 t2 = __floats2bfloat162_rn(s[u * 8 + 4], s[u * 8 + 5]);
        __nv_bfloat162 t3 = __floats2bfloat162_rn(s[u * 8 + 6], s[u * 8 + 7]);
        w.x = *reinterpret_cast<uint32_t *>(&t0);
        w.y = *reinterpret_cast<uint32_t *>(&t1);
        w.z = *reinterpret_cast<uint32_t *>(&t2);
        w.w = *reinterpret_cast<uint32_t *>(&t3);
        const uint32_t off = C::OFF_P + (u / 8) * (C::BM * 128) +
                             swizzle_off(r * 128 + (u % 8) * 16, 128);
        *reinterpret_cast<uint4 *>(smem + off) = w;
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(p_full);
    }

    // ------------------------------------------------------------ epilogue
    if (ok)
      ok = __all_sync(0xffffffffu, mbar_wait(o_done, (n_kv - 1) & 1, wait_ns));
    if (ok) {
      tc_fence_after();
      const float inv_l = (l_sum > 0.f) ? 1.f / l_sum : 0.f;
#pragma unroll
      for (int cb = 0; cb < D / 32; ++cb) {
        float o[32];
        tmem_ld32_wait(t_row + C::TM_O + cb * 32, o);
#pragma unroll
        for (int u4 = 0; u4 < 4; ++u4) {
          uint4 w;
          __nv_bfloat162 t0 = __floats2bfloat162_rn(o[u4 * 8 + 0] * inv_l, o[u4 * 8 + 1] * inv_l);
          __nv_bfloat162 t1 = __floats2bfloat162_rn(o[u4 * 8 + 2] * inv_l, o[u4 * 8 + 3] * inv_l);
          __nv_bfloat162 t2 = __floats2bfloat162_rn(o[u4 * 8 + 4] * inv_l, o[u4 * 8 + 5] * inv_l);
          __nv_bfloat162 t3 = __floats2bfloat162_rn(o[u4 * 8 + 6] * inv_l, o[u4 * 8 + 7] * inv_l);
          w.x = *reinterpret_cast<uint32_t *>(&t0);
          w.y = *reinterpret_cast<uint32_t *>(&t1);
          w.z = *reinterpret_cast<uint32_t *>(&t2);
          w.w = *reinterpret_cast<uint32_t *>(&t3);
          const int col = cb * 32 + u4 * 8;
          const int c = col / C::CHUNK;
          const uint32_t off = C::OFF_Q + c * (C::BM * C::SPAN) +
                               swizzle_off(r * C::SPAN + (col % C::CHUNK) * 2, C::SPAN);
          *reinterpret_cast<uint4 *>(smem + off) = w;
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
    named_barrier_sync(1, C::BM);
    if (threadIdx.x == 0 && !*abort_flag) {
      for (int c = 0; c < C::NCHUNK; ++c)
        tma_store_3d(&tm_o, smem + C::OFF_Q + c * (C::BM * C::SPAN), c * C::CHUNK, q0, bh);
      bulk_commit_group();
      bulk_wait_group_read0();
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
