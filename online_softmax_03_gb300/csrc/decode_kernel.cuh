// decode_kernel.cuh -- one query token per sequence against a KV cache.
//
// Decode attention reads the whole cache once per step and does about one
// multiply-add per cached element per query head, so it is bound by HBM
// bandwidth, not arithmetic ("Attention from scratch + roofline", section
// "Classify prefill vs decode"; "Efficient attention & KV cache", section
// 2.4).  The kernels therefore run on the CUDA cores and are organised
// around moving the cache once, coalesced:
//
//  * decode_split_kernel: grid (split, KV head x head chunk, batch).  One CTA
//    streams a contiguous chunk of keys of one K/V head through shared memory
//    with 1-D bulk copies (a ring of STAGES tiles of 32 keys, filled by one
//    producer thread), and serves all query heads that share that K/V head
//    (grouped-query attention), so each cache byte is read once per group.
//    Each consumer warp takes groups of KG = 32/GP keys: a lane owns D/32
//    head-dim columns and forms partial dot products for the GP x KG
//    (head, key) pairs.  Lane l keeps the partial of pair j at position
//    j XOR l (its query heads and key rows are permuted accordingly), which
//    makes the transpose-and-add network that leaves lane l with the full
//    score of pair l free of selects: 31 shuffles and 31 adds for 32 pairs.
//    The online-softmax update of "Efficient attention & KV cache", section
//    2.1 then runs per head over those lanes, and the value accumulation with
//    lanes over head-dim columns.  Products use packed fp32x2 FMAs.  The
//    warps' partial (m, l, acc) are merged in shared memory and written to
//    the workspace.
//    With kPaged the cache is a pool of pages and each sequence a list of
//    page numbers ("Efficient attention & KV cache", section 2.5): the
//    producer looks each tile's page(s) up in the block table and copies
//    the rows from there, one bulk copy per page piece; everything the
//    consumers do is unchanged.  Per-sequence lengths come from the device,
//    so a split may find no keys at all; it then writes an empty partial
//    (m = -inf, l = 0, acc = 0), which the merge weighs with 0.
//  * decode_combine_kernel: one warp per (batch, query head) merges the
//    splits with the same rescaling (m* = max m_s, weights e^(m_s - m*)),
//    writes O as bf16 and LSE in natural log.
//
// Scores are pre-scaled by scale*log2(e) so exponentials run in base 2.
#pragma once

#include <cuda_bf16.h>

#include "ptx.cuh"

namespace attn_dev {

constexpr unsigned int kDecodeStatusTimeout = 6;  // ATTN_ERR_DEVICE_TIMEOUT
constexpr unsigned int kDecodeStatusBadArg = 1;   // ATTN_ERR_INVALID_ARG

struct DecodeParams {
  const __nv_bfloat16 *q;   // [B, Hq, 1, D]
  const __nv_bfloat16 *k;   // [B, Hkv, Tk, D], paged: [num_pages, Hkv, page, D]
  const __nv_bfloat16 *v;   // same layout as k
  float *part_acc;          // [B*Hq, nsplit, D]
  float *part_ml;           // [B*Hq, nsplit, 2]  (m in log2 units, l)
  unsigned int *status;
  int Hq, Hkv, group, Tk;
  int nsplit, chunk;        // keys per split (multiple of 32)
  int n_hc;                 // head chunks of GP per K/V head
  float scale_log2;
  unsigned long long wait_ns;
  int inject;               // test hook: 2 = CTA (0, 0, 0) withholds its first tile
  // paged cache only (Tk is then the longest allowed sequence)
  const int *block_table;   // [B, max_pages]
  const int *seq_lens;      // [B]
  int page_shift;           // log2(page size)
  int max_pages, num_pages;
};

template <int D, int GP>
struct DecodeCfg {
  static constexpr int CW = 4;                  // consumer warps
  static constexpr int THREADS = (CW + 1) * 32;
  static constexpr int TILE = 32;               // keys per stage
  static constexpr int STAGES = 3;   // 48 KB of ring: four CTAs per SM
  static constexpr int KG = 32 / GP;            // keys per reduce-scatter
  static constexpr int NGRP = TILE / KG;
  static constexpr int VEC = D / 32;            // head-dim columns per lane
  static constexpr uint32_t ROW_BYTES = D * 2;
  static constexpr uint32_t TILE_BYTES = TILE * ROW_BYTES;
  static constexpr uint32_t OFF_K = 0;
  static constexpr uint32_t OFF_V = OFF_K + STAGES * TILE_BYTES;
  static constexpr uint32_t OFF_P = OFF_V + STAGES * TILE_BYTES;   // [CW][32] float2
  static constexpr uint32_t OFF_A = OFF_P + CW * 32 * 8;           // [CW][GP]
  static constexpr uint32_t OFF_BAR = OFF_A + CW * GP * 4;
  static constexpr uint32_t OFF_FAIL = OFF_BAR + 2 * STAGES * 8;   // int: a warp gave up
  static constexpr uint32_t SMEM_BYTES = OFF_BAR + 2 * STAGES * 8 + 128;
  // merge scratch, aliased on the (drained) K/V ring after the main loop
  static constexpr uint32_t OFF_MM = 0;                            // [CW][GP]
  static constexpr uint32_t OFF_LL = OFF_MM + CW * GP * 4;         // [CW][GP]
  static constexpr uint32_t OFF_AA = OFF_LL + CW * GP * 4;         // [CW][GP][D]
  static_assert(OFF_AA + CW * GP * D * 4 <= OFF_P, "merge scratch fits the ring");
  static_assert(GP * KG == 32 && NGRP % CW == 0, "one value per lane");
};

// Transpose-and-add across the warp.  On entry lane l holds at position j
// its partial for pair j XOR l; on exit v[0] is the warp-wide sum for pair l.
// At the step with offset o a lane keeps positions [0, o) and adds what its
// partner l ^ o holds at positions [o, 2o), which is the partner's partial
// for the same pairs, so no lane-dependent select is needed.
__device__ __forceinline__ float warp_reduce_scatter32_xor(float (&v)[32]) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
#pragma unroll
    for (int i = 0; i < off; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i + off], off);
  }
  return v[0];
}

template <int VEC>
__device__ __forceinline__ void load_bf16_row(const uint8_t *src, float (&f)[VEC]) {
  if constexpr (VEC == 4) {
    const uint2 w = *reinterpret_cast<const uint2 *>(src);
    f[0] = __uint_as_float(w.x << 16);
    f[1] = __uint_as_float(w.x & 0xffff0000u);
    f[2] = __uint_as_float(w.y << 16);
    f[3] = __uint_as_float(w.y & 0xffff0000u);
  } else if constexpr (VEC == 2) {
    const uint32_t w = *reinterpret_cast<const uint32_t *>(src);
    f[0] = __uint_as_float(w << 16);
    f[1] = __uint_as_float(w & 0xffff0000u);
  } else {
    const uint32_t w = *reinterpret_cast<const uint16_t *>(src);
    f[0] = __uint_as_float(w << 16);
  }
}

template <int D, int GP, bool kPaged>
__global__ void __launch_bounds__(DecodeCfg<D, GP>::THREADS)
    decode_split_kernel(const DecodeParams p) {
  using C = DecodeCfg<D, GP>;
  constexpr int ST = C::STAGES;
  constexpr int KG = C::KG;
  constexpr int VEC = C::VEC;
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
  uint64_t *empty = full + ST;
  float *pbuf = reinterpret_cast<float *>(smem + C::OFF_P);
  float *abuf = reinterpret_cast<float *>(smem + C::OFF_A);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int sidx = blockIdx.x;
  const int hk = blockIdx.y / p.n_hc;
  const int hc = blockIdx.y - hk * p.n_hc;
  const int b = blockIdx.z;
  const int h0 = hk * p.group + hc * GP;          // first query head served
  const int nh = min(GP, p.group - hc * GP);      // query heads served
  int seq_len = p.Tk;
  if constexpr (kPaged) {
    seq_len = p.seq_lens[b];
    if (seq_len < 1 || seq_len > p.Tk) {  // never used to address memory
      if (threadIdx.x == 0) atomicMax(p.status, kDecodeStatusBadArg);
      seq_len = 0;
    }
  }
  const int k0 = sidx * p.chunk;
  // contiguous: >= 1 (host guarantees); paged: 0 for splits past the end
  const int len = max(0, min(seq_len, k0 + p.chunk) - k0);
  const int ntiles = (len + C::TILE - 1) / C::TILE;
  const size_t kv_off = kPaged ? 0 : ((size_t)(b * p.Hkv + hk) * p.Tk + k0) * D;
  const uint8_t *kg = reinterpret_cast<const uint8_t *>(p.k + kv_off);
  const uint8_t *vg = reinterpret_cast<const uint8_t *>(p.v + kv_off);

  volatile int *failed = reinterpret_cast<volatile int *>(smem + C::OFF_FAIL);
  if (threadIdx.x == 0) {
    for (int s = 0; s < ST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], C::CW);
    }
    *failed = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == C::CW) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int last[ST];
      for (int s = 0; s < ST; ++s) last[s] = -1;
      for (int t = 0; t < ntiles; ++t) {
        const int s = t % ST, u = t / ST;
        if (t >= ST && !mbar_wait(&empty[s], (u - 1) & 1, p.wait_ns)) {
          atomicMax(p.status, kDecodeStatusTimeout);
          break;
        }
        const int rows = min(C::TILE, len - t * C::TILE);
        const uint32_t bytes = rows * C::ROW_BYTES;
        mbar_arrive_expect_tx(&full[s], 2 * bytes);
        uint8_t *dk = smem + C::OFF_K + s * C::TILE_BYTES;
        uint8_t *dv = smem + C::OFF_V + s * C::TILE_BYTES;
        // test hook: the first tile of CTA (0, 0, 0) is never loaded, so the
        // consumers' wait for it must expire
        const bool withhold =
            p.inject == 2 && t == 0 && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0;
        if (withhold) {
        } else if constexpr (kPaged) {
          // The tile's keys k0 + t*TILE + [0, rows) may span several pages:
          // one copy per piece that lies within one page.
          const int page = 1 << p.page_shift;
          const int *table = p.block_table + (size_t)b * p.max_pages;
          for (int r = 0; r < rows;) {
            const int key = k0 + t * C::TILE + r;
            const int off = key & (page - 1);
            const int n = min(rows - r, page - off);
            int phys = __ldg(table + (key >> p.page_shift));
            if ((unsigned)phys >= (unsigned)p.num_pages) {  // read page 0 instead
              atomicMax(p.status, kDecodeStatusBadArg);
              phys = 0;
            }
            const size_t src =
                ((((size_t)phys * p.Hkv + hk) << p.page_shift) + off) * C::ROW_BYTES;
            bulk_load(dk + r * C::ROW_BYTES, kg + src, n * C::ROW_BYTES, &full[s]);
            bulk_load(dv + r * C::ROW_BYTES, vg + src, n * C::ROW_BYTES, &full[s]);
            r += n;
          }
        } else {
          bulk_load(dk, kg + (size_t)t * C::TILE_BYTES, bytes, &full[s]);
          bulk_load(dv, vg + (size_t)t * C::TILE_BYTES, bytes, &full[s]);
        }
        last[s] = t;
      }
      for (int s = 0; s < ST; ++s)
        if (last[s] >= 0) mbar_wait(&full[s], (last[s] / ST) & 1, p.wait_ns);
    }
    __syncwarp();
    return;  // the producer warp takes no part in the merge below
  }

  // -------------------------------------------------------------- consumers
  // Lane l's view of the 32 (head, key) pairs is permuted by XOR with l (see
  // warp_reduce_scatter32_xor): position j holds head (j / KG) ^ hsel and key
  // (j % KG) ^ ksel.  The query vectors are loaded in that permuted head
  // order, pre-scaled by scale * log2(e) and duplicated into fp32x2 pairs.
  static_assert(VEC % 2 == 0 || VEC == 1, "head-dim columns per lane");
  constexpr int VP = (VEC + 1) / 2;  // fp32x2 pairs of head-dim columns
  const int hsel = lane / KG;
  const int ksel = lane % KG;
  float2 qd[GP][VEC];
#pragma unroll
  for (int hp = 0; hp < GP; ++hp) {
    const int hh = hp ^ hsel;
    if (hh < nh) {
      const uint8_t *qrow = reinterpret_cast<const uint8_t *>(
          p.q + ((size_t)b * p.Hq + h0 + hh) * D);
      float f[VEC];
      load_bf16_row<VEC>(qrow + lane * VEC * 2, f);
#pragma unroll
      for (int e = 0; e < VEC; ++e) qd[hp][e] = make_float2(f[e] * p.scale_log2, f[e] * p.scale_log2);
    } else {
#pragma unroll
      for (int e = 0; e < VEC; ++e) qd[hp][e] = make_float2(0.f, 0.f);
    }
  }
  // Byte offsets of the lane's permuted K rows inside a key group.
  uint32_t koff[KG];
#pragma unroll
  for (int jj = 0; jj < KG; ++jj) koff[jj] = (uint32_t)((jj ^ ksel) * C::ROW_BYTES + lane * VEC * 2);
  // acc2[h][.] for the natural head order, lanes over head-dim columns.
  float2 acc2[GP][VP];
#pragma unroll
  for (int hh = 0; hh < GP; ++hh)
#pragma unroll
    for (int e = 0; e < VP; ++e) acc2[hh][e] = make_float2(0.f, 0.f);
  float m = -INFINITY;  // reference max for head lane / KG (log2 units)
  float l = 0.f;
  bool ok = true;
  float2 *pw = reinterpret_cast<float2 *>(pbuf) + warp * 32;
  float *aw = abuf + warp * GP;
  constexpr float kRescale = 8.0f;  // lazy rescale threshold, log2 units

  for (int t = 0; t < ntiles; ++t) {
    const int s = t % ST, u = t / ST;
    ok = __all_sync(0xffffffffu, mbar_wait(&full[s], u & 1, p.wait_ns));
    if (!ok) break;
    const int rows_valid = min(C::TILE, len - t * C::TILE);
    const uint8_t *ks = smem + C::OFF_K + s * C::TILE_BYTES;
    const uint8_t *vs = smem + C::OFF_V + s * C::TILE_BYTES;
#pragma unroll
    for (int gi = warp; gi < C::NGRP; gi += C::CW) {
      const int key0 = gi * KG;
      const uint8_t *kg0 = ks + key0 * C::ROW_BYTES;
      // ---- scores: fp32x2 over key pairs, then the select-free transpose-add
      float2 part2[GP * KG / 2];
#pragma unroll
      for (int jj = 0; jj < KG; jj += 2) {
        float ka[VEC], kb[VEC];
        load_bf16_row<VEC>(kg0 + koff[jj], ka);
        load_bf16_row<VEC>(kg0 + koff[jj + 1], kb);
#pragma unroll
        for (int hp = 0; hp < GP; ++hp) {
          float2 a = __fmul2_rn(qd[hp][0], make_float2(ka[0], kb[0]));
#pragma unroll
          for (int e = 1; e < VEC; ++e) a = __ffma2_rn(qd[hp][e], make_float2(ka[e], kb[e]), a);
          part2[(hp * KG + jj) / 2] = a;
        }
      }
#pragma unroll
      for (int off = 8; off >= 1; off >>= 1) {
#pragma unroll
        for (int i = 0; i < off; ++i) {
          const float2 r = make_float2(__shfl_xor_sync(0xffffffffu, part2[i + off].x, 2 * off),
                                       __shfl_xor_sync(0xffffffffu, part2[i + off].y, 2 * off));
          part2[i] = __fadd2_rn(part2[i], r);
        }
      }
      float sc = part2[0].x + __shfl_xor_sync(0xffffffffu, part2[0].y, 1);
      const bool full_group = key0 + KG <= rows_valid;
      if (!full_group && key0 + ksel >= rows_valid) sc = -INFINITY;
      // ---- online update per head over its KG lanes
      float mx = sc;
#pragma unroll
      for (int off = 1; off < KG; off <<= 1)
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const bool resc = mx > m + kRescale;  // true on the first group (m = -inf)
      if (__any_sync(0xffffffffu, resc)) {
        // move the reference max only where it grew; scale acc and l by alpha
        const float m_new = resc ? mx : m;
        const float alpha = (m == -INFINITY) ? 0.f : ex2_approx(m - m_new);
        l *= alpha;
        m = m_new;
        if (ksel == 0) aw[hsel] = alpha;
        __syncwarp();
#pragma unroll
        for (int hh = 0; hh < GP; ++hh) {
          const float a = aw[hh];
#pragma unroll
          for (int e = 0; e < VP; ++e) acc2[hh][e] = __fmul2_rn(acc2[hh][e], make_float2(a, a));
        }
      }
      const float m_ref = (m == -INFINITY) ? 0.f : m;
      const float pv = ex2_approx(sc - m_ref);
      float ps = pv;
#pragma unroll
      for (int off = 1; off < KG; off <<= 1)
        ps += __shfl_xor_sync(0xffffffffu, ps, off);
      l += ps;
      pw[lane] = make_float2(pv, pv);
      __syncwarp();
      // ---- values: lanes over head-dim columns, fp32x2 over column pairs
      const uint8_t *vg0 = vs + key0 * C::ROW_BYTES + lane * VEC * 2;
      const int kmax = full_group ? KG : max(0, rows_valid - key0);
#pragma unroll
      for (int kk = 0; kk < KG; ++kk) {
        if (full_group || kk < kmax) {
          float vf[VEC];
          load_bf16_row<VEC>(vg0 + kk * C::ROW_BYTES, vf);
#pragma unroll
          for (int hh = 0; hh < GP; ++hh) {
            const float2 pk = pw[hh * KG + kk];
            if constexpr (VEC == 1) {
              acc2[hh][0].x = fmaf(pk.x, vf[0], acc2[hh][0].x);
            } else {
#pragma unroll
              for (int e = 0; e < VP; ++e)
                acc2[hh][e] = __ffma2_rn(pk, make_float2(vf[2 * e], vf[2 * e + 1]), acc2[hh][e]);
            }
          }
        }
      }
      __syncwarp();
    }
    if (lane == 0) mbar_arrive(&empty[s]);
  }
  if (!ok) {
    atomicMax(p.status, kDecodeStatusTimeout);
    if (lane == 0) *failed = 1;
  }
  float acc[GP][VEC];
#pragma unroll
  for (int hh = 0; hh < GP; ++hh) {
    if constexpr (VEC == 1) {
      acc[hh][0] = acc2[hh][0].x;
    } else {
#pragma unroll
      for (int e = 0; e < VP; ++e) {
        acc[hh][2 * e] = acc2[hh][e].x;
        acc[hh][2 * e + 1] = acc2[hh][e].y;
      }
    }
  }

  // ---- merge the consumer warps' states (the K/V ring is free now: every
  // tile was waited for above).
  named_barrier_sync(1, C::CW * 32);
  float *mm = reinterpret_cast<float *>(smem + C::OFF_MM);
  float *ll = reinterpret_cast<float *>(smem + C::OFF_LL);
  float *aa = reinterpret_cast<float *>(smem + C::OFF_AA);
  if ((lane % KG) == 0) {
    mm[warp * GP + lane / KG] = m;
    ll[warp * GP + lane / KG] = l;
  }
#pragma unroll
  for (int hh = 0; hh < GP; ++hh)
#pragma unroll
    for (int e = 0; e < VEC; ++e) aa[(warp * GP + hh) * D + lane * VEC + e] = acc[hh][e];
  named_barrier_sync(1, C::CW * 32);
  // A split whose consumers gave up writes an empty partial (m = -inf, l = 0,
  // acc = 0), which the merge weighs with 0, so no call ever mixes in what an
  // earlier call left in the workspace; the status word reports the timeout.
  const bool merged_ok = *failed == 0;
  for (int idx = threadIdx.x; idx < nh * D; idx += C::CW * 32) {
    const int hh = idx / D, col = idx - hh * D;
    float ms = -INFINITY;
    float a = 0.f, ls = 0.f;
    if (merged_ok) {
#pragma unroll
      for (int w = 0; w < C::CW; ++w) ms = fmaxf(ms, mm[w * GP + hh]);
#pragma unroll
      for (int w = 0; w < C::CW; ++w) {
        const float mw = mm[w * GP + hh];
        const float wt = (mw == -INFINITY) ? 0.f : ex2_approx(mw - ms);
        a = fmaf(wt, aa[(w * GP + hh) * D + col], a);
        ls = fmaf(wt, ll[w * GP + hh], ls);
      }
    }
    const size_t row = (size_t)b * p.Hq + h0 + hh;
    p.part_acc[(row * p.nsplit + sidx) * D + col] = a;
    if (col == 0) {
      p.part_ml[(row * p.nsplit + sidx) * 2 + 0] = ms;
      p.part_ml[(row * p.nsplit + sidx) * 2 + 1] = ls;
    }
  }
}

template <int D>
__global__ void __launch_bounds__(128)
    decode_combine_kernel(const float *__restrict__ part_acc,
                          const float *__restrict__ part_ml,
                          __nv_bfloat16 *__restrict__ o, float *__restrict__ lse,
                          int rows, int nsplit) {
  constexpr int VEC = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * 4 + warp;
  if (row >= rows) return;
  const float *ml = part_ml + (size_t)row * nsplit * 2;
  const float *pa = part_acc + (size_t)row * nsplit * D;
  float ms = -INFINITY;
  for (int s = lane; s < nsplit; s += 32) ms = fmaxf(ms, ml[2 * s]);
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1)
    ms = fmaxf(ms, __shfl_xor_sync(0xffffffffu, ms, off));
  float acc[VEC];
#pragma unroll
  for (int e = 0; e < VEC; ++e) acc[e] = 0.f;
  float ls = 0.f;
  for (int s = 0; s < nsplit; ++s) {
    const float mw = ml[2 * s];
    const float wt = (mw == -INFINITY) ? 0.f : ex2_approx(mw - ms);
    ls = fmaf(wt, ml[2 * s + 1], ls);
#pragma unroll
    for (int e = 0; e < VEC; ++e) acc[e] = fmaf(wt, pa[(size_t)s * D + lane * VEC + e], acc[e]);
  }
  const float inv = (ls > 0.f) ? 1.f / ls : 0.f;
  __nv_bfloat16 *orow = o + (size_t)row * D + lane * VEC;
#pragma unroll
  for (int e = 0; e < VEC; ++e) orow[e] = __float2bfloat16_rn(acc[e] * inv);
  if (lane == 0) lse[row] = (ls > 0.f) ? (ms + log2f(ls)) * 0.6931471805599453f : 0.f;
}

}  // namespace attn_dev
