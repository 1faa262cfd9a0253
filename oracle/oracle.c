/*
 * oracle.c -- plain fp64 CPU oracle for exact scaled-dot-product attention.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke
 * check in __graft_entry__.py and the CPU-baseline / reference leg of
 * bench.py may load or call this library.  It shares no code, header,
 * table or helper with the CUDA library under online_softmax_03_gb300/.
 *
 * What it computes (the plain definition, which the tiled method reaches
 * exactly up to rounding order):
 *
 *   s_ij   = scale * sum_c Q[b,h,i,c] * K[b,g,j,c]          g = h / (Hq/Hkv)
 *   J_i    = { j < Tk : !causal  or  j <= i + (Tk - Tq) }   (visible keys)
 *            and, with a sliding window W > 0 (causal only),
 *            additionally j > i + (Tk - Tq) - W
 *   m_i    = max_{j in J_i} s_ij
 *   P_ij   = exp(s_ij - m_i) / sum_{j in J_i} exp(s_ij - m_i)
 *   O_i    = sum_j P_ij V[b,g,j,:]
 *   LSE_i  = m_i + ln sum_{j in J_i} exp(s_ij - m_i)
 *
 * Sources:
 *  - "4.2 FlashAttention I: IO-Awareness & The Online Softmax", section
 *    "The memory bottleneck: why naive attention is IO-bound" (attention_naive,
 *    softmax_rows with the row-max shift) and the reference_attention used to
 *    verify the tiled forward (lower-triangular causal mask).
 *  - "Explain tiled attention and verify its output", lab.py:
 *    standard_attention (materialised N x N scores, max shift optional).
 *  - "Efficient attention & KV cache", section 3, standard_attention.
 *  - The sliding window (query i sees keys i - W < j <= i): "4.2
 *    FlashAttention I", Exercise 4 (reference_swa), and "Efficient attention
 *    & KV cache", exercise 2.
 *  - Causal with Tq != Tk (bottom-right alignment, query i at key position
 *    i + Tk - Tq) and the GQA head map h -> h / (Hq/Hkv) are readings of
 *    the pages, which define causal only for Tq == Tk and name enable_gqa
 *    without giving its map ("SDPA and FlashAttention's tiling", the fused
 *    function's signature).
 *
 * Inputs are either fp64 arrays or bf16 bit patterns (uint16), upcast
 * exactly to fp64.  All arithmetic is fp64, in the order written here.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_IN_F64 0
#define ORACLE_IN_BF16 1

#define ORACLE_OK 0
#define ORACLE_ERR_ARG 1
#define ORACLE_ERR_OVERFLOW 2
#define ORACLE_ERR_NOMEM 3

static double bf16_bits_to_f64(uint16_t h) {
  uint32_t u = ((uint32_t)h) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Copy rows [r0, r0+nrows) of one (batch, head) slice of a [B, H, T, d]
 * tensor into a dense fp64 buffer. */
static void load_rows(const void *src, int in_type, size_t head_offset, int r0,
                      int nrows, int d, double *dst) {
  size_t base = head_offset + (size_t)r0 * (size_t)d;
  size_t n = (size_t)nrows * (size_t)d;
  if (in_type == ORACLE_IN_BF16) {
    const uint16_t *p = (const uint16_t *)src + base;
    for (size_t x = 0; x < n; ++x) dst[x] = bf16_bits_to_f64(p[x]);
  } else {
    const double *p = (const double *)src + base;
    memcpy(dst, p, n * sizeof(double));
  }
}

static int check_shape(int B, int Hq, int Hkv, int Tq, int Tk, int d,
                       int causal, int window) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Tq < 1 || Tk < 1 || d < 1)
    return ORACLE_ERR_ARG;
  if (Hq % Hkv != 0) return ORACLE_ERR_ARG;
  if (causal && Tq > Tk) return ORACLE_ERR_ARG;
  if (window < 0 || (window > 0 && !causal)) return ORACLE_ERR_ARG;
  return ORACLE_OK;
}

/* Is key j visible to query row i? */
static int visible(int i, int j, int Tq, int Tk, int causal, int window) {
  const int p = i + (Tk - Tq);  /* the query's position among the keys */
  if (!causal) return 1;
  if (j > p) return 0;
  return window == 0 || j > p - window;
}

/*
 * Dense attention: for every (b, h) the full Tq x Tk score matrix S is
 * built, turned in place into the probability matrix P row by row, and
 * multiplied by V.  Masked entries hold -inf in S and 0 in P.
 *
 *   o          [B, Hq, Tq, d] fp64 output
 *   lse        [B, Hq, Tq]    fp64 output (natural log)
 *   p_out      optional [B, Hq, Tq, Tk] fp64 copy of P (NULL to skip)
 *   subtract_max  1: shift by the row max before exp (the stable form);
 *                 0: exponentiate raw scores (overflows for large scores,
 *                    reported as ORACLE_ERR_OVERFLOW).
 *   visible_pairs optional output: number of (row, key) pairs inside the
 *                 mask, summed over all heads.
 */
int oracle_attn_dense(const void *q, const void *k, const void *v, int in_type,
                      int B, int Hq, int Hkv, int Tq, int Tk, int d, int causal,
                      int window, double scale, int subtract_max, double *o,
                      double *lse, double *p_out, long long *visible_pairs) {
  int rc = check_shape(B, Hq, Hkv, Tq, Tk, d, causal, window);
  if (rc) return rc;
  const int group = Hq / Hkv;
  const int nheads = B * Hq;
  int status = ORACLE_OK;
  long long vis_total = 0;

#pragma omp parallel for schedule(dynamic, 1) reduction(+ : vis_total)
  for (int bh = 0; bh < nheads; ++bh) {
    const int b = bh / Hq, h = bh % Hq, g = h / group;
    const size_t qoff = ((size_t)b * Hq + h) * (size_t)Tq * d;
    const size_t kvoff = ((size_t)b * Hkv + g) * (size_t)Tk * d;
    double *Qh = malloc(sizeof(double) * (size_t)Tq * d);
    double *Kh = malloc(sizeof(double) * (size_t)Tk * d);
    double *Vh = malloc(sizeof(double) * (size_t)Tk * d);
    double *S = malloc(sizeof(double) * (size_t)Tq * Tk);
    if (!Qh || !Kh || !Vh || !S) {
#pragma omp atomic write
      status = ORACLE_ERR_NOMEM;
      free(Qh); free(Kh); free(Vh); free(S);
      continue;
    }
    load_rows(q, in_type, qoff, 0, Tq, d, Qh);
    load_rows(k, in_type, kvoff, 0, Tk, d, Kh);
    load_rows(v, in_type, kvoff, 0, Tk, d, Vh);

    /* 1. S = scale * Q K^T, with -inf outside the mask. */
    for (int i = 0; i < Tq; ++i) {
      for (int j = 0; j < Tk; ++j) {
        double *sij = &S[(size_t)i * Tk + j];
        if (!visible(i, j, Tq, Tk, causal, window)) {
          *sij = -INFINITY;
          continue;
        }
        double acc = 0.0;
        for (int c = 0; c < d; ++c) acc += Qh[(size_t)i * d + c] * Kh[(size_t)j * d + c];
        *sij = scale * acc;
        vis_total += 1;
      }
    }

    /* 2. Row softmax of S, written over S, and the row log-sum-exp. */
    for (int i = 0; i < Tq; ++i) {
      double *row = &S[(size_t)i * Tk];
      double m = -INFINITY;
      for (int j = 0; j < Tk; ++j)
        if (row[j] > m) m = row[j];
      double shift = subtract_max ? m : 0.0;
      double denom = 0.0;
      for (int j = 0; j < Tk; ++j) {
        double e = (row[j] == -INFINITY) ? 0.0 : exp(row[j] - shift);
        if (isinf(e)) {
#pragma omp atomic write
          status = ORACLE_ERR_OVERFLOW;
        }
        row[j] = e;
        denom += e;
      }
      for (int j = 0; j < Tk; ++j) row[j] /= denom;
      lse[((size_t)b * Hq + h) * Tq + i] = shift + log(denom);
    }

    /* 3. O = P V. */
    for (int i = 0; i < Tq; ++i) {
      double *oi = &o[qoff + (size_t)i * d];
      for (int c = 0; c < d; ++c) oi[c] = 0.0;
      for (int j = 0; j < Tk; ++j) {
        double pij = S[(size_t)i * Tk + j];
        if (pij == 0.0) continue;
        for (int c = 0; c < d; ++c) oi[c] += pij * Vh[(size_t)j * d + c];
      }
    }

    if (p_out) {
      size_t poff = ((size_t)b * Hq + h) * (size_t)Tq * Tk;
      memcpy(p_out + poff, S, sizeof(double) * (size_t)Tq * Tk);
    }
    free(Qh); free(Kh); free(Vh); free(S);
  }
  if (visible_pairs) *visible_pairs = vis_total;
  return status;
}

/*
 * The same definition evaluated for a list of single output rows, so that
 * large problems can be checked on sampled rows.  Row r is (b[r], h[r], i[r]);
 * its score vector over all Tk keys is materialised, normalised and applied
 * to V.  o_rows is [nrows, d], lse_rows is [nrows].
 */
int oracle_attn_rows(const void *q, const void *k, const void *v, int in_type,
                     int B, int Hq, int Hkv, int Tq, int Tk, int d, int causal,
                     int window, double scale, int nrows, const int *rb,
                     const int *rh, const int *ri, double *o_rows,
                     double *lse_rows) {
  int rc = check_shape(B, Hq, Hkv, Tq, Tk, d, causal, window);
  if (rc) return rc;
  for (int r = 0; r < nrows; ++r)
    if (rb[r] < 0 || rb[r] >= B || rh[r] < 0 || rh[r] >= Hq || ri[r] < 0 ||
        ri[r] >= Tq)
      return ORACLE_ERR_ARG;
  const int group = Hq / Hkv;
  int status = ORACLE_OK;

#pragma omp parallel for schedule(dynamic, 1)
  for (int r = 0; r < nrows; ++r) {
    const int b = rb[r], h = rh[r], i = ri[r], g = h / group;
    const size_t qoff = ((size_t)b * Hq + h) * (size_t)Tq * d;
    const size_t kvoff = ((size_t)b * Hkv + g) * (size_t)Tk * d;
    double *qi = malloc(sizeof(double) * d);
    double *kj = malloc(sizeof(double) * d);
    double *s = malloc(sizeof(double) * (size_t)Tk);
    if (!qi || !kj || !s) {
#pragma omp atomic write
      status = ORACLE_ERR_NOMEM;
      free(qi); free(kj); free(s);
      continue;
    }
    load_rows(q, in_type, qoff, i, 1, d, qi);
    double m = -INFINITY;
    for (int j = 0; j < Tk; ++j) {
      if (!visible(i, j, Tq, Tk, causal, window)) {
        s[j] = -INFINITY;
        continue;
      }
      load_rows(k, in_type, kvoff, j, 1, d, kj);
      double acc = 0.0;
      for (int c = 0; c < d; ++c) acc += qi[c] * kj[c];
      s[j] = scale * acc;
      if (s[j] > m) m = s[j];
    }
    double denom = 0.0;
    for (int j = 0; j < Tk; ++j) {
      s[j] = (s[j] == -INFINITY) ? 0.0 : exp(s[j] - m);
      denom += s[j];
    }
    double *orow = &o_rows[(size_t)r * d];
    for (int c = 0; c < d; ++c) orow[c] = 0.0;
    for (int j = 0; j < Tk; ++j) {
      if (s[j] == 0.0) continue;
      double pij = s[j] / denom;
      load_rows(v, in_type, kvoff, j, 1, d, kj);
      for (int c = 0; c < d; ++c) orow[c] += pij * kj[c];
    }
    lse_rows[r] = m + log(denom);
    free(qi); free(kj); free(s);
  }
  return status;
}

/*
 * Blocked forward with the online softmax: for each query block of bq rows,
 * K/V blocks of bk rows are visited one at a time while per-row running
 * max m, running sum l and unnormalised accumulator acc are kept:
 *
 *   m'   = max(m, rowmax S_blk)            (guard: m' = 0 if still -inf)
 *   a    = exp(m - m')                     (a = 0 while m is -inf)
 *   l'   = a l + rowsum exp(S_blk - m')
 *   acc' = a acc + exp(S_blk - m') V_blk
 *   O    = acc / l,  LSE = m + ln l        (l = 0 is read as 1)
 *
 * Sources: "4.2 FlashAttention I: IO-Awareness & The Online Softmax",
 * section "FlashAttention forward: tiling + online softmax fused into one
 * pass" (the -inf guards and the LSE), and "Efficient attention & KV cache",
 * sections 2.1 and 3 (the recurrence and the causal kv_end stop);
 * "Explain tiled attention and verify its output" (rescale_previous_acc).
 *
 * Under causal masking, K/V blocks that lie wholly above the diagonal of
 * the query block are skipped, and with a window also those wholly left of
 * every row's window ("4.2 FlashAttention I", Exercise 4).
 *
 *   kv_order  optional permutation of the K/V block indices [0, nkb), used
 *             for every query block (NULL: natural order).  The result does
 *             not depend on it ("any m gives the same final ratio").
 *   rescale_acc  1: multiply acc by a (the method); 0: leave it unscaled
 *             (a deliberately wrong variant for the mutation test).
 *   tiles_visited optional output: (query block, K/V block) pairs processed,
 *             summed over all heads.
 */
int oracle_attn_blocked(const void *q, const void *k, const void *v,
                        int in_type, int B, int Hq, int Hkv, int Tq, int Tk,
                        int d, int causal, int window, double scale, int bq,
                        int bk, const int *kv_order, int rescale_acc, double *o,
                        double *lse, long long *tiles_visited) {
  int rc = check_shape(B, Hq, Hkv, Tq, Tk, d, causal, window);
  if (rc) return rc;
  if (bq < 1 || bk < 1) return ORACLE_ERR_ARG;
  const int nkb = (Tk + bk - 1) / bk;
  if (kv_order) {
    char *seen = calloc((size_t)nkb, 1);
    if (!seen) return ORACLE_ERR_NOMEM;
    for (int t = 0; t < nkb; ++t) {
      if (kv_order[t] < 0 || kv_order[t] >= nkb || seen[kv_order[t]]) {
        free(seen);
        return ORACLE_ERR_ARG;
      }
      seen[kv_order[t]] = 1;
    }
    free(seen);
  }
  const int group = Hq / Hkv;
  const int nheads = B * Hq;
  const int delta = Tk - Tq;
  int status = ORACLE_OK;
  long long visited = 0;

#pragma omp parallel for schedule(dynamic, 1) reduction(+ : visited)
  for (int bh = 0; bh < nheads; ++bh) {
    const int b = bh / Hq, h = bh % Hq, g = h / group;
    const size_t qoff = ((size_t)b * Hq + h) * (size_t)Tq * d;
    const size_t kvoff = ((size_t)b * Hkv + g) * (size_t)Tk * d;
    double *Qi = malloc(sizeof(double) * (size_t)bq * d);
    double *Kj = malloc(sizeof(double) * (size_t)bk * d);
    double *Vj = malloc(sizeof(double) * (size_t)bk * d);
    double *Sij = malloc(sizeof(double) * (size_t)bq * bk);
    double *m = malloc(sizeof(double) * bq);
    double *l = malloc(sizeof(double) * bq);
    double *acc = malloc(sizeof(double) * (size_t)bq * d);
    if (!Qi || !Kj || !Vj || !Sij || !m || !l || !acc) {
#pragma omp atomic write
      status = ORACLE_ERR_NOMEM;
      free(Qi); free(Kj); free(Vj); free(Sij); free(m); free(l); free(acc);
      continue;
    }
    for (int q0 = 0; q0 < Tq; q0 += bq) {
      const int rows = (Tq - q0 < bq) ? (Tq - q0) : bq;
      load_rows(q, in_type, qoff, q0, rows, d, Qi);
      for (int r = 0; r < rows; ++r) {
        m[r] = -INFINITY;
        l[r] = 0.0;
        for (int c = 0; c < d; ++c) acc[(size_t)r * d + c] = 0.0;
      }
      for (int t = 0; t < nkb; ++t) {
        const int jb = kv_order ? kv_order[t] : t;
        const int j0 = jb * bk;
        const int cols = (Tk - j0 < bk) ? (Tk - j0) : bk;
        /* causal: the block holds no key visible to any row of this block */
        if (causal && j0 > q0 + rows - 1 + delta) continue;
        /* window: the block lies wholly left of every row's window */
        if (window > 0 && j0 + cols - 1 < q0 + delta - window + 1) continue;
        visited += 1;
        load_rows(k, in_type, kvoff, j0, cols, d, Kj);
        load_rows(v, in_type, kvoff, j0, cols, d, Vj);
        for (int r = 0; r < rows; ++r) {
          const int i = q0 + r;
          double *srow = &Sij[(size_t)r * bk];
          double mblk = -INFINITY;
          for (int cj = 0; cj < cols; ++cj) {
            if (!visible(i, j0 + cj, Tq, Tk, causal, window)) {
              srow[cj] = -INFINITY;
              continue;
            }
            double dot = 0.0;
            for (int c = 0; c < d; ++c)
              dot += Qi[(size_t)r * d + c] * Kj[(size_t)cj * d + c];
            srow[cj] = scale * dot;
            if (srow[cj] > mblk) mblk = srow[cj];
          }
          double mnew = (m[r] > mblk) ? m[r] : mblk;
          if (mnew == -INFINITY) mnew = 0.0;
          const double a = (m[r] == -INFINITY) ? 0.0 : exp(m[r] - mnew);
          double rowsum = 0.0;
          for (int cj = 0; cj < cols; ++cj) {
            srow[cj] = (srow[cj] == -INFINITY) ? 0.0 : exp(srow[cj] - mnew);
            rowsum += srow[cj];
          }
          l[r] = a * l[r] + rowsum;
          const double accscale = rescale_acc ? a : 1.0;
          double *ar = &acc[(size_t)r * d];
          for (int c = 0; c < d; ++c) {
            double val = accscale * ar[c];
            for (int cj = 0; cj < cols; ++cj) val += srow[cj] * Vj[(size_t)cj * d + c];
            ar[c] = val;
          }
          m[r] = mnew;
        }
      }
      for (int r = 0; r < rows; ++r) {
        const double lsafe = (l[r] == 0.0) ? 1.0 : l[r];
        for (int c = 0; c < d; ++c)
          o[qoff + (size_t)(q0 + r) * d + c] = acc[(size_t)r * d + c] / lsafe;
        lse[((size_t)b * Hq + h) * Tq + q0 + r] = m[r] + log(lsafe);
      }
    }
    free(Qi); free(Kj); free(Vj); free(Sij); free(m); free(l); free(acc);
  }
  if (tiles_visited) *tiles_visited = visited;
  return status;
}

/*
 * One-dimensional online softmax over x[0..n) in blocks of `block`
 * ("Efficient attention & KV cache", section 3, online_softmax; worked in
 * "4.2 FlashAttention I", Exercise 2):
 *
 *   m_j = max(m_{j-1}, max x^(j)),  l_j = exp(m_{j-1} - m_j) l_{j-1} + sum exp(x^(j) - m_j)
 *   p   = exp(x - m_n) / l_n
 *
 * Per block j the trace arrays (each of length ceil(n/block), may be NULL)
 * receive m_j, l_j and the correction factor exp(m_{j-1} - m_j) (0 for the
 * first block, where m_0 = -inf).  *lse_out = m_n + ln l_n.
 */
int oracle_online_softmax_1d(const double *x, int n, int block, double *p,
                             double *m_trace, double *l_trace,
                             double *alpha_trace, double *lse_out) {
  if (n < 1 || block < 1) return ORACLE_ERR_ARG;
  double m = -INFINITY, l = 0.0;
  int jb = 0;
  for (int s = 0; s < n; s += block, ++jb) {
    const int e = (s + block < n) ? s + block : n;
    double mb = -INFINITY;
    for (int t = s; t < e; ++t)
      if (x[t] > mb) mb = x[t];
    const double mnew = (m > mb) ? m : mb;
    const double a = (m == -INFINITY) ? 0.0 : exp(m - mnew);
    double sum = 0.0;
    for (int t = s; t < e; ++t) sum += exp(x[t] - mnew);
    l = a * l + sum;
    m = mnew;
    if (m_trace) m_trace[jb] = m;
    if (l_trace) l_trace[jb] = l;
    if (alpha_trace) alpha_trace[jb] = a;
  }
  if (p)
    for (int t = 0; t < n; ++t) p[t] = exp(x[t] - m) / l;
  if (lse_out) *lse_out = m + log(l);
  return ORACLE_OK;
}

/*
 * Decode against a paged KV cache: one query token per sequence, its keys
 * and values gathered through a per-sequence block table ("Efficient
 * attention & KV cache", section 2.5 "Paged and shared caches": the cache
 * lives in fixed-size blocks and the kernel fetches each block from its
 * physical location by looking it up in the sequence's table; the same
 * page's interview answer on what PagedAttention changes in the kernel).
 *
 * Layout (a reading: the page fixes blocks and a table, not the order of
 * the axes inside a block):
 *   q            [B, Hq, d]                    one query row per (b, h)
 *   k_pages      [num_pages, Hkv, page_size, d]
 *   v_pages      [num_pages, Hkv, page_size, d]
 *   block_table  [B, max_pages]  int32, physical page of logical page p
 *   seq_lens     [B]             int32, keys of sequence b (1..max_pages*page_size)
 *
 * Key j of sequence b (j < seq_lens[b]) is row j % page_size of head g in
 * physical page block_table[b][j / page_size].  The result is the plain
 * definition over those keys (no mask: a decode query sees its whole
 * cache):  s_j = scale * q . K_j,  O = sum_j softmax(s)_j V_j,
 * LSE = m + ln sum_j exp(s_j - m).  o is [B, Hq, d], lse is [B, Hq].
 */
int oracle_attn_paged_decode(const void *q, const void *k_pages,
                             const void *v_pages, int in_type,
                             const int *block_table, const int *seq_lens,
                             int B, int Hq, int Hkv, int d, int page_size,
                             int num_pages, int max_pages, double scale,
                             double *o, double *lse) {
  if (B < 1 || Hq < 1 || Hkv < 1 || d < 1 || page_size < 1 || num_pages < 1 ||
      max_pages < 1 || Hq % Hkv != 0)
    return ORACLE_ERR_ARG;
  for (int b = 0; b < B; ++b) {
    const int len = seq_lens[b];
    if (len < 1 || len > max_pages * page_size) return ORACLE_ERR_ARG;
    const int used = (len + page_size - 1) / page_size;
    for (int pg = 0; pg < used; ++pg) {
      const int phys = block_table[(size_t)b * max_pages + pg];
      if (phys < 0 || phys >= num_pages) return ORACLE_ERR_ARG;
    }
  }
  const int group = Hq / Hkv;
  int status = ORACLE_OK;

#pragma omp parallel for collapse(2) schedule(dynamic, 1)
  for (int b = 0; b < B; ++b) {
    for (int h = 0; h < Hq; ++h) {
      const int g = h / group, len = seq_lens[b];
      double *qi = malloc(sizeof(double) * d);
      double *row = malloc(sizeof(double) * d);
      double *s = malloc(sizeof(double) * (size_t)len);
      if (!qi || !row || !s) {
#pragma omp atomic write
        status = ORACLE_ERR_NOMEM;
        free(qi); free(row); free(s);
        continue;
      }
      load_rows(q, in_type, ((size_t)b * Hq + h) * (size_t)d, 0, 1, d, qi);
      double m = -INFINITY;
      for (int j = 0; j < len; ++j) {
        const int phys = block_table[(size_t)b * max_pages + j / page_size];
        const size_t slab = ((size_t)phys * Hkv + g) * (size_t)page_size * d;
        load_rows(k_pages, in_type, slab, j % page_size, 1, d, row);
        double acc = 0.0;
        for (int c = 0; c < d; ++c) acc += qi[c] * row[c];
        s[j] = scale * acc;
        if (s[j] > m) m = s[j];
      }
      double denom = 0.0;
      for (int j = 0; j < len; ++j) {
        s[j] = exp(s[j] - m);
        denom += s[j];
      }
      double *orow = &o[((size_t)b * Hq + h) * d];
      for (int c = 0; c < d; ++c) orow[c] = 0.0;
      for (int j = 0; j < len; ++j) {
        const int phys = block_table[(size_t)b * max_pages + j / page_size];
        const size_t slab = ((size_t)phys * Hkv + g) * (size_t)page_size * d;
        load_rows(v_pages, in_type, slab, j % page_size, 1, d, row);
        const double pj = s[j] / denom;
        for (int c = 0; c < d; ++c) orow[c] += pj * row[c];
      }
      lse[(size_t)b * Hq + h] = m + log(denom);
      free(qi); free(row); free(s);
    }
  }
  return status;
}

/*
 * Packed variable-length batches: B sequences concatenated without padding,
 * sequence b owning query rows cu_q[b] .. cu_q[b+1]-1 and key rows
 * cu_k[b] .. cu_k[b+1]-1 ("SDPA and FlashAttention's tiling", the packed
 * flash_attn_varlen_func call: cumulative int32 offsets of length B+1, and
 * no score between two documents is ever formed).  Each sequence is an
 * independent attention problem with the definition at the top of this
 * file (causal: bottom-right aligned inside the sequence; window > 0: also
 * the sliding window of "4.2 FlashAttention I", Exercise 4, inside it).
 *
 * Layout (token-major, as packed activations come):
 *   q, o  [total_q, Hq, d]      k, v  [total_k, Hkv, d]     lse  [Hq, total_q]
 * Offsets must start at 0, never decrease and end within total_q /
 * total_k; a sequence with queries needs at least one key, and causal
 * needs at most as many queries as keys.  Rows not covered by any sequence
 * are left untouched.
 */
int oracle_attn_varlen(const void *q, const void *k, const void *v, int in_type,
                       const int *cu_q, const int *cu_k, int B, int Hq, int Hkv,
                       int total_q, int total_k, int d, int causal, int window,
                       double scale, double *o, double *lse) {
  if (B < 1 || Hq < 1 || Hkv < 1 || d < 1 || total_q < 0 || total_k < 0 ||
      Hq % Hkv != 0 || cu_q[0] != 0 || cu_k[0] != 0 || window < 0 || (window > 0 && !causal))
    return ORACLE_ERR_ARG;
  for (int b = 0; b < B; ++b) {
    const int nq = cu_q[b + 1] - cu_q[b], nk = cu_k[b + 1] - cu_k[b];
    if (nq < 0 || nk < 0 || cu_q[b + 1] > total_q || cu_k[b + 1] > total_k)
      return ORACLE_ERR_ARG;
    if (nq > 0 && nk < 1) return ORACLE_ERR_ARG;
    if (causal && nq > nk) return ORACLE_ERR_ARG;
  }
  const int group = Hq / Hkv;
  int status = ORACLE_OK;

#pragma omp parallel for collapse(2) schedule(dynamic, 1)
  for (int b = 0; b < B; ++b) {
    for (int h = 0; h < Hq; ++h) {
      const int nq = cu_q[b + 1] - cu_q[b], nk = cu_k[b + 1] - cu_k[b];
      if (nq == 0) continue;
      const int g = h / group;
      double *qi = malloc(sizeof(double) * d);
      double *row = malloc(sizeof(double) * d);
      double *s = malloc(sizeof(double) * (size_t)nk);
      if (!qi || !row || !s) {
#pragma omp atomic write
        status = ORACLE_ERR_NOMEM;
        free(qi); free(row); free(s);
        continue;
      }
      for (int i = 0; i < nq; ++i) {
        const size_t qrow = (size_t)cu_q[b] + i;
        load_rows(q, in_type, (qrow * Hq + h) * (size_t)d, 0, 1, d, qi);
        double m = -INFINITY;
        for (int j = 0; j < nk; ++j) {
          if (!visible(i, j, nq, nk, causal, window)) {
            s[j] = -INFINITY;
            continue;
          }
          const size_t krow = (size_t)cu_k[b] + j;
          load_rows(k, in_type, (krow * Hkv + g) * (size_t)d, 0, 1, d, row);
          double acc = 0.0;
          for (int c = 0; c < d; ++c) acc += qi[c] * row[c];
          s[j] = scale * acc;
          if (s[j] > m) m = s[j];
        }
        double denom = 0.0;
        for (int j = 0; j < nk; ++j) {
          s[j] = (s[j] == -INFINITY) ? 0.0 : exp(s[j] - m);
          denom += s[j];
        }
        double *orow = &o[(qrow * Hq + h) * (size_t)d];
        for (int c = 0; c < d; ++c) orow[c] = 0.0;
        for (int j = 0; j < nk; ++j) {
          if (s[j] == 0.0) continue;
          const size_t krow = (size_t)cu_k[b] + j;
          load_rows(v, in_type, (krow * Hkv + g) * (size_t)d, 0, 1, d, row);
          const double pj = s[j] / denom;
          for (int c = 0; c < d; ++c) orow[c] += pj * row[c];
        }
        lse[(size_t)h * total_q + qrow] = m + log(denom);
      }
      free(qi); free(row); free(s);
    }
  }
  return status;
}

/*
 * Backward pass, the plain definition ("4.2 FlashAttention I", section
 * "The backward pass: recomputation instead of storage": the chain rule
 * through O = P V and the row softmax; "Efficient attention & KV cache",
 * section 2.2, backward with recomputation):
 *
 *   P     = softmax_row(S),  S = scale Q K^T (masked entries -inf, P = 0)
 *   O     = P V,   D_i = sum_c dO_ic O_ic
 *   dV    = P^T dO
 *   dP    = dO V^T
 *   dS    = P o (dP - D)        (o: elementwise; D broadcast along rows)
 *   dQ    = scale dS K,   dK = scale dS^T Q
 *
 * The mask is the forward's: causal, and with window > 0 also the sliding
 * window of "4.2 FlashAttention I", Exercise 4 (masked entries have P = 0,
 * so they carry no gradient).
 * For every (b, h) the full Tq x Tk matrices S, P, dP, dS are materialised.
 * Under grouped-query attention K/V head g serves query heads
 * g*group .. g*group+group-1, so dK_g and dV_g sum their contributions.
 * q, k, v and dO are fp64 or bf16 bits (in_type); dq [B,Hq,Tq,d],
 * dk and dv [B,Hkv,Tk,d], and optionally o [B,Hq,Tq,d] and lse [B,Hq,Tq]
 * (natural log) are written in fp64.
 */
int oracle_attn_bwd_dense(const void *q, const void *k, const void *v, const void *dout,
                          int in_type, int B, int Hq, int Hkv, int Tq, int Tk, int d,
                          int causal, int window, double scale, double *dq, double *dk,
                          double *dv, double *o_out, double *lse_out) {
  int rc = check_shape(B, Hq, Hkv, Tq, Tk, d, causal, window);
  if (rc) return rc;
  const int group = Hq / Hkv;
  int status = ORACLE_OK;

#pragma omp parallel for collapse(2) schedule(dynamic, 1)
  for (int b = 0; b < B; ++b) {
    for (int g = 0; g < Hkv; ++g) {
      const size_t kvoff = ((size_t)b * Hkv + g) * (size_t)Tk * d;
      double *Kh = malloc(sizeof(double) * (size_t)Tk * d);
      double *Vh = malloc(sizeof(double) * (size_t)Tk * d);
      double *Qh = malloc(sizeof(double) * (size_t)Tq * d);
      double *dOh = malloc(sizeof(double) * (size_t)Tq * d);
      double *P = malloc(sizeof(double) * (size_t)Tq * Tk);
      double *dS = malloc(sizeof(double) * (size_t)Tq * Tk);
      double *Oh = malloc(sizeof(double) * (size_t)Tq * d);
      double *Dv = malloc(sizeof(double) * (size_t)Tq);
      if (!Kh || !Vh || !Qh || !dOh || !P || !dS || !Oh || !Dv) {
#pragma omp atomic write
        status = ORACLE_ERR_NOMEM;
        free(Kh); free(Vh); free(Qh); free(dOh); free(P); free(dS); free(Oh); free(Dv);
        continue;
      }
      load_rows(k, in_type, kvoff, 0, Tk, d, Kh);
      load_rows(v, in_type, kvoff, 0, Tk, d, Vh);
      double *dKg = &dk[kvoff], *dVg = &dv[kvoff];
      for (size_t x = 0; x < (size_t)Tk * d; ++x) dKg[x] = dVg[x] = 0.0;
      for (int h = g * group; h < (g + 1) * group; ++h) {
        const size_t qoff = ((size_t)b * Hq + h) * (size_t)Tq * d;
        load_rows(q, in_type, qoff, 0, Tq, d, Qh);
        load_rows(dout, in_type, qoff, 0, Tq, d, dOh);
        /* P = softmax(S) row by row, with the row-max shift */
        for (int i = 0; i < Tq; ++i) {
          double *Pi = &P[(size_t)i * Tk];
          double m = -INFINITY;
          for (int j = 0; j < Tk; ++j) {
            if (!visible(i, j, Tq, Tk, causal, window)) {
              Pi[j] = -INFINITY;
              continue;
            }
            double acc = 0.0;
            for (int c = 0; c < d; ++c) acc += Qh[(size_t)i * d + c] * Kh[(size_t)j * d + c];
            Pi[j] = scale * acc;
            if (Pi[j] > m) m = Pi[j];
          }
          double denom = 0.0;
          for (int j = 0; j < Tk; ++j) {
            Pi[j] = (Pi[j] == -INFINITY) ? 0.0 : exp(Pi[j] - m);
            denom += Pi[j];
          }
          for (int j = 0; j < Tk; ++j) Pi[j] /= denom;
          if (lse_out) lse_out[((size_t)b * Hq + h) * Tq + i] = m + log(denom);
        }
        /* O = P V and D = rowsum(dO o O) */
        for (int i = 0; i < Tq; ++i) {
          double Di = 0.0;
          for (int c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int j = 0; j < Tk; ++j) acc += P[(size_t)i * Tk + j] * Vh[(size_t)j * d + c];
            Oh[(size_t)i * d + c] = acc;
            Di += dOh[(size_t)i * d + c] * acc;
          }
          Dv[i] = Di;
        }
        if (o_out) memcpy(&o_out[qoff], Oh, sizeof(double) * (size_t)Tq * d);
        /* dP = dO V^T, then dS = P o (dP - D) */
        for (int i = 0; i < Tq; ++i)
          for (int j = 0; j < Tk; ++j) {
            double dp = 0.0;
            for (int c = 0; c < d; ++c) dp += dOh[(size_t)i * d + c] * Vh[(size_t)j * d + c];
            dS[(size_t)i * Tk + j] = P[(size_t)i * Tk + j] * (dp - Dv[i]);
          }
        /* dQ = scale dS K */
        double *dQh = &dq[qoff];
        for (int i = 0; i < Tq; ++i)
          for (int c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int j = 0; j < Tk; ++j) acc += dS[(size_t)i * Tk + j] * Kh[(size_t)j * d + c];
            dQh[(size_t)i * d + c] = scale * acc;
          }
        /* dK += scale dS^T Q,  dV += P^T dO */
        for (int j = 0; j < Tk; ++j)
          for (int c = 0; c < d; ++c) {
            double ak = 0.0, av = 0.0;
            for (int i = 0; i < Tq; ++i) {
              ak += dS[(size_t)i * Tk + j] * Qh[(size_t)i * d + c];
              av += P[(size_t)i * Tk + j] * dOh[(size_t)i * d + c];
            }
            dKg[(size_t)j * d + c] += scale * ak;
            dVg[(size_t)j * d + c] += av;
          }
      }
      free(Kh); free(Vh); free(Qh); free(dOh); free(P); free(dS); free(Oh); free(Dv);
    }
  }
  return status;
}

/*
 * Backward with recomputation, in the steps of "4.2 FlashAttention I",
 * section "The backward pass: recomputation instead of storage": D from
 * dO and the forward output O; then for each query block of bq rows and
 * each key block of bk keys, the score tile is recomputed and turned into
 * probabilities with the saved log-sum-exp, P = exp(S - L), never stored
 * beyond the tile; dV and dK accumulate over query blocks, dQ over key
 * blocks.  o [B,Hq,Tq,d] and lse [B,Hq,Tq] are fp64 (what the forward
 * returned); q, k, v, dO follow in_type.  Masking is bottom-right causal.
 */
int oracle_attn_bwd_blocked(const void *q, const void *k, const void *v, const void *dout,
                            int in_type, const double *o, const double *lse, int B, int Hq,
                            int Hkv, int Tq, int Tk, int d, int causal, double scale,
                            int bq, int bk, double *dq, double *dk, double *dv) {
  int rc = check_shape(B, Hq, Hkv, Tq, Tk, d, causal, 0);
  if (rc) return rc;
  if (bq < 1 || bk < 1) return ORACLE_ERR_ARG;
  const int group = Hq / Hkv;
  int status = ORACLE_OK;

#pragma omp parallel for collapse(2) schedule(dynamic, 1)
  for (int b = 0; b < B; ++b) {
    for (int g = 0; g < Hkv; ++g) {
      const size_t kvoff = ((size_t)b * Hkv + g) * (size_t)Tk * d;
      double *Kh = malloc(sizeof(double) * (size_t)Tk * d);
      double *Vh = malloc(sizeof(double) * (size_t)Tk * d);
      double *Qh = malloc(sizeof(double) * (size_t)Tq * d);
      double *dOh = malloc(sizeof(double) * (size_t)Tq * d);
      double *Dv = malloc(sizeof(double) * (size_t)Tq);
      double *Pt = malloc(sizeof(double) * (size_t)bq * bk);
      double *dSt = malloc(sizeof(double) * (size_t)bq * bk);
      if (!Kh || !Vh || !Qh || !dOh || !Dv || !Pt || !dSt) {
#pragma omp atomic write
        status = ORACLE_ERR_NOMEM;
        free(Kh); free(Vh); free(Qh); free(dOh); free(Dv); free(Pt); free(dSt);
        continue;
      }
      load_rows(k, in_type, kvoff, 0, Tk, d, Kh);
      load_rows(v, in_type, kvoff, 0, Tk, d, Vh);
      double *dKg = &dk[kvoff], *dVg = &dv[kvoff];
      for (size_t x = 0; x < (size_t)Tk * d; ++x) dKg[x] = dVg[x] = 0.0;
      for (int h = g * group; h < (g + 1) * group; ++h) {
        const size_t qoff = ((size_t)b * Hq + h) * (size_t)Tq * d;
        load_rows(q, in_type, qoff, 0, Tq, d, Qh);
        load_rows(dout, in_type, qoff, 0, Tq, d, dOh);
        const double *Oh = &o[qoff];
        const double *Lh = &lse[((size_t)b * Hq + h) * Tq];
        double *dQh = &dq[qoff];
        for (int i = 0; i < Tq; ++i) {
          double Di = 0.0;
          for (int c = 0; c < d; ++c) Di += dOh[(size_t)i * d + c] * Oh[(size_t)i * d + c];
          Dv[i] = Di;
        }
        for (size_t x = 0; x < (size_t)Tq * d; ++x) dQh[x] = 0.0;
        for (int i0 = 0; i0 < Tq; i0 += bq) {
          const int rows = (Tq - i0 < bq) ? Tq - i0 : bq;
          for (int j0 = 0; j0 < Tk; j0 += bk) {
            const int cols = (Tk - j0 < bk) ? Tk - j0 : bk;
            /* recompute the probability tile from the saved L */
            for (int r = 0; r < rows; ++r)
              for (int cj = 0; cj < cols; ++cj) {
                const int i = i0 + r, j = j0 + cj;
                double p = 0.0;
                if (visible(i, j, Tq, Tk, causal, 0)) {
                  double acc = 0.0;
                  for (int c = 0; c < d; ++c) acc += Qh[(size_t)i * d + c] * Kh[(size_t)j * d + c];
                  p = exp(scale * acc - Lh[i]);
                }
                Pt[r * bk + cj] = p;
              }
            /* dV_j += P^T dO_i;  dP = dO_i V_j^T;  dS = P o (dP - D) */
            for (int cj = 0; cj < cols; ++cj)
              for (int c = 0; c < d; ++c) {
                double acc = 0.0;
                for (int r = 0; r < rows; ++r)
                  acc += Pt[r * bk + cj] * dOh[(size_t)(i0 + r) * d + c];
                dVg[(size_t)(j0 + cj) * d + c] += acc;
              }
            for (int r = 0; r < rows; ++r)
              for (int cj = 0; cj < cols; ++cj) {
                double dp = 0.0;
                for (int c = 0; c < d; ++c)
                  dp += dOh[(size_t)(i0 + r) * d + c] * Vh[(size_t)(j0 + cj) * d + c];
                dSt[r * bk + cj] = Pt[r * bk + cj] * (dp - Dv[i0 + r]);
              }
            /* dQ_i += scale dS K_j;  dK_j += scale dS^T Q_i */
            for (int r = 0; r < rows; ++r)
              for (int c = 0; c < d; ++c) {
                double acc = 0.0;
                for (int cj = 0; cj < cols; ++cj)
                  acc += dSt[r * bk + cj] * Kh[(size_t)(j0 + cj) * d + c];
                dQh[(size_t)(i0 + r) * d + c] += scale * acc;
              }
            for (int cj = 0; cj < cols; ++cj)
              for (int c = 0; c < d; ++c) {
                double acc = 0.0;
                for (int r = 0; r < rows; ++r)
                  acc += dSt[r * bk + cj] * Qh[(size_t)(i0 + r) * d + c];
                dKg[(size_t)(j0 + cj) * d + c] += scale * acc;
              }
          }
        }
      }
      free(Kh); free(Vh); free(Qh); free(dOh); free(Dv); free(Pt); free(dSt);
    }
  }
  return status;
}
