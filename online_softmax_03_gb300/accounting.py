"""Work and traffic accounting for attention forward (pure Python, no GPU).

These are the measurement definitions the benchmark divides by:

* FLOPs of one forward call: the two matrix products QK^T and PV cost
  2 * Tq * Tk * d each per (batch, head), 4 * B * Hq * Tq * Tk * d in all
  ("Attention from scratch + roofline", section "FLOPs / bytes / arithmetic
  intensity"); under a causal mask half of that is counted (its exercise 3,
  and the causal skip in "4.2 FlashAttention I", section "FlashAttention
  forward").
* Compulsory bytes: every input read once and every output written once,
  Q + K + V + O in bf16 plus the fp32 row log-sum-exp.
* The logical access model of "Explain tiled attention and verify its
  output" (lab.py, estimate_hbm_bytes): the standard method's Q, K, V, O plus
  four T x T passes (write S, read S, write P, read P), against the causal
  outer-Q tiled loop that rereads the visible K/V rows once per query block.
"""
from __future__ import annotations

import math

BF16_BYTES = 2
LSE_BYTES = 4


def attention_flops(B: int, Hq: int, Tq: int, Tk: int, d: int, causal: bool) -> float:
    """4*B*Hq*Tq*Tk*d, halved for a causal mask."""
    f = 4.0 * B * Hq * Tq * Tk * d
    return f / 2.0 if causal else f


def backward_flops(B: int, Hq: int, Tq: int, Tk: int, d: int, causal: bool) -> float:
    """Five Tq x Tk x d products per (batch, head) -- S recomputed, dP, dV,
    dK, dQ -- 2*Tq*Tk*d each: 10*B*Hq*Tq*Tk*d, halved for a causal mask
    (2.5 times the forward's count)."""
    f = 10.0 * B * Hq * Tq * Tk * d
    return f / 2.0 if causal else f


def backward_dq_reduction_bytes(B: int, Hq: int, Tq: int, Tk: int, d: int, causal: bool,
                                key_tile: int = 128, query_tile: int = 128,
                                window: int = 0) -> int:
    """Bytes of fp32 dQ the keys-outer backward adds into its global
    accumulator: every (key tile, query tile) pair a CTA visits contributes a
    partial for each query row of the tile that exists (rows past Tq are not
    added), d fp32 values each.  Under causal masking key tile j visits the
    query tiles from the first one that sees its first key; under a sliding
    window of W keys only up to the last one whose window reaches its last
    key (query j*key_tile + key_tile - 2 - (Tk - Tq) + W)."""
    n_kt = -(-Tk // key_tile)
    n_qt = -(-Tq // query_tile)
    delta = Tk - Tq
    rows = 0
    for j in range(n_kt):
        lo = max(0, j * key_tile - delta) // query_tile if causal or window else 0
        hi = n_qt
        if window:
            last = j * key_tile + key_tile - 2 - delta + window
            hi = 0 if last < 0 else min(n_qt, last // query_tile + 1)
        for t in range(lo, hi):
            rows += min(query_tile, Tq - t * query_tile)
    return B * Hq * rows * d * 4


def visible_pairs(Tq: int, Tk: int, causal: bool, window: int = 0) -> int:
    """(row, key) pairs inside the mask of one (batch, head): all Tq*Tk, the
    bottom-right causal triangle, or the causal band of `window` keys."""
    if not causal:
        return Tq * Tk
    total = 0
    for i in range(Tq):
        p = i + Tk - Tq  # the query's position among the keys
        total += (p + 1) if window <= 0 else min(window, p + 1)
    return total


def window_flops(B: int, Hq: int, Tq: int, Tk: int, d: int, window: int) -> float:
    """Sliding-window forward: 4*d per visible (row, key) pair (QK^T and PV
    each cost 2*d per pair), counted exactly rather than halved."""
    return 4.0 * d * B * Hq * visible_pairs(Tq, Tk, True, window)


def varlen_flops(lens_q, lens_k, Hq: int, d: int, causal: bool) -> float:
    """Packed batch: 4*d per visible (row, key) pair of every sequence and
    head (causal pairs counted exactly, bottom-right aligned)."""
    pairs = 0
    for nq, nk in zip(lens_q, lens_k):
        nq, nk = int(nq), int(nk)
        if not causal:
            pairs += nq * nk
        else:  # row i sees i + (nk - nq) + 1 keys
            pairs += nq * (nk - nq) + nq * (nq + 1) // 2
    return 4.0 * d * Hq * pairs


def prefill_compulsory_bytes(B: int, Hq: int, Hkv: int, Tq: int, Tk: int, d: int) -> int:
    """Read Q, K, V once and write O (bf16) and LSE (fp32) once."""
    q = B * Hq * Tq * d * BF16_BYTES
    kv = 2 * B * Hkv * Tk * d * BF16_BYTES
    o = B * Hq * Tq * d * BF16_BYTES
    lse = B * Hq * Tq * LSE_BYTES
    return q + kv + o + lse


def decode_bytes(B: int, Hq: int, Hkv: int, Tk: int, d: int) -> int:
    """Algorithmic bytes of one decode call: the KV cache read once, q read,
    o and lse written.  Split-KV partials are not counted (they are an
    implementation choice, reported separately)."""
    return prefill_compulsory_bytes(B, Hq, Hkv, 1, Tk, d)


def paged_decode_bytes(B: int, Hq: int, Hkv: int, seq_lens, d: int, page_size: int) -> int:
    """Algorithmic bytes of one paged decode call: every sequence's keys and
    values once (per K/V head), the block-table entries of its pages, its
    length, q read and o, lse written."""
    lens = [int(n) for n in seq_lens]
    kv = sum(2 * Hkv * n * d * BF16_BYTES for n in lens)
    table = sum(-(-n // page_size) for n in lens) * 4
    q_o = 2 * B * Hq * d * BF16_BYTES
    return kv + table + 4 * B + q_o + B * Hq * LSE_BYTES


def decode_flops(B: int, Hq: int, Tk: int, d: int) -> float:
    return attention_flops(B, Hq, 1, Tk, d, causal=False)


def logical_access_model(seq_len: int, num_heads: int = 32, head_dim: int = 128,
                         bytes_per_elem: int = 2, block_q: int = 128) -> dict:
    """Logical (not measured) HBM access counts for one layer, in bytes.

    standard: Q, K, V, O plus S and P each written and read once (4 T^2 per head).
    tiled_causal: Q and O once, plus K and V rows [0, min(T, q0 + block_q))
    for every query block starting at q0 (no reuse between blocks assumed).
    """
    qkvo = 4 * num_heads * seq_len * head_dim * bytes_per_elem
    nxn = 4 * num_heads * seq_len * seq_len * bytes_per_elem
    kv_rows = sum(min(seq_len, q0 + block_q) for q0 in range(0, seq_len, block_q))
    tiled = (2 * num_heads * seq_len * head_dim
             + 2 * num_heads * kv_rows * head_dim) * bytes_per_elem
    return {
        "qkvo_bytes": qkvo,
        "standard_nxn_bytes": nxn,
        "standard_total_bytes": qkvo + nxn,
        "tiled_causal_bytes": tiled,
        "num_q_blocks": math.ceil(seq_len / block_q),
    }
