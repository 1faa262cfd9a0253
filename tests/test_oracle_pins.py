"""Pins for the fp64 CPU oracle, against what the pages and mathematics fix.

Each test ties the oracle to something other than itself: values printed on
the pages, closed forms, invariants, library routines on special cases, or
the agreement of two independently written algorithms (dense and blocked).
Every plausible slip in the oracle (a dropped rescale, a wrong causal index,
a transposed operand, a wrong GQA map, a missing max shift, a wrong LSE base)
fails at least one of them.
"""
import json
import math
import os
import random

import numpy as np
import pytest
import scipy.special

from oracle import oracle as ora

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _bhtd(x):
    """[T, d] list/array -> [1, 1, T, d] float64."""
    return np.asarray(x, dtype=np.float64)[None, None]


def _lab_qkv(seq_len, head_dim, seed):
    """The lab's input recipe: one random.Random stream, q then k then v,
    row-major, each entry uniform on (-0.8, 0.8)."""
    rng = random.Random(seed)
    out = []
    for _ in range(3):
        out.append([[rng.uniform(-0.8, 0.8) for _ in range(head_dim)]
                    for _ in range(seq_len)])
    return out


# --- values printed on the pages -------------------------------------------

def test_p2_recorded_run_sample_rows_and_counts():
    """'Explain tiled attention and verify its output': recorded result."""
    gold = _golden("p2_lab_recorded.json")
    q, k, v = _lab_qkv(gold["seq_len"], gold["head_dim"], gold["seed"])
    q, k, v = _bhtd(q), _bhtd(k), _bhtd(v)
    o, lse, ex = ora.attention_dense(q, k, v, causal=True)
    half_ulp = 0.5 * 10.0 ** -gold["printed_decimals"] + 1e-12
    np.testing.assert_allclose(o[0, 0, 0, :4], gold["sample_row0_first4"], rtol=0,
                               atol=half_ulp)
    np.testing.assert_allclose(o[0, 0, -1, :4], gold["sample_last_row_first4"],
                               rtol=0, atol=half_ulp)
    # the standard method keeps one score and one probability per visible pair
    assert 2 * ex["visible_pairs"] == gold["standard_materialized_elements"]
    ob, lseb, visited = ora.attention_blocked(q, k, v, gold["block_q"],
                                              gold["block_kv"], causal=True)
    assert visited == gold["flash_tiles_visited"]
    assert np.abs(ob - o).max() < 1e-12
    assert np.abs(lseb - lse).max() < 1e-12


def test_p3_exercise2_online_softmax_trace():
    """'4.2 FlashAttention I', Exercise 2: x=[3,1,6,2], block 2."""
    gold = _golden("p3_exercise2.json")
    p, lse, tr = ora.online_softmax_1d(gold["x"], gold["block"])
    tol = gold["tolerance"]
    assert tr["m"][0] == gold["m_after_block1"]
    assert abs(tr["l"][0] - gold["l_after_block1"]) < tol
    assert abs(tr["alpha"][1] - gold["alpha_block2"]) < tol
    assert tr["m"][1] == gold["m_final"]
    assert abs(tr["l"][1] - gold["l_final"]) < tol
    assert abs(lse - gold["lse"]) < tol
    # (a): the streamed denominator equals the two-pass one
    x = np.asarray(gold["x"])
    assert abs(tr["l"][1] - np.exp(x - x.max()).sum()) < 1e-15
    assert abs(p.sum() - 1.0) < 1e-15


def test_hand_example_t4_d2():
    gold = _golden("hand_t4_d2.json")
    q = _bhtd([[math.sqrt(2.0), 0.0]] * 4)
    k = _bhtd([[math.log(j + 1.0), 0.0] for j in range(4)])
    v = _bhtd(gold["v"])
    scale = 1.0 / math.sqrt(2.0)
    o, lse, _ = ora.attention_dense(q, k, v, causal=True, scale=scale)
    np.testing.assert_allclose(o[0, 0], gold["causal_o"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse[0, 0], gold["causal_lse"], rtol=0, atol=1e-14)
    o, lse, _ = ora.attention_dense(q, k, v, causal=False, scale=scale)
    for i in range(4):
        np.testing.assert_allclose(o[0, 0, i], gold["noncausal_o_every_row"], rtol=0,
                                   atol=1e-14)
        assert abs(lse[0, 0, i] - gold["noncausal_lse_every_row"]) < 1e-14
    ob, lseb, _ = ora.attention_blocked(q, k, v, 3, 3, causal=True, scale=scale)
    np.testing.assert_allclose(ob[0, 0], gold["causal_o"], rtol=0, atol=1e-14)


# --- closed forms and invariants ---------------------------------------------

def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def test_causal_row0_is_v0_and_lse0_is_s00():
    q, k, v = _rand((2, 3, 9, 8), 1), _rand((2, 3, 9, 8), 2), _rand((2, 3, 9, 8), 3)
    o, lse, _ = ora.attention_dense(q, k, v, causal=True)
    np.testing.assert_allclose(o[:, :, 0], v[:, :, 0], rtol=0, atol=1e-15)
    s00 = (q[:, :, 0] * k[:, :, 0]).sum(-1) / math.sqrt(8)
    np.testing.assert_allclose(lse[:, :, 0], s00, rtol=0, atol=1e-14)


def test_equal_keys_give_prefix_mean():
    T, d = 37, 8
    q = _rand((1, 2, T, d), 4)
    k = np.broadcast_to(_rand((1, 2, 1, d), 5), (1, 2, T, d)).copy()
    v = _rand((1, 2, T, d), 6)
    s = (q * k).sum(-1) / math.sqrt(d)  # every key scores the same per row
    o, lse, _ = ora.attention_dense(q, k, v, causal=True)
    prefix_mean = np.cumsum(v, axis=2) / np.arange(1, T + 1)[None, None, :, None]
    np.testing.assert_allclose(o, prefix_mean, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, s + np.log(np.arange(1, T + 1)), rtol=0,
                               atol=1e-13)
    o, lse, _ = ora.attention_dense(q, k, v, causal=False)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(2, keepdims=True), o.shape),
                               rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, s + math.log(T), rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_p_rows_sum_to_one_and_equal_exp_s_minus_lse(causal):
    """Rows of P sum to 1; P_ij = exp(s_ij - L_i) on visible entries
    ('4.2 FlashAttention I', Exercise 5; 'Efficient attention & KV cache',
    exercise 3)."""
    T, d = 23, 16
    q, k, v = _rand((1, 2, T, d), 7), _rand((1, 2, T, d), 8), _rand((1, 2, T, d), 9)
    o, lse, ex = ora.attention_dense(q, k, v, causal=causal, return_p=True)
    p = ex["p"]
    np.testing.assert_allclose(p.sum(-1), 1.0, rtol=0, atol=1e-14)
    s = np.einsum("bhid,bhjd->bhij", q, k) / math.sqrt(d)
    vis = np.tril(np.ones((T, T), bool)) if causal else np.ones((T, T), bool)
    ref = np.where(vis, np.exp(s - lse[..., None]), 0.0)
    np.testing.assert_allclose(p, ref, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(o, np.einsum("bhij,bhjd->bhid", p, v), rtol=0,
                               atol=1e-13)
    assert ex["visible_pairs"] == 2 * (T * (T + 1) // 2 if causal else T * T)


def test_special_case_single_row_matches_scipy_softmax_and_logsumexp():
    """With one query row the method is softmax(s) @ V; scipy supplies both
    the softmax and the log-sum-exp."""
    Tk, d = 50, 12
    q, k, v = _rand((1, 1, 1, d), 10, 3.0), _rand((1, 1, Tk, d), 11), _rand((1, 1, Tk, d), 12)
    s = (k[0, 0] @ q[0, 0, 0]) * 0.37
    o, lse, _ = ora.attention_dense(q, k, v, causal=False, scale=0.37)
    assert abs(lse[0, 0, 0] - scipy.special.logsumexp(s)) < 1e-13
    np.testing.assert_allclose(o[0, 0, 0], scipy.special.softmax(s) @ v[0, 0], rtol=0,
                               atol=1e-14)


def test_online_softmax_1d_matches_scipy():
    """'Efficient attention & KV cache', section 3: online_softmax against the
    library softmax and logsumexp, for chunks that do not divide the length."""
    x = _rand((101,), 13, 5.0)
    for chunk in (1, 4, 7, 101, 200):
        p, lse, _ = ora.online_softmax_1d(x, chunk)
        np.testing.assert_allclose(p, scipy.special.softmax(x), rtol=1e-13, atol=0)
        assert abs(lse - scipy.special.logsumexp(x)) < 1e-13


def test_gqa_head_map_is_consecutive_grouping():
    """Query head h reads K/V head h // (Hq/Hkv): the same as repeating every
    K/V head Hq/Hkv times in place (enable_gqa)."""
    q = _rand((2, 8, 11, 8), 14)
    k, v = _rand((2, 2, 13, 8), 15), _rand((2, 2, 13, 8), 16)
    o, lse, _ = ora.attention_dense(q, k, v, causal=True)
    kr, vr = np.repeat(k, 4, axis=1), np.repeat(v, 4, axis=1)
    o2, lse2, _ = ora.attention_dense(q, kr, vr, causal=True)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, lse2)
    # the other map (h % Hkv) would differ
    kt, vt = np.tile(k, (1, 4, 1, 1)), np.tile(v, (1, 4, 1, 1))
    o3, _, _ = ora.attention_dense(q, kt, vt, causal=True)
    assert np.abs(o3 - o).max() > 1e-3


def test_causal_alignment_is_bottom_right():
    """Query i of Tq sits at key position i + Tk - Tq; with Tq = 1 causal is
    attention over the whole cache."""
    Tq, Tk, d = 3, 7, 4
    q, k, v = _rand((1, 1, Tq, d), 17), _rand((1, 1, Tk, d), 18), _rand((1, 1, Tk, d), 19)
    o, lse, _ = ora.attention_dense(q, k, v, causal=True)
    for i in range(Tq):
        last = i + Tk - Tq
        oi, li, _ = ora.attention_dense(q[:, :, i:i + 1], k[:, :, :last + 1],
                                        v[:, :, :last + 1], causal=False)
        np.testing.assert_allclose(o[:, :, i], oi[:, :, 0], rtol=0, atol=1e-15)
        np.testing.assert_allclose(lse[:, :, i], li[:, :, 0], rtol=0, atol=1e-15)
    o1, l1, _ = ora.attention_dense(q[:, :, :1], k, v, causal=True)
    o0, l0, _ = ora.attention_dense(q[:, :, :1], k, v, causal=False)
    np.testing.assert_array_equal(o1, o0)
    with pytest.raises(ValueError):
        ora.attention_dense(k, q, q, causal=True)  # Tq > Tk under causal


def test_bf16_inputs_are_upcast_exactly():
    rng = np.random.default_rng(20)
    bits = [rng.integers(0x3000, 0x4000, size=(1, 2, 9, 8), dtype=np.uint16) for _ in range(3)]
    bits = [b | (rng.integers(0, 2, size=b.shape, dtype=np.uint16) << 15) for b in bits]
    f64 = [(b.astype(np.uint32) << 16).view(np.float32).astype(np.float64) for b in bits]
    o, lse, _ = ora.attention_dense(*bits, causal=True)
    o2, lse2, _ = ora.attention_dense(*f64, causal=True)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, lse2)


def test_rows_entry_point_matches_dense():
    q, k, v = _rand((2, 4, 19, 8), 21), _rand((2, 2, 23, 8), 22), _rand((2, 2, 23, 8), 23)
    for causal in (False, True):
        o, lse, _ = ora.attention_dense(q, k, v, causal=causal)
        rb, rh, ri = [0, 1, 1, 0, 1], [0, 3, 2, 1, 0], [0, 18, 7, 5, 12]
        orow, lrow = ora.attention_rows(q, k, v, rb, rh, ri, causal=causal)
        np.testing.assert_allclose(orow, o[rb, rh, ri], rtol=0, atol=1e-14)
        np.testing.assert_allclose(lrow, lse[rb, rh, ri], rtol=0, atol=1e-14)


@pytest.mark.parametrize("window", [1, 3, 7, 30])
def test_rows_entry_point_matches_dense_with_a_window(window):
    """The sampled-rows routine under a sliding window equals the dense
    windowed definition on every row (GQA, Tq < Tk, and windows from one key
    to past every row), so tests that check rows instead of whole tensors
    rest on a pinned routine."""
    q, k, v = _rand((2, 4, 19, 8), 31), _rand((2, 2, 23, 8), 32), _rand((2, 2, 23, 8), 33)
    o, lse, _ = ora.attention_dense(q, k, v, causal=True, window=window)
    rb, rh, ri = np.meshgrid(np.arange(2), np.arange(4), np.arange(19), indexing="ij")
    rb, rh, ri = rb.ravel(), rh.ravel(), ri.ravel()
    orow, lrow = ora.attention_rows(q, k, v, rb, rh, ri, causal=True, window=window)
    np.testing.assert_allclose(orow, o[rb, rh, ri], rtol=0, atol=1e-14)
    np.testing.assert_allclose(lrow, lse[rb, rh, ri], rtol=0, atol=1e-14)
    if window == 1:
        # one visible key: the value at the query's position (bottom-right
        # aligned, 23 - 19 = 4 keys ahead) and its single scaled score
        g = rh // 2
        np.testing.assert_array_equal(orow, v[rb, g, ri + 4])
        s = (q[rb, rh, ri] * k[rb, g, ri + 4]).sum(-1) / np.sqrt(8)
        np.testing.assert_allclose(lrow, s, rtol=0, atol=1e-14)


# --- blocked online softmax against dense ------------------------------------

@pytest.mark.parametrize("bq,bk", [(8, 8), (16, 16), (13, 19), (32, 8), (1, 1), (64, 64)])
@pytest.mark.parametrize("causal", [False, True])
def test_blocked_equals_dense_any_tile(bq, bk, causal):
    """Tile pairs from the lab's unit test, (1, 1), and a ragged T = 61."""
    q, k, v = _rand((1, 2, 61, 16), 24), _rand((1, 2, 61, 16), 25), _rand((1, 2, 61, 16), 26)
    o, lse, _ = ora.attention_dense(q, k, v, causal=causal)
    ob, lseb, _ = ora.attention_blocked(q, k, v, bq, bk, causal=causal)
    assert np.abs(ob - o).max() < 1e-12
    assert np.abs(lseb - lse).max() < 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_blocked_random_block_order_with_scores_times_20(causal):
    """'Efficient attention & KV cache', failure modes: scores scaled x20 and
    random block orders must not change the result."""
    T, d, bk = 70, 8, 9
    q, k, v = _rand((1, 3, T, d), 27, 20.0), _rand((1, 3, T, d), 28), _rand((1, 3, T, d), 29)
    o, lse, _ = ora.attention_dense(q, k, v, causal=causal)
    rng = np.random.default_rng(30)
    for _ in range(4):
        order = rng.permutation((T + bk - 1) // bk)
        ob, lseb, _ = ora.attention_blocked(q, k, v, 16, bk, causal=causal,
                                            kv_order=order)
        assert np.abs(ob - o).max() < 1e-12
        assert np.abs(lseb - lse).max() < 1e-11


def test_blocked_gqa_and_tq_lt_tk():
    q = _rand((2, 6, 20, 8), 31)
    k, v = _rand((2, 3, 45, 8), 32), _rand((2, 3, 45, 8), 33)
    for causal in (False, True):
        o, lse, _ = ora.attention_dense(q, k, v, causal=causal)
        ob, lseb, _ = ora.attention_blocked(q, k, v, 7, 10, causal=causal)
        assert np.abs(ob - o).max() < 1e-12
        assert np.abs(lseb - lse).max() < 1e-12


def test_mutation_without_accumulator_rescale_is_caught():
    """The lab's failure-boundary test: emphasise a late key so the running
    max grows on a later tile; dropping the rescale of acc is then wrong by
    more than 0.1 while the correct variant agrees to 1e-12."""
    q, k, v = _lab_qkv(32, 8, 99)
    k[-1] = [4.0] * 8
    q, k, v = _bhtd(q), _bhtd(k), _bhtd(v)
    o, _, _ = ora.attention_dense(q, k, v, causal=True)
    good, _, _ = ora.attention_blocked(q, k, v, 8, 8, causal=True, rescale_acc=True)
    bad, _, _ = ora.attention_blocked(q, k, v, 8, 8, causal=True, rescale_acc=False)
    assert np.abs(good - o).max() < 1e-12
    assert np.abs(bad - o).max() > 0.1


def test_unshifted_softmax_overflows_while_stable_forms_agree():
    """The lab's overflow test: logits near 1414 overflow exp() without the
    max shift; the shifted dense form and the 1x1-blocked form agree."""
    q = _bhtd([[500.0, 500.0], [500.0, 500.0]])
    k = _bhtd([[1.0, 1.0], [2.0, 2.0]])
    v = _bhtd([[1.0, 0.0], [0.0, 1.0]])
    with pytest.raises(ora.OracleOverflow):
        ora.attention_dense(q, k, v, causal=False, subtract_max=False)
    o, lse, _ = ora.attention_dense(q, k, v, causal=False)
    ob, lseb, _ = ora.attention_blocked(q, k, v, 1, 1, causal=False)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    assert np.abs(ob - o).max() < 1e-12


def test_causal_tiles_visited_half_the_grid():
    """Causal skipping visits only blocks at or below the diagonal."""
    q = k = v = _rand((1, 1, 64, 4), 34)
    _, _, visited = ora.attention_blocked(q, k, v, 16, 16, causal=True)
    assert visited == 1 + 2 + 3 + 4
    _, _, visited = ora.attention_blocked(q, k, v, 16, 16, causal=False)
    assert visited == 16


# --- sliding window ("4.2 FlashAttention I", Exercise 4) ---------------------

def test_window_one_sees_only_the_diagonal_key():
    """W = 1: each query sees exactly its own position, so O_i = v_{i+d} and
    LSE_i = s_{i,i+d} with d = Tk - Tq."""
    Tq, Tk, d = 9, 13, 8
    q, k, v = _rand((2, 2, Tq, d), 40), _rand((2, 2, Tk, d), 41), _rand((2, 2, Tk, d), 42)
    o, lse, ex = ora.attention_dense(q, k, v, causal=True, window=1)
    idx = np.arange(Tq) + (Tk - Tq)
    np.testing.assert_allclose(o, v[:, :, idx], rtol=0, atol=1e-15)
    s_diag = (q * k[:, :, idx]).sum(-1) / math.sqrt(d)
    np.testing.assert_allclose(lse, s_diag, rtol=0, atol=1e-14)
    assert ex["visible_pairs"] == 2 * 2 * Tq


def test_window_at_least_tk_is_plain_causal():
    q, k, v = _rand((1, 3, 20, 8), 43), _rand((1, 3, 27, 8), 44), _rand((1, 3, 27, 8), 45)
    o, lse, _ = ora.attention_dense(q, k, v, causal=True)
    for w in (27, 40):
        ow, lw, _ = ora.attention_dense(q, k, v, causal=True, window=w)
        np.testing.assert_array_equal(o, ow)
        np.testing.assert_array_equal(lse, lw)


def test_window_equal_keys_give_windowed_mean():
    T, d, W = 30, 4, 7
    q = _rand((1, 1, T, d), 46)
    k = np.broadcast_to(_rand((1, 1, 1, d), 47), (1, 1, T, d)).copy()
    v = _rand((1, 1, T, d), 48)
    o, _, _ = ora.attention_dense(q, k, v, causal=True, window=W)
    for i in range(T):
        lo = max(0, i - W + 1)
        np.testing.assert_allclose(o[0, 0, i], v[0, 0, lo:i + 1].mean(0), rtol=0, atol=1e-14)


def test_window_exercise_setup_blocked_equals_dense():
    """The exercise's check: N = 100, d = 16, W = 24, 32 x 32 blocks."""
    q, k, v = _rand((1, 1, 100, 16), 7), _rand((1, 1, 100, 16), 8), _rand((1, 1, 100, 16), 9)
    o, lse, ex = ora.attention_dense(q, k, v, causal=True, window=24)
    ob, lseb, visited = ora.attention_blocked(q, k, v, 32, 32, causal=True, window=24)
    assert np.abs(ob - o).max() < 1e-12
    assert np.abs(lseb - lse).max() < 1e-12
    _, _, visited_causal = ora.attention_blocked(q, k, v, 32, 32, causal=True)
    assert visited < visited_causal


@pytest.mark.parametrize("bq,bk", [(8, 8), (13, 19), (32, 8), (1, 1), (16, 64)])
@pytest.mark.parametrize("W", [1, 5, 24, 64])
def test_window_blocked_skips_exactly_the_empty_blocks(bq, bk, W):
    """Blocked with the left-edge skip equals dense, and the blocks it
    visits are exactly those holding at least one visible (row, key) pair
    (found by brute force from the dense probability matrix)."""
    Tq, Tk, d = 45, 61, 8
    q, k, v = _rand((1, 1, Tq, d), 49), _rand((1, 1, Tk, d), 50), _rand((1, 1, Tk, d), 51)
    o, lse, ex = ora.attention_dense(q, k, v, causal=True, window=W, return_p=True)
    ob, lseb, visited = ora.attention_blocked(q, k, v, bq, bk, causal=True, window=W)
    assert np.abs(ob - o).max() < 1e-12
    assert np.abs(lseb - lse).max() < 1e-12
    vis = ex["p"][0, 0] > 0
    nonempty = sum(vis[i0:i0 + bq, j0:j0 + bk].any()
                   for i0 in range(0, Tq, bq) for j0 in range(0, Tk, bk))
    assert visited == nonempty


def test_window_requires_causal():
    q = k = v = _rand((1, 1, 8, 4), 52)
    with pytest.raises(ValueError):
        ora.attention_dense(q, k, v, causal=False, window=3)


# --- paged-KV decode ("Efficient attention & KV cache", section 2.5) -------

def _paginate(k, v, page_size, seed=None):
    """Cut a contiguous cache [B, Hkv, Tk, d] into pages [num_pages, Hkv,
    page_size, d] (sequence b owns pages b*npp .. b*npp + npp - 1, the tail
    of its last page zero) and return (k_pages, v_pages, table).  With a
    seed the physical pages are shuffled and the table follows them."""
    B, Hkv, Tk, d = k.shape
    npp = -(-Tk // page_size)
    pad = npp * page_size - Tk
    kp = np.pad(k, ((0, 0), (0, 0), (0, pad), (0, 0)))
    vp = np.pad(v, ((0, 0), (0, 0), (0, pad), (0, 0)))
    # [B, Hkv, npp, ps, d] -> [B, npp, Hkv, ps, d] -> [B*npp, Hkv, ps, d]
    kp = kp.reshape(B, Hkv, npp, page_size, d).transpose(0, 2, 1, 3, 4).reshape(-1, Hkv, page_size, d)
    vp = vp.reshape(B, Hkv, npp, page_size, d).transpose(0, 2, 1, 3, 4).reshape(-1, Hkv, page_size, d)
    table = np.arange(B * npp, dtype=np.int32).reshape(B, npp)
    if seed is not None:
        perm = np.random.default_rng(seed).permutation(B * npp)
        kp2, vp2 = np.empty_like(kp), np.empty_like(vp)
        kp2[perm], vp2[perm] = kp, vp
        kp, vp, table = kp2, vp2, perm[table].astype(np.int32)
    return np.ascontiguousarray(kp), np.ascontiguousarray(vp), table


@pytest.mark.parametrize("page_size", [1, 4, 16, 7])
def test_paged_decode_identity_table_equals_dense(page_size):
    """Pages laid out in order with full lengths: the result is the dense
    definition on the contiguous cache (GQA group 3, Tk not a multiple of the
    page size)."""
    B, Hq, Hkv, Tk, d = 2, 6, 2, 37, 8
    q, k, v = _rand((B, Hq, 1, d), 60), _rand((B, Hkv, Tk, d), 61), _rand((B, Hkv, Tk, d), 62)
    o, lse, _ = ora.attention_dense(q, k, v, causal=False)
    kp, vp, table = _paginate(k, v, page_size)
    op, lp = ora.attention_paged_decode(q[:, :, 0], kp, vp, table, np.full(B, Tk))
    np.testing.assert_allclose(op, o[:, :, 0], rtol=0, atol=1e-14)
    np.testing.assert_allclose(lp, lse[:, :, 0], rtol=0, atol=1e-14)


def test_paged_decode_shuffled_pages_change_nothing():
    """Moving physical pages and updating the table is invisible."""
    B, Hq, Hkv, Tk, d = 3, 4, 4, 50, 16
    q, k, v = _rand((B, Hq, 1, d), 63), _rand((B, Hkv, Tk, d), 64), _rand((B, Hkv, Tk, d), 65)
    lens = np.array([50, 17, 1])
    a = ora.attention_paged_decode(q[:, :, 0], *_paginate(k, v, 8), lens)
    b = ora.attention_paged_decode(q[:, :, 0], *_paginate(k, v, 8, seed=5), lens)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_paged_decode_ragged_lengths_read_only_their_keys():
    """Sequence b sees exactly its first seq_lens[b] keys: every slot past
    them (the rest of the last page, whole unused pages) holds NaN and the
    result equals the dense definition on the truncated cache."""
    B, Hq, Hkv, Tk, d, ps = 4, 4, 2, 40, 8, 16
    q, k, v = _rand((B, Hq, 1, d), 66), _rand((B, Hkv, Tk, d), 67), _rand((B, Hkv, Tk, d), 68)
    lens = np.array([40, 33, 16, 5])
    kn, vn = k.copy(), v.copy()
    for b, n in enumerate(lens):
        kn[b, :, n:] = np.nan
        vn[b, :, n:] = np.nan
    kp, vp, table = _paginate(kn, vn, ps, seed=9)
    op, lp = ora.attention_paged_decode(q[:, :, 0], kp, vp, table, lens)
    assert np.isfinite(op).all() and np.isfinite(lp).all()
    for b, n in enumerate(lens):
        o, lse, _ = ora.attention_dense(q[b:b + 1], k[b:b + 1, :, :n], v[b:b + 1, :, :n])
        np.testing.assert_allclose(op[b], o[0, :, 0], rtol=0, atol=1e-14)
        np.testing.assert_allclose(lp[b], lse[0, :, 0], rtol=0, atol=1e-14)


def test_paged_decode_single_key_and_shared_prefix():
    """seq_len 1: O is that key's value row and LSE its scaled score.  Two
    sequences whose tables point at the same pages (a shared prefix) with
    the same query give identical rows."""
    Hq = Hkv = 2
    d, ps = 8, 4
    kp, vp = _rand((3, Hkv, ps, d), 69), _rand((3, Hkv, ps, d), 70)
    q = _rand((2, Hq, d), 71)
    q[1] = q[0]
    table = np.array([[2, 0], [2, 0]], dtype=np.int32)
    o, lse = ora.attention_paged_decode(q, kp, vp, table, np.array([1, 1]))
    for h in range(Hq):
        np.testing.assert_array_equal(o[0, h], vp[2, h, 0])
        np.testing.assert_allclose(lse[0, h], q[0, h] @ kp[2, h, 0] / math.sqrt(d), rtol=0, atol=1e-15)
    o, lse = ora.attention_paged_decode(q, kp, vp, table, np.array([6, 6]))
    np.testing.assert_array_equal(o[0], o[1])
    np.testing.assert_array_equal(lse[0], lse[1])


def test_paged_decode_bf16_inputs_match_the_upcast_f64_inputs():
    rng = np.random.default_rng(72)
    bits = lambda shape: rng.integers(0x3c00, 0x4000, size=shape, dtype=np.uint16) ^ (
        rng.integers(0, 2, size=shape, dtype=np.uint16) << 15)
    qb, kb, vb = bits((2, 4, 32)), bits((5, 2, 16, 32)), bits((5, 2, 16, 32))
    up = lambda x: (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    table = np.array([[4, 1, 0], [3, 2, 0]], dtype=np.int32)
    lens = np.array([40, 20])
    a = ora.attention_paged_decode(qb, kb, vb, table, lens)
    b = ora.attention_paged_decode(up(qb), up(kb), up(vb), table, lens)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


@pytest.mark.parametrize("lens,table_fix", [([0], None), ([9], None), ([3], -1), ([3], 2)])
def test_paged_decode_rejects_bad_lengths_and_pages(lens, table_fix):
    q, kp, vp = _rand((1, 1, 4), 73), _rand((2, 1, 4, 4), 74), _rand((2, 1, 4, 4), 75)
    table = np.array([[0, 1]], dtype=np.int32)
    if table_fix is not None:
        table[0, 0] = table_fix
    with pytest.raises(ValueError):
        ora.attention_paged_decode(q, kp, vp, table, np.array(lens))


# --- packed variable-length batches ("SDPA and FlashAttention's tiling",
# flash_attn_varlen_func with cu_seqlens) ---------------------------------

def _pack(xs):
    """List of [H, T_b, d] arrays -> packed [sum T_b, H, d] and offsets."""
    cu = np.concatenate([[0], np.cumsum([x.shape[1] for x in xs])]).astype(np.int32)
    return np.concatenate([x.transpose(1, 0, 2) for x in xs], axis=0), cu


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_each_sequence_is_its_own_dense_problem(causal):
    """Every sequence of the pack equals the dense definition run on that
    sequence alone (GQA 3, Tq < Tk per sequence, ragged lengths, an empty
    query sequence)."""
    Hq, Hkv, d = 6, 2, 8
    lq, lk = [5, 0, 17, 1], [9, 4, 17, 3]
    qs = [_rand((Hq, n, d), 80 + i) for i, n in enumerate(lq)]
    ks = [_rand((Hkv, n, d), 90 + i) for i, n in enumerate(lk)]
    vs = [_rand((Hkv, n, d), 100 + i) for i, n in enumerate(lk)]
    (q, cq), (k, ck), (v, _) = _pack(qs), _pack(ks), _pack(vs)
    o, lse = ora.attention_varlen(q, k, v, cq, ck, causal=causal)
    for b in range(len(lq)):
        if lq[b] == 0:
            continue
        od, ld, _ = ora.attention_dense(qs[b][None], ks[b][None], vs[b][None], causal=causal)
        np.testing.assert_allclose(o[cq[b]:cq[b + 1]], od[0].transpose(1, 0, 2), rtol=0, atol=1e-14)
        np.testing.assert_allclose(lse[:, cq[b]:cq[b + 1]], ld[0], rtol=0, atol=1e-14)


def test_varlen_no_score_crosses_documents():
    """Changing one document's keys and values leaves every other document's
    rows bit-identical (nothing attends across the pack)."""
    lens = [7, 12, 3]
    H, d = 2, 4
    q, cu = _pack([_rand((H, n, d), 110 + i) for i, n in enumerate(lens)])
    k, _ = _pack([_rand((H, n, d), 120 + i) for i, n in enumerate(lens)])
    v, _ = _pack([_rand((H, n, d), 130 + i) for i, n in enumerate(lens)])
    o, lse = ora.attention_varlen(q, k, v, cu, cu, causal=True)
    k2, v2 = k.copy(), v.copy()
    k2[cu[1]:cu[2]] *= -3.0
    v2[cu[1]:cu[2]] += 5.0
    o2, lse2 = ora.attention_varlen(q, k2, v2, cu, cu, causal=True)
    for b in (0, 2):
        sl = slice(cu[b], cu[b + 1])
        np.testing.assert_array_equal(o[sl], o2[sl])
        np.testing.assert_array_equal(lse[:, sl], lse2[:, sl])
    assert np.abs(o[cu[1]:cu[2]] - o2[cu[1]:cu[2]]).max() > 0.1


def test_varlen_equal_lengths_is_the_batched_dense_problem():
    B, H, T, d = 3, 4, 11, 8
    q4, k4, v4 = _rand((B, H, T, d), 140), _rand((B, H, T, d), 141), _rand((B, H, T, d), 142)
    od, ld, _ = ora.attention_dense(q4, k4, v4, causal=True)
    pk = lambda x: x.transpose(0, 2, 1, 3).reshape(B * T, H, d)
    cu = np.arange(0, B * T + 1, T, dtype=np.int32)
    o, lse = ora.attention_varlen(pk(q4), pk(k4), pk(v4), cu, cu, causal=True)
    np.testing.assert_allclose(o, pk(od), rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, ld.transpose(1, 0, 2).reshape(H, B * T), rtol=0, atol=1e-14)


@pytest.mark.parametrize("cq,ck,causal", [
    ([1, 3], [0, 3], False),      # must start at 0
    ([0, 3, 2], [0, 3, 5], False),  # decreasing
    ([0, 3], [0, 0], False),      # queries without keys
    ([0, 4], [0, 3], True),       # causal with more queries than keys
    ([0, 9], [0, 3], False),      # past total_q
])
def test_varlen_rejects_bad_offsets(cq, ck, causal):
    q, k = _rand((8, 1, 4), 150), _rand((5, 1, 4), 151)
    with pytest.raises(ValueError):
        ora.attention_varlen(q, k, k, cq, ck, causal=causal)


# --- backward ("4.2 FlashAttention I", "The backward pass: recomputation
# instead of storage") -----------------------------------------------------

def _fd_grad(f, x, idx, eps=1e-6):
    """Central difference of the scalar f at x[idx]."""
    xp, xm = x.copy(), x.copy()
    xp[idx] += eps
    xm[idx] -= eps
    return (f(xp) - f(xm)) / (2 * eps)


@pytest.mark.parametrize("causal,Tq,Tk,Hq,Hkv", [
    (True, 9, 9, 2, 2), (True, 7, 12, 4, 2), (False, 6, 10, 3, 1)])
def test_backward_matches_finite_differences(causal, Tq, Tk, Hq, Hkv):
    """The page's own check: the gradients of sum(dO * O) agree with central
    differences of the forward definition, coordinate by coordinate (every
    entry of a small problem, GQA and Tq < Tk included)."""
    B, d = 1, 4
    q, k, v = _rand((B, Hq, Tq, d), 160), _rand((B, Hkv, Tk, d), 161), _rand((B, Hkv, Tk, d), 162)
    do = _rand((B, Hq, Tq, d), 163)
    dq, dk, dv, o, lse = ora.attention_backward(q, k, v, do, causal=causal)
    o_fwd, lse_fwd, _ = ora.attention_dense(q, k, v, causal=causal)
    np.testing.assert_allclose(o, o_fwd, rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, lse_fwd, rtol=0, atol=1e-14)
    loss = lambda qq, kk, vv: float((do * ora.attention_dense(qq, kk, vv, causal=causal)[0]).sum())
    for idx in np.ndindex(q.shape):
        assert abs(_fd_grad(lambda x: loss(x, k, v), q, idx) - dq[idx]) < 1e-7
    for idx in np.ndindex(k.shape):
        assert abs(_fd_grad(lambda x: loss(q, x, v), k, idx) - dk[idx]) < 1e-7
        assert abs(_fd_grad(lambda x: loss(q, k, x), v, idx) - dv[idx]) < 1e-7


def test_backward_matches_torch_autograd():
    """Special case that reduces to a library routine: torch's float64
    autograd through softmax(scale Q K^T + mask) V, with K/V repeated per
    query head (GQA) and the bottom-right causal mask built explicitly."""
    torch = pytest.importorskip("torch")
    B, Hq, Hkv, Tq, Tk, d = 2, 4, 2, 11, 15, 8
    q, k, v = _rand((B, Hq, Tq, d), 164), _rand((B, Hkv, Tk, d), 165), _rand((B, Hkv, Tk, d), 166)
    do = _rand((B, Hq, Tq, d), 167)
    dq, dk, dv, _, _ = ora.attention_backward(q, k, v, do, causal=True)
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    kk = tk.repeat_interleave(Hq // Hkv, dim=1)
    vv = tv.repeat_interleave(Hq // Hkv, dim=1)
    mask = torch.tril(torch.ones(Tq, Tk, dtype=torch.bool), diagonal=Tk - Tq)
    s = (tq @ kk.transpose(-1, -2)) / math.sqrt(d)
    out = torch.softmax(s.masked_fill(~mask, float("-inf")), dim=-1) @ vv
    out.backward(torch.tensor(do))
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("bq,bk", [(16, 16), (5, 7), (1, 1), (32, 8), (64, 64)])
@pytest.mark.parametrize("causal", [False, True])
def test_backward_blocked_recomputation_equals_dense(bq, bk, causal):
    """The page's algorithm (P rebuilt per tile from the saved L, dK/dV
    accumulated over query blocks) equals the dense definition."""
    B, Hq, Hkv, Tq, Tk, d = 1, 4, 2, 29, 37, 8
    q, k, v = _rand((B, Hq, Tq, d), 168), _rand((B, Hkv, Tk, d), 169), _rand((B, Hkv, Tk, d), 170)
    do = _rand((B, Hq, Tq, d), 171)
    dq, dk, dv, o, lse = ora.attention_backward(q, k, v, do, causal=causal)
    bq_, bk_, bv_ = ora.attention_backward_blocked(q, k, v, do, o, lse, bq, bk, causal=causal)
    for a, b in ((dq, bq_), (dk, bk_), (dv, bv_)):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


def test_backward_invariants():
    """Rows of dS sum to zero (the softmax Jacobian annihilates constants),
    so the dK rows of a head sum to zero; the dV rows sum to the dO rows
    (P rows sum to one); and with one visible key per row (causal row 0)
    dQ vanishes."""
    B, Hq, Hkv, T, d = 2, 6, 3, 13, 8
    q, k, v = _rand((B, Hq, T, d), 172), _rand((B, Hkv, T, d), 173), _rand((B, Hkv, T, d), 174)
    do = _rand((B, Hq, T, d), 175)
    for causal in (False, True):
        dq, dk, dv, _, _ = ora.attention_backward(q, k, v, do, causal=causal)
        np.testing.assert_allclose(dk.sum(axis=2), 0.0, atol=1e-12)
        want = do.reshape(B, Hkv, Hq // Hkv, T, d).sum(axis=(2, 3))
        np.testing.assert_allclose(dv.sum(axis=2), want, rtol=0, atol=1e-12)
        if causal:
            np.testing.assert_allclose(dq[:, :, 0], 0.0, atol=1e-15)


def test_backward_bf16_inputs_match_the_upcast_f64_inputs():
    rng = np.random.default_rng(176)
    bits = lambda shape: rng.integers(0x3c00, 0x4000, size=shape, dtype=np.uint16) ^ (
        rng.integers(0, 2, size=shape, dtype=np.uint16) << 15)
    up = lambda x: (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    q, k, v, do = bits((1, 2, 9, 16)), bits((1, 2, 9, 16)), bits((1, 2, 9, 16)), bits((1, 2, 9, 16))
    a = ora.attention_backward(q, k, v, do, causal=True)
    b = ora.attention_backward(up(q), up(k), up(v), up(do), causal=True)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


# --- backward under the sliding window ("4.2 FlashAttention I", Exercise 4:
# query i sees keys i - W < j <= i; the backward inherits the forward's mask)

@pytest.mark.parametrize("Tq,Tk,Hq,Hkv,window", [(9, 9, 2, 2, 3), (7, 12, 4, 2, 4), (6, 6, 1, 1, 1)])
def test_window_backward_matches_finite_differences(Tq, Tk, Hq, Hkv, window):
    """Central differences of sum(dO * O) through the windowed forward
    definition, every coordinate of a small problem (GQA and Tq < Tk
    included)."""
    B, d = 1, 4
    q, k, v = _rand((B, Hq, Tq, d), 180), _rand((B, Hkv, Tk, d), 181), _rand((B, Hkv, Tk, d), 182)
    do = _rand((B, Hq, Tq, d), 183)
    dq, dk, dv, o, lse = ora.attention_backward(q, k, v, do, causal=True, window=window)
    o_fwd, lse_fwd, _ = ora.attention_dense(q, k, v, causal=True, window=window)
    np.testing.assert_allclose(o, o_fwd, rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, lse_fwd, rtol=0, atol=1e-14)
    loss = lambda qq, kk, vv: float(
        (do * ora.attention_dense(qq, kk, vv, causal=True, window=window)[0]).sum())
    for idx in np.ndindex(q.shape):
        assert abs(_fd_grad(lambda x: loss(x, k, v), q, idx) - dq[idx]) < 1e-7
    for idx in np.ndindex(k.shape):
        assert abs(_fd_grad(lambda x: loss(q, x, v), k, idx) - dk[idx]) < 1e-7
        assert abs(_fd_grad(lambda x: loss(q, k, x), v, idx) - dv[idx]) < 1e-7


def test_window_backward_reduces_to_causal_and_to_the_diagonal():
    """A window of at least Tk keys is the causal mask (identical results);
    a window of one key leaves each query only the key at its own position,
    so O_i = V_{i+Tk-Tq}, P is that one-hot row, dS = P (dO.V - dO.O) = 0
    (dQ = dK = 0) and dV_j sums dO over the query rows (and query heads) at
    position j."""
    B, Hq, Hkv, Tq, Tk, d = 2, 4, 2, 7, 11, 8
    q, k, v = _rand((B, Hq, Tq, d), 184), _rand((B, Hkv, Tk, d), 185), _rand((B, Hkv, Tk, d), 186)
    do = _rand((B, Hq, Tq, d), 187)
    full = ora.attention_backward(q, k, v, do, causal=True)
    wide = ora.attention_backward(q, k, v, do, causal=True, window=Tk)
    for a, b in zip(full, wide):
        np.testing.assert_array_equal(a, b)
    dq, dk, dv, o, _ = ora.attention_backward(q, k, v, do, causal=True, window=1)
    delta, G = Tk - Tq, Hq // Hkv
    np.testing.assert_allclose(o, np.repeat(v, G, axis=1)[:, :, delta:], rtol=0, atol=1e-15)
    np.testing.assert_allclose(dq, 0.0, atol=1e-15)
    np.testing.assert_allclose(dk, 0.0, atol=1e-15)
    want = np.zeros_like(dv)
    want[:, :, delta:] = do.reshape(B, Hkv, G, Tq, d).sum(axis=2)
    np.testing.assert_allclose(dv, want, rtol=0, atol=1e-15)


def test_window_backward_rejects_a_window_without_causal():
    q = _rand((1, 1, 4, 4), 188)
    with pytest.raises(ValueError):
        ora.attention_backward(q, q, q, q, causal=False, window=2)


@pytest.mark.parametrize("window", [1, 3, 6, 40])
def test_varlen_window_is_the_dense_window_per_sequence(window):
    """With a sliding window each sequence of the pack equals the dense
    windowed definition on that sequence alone (the window counted inside
    the sequence, bottom-right aligned; W past every length is causal)."""
    Hq, Hkv, d = 4, 2, 8
    lq, lk = [5, 0, 17, 1, 9], [9, 4, 17, 3, 9]
    qs = [_rand((Hq, n, d), 200 + i) for i, n in enumerate(lq)]
    ks = [_rand((Hkv, n, d), 210 + i) for i, n in enumerate(lk)]
    vs = [_rand((Hkv, n, d), 220 + i) for i, n in enumerate(lk)]
    (q, cq), (k, ck), (v, _) = _pack(qs), _pack(ks), _pack(vs)
    o, lse = ora.attention_varlen(q, k, v, cq, ck, causal=True, window=window)
    for b in range(len(lq)):
        if lq[b] == 0:
            continue
        od, ld, _ = ora.attention_dense(qs[b][None], ks[b][None], vs[b][None], causal=True,
                                        window=window)
        np.testing.assert_allclose(o[cq[b]:cq[b + 1]], od[0].transpose(1, 0, 2), rtol=0, atol=1e-14)
        np.testing.assert_allclose(lse[:, cq[b]:cq[b + 1]], ld[0], rtol=0, atol=1e-14)
    if window == 40:
        oc, lc = ora.attention_varlen(q, k, v, cq, ck, causal=True)
        rows = ~np.isnan(oc[:, 0, 0])
        np.testing.assert_array_equal(o[rows], oc[rows])


def test_varlen_window_one_key_copies_the_value_at_each_position():
    """W = 1: every query sees only the key at its own position, so O is that
    value row and LSE the single scaled score (closed form)."""
    H, d = 2, 4
    lens = [3, 7]
    q, cu = _pack([_rand((H, n, d), 230 + i) for i, n in enumerate(lens)])
    k, _ = _pack([_rand((H, n, d), 232 + i) for i, n in enumerate(lens)])
    v, _ = _pack([_rand((H, n, d), 234 + i) for i, n in enumerate(lens)])
    o, lse = ora.attention_varlen(q, k, v, cu, cu, causal=True, window=1, scale=0.5)
    np.testing.assert_allclose(o, v, rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse, 0.5 * (q * k).sum(axis=2).T, rtol=0, atol=1e-14)


def test_varlen_window_requires_causal():
    q, cu = _pack([_rand((1, 4, 4), 236)])
    with pytest.raises(ValueError):
        ora.attention_varlen(q, q, q, cu, cu, causal=False, window=2)
