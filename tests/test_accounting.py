"""Pins for the work/traffic accounting the benchmark divides by."""
import json
import os

from online_softmax_03_gb300 import accounting as acc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_logical_access_model_matches_recorded_sweep():
    """'Explain tiled attention and verify its output', recorded
    hbm_traffic_sweep (MB = 1e6 bytes, two decimals)."""
    with open(os.path.join(GOLDEN, "p2_hbm_sweep.json")) as f:
        gold = json.load(f)
    for row in gold["rows"]:
        m = acc.logical_access_model(row["seq_len"], 32, 128, 2, 128)
        assert round(m["qkvo_bytes"] / 1e6, 2) == row["standard_qkv_o_mb"]
        assert round(m["standard_nxn_bytes"] / 1e6, 2) == row["standard_nxn_matrix_hbm_mb"]
        assert round(m["standard_total_bytes"] / 1e6, 2) == row["standard_total_hbm_mb"]
        assert (round(m["tiled_causal_bytes"] / 1e6, 2)
                == row["tiled_logical_access_mb_no_cache_reuse"])
        assert m["num_q_blocks"] == row["num_q_blocks"]


def test_flops_and_intensity():
    """'Attention from scratch + roofline': 4*B*H*T*T*D FLOPs over Q+K+V+O
    bytes; intensity doubles with T; decode stays memory-bound."""
    def ai(T):
        return acc.attention_flops(1, 32, T, T, 128, False) / (2 * 32 * 128 * 4 * T)
    assert 1.8 <= ai(2048) / ai(1024) <= 2.2
    assert acc.attention_flops(4, 32, 4096, 4096, 128, True) == 4 * 32 * 4096 * 4096 * 128 * 2
    assert acc.decode_bytes(64, 32, 8, 8192, 128) == 2147483648 + 2 * 64 * 32 * 128 * 2 + 64 * 32 * 4
    # GQA decode: 4 query heads share each K/V head, AI about 4 FLOP/byte
    ai_dec = acc.decode_flops(64, 32, 8192, 128) / acc.decode_bytes(64, 32, 8, 8192, 128)
    assert 3.9 < ai_dec < 4.1


def test_visible_pairs_and_window_flops():
    """Pair counts match brute force over the mask definition, and the
    window count has the closed form W(W+1)/2 + (T-W)W for Tq = Tk = T >= W."""
    import numpy as np

    for Tq, Tk, W in ((5, 5, 0), (7, 11, 0), (7, 11, 3), (16, 16, 4), (9, 9, 20)):
        i = np.arange(Tq)[:, None] + (Tk - Tq)
        j = np.arange(Tk)[None, :]
        mask = j <= i
        if W:
            mask &= j > i - W
        assert acc.visible_pairs(Tq, Tk, True, W) == int(mask.sum())
    T, W = 8192, 1024
    assert acc.visible_pairs(T, T, True, W) == W * (W + 1) // 2 + (T - W) * W
    assert acc.window_flops(4, 32, T, T, 128, W) == 4.0 * 128 * 4 * 32 * acc.visible_pairs(T, T, True, W)
    assert acc.visible_pairs(6, 9, False) == 54


def test_paged_decode_bytes():
    """Full-length sequences cost the contiguous decode bytes plus one 4-byte
    table entry per page and one length per sequence."""
    base = acc.decode_bytes(64, 32, 8, 8192, 128)
    assert acc.paged_decode_bytes(64, 32, 8, [8192] * 64, 128, 16) == base + 64 * 512 * 4 + 64 * 4
    # ragged: K/V bytes follow the lengths, pages round up
    assert acc.paged_decode_bytes(2, 4, 2, [1, 17], 64, 16) == (
        2 * 2 * 18 * 64 * 2 + (1 + 2) * 4 + 2 * 4 + 2 * 2 * 4 * 64 * 2 + 2 * 4 * 4)


def test_varlen_flops_counts_each_document_alone():
    lq, lk = [5, 0, 17, 1], [9, 4, 17, 3]
    for causal in (False, True):
        want = sum(acc.visible_pairs(a, b, causal) for a, b in zip(lq, lk) if a) * 4.0 * 8 * 6
        assert acc.varlen_flops(lq, lk, 6, 8, causal) == want
    # one document of T tokens is the dense causal count, T(T+1)/2 pairs
    assert acc.varlen_flops([4096], [4096], 32, 128, True) == 4.0 * 128 * 32 * 4096 * 4097 // 2


def test_backward_flops_are_five_products():
    assert acc.backward_flops(4, 32, 4096, 4096, 128, True) == 2.5 * acc.attention_flops(
        4, 32, 4096, 4096, 128, True)
    assert acc.backward_flops(1, 1, 3, 5, 2, False) == 5 * 2 * 3 * 5 * 2


def test_backward_dq_reduction_bytes():
    # square causal case: key tile j visits the n - j query tiles from its own
    # diagonal on, n (n + 1) / 2 pairs of 128 x 128 rows x columns; for the
    # bench shape this is 4,429,185,024 bytes (ncu counted 138,412,032
    # 32-byte reduction sectors per backward launch, the same bytes)
    n = 4096 // 128
    assert acc.backward_dq_reduction_bytes(4, 32, 4096, 4096, 128, True) == \
        4 * 32 * (n * (n + 1) // 2) * 128 * 128 * 4 == 138412032 * 32
    # non-causal: every key tile adds a partial for every query row
    assert acc.backward_dq_reduction_bytes(2, 3, 200, 300, 64, False) == 2 * 3 * 3 * 200 * 64 * 4
    # causal with more keys than queries: Tq = 130 (query tiles of 128 and 2
    # rows), Tk = 300 (delta 170); the first query to see key tile 2 (keys
    # 256..299) is row 86, in tile 0, so all three key tiles visit all 130 rows
    assert acc.backward_dq_reduction_bytes(1, 1, 130, 300, 32, True) == 3 * 130 * 32 * 4


def test_backward_dq_reduction_bytes_under_a_window():
    # a window of at least Tk keys is the causal count
    assert acc.backward_dq_reduction_bytes(2, 4, 1000, 1000, 64, True, window=1000) == \
        acc.backward_dq_reduction_bytes(2, 4, 1000, 1000, 64, True)
    # T = 8192, W = 1024: key tile j (keys 128j .. 128j+127) is seen by queries
    # 128j .. 128j+126+1024, i.e. query tiles j .. j+8 (9 tiles), clipped at the
    # last of the 64 tiles; every tile is a full 128 rows
    steps = sum(min(64, j + 9) - j for j in range(64))
    assert steps == 64 * 9 - 36
    assert acc.backward_dq_reduction_bytes(4, 32, 8192, 8192, 128, True, window=1024) == \
        4 * 32 * steps * 128 * 128 * 4
    # W = 1: each key tile reaches only its own query tile
    assert acc.backward_dq_reduction_bytes(1, 1, 256, 256, 32, True, window=1) == 2 * 128 * 32 * 4
