"""Packed variable-length forward on the GPU (attn_fwd_varlen through the C
ABI) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import synth
from oracle import oracle as ora
from online_softmax_03_gb300 import binding
from parity import assert_close

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from online_softmax_03_gb300 import build as cuda_build

    cuda_build.build()
    binding.load_library()
    assert binding.attn_device_status() == binding.ATTN_OK
    yield
    assert binding.attn_device_status() == binding.ATTN_OK


def _oracle(q, k, v, cq, ck, causal, scale=None):
    return ora.attention_varlen(synth.bf16_bits(q), synth.bf16_bits(k), synth.bf16_bits(v),
                                cq.cpu().numpy(), ck.cpu().numpy(), causal=causal, scale=scale)


def _rows(cu):
    """Row ranges of the sequences as one index array."""
    c = cu.cpu().numpy()
    return np.concatenate([np.arange(c[b], c[b + 1]) for b in range(len(c) - 1)])


@pytest.mark.parametrize("lens_q,lens_k,Hq,Hkv,d,causal", [
    ((100, 1, 300, 257), (100, 1, 300, 257), 4, 4, 128, True),
    ((5, 0, 700), (9, 4, 700), 8, 2, 64, True),        # Tq < Tk, an empty sequence
    ((1000, 37, 1), (1000, 50, 3000), 6, 2, 128, False),
    ((128, 256, 384), (128, 256, 384), 2, 1, 32, True),  # whole tiles, GQA 2
    ((513, 255, 2), (513, 255, 2), 3, 3, 64, False),
    ((1, 1, 1, 1, 1), (1, 2, 3, 4, 130), 8, 8, 128, True),
])
def test_varlen_against_oracle(lens_q, lens_k, Hq, Hkv, d, causal):
    q, k, v, cq, ck = synth.make_varlen_inputs(lens_q, lens_k, Hq, Hkv, d,
                                               seed=sum(lens_q) + d, device=DEV)
    o, lse = binding.fwd_varlen(q, k, v, cq, ck, max(lens_q), max(lens_k), causal=causal)
    torch.cuda.synchronize()
    o_ref, lse_ref = _oracle(q, k, v, cq, ck, causal)
    r = _rows(cq)
    assert_close(o[r], lse[:, r], o_ref[r], lse_ref[:, r], f"varlen {lens_q}/{lens_k}")


def test_varlen_single_sequence_matches_attn_fwd_bit_for_bit():
    """One sequence of the pack is the padded-free [1, H, T, d] problem: the
    same tiles, products and softmax, so the same bits as attn_fwd."""
    w = synth.Workload("vl_single", 1, 16, 4, 1500, 2000, 128, True, "normal", 40)
    q4, k4, v4 = synth.make_inputs(w, DEV)
    o4, l4 = binding.fwd(q4, k4, v4, causal=True)
    tok = lambda x: x[0].transpose(0, 1).contiguous()
    cq = torch.tensor([0, w.Tq], dtype=torch.int32, device=DEV)
    ck = torch.tensor([0, w.Tk], dtype=torch.int32, device=DEV)
    o, lse = binding.fwd_varlen(tok(q4), tok(k4), tok(v4), cq, ck, w.Tq, w.Tk, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o, tok(o4)) and torch.equal(lse, l4[0])


def test_varlen_documents_do_not_see_each_other():
    """Scaling another document's keys and values leaves a document's rows
    bit-identical, although its last K/V tile reads the neighbour's rows."""
    lens = (200, 300, 100)
    q, k, v, cq, ck = synth.make_varlen_inputs(lens, lens, 4, 2, 64, seed=41, device=DEV)
    o1, l1 = binding.fwd_varlen(q, k, v, cq, ck, 300, 300, causal=True)
    k2, v2 = k.clone(), v.clone()
    k2[200:500] *= -4
    v2[200:500] *= 8
    o2, l2 = binding.fwd_varlen(q, k2, v2, cq, ck, 300, 300, causal=True)
    torch.cuda.synchronize()
    for a, b in ((0, 200), (500, 600)):
        assert torch.equal(o1[a:b], o2[a:b]) and torch.equal(l1[:, a:b], l2[:, a:b])
    assert not torch.equal(o1[200:500], o2[200:500])


def test_varlen_rows_outside_sequences_are_not_written():
    lens = (70, 130)
    q, k, v, cq, ck = synth.make_varlen_inputs(lens, lens, 4, 4, 128, seed=42, device=DEV,
                                               pad_q=50, pad_k=20)
    o = torch.full_like(q, 7.0)
    lse = torch.full((4, q.shape[0]), 7.0, dtype=torch.float32, device=DEV)
    binding.fwd_varlen(q, k, v, cq, ck, 130, 130, causal=False, out=o, lse=lse)
    torch.cuda.synchronize()
    assert (o[200:] == 7.0).all() and (lse[:, 200:] == 7.0).all()
    o_ref, lse_ref = _oracle(q, k, v, cq, ck, False)
    assert_close(o[:200], lse[:, :200], o_ref[:200], lse_ref[:, :200], "varlen padded")


def test_varlen_packed_documents_sampled_rows():
    """The benchmarked packed batch (65,536 tokens of documents of 64 to 8192
    tokens, H=32, d=128, causal): sampled rows of sampled documents against
    the dense oracle on each document alone."""
    w = synth.VARLEN
    lens = synth.packed_lengths(synth.VARLEN_TOKENS, w.seed)
    q, k, v, cq, ck = synth.make_varlen_inputs(lens, lens, w.Hq, w.Hkv, w.d, w.seed, DEV)
    o, lse = binding.fwd_varlen(q, k, v, cq, ck, max(lens), max(lens), causal=True,
                                scale=w.scale)
    torch.cuda.synchronize()
    c = cq.cpu().numpy()
    docs = sorted({0, len(lens) - 1, int(np.argmax(lens)), 5, 11})
    g = np.random.default_rng(43)
    for b in docs:
        n = lens[b]
        sl = slice(int(c[b]), int(c[b + 1]))
        doc = lambda x: x[sl].transpose(0, 1).contiguous()[None]
        ri = np.unique(np.concatenate([[0, n - 1], g.integers(0, n, 24)]))
        rh = g.integers(0, w.Hq, ri.size)
        rb = np.zeros_like(ri)
        o_ref, lse_ref = ora.attention_rows(synth.bf16_bits(doc(q)), synth.bf16_bits(doc(k)),
                                            synth.bf16_bits(doc(v)), rb, rh, ri, causal=True,
                                            scale=w.scale)
        rows = torch.as_tensor(c[b] + ri, device=DEV)
        heads = torch.as_tensor(rh, device=DEV)
        assert_close(o[rows, heads], lse[heads, rows], o_ref, lse_ref, f"doc {b} (len {n})")


@pytest.mark.parametrize("cq_list,ck_list,causal", [
    ([0, 50, 40], [0, 50, 90], False),     # decreasing query offsets
    ([0, 60, 100], [0, 50, 100], True),    # causal, more queries than keys
    ([1, 50, 100], [0, 50, 100], False),   # does not start at 0
    ([0, 50, 100], [0, 0, 100], False),    # queries without keys
])
def test_varlen_bad_device_offsets_are_reported_and_nothing_is_written(cq_list, ck_list,
                                                                        causal):
    q, k, v, _, _ = synth.make_varlen_inputs((100,), (100,), 4, 4, 64, seed=44, device=DEV)
    cq = torch.tensor(cq_list, dtype=torch.int32, device=DEV)
    ck = torch.tensor(ck_list, dtype=torch.int32, device=DEV)
    o = torch.full_like(q, 3.0)
    lse = torch.full((4, 100), 3.0, dtype=torch.float32, device=DEV)
    binding.fwd_varlen(q, k, v, cq, ck, 100, 100, causal=causal, out=o, lse=lse)
    torch.cuda.synchronize()
    assert binding.attn_device_status() == binding.ATTN_ERR_INVALID_ARG
    assert (o == 3.0).all() and (lse == 3.0).all()


# --- sliding window inside each sequence (attn_fwd_varlen_window)

@pytest.mark.parametrize("lens_q,lens_k,Hq,Hkv,d,window", [
    ((100, 1, 300, 257), (100, 1, 300, 257), 4, 4, 128, 64),
    ((5, 0, 700), (9, 4, 700), 8, 2, 64, 129),          # Tq < Tk, an empty sequence
    ((128, 256, 384), (128, 256, 384), 2, 1, 32, 1),    # one key per query
    ((513, 255, 2), (513, 255, 2), 3, 3, 64, 300),
    ((1000, 37, 1), (1000, 50, 3000), 6, 2, 128, 5000),  # window past every length: causal
])
def test_varlen_window_against_oracle(lens_q, lens_k, Hq, Hkv, d, window):
    q, k, v, cq, ck = synth.make_varlen_inputs(lens_q, lens_k, Hq, Hkv, d,
                                               seed=sum(lens_q) + window, device=DEV)
    o, lse = binding.fwd_varlen(q, k, v, cq, ck, max(lens_q), max(lens_k), window=window)
    torch.cuda.synchronize()
    ref = ora.attention_varlen(synth.bf16_bits(q), synth.bf16_bits(k), synth.bf16_bits(v),
                               cq.cpu().numpy(), ck.cpu().numpy(), causal=True, window=window)
    r = _rows(cq)
    assert_close(o[r], lse[:, r], ref[0][r], ref[1][:, r], f"varlen w{window} {lens_q}/{lens_k}")


def test_varlen_window_single_sequence_matches_attn_fwd_window_bit_for_bit():
    w = synth.Workload("vl_win_single", 1, 8, 2, 1500, 2000, 128, True, "normal", 43)
    q4, k4, v4 = synth.make_inputs(w, DEV)
    o4, l4 = binding.fwd(q4, k4, v4, window=300)
    tok = lambda x: x[0].transpose(0, 1).contiguous()
    cq = torch.tensor([0, w.Tq], dtype=torch.int32, device=DEV)
    ck = torch.tensor([0, w.Tk], dtype=torch.int32, device=DEV)
    o, lse = binding.fwd_varlen(tok(q4), tok(k4), tok(v4), cq, ck, w.Tq, w.Tk, window=300)
    torch.cuda.synchronize()
    assert torch.equal(o, tok(o4)) and torch.equal(lse, l4[0])


def test_varlen_window_packed_documents_sampled_rows():
    """The bench pack (27 documents, 65,536 tokens, H=32, d=128) with a
    1024-key window: sampled rows of every document, on sampled heads,
    against the oracle's windowed definition on that document alone."""
    lens = synth.packed_lengths(synth.VARLEN_TOKENS, synth.VARLEN.seed)
    q, k, v, cq, ck = synth.make_varlen_inputs(lens, lens, 32, 32, 128, seed=44, device=DEV)
    o, lse = binding.fwd_varlen(q, k, v, cq, ck, max(lens), max(lens), window=1024)
    torch.cuda.synchronize()
    c = cq.cpu().numpy()
    rng = np.random.default_rng(45)
    head_major = lambda x: x.transpose(0, 1).unsqueeze(0).contiguous()  # [1, H, n, d]
    for b in range(len(lens)):
        n = int(c[b + 1] - c[b])
        sl = slice(int(c[b]), int(c[b + 1]))
        ri = np.concatenate([[0, n - 1], rng.integers(0, n, size=4)]).astype(np.int32)
        rh = rng.integers(0, 32, size=ri.size).astype(np.int32)
        ref_o, ref_l = ora.attention_rows(synth.bf16_bits(head_major(q[sl])),
                                          synth.bf16_bits(head_major(k[sl])),
                                          synth.bf16_bits(head_major(v[sl])),
                                          np.zeros_like(ri), rh, ri, causal=True, window=1024)
        got_o = o[sl][torch.as_tensor(ri, device=DEV).long(), torch.as_tensor(rh, device=DEV).long()]
        got_l = lse[:, sl][torch.as_tensor(rh, device=DEV).long(), torch.as_tensor(ri, device=DEV).long()]
        assert_close(got_o, got_l, ref_o, ref_l, f"window pack doc {b}")
