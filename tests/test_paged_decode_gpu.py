"""Decode against a paged KV cache on the GPU (attn_decode_paged through the
C ABI) against the fp64 oracle's paged decode."""
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


def _oracle(q, kp, vp, table, lens, scale=None, rows=None):
    """Oracle result as [B, Hq, 1, d] / [B, Hq, 1] (for the sequences `rows`)."""
    qb = synth.bf16_bits(q)[:, :, 0]
    t = table.cpu().numpy()
    n = lens.cpu().numpy()
    if rows is not None:
        qb, t, n = qb[rows], t[rows], n[rows]
    o, lse = ora.attention_paged_decode(qb, synth.bf16_bits(kp), synth.bf16_bits(vp), t, n,
                                        scale=scale)
    return o[:, :, None], lse[:, :, None]


@pytest.mark.parametrize("B,Hq,Hkv,d,page,lens", [
    (3, 8, 2, 128, 16, (100, 1, 37)),        # GQA 4, one-token sequence
    (2, 32, 8, 64, 1, (70, 64)),              # one token per page
    (4, 8, 1, 32, 8, (9, 17, 300, 1000)),     # GQA 8
    (2, 4, 4, 128, 64, (64, 65)),             # no grouping; page boundary +-1
    (2, 16, 2, 128, 256, (1000, 513)),
    (1, 4, 4, 64, 4096, (5000,)),             # largest page size, two pages
    (2, 12, 2, 128, 32, (2000, 3333)),        # GQA 6 (padded head chunk)
    (5, 8, 8, 32, 2, (1, 2, 3, 31, 33)),
])
def test_paged_decode_shapes(B, Hq, Hkv, d, page, lens):
    q, kp, vp, table, sl = synth.make_paged_inputs(B, Hq, Hkv, d, page, lens,
                                                   seed=B * 97 + page, device=DEV,
                                                   spare_pages=3)
    o, lse = binding.decode_paged(q, kp, vp, table, sl, max_seq_len=max(lens))
    torch.cuda.synchronize()
    assert_close(o, lse, *_oracle(q, kp, vp, table, sl), f"paged b{B} p{page} {lens}")


def test_paged_decode_reads_nothing_outside_the_sequences():
    """Every slot past a sequence's length (the tail of its last page) and
    every spare page holds NaN, unused table entries are -1, and max_seq_len
    is the table's full capacity (so trailing splits find no keys): the
    result is finite, matches the oracle, and no invalid index is reported."""
    B, Hq, Hkv, d, page = 4, 8, 2, 128, 16
    lens = (45, 16, 3, 200)
    q, kp, vp, table, sl = synth.make_paged_inputs(B, Hq, Hkv, d, page, lens, seed=11,
                                                   device=DEV, spare_pages=5, max_pages=40)
    used = torch.zeros(kp.shape[0], page, dtype=torch.bool)
    t = table.cpu()
    for b, n in enumerate(lens):
        for j in range(n):
            used[t[b, j // page], j % page] = True
    poison = (~used).to(DEV)[:, None, :, None].expand_as(kp)
    kp = kp.masked_fill(poison, float("nan"))
    vp = vp.masked_fill(poison, float("nan"))
    o, lse = binding.decode_paged(q, kp, vp, table, sl, max_seq_len=40 * page)
    torch.cuda.synchronize()
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    assert_close(o, lse, *_oracle(q, kp, vp, table, sl), "paged poisoned slack")
    assert binding.attn_device_status() == binding.ATTN_OK


def test_paged_decode_shared_prefix_pages():
    """Sequences whose tables share their first pages (a common prefix)."""
    B, Hq, Hkv, d, page = 3, 8, 2, 64, 16
    lens = (80, 80, 50)
    q, kp, vp, table, sl = synth.make_paged_inputs(B, Hq, Hkv, d, page, lens, seed=12,
                                                   device=DEV)
    table[1, :3] = table[0, :3]
    table[2, :2] = table[0, :2]
    q[1] = q[0]
    o, lse = binding.decode_paged(q, kp, vp, table, sl)
    torch.cuda.synchronize()
    assert_close(o, lse, *_oracle(q, kp, vp, table, sl), "paged shared prefix")


def test_paged_decode_bench_workload_matches_oracle_and_contiguous_decode():
    """The benchmarked paged workload (B=64, Hq=32, Hkv=8, 8192 tokens per
    sequence, d=128, 16-token pages in a shuffled pool): 8 sequences against
    the oracle, and every row bit-identical to attn_decode on the same cache
    laid out contiguously (same split plan, same arithmetic)."""
    w, page = synth.PAGED_DECODE, synth.PAGED_PAGE_SIZE
    lens = [w.Tk] * w.B
    q, kp, vp, table, sl = synth.make_paged_inputs(w.B, w.Hq, w.Hkv, w.d, page, lens,
                                                   seed=w.seed, device=DEV)
    o, lse = binding.decode_paged(q, kp, vp, table, sl, max_seq_len=w.Tk, scale=w.scale)
    torch.cuda.synchronize()
    rows = np.array([0, 1, 17, 30, 31, 45, 62, 63])
    o_ref, lse_ref = _oracle(q, kp, vp, table, sl, scale=w.scale, rows=rows)
    idx = torch.as_tensor(rows, device=DEV)
    assert_close(o[idx], lse[idx], o_ref, lse_ref, w.name)
    # gather the pages into [B, Hkv, Tk, d] and decode contiguously
    tl = table.long()
    kc = kp[tl].permute(0, 2, 1, 3, 4).reshape(w.B, w.Hkv, w.Tk, w.d).contiguous()
    vc = vp[tl].permute(0, 2, 1, 3, 4).reshape(w.B, w.Hkv, w.Tk, w.d).contiguous()
    oc, lc = binding.decode(q, kc, vc, scale=w.scale)
    torch.cuda.synchronize()
    assert torch.equal(o, oc) and torch.equal(lse, lc)


def test_paged_decode_invalid_device_entries_are_reported_not_used():
    """A page number outside the pool and lengths outside 1..max_seq_len are
    found on the device: nothing outside the pool is read, the status word
    reports ATTN_ERR_INVALID_ARG, and the other sequences are unaffected."""
    B, Hq, Hkv, d, page = 4, 8, 2, 64, 16
    lens = (40, 40, 40, 40)
    q, kp, vp, table, sl = synth.make_paged_inputs(B, Hq, Hkv, d, page, lens, seed=13,
                                                   device=DEV)
    good_o, good_l = binding.decode_paged(q, kp, vp, table, sl, max_seq_len=40)
    torch.cuda.synchronize()
    assert binding.attn_device_status() == binding.ATTN_OK
    bad_t = table.clone()
    bad_t[1, 1] = kp.shape[0]          # one past the pool
    bad_l = sl.clone()
    bad_l[2] = 0                       # empty sequence
    bad_l[3] = 41                      # longer than max_seq_len
    o, lse = binding.decode_paged(q, kp, vp, bad_t, bad_l, max_seq_len=40)
    torch.cuda.synchronize()
    assert binding.attn_device_status() == binding.ATTN_ERR_INVALID_ARG
    assert torch.equal(o[0], good_o[0]) and torch.equal(lse[0], good_l[0])
    # the context is still usable and a clean call reports nothing
    o2, l2 = binding.decode_paged(q, kp, vp, table, sl, max_seq_len=40)
    torch.cuda.synchronize()
    assert binding.attn_device_status() == binding.ATTN_OK
    assert torch.equal(o2, good_o) and torch.equal(l2, good_l)


def test_paged_decode_rejects_bad_host_arguments():
    q, kp, vp, table, sl = synth.make_paged_inputs(1, 4, 4, 64, 16, (20,), seed=14, device=DEV)
    with pytest.raises(binding.AttnError):
        binding.decode_paged(q, kp, vp, table, sl, max_seq_len=33)  # > 2 pages of 16
    with pytest.raises(ValueError):
        binding.decode_paged(q, kp, vp, table.long(), sl)


def test_dense_cache_with_per_sequence_lengths_as_one_page_per_sequence():
    """A dense cache [B, Hkv, T, d] whose T is a power of two <= 4096 is a
    page pool with page_size = T and the table b -> b, so decode over
    sequences of different lengths in a dense cache is attn_decode_paged with
    one page per sequence: it must equal the dense definition on each
    sequence's first seq_lens[b] keys."""
    B, Hq, Hkv, T, d = 5, 16, 4, 2048, 128
    w = synth.Workload("dense_lens", B, Hq, Hkv, 1, T, d, False, "normal", 70)
    q, k, v = synth.make_inputs(w, DEV)
    lens = torch.tensor([2048, 1, 777, 1500, 64], dtype=torch.int32, device=DEV)
    table = torch.arange(B, dtype=torch.int32, device=DEV).reshape(B, 1)
    o, lse = binding.decode_paged(q, k, v, table, lens, max_seq_len=T)
    torch.cuda.synchronize()
    for b, n in enumerate(lens.tolist()):
        ref_o, ref_l, _ = ora.attention_dense(synth.bf16_bits(q[b:b + 1]),
                                              synth.bf16_bits(k[b:b + 1, :, :n]),
                                              synth.bf16_bits(v[b:b + 1, :, :n]), causal=False)
        assert_close(o[b:b + 1], lse[b:b + 1], ref_o, ref_l, f"dense lens b{b} n{n}")
