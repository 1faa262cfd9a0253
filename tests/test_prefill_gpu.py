"""Prefill forward on the GPU (through the C ABI) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import synth
from online_softmax_03_gb300 import binding
from parity import assert_close, oracle_full, oracle_rows

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from online_softmax_03_gb300 import build as cuda_build

    cuda_build.build()
    binding.load_library()
    yield
    assert binding.attn_device_status() == binding.ATTN_OK


def _run(w):
    q, k, v = synth.make_inputs(w, DEV)
    o, lse = binding.fwd(q, k, v, causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    return q, k, v, o, lse


@pytest.mark.parametrize("w", [synth.TINY, synth.TINY_NONCAUSAL], ids=lambda w: w.name)
def test_tiny_full(w):
    q, k, v, o, lse = _run(w)
    assert_close(o, lse, *oracle_full(q, k, v, w.causal, w.scale), w.name)


def test_prefill_1k_full():
    w = synth.PREFILL_1K
    q, k, v, o, lse = _run(w)
    assert_close(o, lse, *oracle_full(q, k, v, w.causal, w.scale), w.name)


@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("T", [1, 17, 129, 255])
@pytest.mark.parametrize("causal", [False, True])
def test_odd_shapes(d, T, causal):
    w = synth.Workload(f"odd_t{T}_d{d}", 1, 2, 2, T, T, d, causal, "normal", 100 + T + d)
    q, k, v, o, lse = _run(w)
    assert_close(o, lse, *oracle_full(q, k, v, causal, w.scale), w.name)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_gqa_prefill(causal, d):
    w = synth.Workload("gqa_b2_hq8_hkv2_t300", 2, 8, 2, 300, 300, d, causal, "normal", 7)
    q, k, v, o, lse = _run(w)
    assert_close(o, lse, *oracle_full(q, k, v, causal, w.scale), w.name)


@pytest.mark.parametrize("causal", [False, True])
def test_tq_shorter_than_tk_bottom_right(causal):
    w = synth.Workload("tq100_tk333", 2, 4, 4, 100, 333, 64, causal, "normal", 8)
    q, k, v, o, lse = _run(w)
    assert_close(o, lse, *oracle_full(q, k, v, causal, w.scale), w.name)


@pytest.mark.parametrize("mult", [8.0, 20.0])
def test_large_scores_and_late_growing_max(mult):
    """Scores scaled up and a dominant late key: the running max grows late
    in rows, which exercises the accumulator rescale."""
    w = synth.Workload("stress", 1, 4, 4, 700, 700, 64, True, "normal", 9, q_mult=mult)
    q, k, v = synth.make_inputs(w, DEV)
    k[:, :, 650] = (q[:, :, 699] * 3).to(torch.bfloat16)
    o, lse = binding.fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    # scores reach ~1e4 here: allow 4 fp32 ulps of |LSE| on top of 1e-3
    assert_close(o, lse, *oracle_full(q, k, v, True, w.scale), "late key", lse_rel=4.8e-7)


@pytest.mark.parametrize("w", [synth.LONG_8K_CAUSAL, synth.LONG_8K_FULL,
                               synth.LONG_8000_CAUSAL, synth.LONG_8000_FULL],
                         ids=lambda w: w.name)
def test_long_d64_every_row(w):
    """The long d = 64 workloads (T = 8192 and the ragged 8000, causal and
    full, scores up to |s| ~ 30): every row of O and LSE against the full
    oracle."""
    q, k, v, o, lse = _run(w)
    assert_close(o, lse, *oracle_full(q, k, v, w.causal, w.scale), w.name)


def test_prefill_4k_every_row():
    """The benchmarked causal prefill (B=4, H=32, T=4096, d=128): every row
    of O and LSE against the full oracle, and causal row 0 of every head
    exactly v_0 (one visible key)."""
    w = synth.PREFILL_4K
    q, k, v, o, lse = _run(w)
    assert_close(o, lse, *oracle_full(q, k, v, w.causal, w.scale), w.name)
    assert torch.equal(o[:, :, 0], v[:, :, 0])


def test_prefill_32k_context_sampled_rows():
    """A 32,768-token causal sequence (B=1, H=8, d=128): the last rows visit
    256 key tiles and the 1024 items range from 2 to 512 tile products;
    sampled rows against the oracle and every output finite."""
    w = synth.Workload("prefill_b1_h8_t32768_d128_causal", 1, 8, 8, 32768, 32768, 128, True,
                       "normal", 21)
    q, k, v, o, lse = _run(w)
    rb, rh, ri = synth.sample_rows(w, 28)
    o_ref, lse_ref = oracle_rows(q, k, v, w.causal, w.scale, rb, rh, ri)
    assert_close(o[rb, rh, ri], lse[rb, rh, ri], o_ref, lse_ref, w.name)
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()


def test_outputs_stay_inside_their_buffers():
    """Guard canaries around O and LSE are left untouched."""
    w = synth.Workload("canary", 2, 3, 3, 200, 200, 128, True, "normal", 10)
    q, k, v = synth.make_inputs(w, DEV)
    pad = 4096
    n_o = q.numel()
    o_buf = torch.full((n_o + 2 * pad,), 7.0, dtype=torch.bfloat16, device=DEV)
    l_buf = torch.full((w.B * w.Hq * w.Tq + 2 * pad,), -5.0, dtype=torch.float32, device=DEV)
    o = o_buf[pad:pad + n_o].view(q.shape)
    lse = l_buf[pad:pad + w.B * w.Hq * w.Tq].view(w.B, w.Hq, w.Tq)
    binding.fwd(q, k, v, causal=True, out=o, lse=lse)
    torch.cuda.synchronize()
    assert (o_buf[:pad] == 7.0).all() and (o_buf[-pad:] == 7.0).all()
    assert (l_buf[:pad] == -5.0).all() and (l_buf[-pad:] == -5.0).all()
    assert_close(o, lse, *oracle_full(q, k, v, True, w.scale), w.name)


def test_deterministic_and_allocation_free():
    w = synth.PREFILL_1K
    q, k, v = synth.make_inputs(w, DEV)
    o1 = torch.empty_like(q)
    l1 = torch.empty((w.B, w.Hq, w.Tq), dtype=torch.float32, device=DEV)
    o2, l2 = torch.empty_like(o1), torch.empty_like(l1)
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats()
    before = torch.cuda.memory_allocated()
    binding.fwd(q, k, v, causal=True, out=o1, lse=l1)
    binding.fwd(q, k, v, causal=True, out=o2, lse=l2)
    torch.cuda.synchronize()
    assert torch.cuda.max_memory_allocated() == before  # no T x T anything
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_stream_argument_is_honoured():
    w = synth.TINY
    q, k, v = synth.make_inputs(w, DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o, lse = binding.fwd(q, k, v, causal=True)
    s.synchronize()
    assert_close(o, lse, *oracle_full(q, k, v, True, w.scale), "side stream")


def test_cuda_graph_replays_recompute_every_item():
    """A forward captured in a CUDA graph and replayed: every replay takes
    its work slot afresh (the last CTA of each launch frees it), so new
    inputs copied in before each replay give new, correct outputs."""
    w = synth.Workload("graph_b1_h4_t640_d128", 1, 4, 4, 640, 640, 128, True, "normal", 40)
    q, k, v = synth.make_inputs(w, DEV)
    o, lse = binding.fwd(q, k, v, causal=True)  # first call on the device: before capture
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        binding.fwd(q, k, v, causal=True, out=o, lse=lse)
    for seed in (41, 42, 43):
        qn, kn, vn = synth.make_inputs(w.with_(seed=seed), DEV)
        q.copy_(qn)
        k.copy_(kn)
        v.copy_(vn)
        o.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert_close(o, lse, *oracle_full(qn, kn, vn, True, w.scale), f"replay seed {seed}")
    assert binding.attn_device_status() == binding.ATTN_OK


def test_concurrent_launches_on_many_streams():
    """Sixteen small forwards in flight at once on sixteen streams, each on
    its own work slot, all correct and equal to the same calls made one at
    a time."""
    ws = [synth.Workload(f"conc_{i}", 1, 2, 2, 300 + 37 * i, 300 + 37 * i, 64, i % 2 == 0,
                         "normal", 50 + i) for i in range(16)]
    ins = [synth.make_inputs(w, DEV) for w in ws]
    ref = [binding.fwd(q, k, v, causal=w.causal) for w, (q, k, v) in zip(ws, ins)]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in ws]
    outs = []
    for st, w, (q, k, v) in zip(streams, ws, ins):
        st.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(st):
            outs.append(binding.fwd(q, k, v, causal=w.causal))
    torch.cuda.synchronize()
    for (o, l), (o_r, l_r) in zip(outs, ref):
        assert torch.equal(o, o_r) and torch.equal(l, l_r)
    assert binding.attn_device_status() == binding.ATTN_OK
