"""GQA split-KV decode on the GPU (through the C ABI) against the fp64 oracle."""
import pytest
import torch

import synth
from online_softmax_03_gb300 import binding
from parity import assert_close, oracle_full

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from online_softmax_03_gb300 import build as cuda_build

    cuda_build.build()
    binding.load_library()
    yield
    assert binding.attn_device_status() == binding.ATTN_OK


def _decode_case(B, Hq, Hkv, Tk, d, seed):
    return synth.Workload(f"dec_b{B}_hq{Hq}_hkv{Hkv}_tk{Tk}_d{d}", B, Hq, Hkv, 1, Tk, d,
                          False, "normal", seed, decode=True)


def test_decode_gqa_full_size_all_rows():
    w = synth.DECODE_GQA
    q, k, v = synth.make_inputs(w, DEV)
    ws = binding.decode_workspace(k, w.Hq)
    torch.cuda.synchronize()
    before = torch.cuda.memory_allocated()
    torch.cuda.reset_peak_memory_stats()
    o, lse = binding.decode(q, k, v, scale=w.scale, workspace=ws)
    torch.cuda.synchronize()
    # only the outputs are allocated by the binding; the library allocates nothing
    out_bytes = o.numel() * 2 + lse.numel() * 4
    assert torch.cuda.max_memory_allocated() - before <= out_bytes + 2 * 512
    assert_close(o, lse, *oracle_full(q, k, v, False, w.scale), w.name)


@pytest.mark.parametrize("B,Hq,Hkv,Tk,d", [
    (1, 1, 1, 1, 128),
    (2, 4, 4, 31, 64),
    (3, 8, 2, 33, 32),
    (2, 16, 2, 1000, 128),
    (1, 32, 2, 777, 64),
    (2, 6, 2, 500, 128),
    (1, 5, 1, 300, 64),
    (4, 32, 8, 4099, 128),
])
def test_decode_shapes(B, Hq, Hkv, Tk, d):
    w = _decode_case(B, Hq, Hkv, Tk, d, B * 1000 + Tk)
    q, k, v = synth.make_inputs(w, DEV)
    o, lse = binding.decode(q, k, v)
    torch.cuda.synchronize()
    assert_close(o, lse, *oracle_full(q, k, v, False, w.scale), w.name)


def test_decode_128k_context():
    """131,072 cached tokens per sequence (B=2, Hq=32, Hkv=8, d=128): only 16
    (sequence, K/V head) pairs, so the plan cuts each into tens of splits of
    a few thousand keys; every row, after the merge, against the oracle."""
    w = _decode_case(2, 32, 8, 131072, 128, 77)
    q, k, v = synth.make_inputs(w, DEV)
    o, lse = binding.decode(q, k, v)
    torch.cuda.synchronize()
    assert_close(o, lse, *oracle_full(q, k, v, False, w.scale), w.name)


def test_decode_matches_prefill_entry_point_with_one_query():
    w = _decode_case(2, 8, 2, 640, 128, 77)
    q, k, v = synth.make_inputs(w, DEV)
    o1, l1 = binding.decode(q, k, v)
    o2, l2 = binding.fwd(q, k, v, causal=True)  # causal with Tq=1 sees the whole cache
    torch.cuda.synchronize()
    ref = oracle_full(q, k, v, False, w.scale)
    assert_close(o1, l1, *ref, "decode")
    assert_close(o2, l2, *ref, "fwd Tq=1")


def test_decode_large_scores():
    w = _decode_case(4, 16, 4, 2000, 128, 78).with_(q_mult=6.0)
    q, k, v = synth.make_inputs(w, DEV)
    o, lse = binding.decode(q, k, v)
    torch.cuda.synchronize()
    assert_close(o, lse, *oracle_full(q, k, v, False, w.scale), "decode q x6")
