"""Causal sliding-window forward (attn_fwd_window) on the GPU against the
fp64 oracle ("4.2 FlashAttention I", Exercise 4)."""
import pytest
import torch

import synth
from online_softmax_03_gb300 import binding
from parity import assert_close
from oracle import oracle as ora

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from online_softmax_03_gb300 import build as cuda_build

    cuda_build.build()
    binding.load_library()
    yield
    assert binding.attn_device_status() == binding.ATTN_OK


def _ref(q, k, v, w, window):
    o, lse, _ = ora.attention_dense(synth.bf16_bits(q), synth.bf16_bits(k), synth.bf16_bits(v),
                                    causal=True, scale=w.scale, window=window)
    return o, lse


@pytest.mark.parametrize("B,Hq,Hkv,Tq,Tk,d,window", [
    (1, 2, 2, 1000, 1000, 64, 100),
    (1, 2, 2, 300, 300, 128, 1),
    (1, 2, 2, 257, 257, 32, 300),
    (2, 4, 4, 100, 333, 64, 50),
    (2, 8, 2, 700, 700, 128, 129),
    (1, 4, 4, 1024, 1024, 128, 256),
    (1, 2, 2, 129, 129, 64, 128),
])
def test_window_against_oracle(B, Hq, Hkv, Tq, Tk, d, window):
    w = synth.Workload(f"win_b{B}_t{Tq}_{Tk}_d{d}_w{window}", B, Hq, Hkv, Tq, Tk, d, True,
                       "normal", 60 + window)
    q, k, v = synth.make_inputs(w, "cuda")
    o, lse = binding.fwd(q, k, v, window=window)
    torch.cuda.synchronize()
    assert_close(o, lse, *_ref(q, k, v, w, window), w.name)


def test_window_long_sequence_every_row():
    w = synth.Workload("win_b2_h16_t8192_d128_w2048", 2, 16, 16, 8192, 8192, 128, True,
                       "normal", 61)
    q, k, v = synth.make_inputs(w, "cuda")
    o, lse = binding.fwd(q, k, v, window=2048)
    torch.cuda.synchronize()
    assert_close(o, lse, *_ref(q, k, v, w, 2048), w.name)


def test_window_at_least_tk_matches_causal_entry_point():
    w = synth.Workload("win_eq_causal", 1, 4, 4, 500, 500, 128, True, "normal", 62)
    q, k, v = synth.make_inputs(w, "cuda")
    o1, l1 = binding.fwd(q, k, v, causal=True)
    o2, l2 = binding.fwd(q, k, v, window=500)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_window_rejects_bad_windows():
    w = synth.Workload("win_bad", 1, 1, 1, 8, 8, 64, True, "normal", 63)
    q, k, v = synth.make_inputs(w, "cuda")
    with pytest.raises(binding.AttnError):
        binding.fwd(q, k, v, window=0)


def test_window_benchmarked_workload_every_row():
    """The sliding-window workload the benchmark times (B=4, H=32, T=8192,
    d=128, 1024-key window): every row of O and LSE against the full oracle."""
    w = synth.WINDOW_8K
    q, k, v = synth.make_inputs(w, "cuda")
    o, lse = binding.fwd(q, k, v, window=synth.WINDOW_KEYS)
    torch.cuda.synchronize()
    assert_close(o, lse, *_ref(q, k, v, w, synth.WINDOW_KEYS), w.name)
