"""Bounded waits: a kernel that never receives a tile gives up, reports
ATTN_ERR_DEVICE_TIMEOUT through the device status word, and leaves the CUDA
context usable.  The failure is made on the host (a test hook withholds one
load: the forward's first V tile, the decode's first K/V tile, the
backward's first dO tile); nothing faults, traps or hangs."""
import numpy as np
import pytest
import torch

import synth
from online_softmax_03_gb300 import binding
from parity import assert_close, oracle_full

pytestmark = pytest.mark.gpu

WAIT_NS = 50_000_000  # 50 ms per wait while a hook is set


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from online_softmax_03_gb300 import build as cuda_build

    cuda_build.build()
    binding.load_library()
    binding.attn_device_status()  # start from a clear status word
    yield
    binding.attn_debug_set(0, 0)


def _with_hook(inject, fn):
    """Run fn with the hook set, then restore the defaults; returns the
    status word the call left."""
    try:
        binding.attn_debug_set(WAIT_NS, inject)
        fn()
        torch.cuda.synchronize()  # returns: the waits are bounded
    finally:
        binding.attn_debug_set(0, 0)
    status = binding.attn_device_status()
    assert binding.attn_device_status() == binding.ATTN_OK  # read clears it
    return status


def test_withheld_tile_times_out_and_context_survives():
    w = synth.Workload("timeout_b1_h1_t384_d128", 1, 1, 1, 384, 384, 128, False, "normal", 30)
    q, k, v = synth.make_inputs(w, "cuda")
    status = _with_hook(1, lambda: binding.fwd(q, k, v, causal=False))
    assert status == binding.ATTN_ERR_DEVICE_TIMEOUT
    o, lse = binding.fwd(q, k, v, causal=False)
    torch.cuda.synchronize()
    assert_close(o, lse, *oracle_full(q, k, v, False, w.scale), "after timeout")


@pytest.mark.parametrize("d", [64, 128])
def test_decode_withheld_tile_times_out_and_context_survives(d):
    w = synth.Workload(f"timeout_decode_d{d}", 2, 8, 2, 1, 3000, d, False, "normal", 31,
                       decode=True)
    q, k, v = synth.make_inputs(w, "cuda")
    ws = binding.decode_workspace(k, w.Hq)
    status = _with_hook(2, lambda: binding.decode(q, k, v, workspace=ws))
    assert status == binding.ATTN_ERR_DEVICE_TIMEOUT
    o, lse = binding.decode(q, k, v, workspace=ws)
    torch.cuda.synchronize()
    assert binding.attn_device_status() == binding.ATTN_OK
    assert_close(o, lse, *oracle_full(q, k, v, False, w.scale), "decode after timeout")


def test_paged_decode_withheld_tile_times_out():
    pq, pk, pv, tab, lens = synth.make_paged_inputs(2, 8, 2, 128, 16, [700, 1200], 32, "cuda")
    status = _with_hook(2, lambda: binding.decode_paged(pq, pk, pv, tab, lens))
    assert status == binding.ATTN_ERR_DEVICE_TIMEOUT
    o1, l1 = binding.decode_paged(pq, pk, pv, tab, lens)
    o2, l2 = binding.decode_paged(pq, pk, pv, tab, lens)
    torch.cuda.synchronize()
    assert binding.attn_device_status() == binding.ATTN_OK
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("d", [32, 128])
def test_backward_withheld_tile_times_out_and_context_survives(d):
    """d = 32 runs the single-buffered kernel, d = 128 the 128-query one."""
    w = synth.Workload(f"timeout_bwd_d{d}", 1, 2, 2, 256, 256, d, False, "normal", 33)
    q, k, v = synth.make_inputs(w, "cuda")
    g = torch.Generator(device="cuda").manual_seed(34)
    do = torch.randn(q.shape, generator=g, device="cuda", dtype=torch.float32).to(torch.bfloat16)
    o, lse = binding.fwd(q, k, v, causal=False)
    status = _with_hook(3, lambda: binding.bwd(q, k, v, o, lse, do, causal=False))
    assert status == binding.ATTN_ERR_DEVICE_TIMEOUT
    # the context still works: a call without the hook gives the oracle's gradients
    from oracle import oracle as ora

    dq, dk, dv = binding.bwd(q, k, v, o, lse, do, causal=False)
    torch.cuda.synchronize()
    assert binding.attn_device_status() == binding.ATTN_OK
    rq, rk, rv, _, _ = ora.attention_backward(synth.bf16_bits(q), synth.bf16_bits(k),
                                        synth.bf16_bits(v), synth.bf16_bits(do), causal=False,
                                        scale=w.scale)
    for name, x, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        err = np.abs(x.float().cpu().numpy().astype(np.float64) - ref)
        assert err.max() <= 1.5e-2 * np.abs(ref).max() + 1e-4, name
