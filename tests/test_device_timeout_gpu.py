"""Bounded waits: a kernel that never receives a tile gives up, reports
ATTN_ERR_DEVICE_TIMEOUT through the device status word, and leaves the CUDA
context usable.  The failure is made on the host (a test hook withholds the
first V tile); nothing faults, traps or hangs."""
import pytest
import torch

import synth
from online_softmax_03_gb300 import binding
from parity import assert_close, oracle_full

pytestmark = pytest.mark.gpu


def test_withheld_tile_times_out_and_context_survives():
    from online_softmax_03_gb300 import build as cuda_build

    cuda_build.build()
    binding.load_library()
    binding.attn_device_status()  # start from a clear status word
    w = synth.Workload("timeout_b1_h1_t384_d128", 1, 1, 1, 384, 384, 128, False, "normal", 30)
    q, k, v = synth.make_inputs(w, "cuda")
    try:
        binding.attn_debug_set(50_000_000, 1)  # 50 ms per wait, withhold V tile 0
        binding.fwd(q, k, v, causal=False)
        torch.cuda.synchronize()  # returns: the waits are bounded
    finally:
        binding.attn_debug_set(0, 0)
    assert binding.attn_device_status() == binding.ATTN_ERR_DEVICE_TIMEOUT
    assert binding.attn_device_status() == binding.ATTN_OK  # read clears it
    o, lse = binding.fwd(q, k, v, causal=False)
    torch.cuda.synchronize()
    assert_close(o, lse, *oracle_full(q, k, v, False, w.scale), "after timeout")
