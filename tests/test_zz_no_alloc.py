"""attn_decode_noalloc: decode for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc where they decode (a host framework owns
all device allocations, a serving loop cannot afford the implicit device
synchronisation, or the memory plan is frozen at start-up).  The library
gives them an entry point whose scratch is a fixed 16 MiB array inside the
library image.  These tests call it through the C ABI on two different
problems in a row, the first one larger, so every partial the second call
reads sits where the first call left data of another problem.  Each result
must be bit-identical to attn_decode with a caller workspace (the same split
plan and the same kernels) and must match the fp64 oracle.  The file is
named to be collected last.
"""
import ctypes
import os
import re

import pytest
import torch

import synth
from online_softmax_03_gb300 import binding
from online_softmax_03_gb300 import build as cuda_build
from parity import assert_close, oracle_full

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _entry():
    cuda_build.build()
    lib = binding.load_library()
    f = lib.attn_decode_noalloc
    vp, i = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, ctypes.c_float, vp]
    f.restype = i
    return f


def _max_bytes():
    with open(os.path.join(ROOT, "include", "attn.h")) as fh:
        m = re.search(r"#define ATTN_DECODE_NOALLOC_MAX_BYTES \(\(size_t\)(\d+) << (\d+)\)", fh.read())
    return int(m.group(1)) << int(m.group(2))


def _call(f, q, k, v):
    B, Hq, _, d = q.shape
    _, Hkv, Tk, _ = k.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, 1), dtype=torch.float32, device=q.device)
    rc = f(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
           B, Hq, Hkv, Tk, d, 0.0, torch.cuda.current_stream().cuda_stream)
    return rc, o, lse


def test_noalloc_decode_matches_attn_decode_on_two_calls_in_a_row():
    f = _entry()
    binding.attn_device_status()  # start from a clear status word
    problems = [
        synth.DECODE_GQA,  # B=64 Hq=32 Hkv=8 Tk=8192 d=128: the larger footprint first
        synth.Workload("dec_b4_hq16_hkv2_tk1500_d64", 4, 16, 2, 1, 1500, 64, False,
                       "normal", 21, decode=True),
    ]
    for w in problems:
        q, k, v = synth.make_inputs(w, "cuda")
        o_ref, lse_ref = binding.decode(q, k, v)
        rc, o, lse = _call(f, q, k, v)
        assert rc == binding.ATTN_OK, binding.attn_status_string(rc)
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref), w.name
        assert_close(o, lse, *oracle_full(q, k, v, False, w.scale), w.name)
        del q, k, v
    assert binding.attn_device_status() == binding.ATTN_OK


def test_noalloc_decode_timeout_reports_and_next_call_is_clean():
    """A withheld tile (host-set hook, 50 ms wait limit) makes one split give
    up: the call reports ATTN_ERR_DEVICE_TIMEOUT, and the next call, on the
    same shared array, is bit-identical to attn_decode."""
    f = _entry()
    binding.attn_device_status()
    w = synth.Workload("dec_b2_hq8_hkv2_tk3000_d128", 2, 8, 2, 1, 3000, 128, False, "normal",
                       23, decode=True)
    q, k, v = synth.make_inputs(w, "cuda")
    try:
        binding.attn_debug_set(50_000_000, 2)
        rc, _, _ = _call(f, q, k, v)
        torch.cuda.synchronize()
    finally:
        binding.attn_debug_set(0, 0)
    assert rc == binding.ATTN_OK
    assert binding.attn_device_status() == binding.ATTN_ERR_DEVICE_TIMEOUT
    rc, o, lse = _call(f, q, k, v)
    o_ref, lse_ref = binding.decode(q, k, v)
    torch.cuda.synchronize()
    assert rc == binding.ATTN_OK
    assert binding.attn_device_status() == binding.ATTN_OK
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)


def test_noalloc_decode_rejects_plans_beyond_its_scratch():
    f = _entry()
    # 1024 x 32 rows, one split (Tk = 1), (128 + 2) floats each: just over 16 MiB
    w = synth.Workload("dec_oversize", 1024, 32, 32, 1, 1, 128, False, "normal", 22,
                       decode=True)
    assert w.B * w.Hq * (w.d + 2) * 4 > _max_bytes()
    q, k, v = synth.make_inputs(w, "cuda")
    rc, _, _ = _call(f, q, k, v)
    assert rc == binding.ATTN_ERR_WORKSPACE
