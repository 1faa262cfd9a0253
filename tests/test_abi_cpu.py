"""The C ABI without a GPU: the library loads, exports every entry point
include/attn.h declares, and rejects bad arguments before any CUDA call."""
import os
import re

import pytest

from online_softmax_03_gb300 import binding
from online_softmax_03_gb300 import build as cuda_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    cuda_build.build()
    return binding.load_library()


def _declared_functions():
    with open(os.path.join(ROOT, "include", "attn.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for n in ("attn_fwd", "attn_fwd_window", "attn_fwd_varlen", "attn_decode",
              "attn_decode_paged", "attn_fwd_varlen_workspace_bytes",
              "attn_decode_noalloc", "attn_decode_workspace_bytes",
              "attn_status_string", "attn_device_status", "attn_debug_set"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_status_strings_cover_every_code(lib):
    seen = set()
    for code in binding.STATUS_CODES:
        s = binding.attn_status_string(code)
        assert s.startswith("ATTN_") and "UNKNOWN" not in s
        seen.add(s)
    assert len(seen) == len(binding.STATUS_CODES)
    assert "UNKNOWN" in binding.attn_status_string(99)


# Fake, 16-byte aligned "device" addresses: every call below must be rejected
# by host validation, so nothing ever dereferences them.
Q, K, V, O, L, W = (0x10000 * i for i in range(1, 7))
OK_ARGS = dict(B=1, Hq=4, Hkv=2, Tq=8, Tk=16, d=64, causal=1, scale=0.0)


def _fwd(**kw):
    a = dict(q=Q, k=K, v=V, o=O, lse=L, **OK_ARGS)
    a.update(kw)
    return binding.attn_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["Hq"],
                            a["Hkv"], a["Tq"], a["Tk"], a["d"], a["causal"], a["scale"],
                            None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), binding.ATTN_ERR_INVALID_ARG),
    (dict(k=None), binding.ATTN_ERR_INVALID_ARG),
    (dict(v=None), binding.ATTN_ERR_INVALID_ARG),
    (dict(o=None), binding.ATTN_ERR_INVALID_ARG),
    (dict(lse=None), binding.ATTN_ERR_INVALID_ARG),
    (dict(B=0), binding.ATTN_ERR_INVALID_ARG),
    (dict(Hq=0), binding.ATTN_ERR_INVALID_ARG),
    (dict(Tq=0), binding.ATTN_ERR_INVALID_ARG),
    (dict(Tk=-1), binding.ATTN_ERR_INVALID_ARG),
    (dict(Hq=6, Hkv=4), binding.ATTN_ERR_INVALID_ARG),
    (dict(Tq=17, Tk=16), binding.ATTN_ERR_INVALID_ARG),
    (dict(causal=2), binding.ATTN_ERR_INVALID_ARG),
    (dict(scale=-1.0), binding.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("nan")), binding.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("inf")), binding.ATTN_ERR_INVALID_ARG),
    (dict(d=96), binding.ATTN_ERR_UNSUPPORTED),
    (dict(d=256), binding.ATTN_ERR_UNSUPPORTED),
    (dict(q=Q + 8), binding.ATTN_ERR_MISALIGNED),
    (dict(k=K + 2), binding.ATTN_ERR_MISALIGNED),
    (dict(v=V + 4), binding.ATTN_ERR_MISALIGNED),
    (dict(o=O + 8), binding.ATTN_ERR_MISALIGNED),
    (dict(lse=L + 2), binding.ATTN_ERR_MISALIGNED),
])
def test_fwd_rejects_bad_arguments_on_the_host(lib, kw, code):
    assert _fwd(**kw) == code


def test_valid_arguments_reach_the_device_check(lib):
    # Valid arguments get past validation, and without a GPU the device query
    # then fails.  Only run where no GPU exists: the pointers are fake.
    import torch

    if torch.cuda.is_available():
        pytest.skip("fake pointers must never reach a real device")
    assert _fwd(Tq=16, Tk=16) == binding.ATTN_ERR_CUDA


def test_decode_workspace_bytes(lib):
    n = binding.attn_decode_workspace_bytes(64, 32, 8, 8192, 128)
    # 32 splits at most for 8192 keys; (d + 2) floats per split and head
    assert n == 64 * 32 * 32 * (128 + 2) * 4
    assert binding.attn_decode_workspace_bytes(0, 32, 8, 8192, 128) == 0
    assert binding.attn_decode_workspace_bytes(1, 6, 4, 10, 64) == 0
    assert binding.attn_decode_workspace_bytes(1, 8, 8, 10, 48) == 0
    assert binding.attn_decode_workspace_bytes(1, 1, 1, 1, 32) == (32 + 2) * 4


def _decode(**kw):
    a = dict(q=Q, k=K, v=V, o=O, lse=L, B=2, Hq=8, Hkv=2, Tk=100, d=128, scale=0.0,
             ws=W, ws_bytes=1 << 20)
    a.update(kw)
    return binding.attn_decode(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["Hq"],
                               a["Hkv"], a["Tk"], a["d"], a["scale"], a["ws"],
                               a["ws_bytes"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), binding.ATTN_ERR_INVALID_ARG),
    (dict(Hq=8, Hkv=3), binding.ATTN_ERR_INVALID_ARG),
    (dict(Tk=0), binding.ATTN_ERR_INVALID_ARG),
    (dict(d=16), binding.ATTN_ERR_UNSUPPORTED),
    (dict(k=K + 8), binding.ATTN_ERR_MISALIGNED),
    (dict(ws=None), binding.ATTN_ERR_WORKSPACE),
    (dict(ws=W + 4), binding.ATTN_ERR_WORKSPACE),
    (dict(ws_bytes=16), binding.ATTN_ERR_WORKSPACE),
])
def test_decode_rejects_bad_arguments_on_the_host(lib, kw, code):
    assert _decode(**kw) == code


T_, S_ = 0x70000, 0x80000  # fake table and length addresses (4-byte aligned)


def _decode_paged(**kw):
    a = dict(q=Q, k=K, v=V, table=T_, lens=S_, o=O, lse=L, B=2, Hq=8, Hkv=2, d=128,
             page_size=16, num_pages=64, max_pages=8, max_len=100, scale=0.0, ws=W,
             ws_bytes=1 << 20)
    a.update(kw)
    return binding.attn_decode_paged(a["q"], a["k"], a["v"], a["table"], a["lens"], a["o"],
                                     a["lse"], a["B"], a["Hq"], a["Hkv"], a["d"],
                                     a["page_size"], a["num_pages"], a["max_pages"],
                                     a["max_len"], a["scale"], a["ws"], a["ws_bytes"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), binding.ATTN_ERR_INVALID_ARG),
    (dict(table=None), binding.ATTN_ERR_INVALID_ARG),
    (dict(lens=None), binding.ATTN_ERR_INVALID_ARG),
    (dict(Hq=8, Hkv=3), binding.ATTN_ERR_INVALID_ARG),
    (dict(max_len=0), binding.ATTN_ERR_INVALID_ARG),
    (dict(max_len=129), binding.ATTN_ERR_INVALID_ARG),   # > max_pages * page_size
    (dict(page_size=0), binding.ATTN_ERR_INVALID_ARG),
    (dict(page_size=24), binding.ATTN_ERR_INVALID_ARG),  # not a power of two
    (dict(page_size=8192), binding.ATTN_ERR_INVALID_ARG),
    (dict(num_pages=0), binding.ATTN_ERR_INVALID_ARG),
    (dict(max_pages=0), binding.ATTN_ERR_INVALID_ARG),
    (dict(d=96), binding.ATTN_ERR_UNSUPPORTED),
    (dict(v=V + 8), binding.ATTN_ERR_MISALIGNED),
    (dict(table=T_ + 2), binding.ATTN_ERR_MISALIGNED),
    (dict(lens=S_ + 1), binding.ATTN_ERR_MISALIGNED),
    (dict(ws=None), binding.ATTN_ERR_WORKSPACE),
    (dict(ws_bytes=64), binding.ATTN_ERR_WORKSPACE),
])
def test_decode_paged_rejects_bad_arguments_on_the_host(lib, kw, code):
    assert _decode_paged(**kw) == code


def test_varlen_workspace_bytes(lib):
    # list capacity min(B * ceil(max_q / 256), ceil(total_q / 256) + B) entries of two ints
    assert binding.attn_fwd_varlen_workspace_bytes(4, 1000, 600) == (2 + 2 * 8) * 4 + 8
    assert binding.attn_fwd_varlen_workspace_bytes(4, 5000, 300) == (2 + 2 * 8) * 4 + 8
    assert binding.attn_fwd_varlen_workspace_bytes(64, 4096, 4096) == (2 + 2 * 80) * 4 + 8
    assert binding.attn_fwd_varlen_workspace_bytes(0, 10, 10) == 0
    assert binding.attn_fwd_varlen_workspace_bytes(1, 0, 10) == 0


CQ, CK = 0x90000, 0xA0000  # fake offset arrays


def _fwd_varlen(**kw):
    a = dict(q=Q, k=K, v=V, o=O, lse=L, cq=CQ, ck=CK, B=3, Hq=8, Hkv=2, total_q=300,
             total_k=400, max_q=200, max_k=200, d=64, causal=1, scale=0.0, ws=W,
             ws_bytes=1 << 16)
    a.update(kw)
    return binding.attn_fwd_varlen(a["q"], a["k"], a["v"], a["o"], a["lse"], a["cq"], a["ck"],
                                   a["B"], a["Hq"], a["Hkv"], a["total_q"], a["total_k"],
                                   a["max_q"], a["max_k"], a["d"], a["causal"], a["scale"],
                                   a["ws"], a["ws_bytes"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), binding.ATTN_ERR_INVALID_ARG),
    (dict(cq=None), binding.ATTN_ERR_INVALID_ARG),
    (dict(ck=None), binding.ATTN_ERR_INVALID_ARG),
    (dict(B=0), binding.ATTN_ERR_INVALID_ARG),
    (dict(total_q=0), binding.ATTN_ERR_INVALID_ARG),
    (dict(total_k=0), binding.ATTN_ERR_INVALID_ARG),
    (dict(max_q=0), binding.ATTN_ERR_INVALID_ARG),
    (dict(causal=3), binding.ATTN_ERR_INVALID_ARG),
    (dict(Hq=8, Hkv=3), binding.ATTN_ERR_INVALID_ARG),
    (dict(d=80), binding.ATTN_ERR_UNSUPPORTED),
    (dict(o=O + 8), binding.ATTN_ERR_MISALIGNED),
    (dict(cq=CQ + 2), binding.ATTN_ERR_MISALIGNED),
    (dict(ws=None), binding.ATTN_ERR_WORKSPACE),
    (dict(ws_bytes=16), binding.ATTN_ERR_WORKSPACE),
])
def test_fwd_varlen_rejects_bad_arguments_on_the_host(lib, kw, code):
    assert _fwd_varlen(**kw) == code


def test_library_has_no_oracle_dependency():
    """The CUDA path neither links, loads nor imports the oracle."""
    pkg = os.path.join(ROOT, "online_softmax_03_gb300")
    pat = re.compile(r"(from\s+oracle|import\s+oracle|liboracle|oracle\.c)")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                with open(os.path.join(dirpath, f)) as fh:
                    assert not pat.search(fh.read()), f


# ---------------------------------------------------- host-buffer entry points

def test_host_workspace_bytes(lib):
    # device copies of q, k, v, o (bf16) and lse (fp32), each region rounded
    # up to 256 bytes
    qb, kb, lb = 4 * 32 * 4096 * 128 * 2, 4 * 32 * 4096 * 128 * 2, 4 * 32 * 4096 * 4
    assert binding.attn_fwd_host_workspace_bytes(4, 32, 32, 4096, 4096, 128) == 2 * qb + 2 * kb + lb
    r = lambda x: (x + 255) // 256 * 256
    assert binding.attn_fwd_host_workspace_bytes(1, 2, 1, 3, 5, 32) == \
        2 * r(2 * 3 * 32 * 2) + 2 * r(5 * 32 * 2) + r(2 * 3 * 4)
    assert binding.attn_fwd_host_workspace_bytes(1, 6, 4, 8, 8, 64) == 0
    assert binding.attn_fwd_host_workspace_bytes(1, 4, 4, 8, 8, 48) == 0
    # decode: the same device copies plus attn_decode's split partials
    part = binding.attn_decode_workspace_bytes(64, 32, 8, 8192, 128)
    assert binding.attn_decode_host_workspace_bytes(64, 32, 8, 8192, 128) == \
        2 * r(64 * 32 * 128 * 2) + 2 * r(64 * 8 * 8192 * 128 * 2) + r(64 * 32 * 4) + r(part)
    assert binding.attn_decode_host_workspace_bytes(0, 32, 8, 8192, 128) == 0


HW = 0x100000  # fake 256-byte aligned device workspace


def _fwd_host(**kw):
    a = dict(q=Q, k=K, v=V, o=O, lse=L, B=1, Hq=4, Hkv=2, Tq=8, Tk=16, d=64, causal=1,
             scale=0.0, ws=HW, ws_bytes=1 << 30)
    a.update(kw)
    return binding.attn_fwd_host(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["Hq"],
                                 a["Hkv"], a["Tq"], a["Tk"], a["d"], a["causal"], a["scale"],
                                 a["ws"], a["ws_bytes"], None)


def _decode_host(**kw):
    a = dict(q=Q, k=K, v=V, o=O, lse=L, B=2, Hq=8, Hkv=2, Tk=100, d=128, scale=0.0,
             ws=HW, ws_bytes=1 << 30)
    a.update(kw)
    return binding.attn_decode_host(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"],
                                    a["Hq"], a["Hkv"], a["Tk"], a["d"], a["scale"], a["ws"],
                                    a["ws_bytes"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), binding.ATTN_ERR_INVALID_ARG),
    (dict(lse=None), binding.ATTN_ERR_INVALID_ARG),
    (dict(B=0), binding.ATTN_ERR_INVALID_ARG),
    (dict(Hq=6, Hkv=4), binding.ATTN_ERR_INVALID_ARG),
    (dict(Tq=17, Tk=16), binding.ATTN_ERR_INVALID_ARG),
    (dict(causal=2), binding.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("nan")), binding.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("inf")), binding.ATTN_ERR_INVALID_ARG),
    (dict(scale=-0.5), binding.ATTN_ERR_INVALID_ARG),
    (dict(d=96), binding.ATTN_ERR_UNSUPPORTED),
    (dict(ws=None), binding.ATTN_ERR_WORKSPACE),
    (dict(ws=HW + 16), binding.ATTN_ERR_WORKSPACE),
    (dict(ws_bytes=1024), binding.ATTN_ERR_WORKSPACE),
])
def test_fwd_host_rejects_bad_arguments_on_the_host(lib, kw, code):
    assert _fwd_host(**kw) == code


@pytest.mark.parametrize("kw,code", [
    (dict(k=None), binding.ATTN_ERR_INVALID_ARG),
    (dict(Tk=0), binding.ATTN_ERR_INVALID_ARG),
    (dict(Hq=8, Hkv=3), binding.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("nan")), binding.ATTN_ERR_INVALID_ARG),
    (dict(d=16), binding.ATTN_ERR_UNSUPPORTED),
    (dict(ws=None), binding.ATTN_ERR_WORKSPACE),
    (dict(ws_bytes=4096), binding.ATTN_ERR_WORKSPACE),
])
def test_decode_host_rejects_bad_arguments_on_the_host(lib, kw, code):
    assert _decode_host(**kw) == code


def test_host_entry_points_with_valid_arguments_reach_cuda(lib):
    # Past validation the first CUDA call (a stream) fails without a GPU.
    import torch

    if torch.cuda.is_available():
        pytest.skip("fake pointers must never reach a real device")
    assert _fwd_host() == binding.ATTN_ERR_CUDA
    assert _decode_host() == binding.ATTN_ERR_CUDA


def test_host_wrappers_require_pinned_cpu_tensors():
    import torch

    x = torch.zeros(1, 2, 8, 64, dtype=torch.bfloat16)  # pageable
    with pytest.raises(ValueError):
        binding.fwd_host(x, x, x)
    with pytest.raises(ValueError):
        binding.decode_host(x[:, :, :1], x, x)


def test_bwd_window_rejects_bad_windows_on_the_host(lib):
    for bad in (0, -1):
        rc = binding.attn_bwd_window(Q, K, V, O, L, Q, K, V, O, 1, 2, 2, 16, 16, 64, bad, 0.0,
                                     W, 1 << 20, None)
        assert rc == binding.ATTN_ERR_INVALID_ARG
    # causal is implied: more queries than keys is rejected like attn_bwd's causal case
    rc = binding.attn_bwd_window(Q, K, V, O, L, Q, K, V, O, 1, 2, 2, 17, 16, 64, 4, 0.0,
                                 W, 1 << 20, None)
    assert rc == binding.ATTN_ERR_INVALID_ARG


def test_varlen_window_rejects_bad_windows_on_the_host(lib):
    for bad in (0, -2):
        rc = binding.attn_fwd_varlen_window(Q, K, V, O, L, T_, S_, 2, 4, 2, 64, 64, 32, 32, 64,
                                            bad, 0.0, W, 1 << 20, None)
        assert rc == binding.ATTN_ERR_INVALID_ARG
