"""Python access to the fp64 CPU attention oracle (oracle.c).

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only tests/, the smoke check in
__graft_entry__.py and the CPU-baseline / reference leg of bench.py may
import this module.  The oracle shares no code with the CUDA library: it is
a separate C file, compiled by gcc into its own shared object.

Every function takes numpy arrays laid out [B, H, T, d] (row-major) either
as float64 or as bf16 bit patterns (uint16) and returns float64 results.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

IN_F64 = 0
IN_BF16 = 1

OK = 0
ERR_ARG = 1
ERR_OVERFLOW = 2
ERR_NOMEM = 3

_lock = threading.Lock()
_lib = None


class OracleOverflow(ArithmeticError):
    """exp() overflowed: raised for the unshifted softmax on large scores."""


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with gcc (fp64, OpenMP, no fast-math)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-fopenmp",
           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            vp, ip, dp = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
            llp = ctypes.POINTER(ctypes.c_longlong)
            lib.oracle_attn_dense.argtypes = [vp, vp, vp, ip, ip, ip, ip, ip, ip,
                                              ip, ip, ip, dp, ip, vp, vp, vp, llp]
            lib.oracle_attn_rows.argtypes = [vp, vp, vp, ip, ip, ip, ip, ip, ip,
                                             ip, ip, ip, dp, ip, vp, vp, vp, vp, vp]
            lib.oracle_attn_blocked.argtypes = [vp, vp, vp, ip, ip, ip, ip, ip,
                                                ip, ip, ip, ip, dp, ip, ip, vp, ip,
                                                vp, vp, llp]
            lib.oracle_online_softmax_1d.argtypes = [vp, ip, ip, vp, vp, vp, vp,
                                                     vp]
            lib.oracle_attn_paged_decode.argtypes = [vp, vp, vp, ip, vp, vp, ip, ip,
                                                     ip, ip, ip, ip, ip, dp, vp, vp]
            lib.oracle_attn_varlen.argtypes = [vp, vp, vp, ip, vp, vp, ip, ip, ip, ip,
                                               ip, ip, ip, ip, dp, vp, vp]
            lib.oracle_attn_bwd_dense.argtypes = [vp, vp, vp, vp, ip, ip, ip, ip, ip, ip, ip,
                                                  ip, ip, dp, vp, vp, vp, vp, vp]
            lib.oracle_attn_bwd_blocked.argtypes = [vp, vp, vp, vp, ip, vp, vp, ip, ip, ip,
                                                    ip, ip, ip, ip, dp, ip, ip, vp, vp, vp]
            for f in (lib.oracle_attn_dense, lib.oracle_attn_rows,
                      lib.oracle_attn_blocked, lib.oracle_online_softmax_1d,
                      lib.oracle_attn_paged_decode, lib.oracle_attn_varlen,
                      lib.oracle_attn_bwd_dense, lib.oracle_attn_bwd_blocked):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def _as_input(x: np.ndarray) -> tuple[np.ndarray, int]:
    if x.dtype == np.float64:
        return np.ascontiguousarray(x), IN_F64
    if x.dtype == np.uint16:
        return np.ascontiguousarray(x), IN_BF16
    raise TypeError(f"oracle inputs are float64 or bf16 bits (uint16), not {x.dtype}")


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int):
    if rc == ERR_OVERFLOW:
        raise OracleOverflow("exp overflow in the unshifted softmax")
    if rc == ERR_ARG:
        raise ValueError("oracle: invalid shape or argument")
    if rc == ERR_NOMEM:
        raise MemoryError("oracle: allocation failed")
    if rc != OK:
        raise RuntimeError(f"oracle returned {rc}")


def _shapes(q, k, v):
    if q.ndim != 4 or k.ndim != 4 or v.ndim != 4:
        raise ValueError("q, k, v must be [B, H, T, d]")
    B, Hq, Tq, d = q.shape
    Bk, Hkv, Tk, dk = k.shape
    if (Bk, dk) != (B, d) or v.shape != k.shape:
        raise ValueError("inconsistent q/k/v shapes")
    return B, Hq, Hkv, Tq, Tk, d


def _inputs(q, k, v):
    (q, tq), (k, tk), (v, tv) = _as_input(q), _as_input(k), _as_input(v)
    if not tq == tk == tv:
        raise TypeError("q, k, v must share one input type")
    return q, k, v, tq


def attention_dense(q, k, v, causal=False, scale=None, subtract_max=True,
                    return_p=False, window=0):
    """Dense fp64 attention with materialised S and P (window > 0: causal
    sliding window of that many keys).

    Returns (o [B,Hq,Tq,d], lse [B,Hq,Tq], extras) where extras holds
    'visible_pairs' and, if return_p, 'p' [B,Hq,Tq,Tk].
    """
    B, Hq, Hkv, Tq, Tk, d = _shapes(q, k, v)
    q, k, v, t = _inputs(q, k, v)
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    o = np.empty((B, Hq, Tq, d), np.float64)
    lse = np.empty((B, Hq, Tq), np.float64)
    p = np.empty((B, Hq, Tq, Tk), np.float64) if return_p else None
    vis = ctypes.c_longlong(0)
    rc = _load().oracle_attn_dense(_ptr(q), _ptr(k), _ptr(v), t, B, Hq, Hkv, Tq,
                                   Tk, d, int(bool(causal)), int(window), scale,
                                   int(bool(subtract_max)), _ptr(o), _ptr(lse),
                                   _ptr(p), ctypes.byref(vis))
    _check(rc)
    extras = {"visible_pairs": vis.value}
    if return_p:
        extras["p"] = p
    return o, lse, extras


def attention_rows(q, k, v, rows_b, rows_h, rows_i, causal=False, scale=None,
                   window=0):
    """The dense definition evaluated for selected rows (b, h, i) only.

    Returns (o_rows [n, d], lse_rows [n]).
    """
    B, Hq, Hkv, Tq, Tk, d = _shapes(q, k, v)
    q, k, v, t = _inputs(q, k, v)
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    rb = np.ascontiguousarray(rows_b, dtype=np.int32)
    rh = np.ascontiguousarray(rows_h, dtype=np.int32)
    ri = np.ascontiguousarray(rows_i, dtype=np.int32)
    n = rb.size
    if not (rh.size == ri.size == n):
        raise ValueError("row index arrays differ in length")
    o = np.empty((n, d), np.float64)
    lse = np.empty((n,), np.float64)
    rc = _load().oracle_attn_rows(_ptr(q), _ptr(k), _ptr(v), t, B, Hq, Hkv, Tq,
                                  Tk, d, int(bool(causal)), int(window), scale, n,
                                  _ptr(rb),
                                  _ptr(rh), _ptr(ri), _ptr(o), _ptr(lse))
    _check(rc)
    return o, lse


def attention_blocked(q, k, v, block_q, block_kv, causal=False, scale=None,
                      kv_order=None, rescale_acc=True, window=0):
    """Blocked online-softmax forward (fp64).

    Returns (o, lse, tiles_visited).
    """
    B, Hq, Hkv, Tq, Tk, d = _shapes(q, k, v)
    q, k, v, t = _inputs(q, k, v)
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    order = None
    if kv_order is not None:
        order = np.ascontiguousarray(kv_order, dtype=np.int32)
        if order.size != (Tk + block_kv - 1) // block_kv:
            raise ValueError("kv_order must list every K/V block once")
    o = np.empty((B, Hq, Tq, d), np.float64)
    lse = np.empty((B, Hq, Tq), np.float64)
    visited = ctypes.c_longlong(0)
    rc = _load().oracle_attn_blocked(_ptr(q), _ptr(k), _ptr(v), t, B, Hq, Hkv,
                                     Tq, Tk, d, int(bool(causal)), int(window), scale,
                                     int(block_q), int(block_kv), _ptr(order),
                                     int(bool(rescale_acc)), _ptr(o), _ptr(lse),
                                     ctypes.byref(visited))
    _check(rc)
    return o, lse, visited.value


def attention_paged_decode(q, k_pages, v_pages, block_table, seq_lens, scale=None):
    """Decode of one query token per sequence against a paged KV cache.

    q [B, Hq, d]; k_pages, v_pages [num_pages, Hkv, page_size, d];
    block_table int [B, max_pages]; seq_lens int [B].
    Returns (o [B, Hq, d], lse [B, Hq]) in float64.
    """
    if q.ndim != 3 or k_pages.ndim != 4 or v_pages.shape != k_pages.shape:
        raise ValueError("q must be [B, Hq, d] and the pages [num_pages, Hkv, page_size, d]")
    B, Hq, d = q.shape
    num_pages, Hkv, page_size, dk = k_pages.shape
    if dk != d:
        raise ValueError("head dims differ")
    (qa, tq), (ka, tk), (va, tv) = _as_input(q), _as_input(k_pages), _as_input(v_pages)
    if not tq == tk == tv:
        raise TypeError("q, k, v must share one input type")
    table = np.ascontiguousarray(block_table, dtype=np.int32)
    lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    if table.ndim != 2 or table.shape[0] != B or lens.shape != (B,):
        raise ValueError("block_table must be [B, max_pages] and seq_lens [B]")
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    o = np.empty((B, Hq, d), np.float64)
    lse = np.empty((B, Hq), np.float64)
    rc = _load().oracle_attn_paged_decode(_ptr(qa), _ptr(ka), _ptr(va), tq, _ptr(table),
                                          _ptr(lens), B, Hq, Hkv, d, page_size, num_pages,
                                          table.shape[1], scale, _ptr(o), _ptr(lse))
    _check(rc)
    return o, lse


def attention_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, causal=False, scale=None, window=0):
    """Packed variable-length attention.

    q [total_q, Hq, d]; k, v [total_k, Hkv, d]; cu_seqlens_q / _k int [B+1];
    window > 0 (causal only) applies the sliding window inside each sequence.
    Returns (o [total_q, Hq, d], lse [Hq, total_q]) in float64; rows outside
    every sequence are NaN.
    """
    if q.ndim != 3 or k.ndim != 3 or v.shape != k.shape or q.shape[2] != k.shape[2]:
        raise ValueError("q must be [total_q, Hq, d] and k, v [total_k, Hkv, d]")
    total_q, Hq, d = q.shape
    total_k, Hkv, _ = k.shape
    (qa, tq), (ka, tk), (va, tv) = _as_input(q), _as_input(k), _as_input(v)
    if not tq == tk == tv:
        raise TypeError("q, k, v must share one input type")
    cq = np.ascontiguousarray(cu_seqlens_q, dtype=np.int32)
    ck = np.ascontiguousarray(cu_seqlens_k, dtype=np.int32)
    if cq.ndim != 1 or cq.shape != ck.shape or cq.size < 2:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must both be [B+1]")
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    o = np.full((total_q, Hq, d), np.nan)
    lse = np.full((Hq, total_q), np.nan)
    rc = _load().oracle_attn_varlen(_ptr(qa), _ptr(ka), _ptr(va), tq, _ptr(cq), _ptr(ck),
                                    cq.size - 1, Hq, Hkv, total_q, total_k, d,
                                    int(bool(causal)), int(window), scale, _ptr(o), _ptr(lse))
    _check(rc)
    return o, lse


def attention_backward(q, k, v, dout, causal=False, scale=None, window=0):
    """Gradients of attention from the plain definition (S, P, dP, dS
    materialised).  q, dout [B,Hq,Tq,d]; k, v [B,Hkv,Tk,d]; float64 or bf16
    bits, all of one type.  window > 0 (causal only) applies the forward's
    sliding-window mask.  Returns (dq, dk, dv, o, lse) in float64."""
    B, Hq, Hkv, Tq, Tk, d = _shapes(q, k, v)
    q, k, v, t = _inputs(q, k, v)
    do, td = _as_input(dout)
    if td != t or do.shape != q.shape:
        raise ValueError("dout must match q in shape and type")
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    dq = np.empty((B, Hq, Tq, d), np.float64)
    dk = np.empty((B, Hkv, Tk, d), np.float64)
    dv = np.empty((B, Hkv, Tk, d), np.float64)
    o = np.empty((B, Hq, Tq, d), np.float64)
    lse = np.empty((B, Hq, Tq), np.float64)
    rc = _load().oracle_attn_bwd_dense(_ptr(q), _ptr(k), _ptr(v), _ptr(do), t, B, Hq, Hkv, Tq,
                                       Tk, d, int(bool(causal)), int(window), scale, _ptr(dq),
                                       _ptr(dk), _ptr(dv), _ptr(o), _ptr(lse))
    _check(rc)
    return dq, dk, dv, o, lse


def attention_backward_blocked(q, k, v, dout, o, lse, block_q, block_kv, causal=False,
                               scale=None):
    """Backward with the probability tiles recomputed from the saved
    log-sum-exp, block by block.  o [B,Hq,Tq,d] and lse [B,Hq,Tq] are the
    forward's outputs (float64).  Returns (dq, dk, dv) in float64."""
    B, Hq, Hkv, Tq, Tk, d = _shapes(q, k, v)
    q, k, v, t = _inputs(q, k, v)
    do, td = _as_input(dout)
    if td != t or do.shape != q.shape:
        raise ValueError("dout must match q in shape and type")
    o = np.ascontiguousarray(o, dtype=np.float64)
    lse = np.ascontiguousarray(lse, dtype=np.float64)
    if o.shape != (B, Hq, Tq, d) or lse.shape != (B, Hq, Tq):
        raise ValueError("o must be [B,Hq,Tq,d] and lse [B,Hq,Tq]")
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    dq = np.empty((B, Hq, Tq, d), np.float64)
    dk = np.empty((B, Hkv, Tk, d), np.float64)
    dv = np.empty((B, Hkv, Tk, d), np.float64)
    rc = _load().oracle_attn_bwd_blocked(_ptr(q), _ptr(k), _ptr(v), _ptr(do), t, _ptr(o),
                                         _ptr(lse), B, Hq, Hkv, Tq, Tk, d, int(bool(causal)),
                                         scale, int(block_q), int(block_kv), _ptr(dq), _ptr(dk),
                                         _ptr(dv))
    _check(rc)
    return dq, dk, dv


def online_softmax_1d(x, block):
    """Streaming softmax of a 1-D vector in blocks.

    Returns (p, lse, trace) with trace = {'m': [...], 'l': [...], 'alpha': [...]}
    holding the state after each block.
    """
    x = np.ascontiguousarray(x, dtype=np.float64)
    n = x.size
    nb = (n + block - 1) // block
    p = np.empty(n, np.float64)
    mt, lt, at = (np.empty(nb, np.float64) for _ in range(3))
    lse = ctypes.c_double(0.0)
    rc = _load().oracle_online_softmax_1d(_ptr(x), n, int(block), _ptr(p),
                                          _ptr(mt), _ptr(lt), _ptr(at),
                                          ctypes.byref(lse))
    _check(rc)
    return p, lse.value, {"m": mt, "l": lt, "alpha": at}
