"""Thin ctypes binding over libattn.so (the C ABI in include/attn.h).

The functions named like the C entry points (attn_fwd, attn_decode, ...)
take raw integers and pointers exactly as the C ABI does.  `fwd`,
`fwd_varlen`, `bwd`, `decode` and `decode_paged` marshal torch CUDA tensors into those calls: they check dtype,
device, layout and shapes, allocate the outputs with torch, and pass the
current CUDA stream.  All attention arithmetic runs in the library's
kernels; if the library is missing these functions raise instead of
computing anything elsewhere.
"""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libattn.so")

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_MISALIGNED = 3
ATTN_ERR_WORKSPACE = 4
ATTN_ERR_CUDA = 5
ATTN_ERR_DEVICE_TIMEOUT = 6
ATTN_ERR_IN_FLIGHT_LIMIT = 7
STATUS_CODES = (ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED, ATTN_ERR_MISALIGNED,
                ATTN_ERR_WORKSPACE, ATTN_ERR_CUDA, ATTN_ERR_DEVICE_TIMEOUT,
                ATTN_ERR_IN_FLIGHT_LIMIT)

_lock = threading.Lock()
_lib = None


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {attn_status_string(status)}")


def load_library():
    """Load libattn.so (built by __graft_entry__.build()); raise if absent."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build the CUDA library first "
                    "(python -c 'import __graft_entry__ as g; g.build()')")
            lib = ctypes.CDLL(LIB_PATH)
            vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
            lib.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, vp]
            lib.attn_fwd.restype = i
            lib.attn_fwd_window.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, vp]
            lib.attn_fwd_window.restype = i
            lib.attn_fwd_varlen_workspace_bytes.argtypes = [i, i, i]
            lib.attn_fwd_varlen_workspace_bytes.restype = ctypes.c_size_t
            lib.attn_fwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i,
                                            i, i, f, vp, ctypes.c_size_t, vp]
            lib.attn_fwd_varlen.restype = i
            lib.attn_fwd_varlen_window.argtypes = lib.attn_fwd_varlen.argtypes
            lib.attn_fwd_varlen_window.restype = i
            lib.attn_decode_workspace_bytes.argtypes = [i, i, i, i, i]
            lib.attn_decode_workspace_bytes.restype = ctypes.c_size_t
            lib.attn_decode.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, vp,
                                        ctypes.c_size_t, vp]
            lib.attn_decode.restype = i
            lib.attn_decode_paged.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i,
                                              i, i, f, vp, ctypes.c_size_t, vp]
            lib.attn_decode_paged.restype = i
            lib.attn_bwd_workspace_bytes.argtypes = [i, i, i, i]
            lib.attn_bwd_workspace_bytes.restype = ctypes.c_size_t
            lib.attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f,
                                     vp, ctypes.c_size_t, vp]
            lib.attn_bwd.restype = i
            lib.attn_bwd_window.argtypes = lib.attn_bwd.argtypes
            lib.attn_bwd_window.restype = i
            lib.attn_fwd_host_workspace_bytes.argtypes = [i, i, i, i, i, i]
            lib.attn_fwd_host_workspace_bytes.restype = ctypes.c_size_t
            lib.attn_fwd_host.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, vp,
                                          ctypes.c_size_t, vp]
            lib.attn_fwd_host.restype = i
            lib.attn_decode_host_workspace_bytes.argtypes = [i, i, i, i, i]
            lib.attn_decode_host_workspace_bytes.restype = ctypes.c_size_t
            lib.attn_decode_host.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, vp,
                                             ctypes.c_size_t, vp]
            lib.attn_decode_host.restype = i
            lib.attn_status_string.argtypes = [i]
            lib.attn_status_string.restype = ctypes.c_char_p
            lib.attn_device_status.argtypes = [vp, ctypes.POINTER(i)]
            lib.attn_device_status.restype = i
            lib.attn_debug_set.argtypes = [ctypes.c_ulonglong, i]
            lib.attn_debug_set.restype = None
            _lib = lib
    return _lib


# ---------------------------------------------------------------- raw C ABI

def attn_fwd(q, k, v, o, lse, B, Hq, Hkv, Tq, Tk, d, causal, scale, stream) -> int:
    return load_library().attn_fwd(q, k, v, o, lse, B, Hq, Hkv, Tq, Tk, d, causal,
                                   scale, stream)


def attn_fwd_window(q, k, v, o, lse, B, Hq, Hkv, Tq, Tk, d, window, scale, stream) -> int:
    return load_library().attn_fwd_window(q, k, v, o, lse, B, Hq, Hkv, Tq, Tk, d, window,
                                          scale, stream)


def attn_fwd_varlen_workspace_bytes(B, total_q, max_seqlen_q) -> int:
    return load_library().attn_fwd_varlen_workspace_bytes(B, total_q, max_seqlen_q)


def attn_fwd_varlen(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, B, Hq, Hkv, total_q, total_k,
                    max_seqlen_q, max_seqlen_k, d, causal, scale, workspace, workspace_bytes,
                    stream) -> int:
    return load_library().attn_fwd_varlen(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, B, Hq,
                                          Hkv, total_q, total_k, max_seqlen_q, max_seqlen_k, d,
                                          causal, scale, workspace, workspace_bytes, stream)


def attn_fwd_varlen_window(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, B, Hq, Hkv, total_q,
                           total_k, max_seqlen_q, max_seqlen_k, d, window, scale, workspace,
                           workspace_bytes, stream) -> int:
    return load_library().attn_fwd_varlen_window(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k,
                                                 B, Hq, Hkv, total_q, total_k, max_seqlen_q,
                                                 max_seqlen_k, d, window, scale, workspace,
                                                 workspace_bytes, stream)


def attn_decode_workspace_bytes(B, Hq, Hkv, Tk, d) -> int:
    return load_library().attn_decode_workspace_bytes(B, Hq, Hkv, Tk, d)


def attn_decode(q, k_cache, v_cache, o, lse, B, Hq, Hkv, Tk, d, scale, workspace,
                workspace_bytes, stream) -> int:
    return load_library().attn_decode(q, k_cache, v_cache, o, lse, B, Hq, Hkv, Tk, d,
                                      scale, workspace, workspace_bytes, stream)


def attn_decode_paged(q, k_pages, v_pages, block_table, seq_lens, o, lse, B, Hq, Hkv, d,
                      page_size, num_pages, max_pages_per_seq, max_seq_len, scale, workspace,
                      workspace_bytes, stream) -> int:
    return load_library().attn_decode_paged(q, k_pages, v_pages, block_table, seq_lens, o, lse,
                                            B, Hq, Hkv, d, page_size, num_pages,
                                            max_pages_per_seq, max_seq_len, scale, workspace,
                                            workspace_bytes, stream)


def attn_bwd_workspace_bytes(B, Hq, Tq, d) -> int:
    return load_library().attn_bwd_workspace_bytes(B, Hq, Tq, d)


def attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, Tq, Tk, d, causal, scale, workspace,
             workspace_bytes, stream) -> int:
    return load_library().attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, Tq, Tk, d,
                                   causal, scale, workspace, workspace_bytes, stream)


def attn_fwd_host_workspace_bytes(B, Hq, Hkv, Tq, Tk, d) -> int:
    return load_library().attn_fwd_host_workspace_bytes(B, Hq, Hkv, Tq, Tk, d)


def attn_fwd_host(q, k, v, o, lse, B, Hq, Hkv, Tq, Tk, d, causal, scale, workspace,
                  workspace_bytes, stream) -> int:
    return load_library().attn_fwd_host(q, k, v, o, lse, B, Hq, Hkv, Tq, Tk, d, causal, scale,
                                        workspace, workspace_bytes, stream)


def attn_decode_host_workspace_bytes(B, Hq, Hkv, Tk, d) -> int:
    return load_library().attn_decode_host_workspace_bytes(B, Hq, Hkv, Tk, d)


def attn_decode_host(q, k_cache, v_cache, o, lse, B, Hq, Hkv, Tk, d, scale, workspace,
                     workspace_bytes, stream) -> int:
    return load_library().attn_decode_host(q, k_cache, v_cache, o, lse, B, Hq, Hkv, Tk, d,
                                           scale, workspace, workspace_bytes, stream)


def attn_bwd_window(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, Tq, Tk, d, window, scale,
                    workspace, workspace_bytes, stream) -> int:
    return load_library().attn_bwd_window(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, Tq, Tk,
                                          d, window, scale, workspace, workspace_bytes, stream)


def attn_status_string(status: int) -> str:
    return load_library().attn_status_string(status).decode()


def attn_device_status(stream=None) -> int:
    out = ctypes.c_int(0)
    rc = load_library().attn_device_status(stream, ctypes.byref(out))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_device_status")
    return out.value


def attn_debug_set(wait_limit_ns: int = 0, inject: int = 0) -> None:
    load_library().attn_debug_set(wait_limit_ns, inject)


# ------------------------------------------------------- torch marshalling

def _check_tensor(t, name, ndim):
    import torch

    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be on a CUDA device")
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16")
    if t.dim() != ndim or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {ndim}-d tensor")


def _check_host_tensor(t, name, ndim):
    import torch

    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cpu" or not t.is_pinned():
        raise ValueError(f"{name} must be a page-locked (pinned) CPU tensor")
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16")
    if t.dim() != ndim or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {ndim}-d tensor")


def _host_workspace(n, workspace, device):
    import torch

    if n == 0:
        raise ValueError("invalid sizes")
    if workspace is None:
        # torch's caching allocator returns 512-byte aligned blocks
        workspace = torch.empty(n, dtype=torch.uint8, device=device)
    return workspace


def _stream_handle(stream):
    import torch

    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def fwd(q, k, v, causal: bool = False, scale: float | None = None, out=None,
        lse=None, stream=None, window: int | None = None):
    """O, LSE = attention(q [B,Hq,Tq,d], k/v [B,Hkv,Tk,d]) through attn_fwd, or
    through attn_fwd_window (causal, `window` most recent keys) if window is
    given."""
    import torch

    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check_tensor(t, n, 4)
    B, Hq, Tq, d = q.shape
    Bk, Hkv, Tk, dk = k.shape
    if (Bk, dk) != (B, d) or tuple(v.shape) != tuple(k.shape):
        raise ValueError("inconsistent q/k/v shapes")
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, Tq), dtype=torch.float32, device=q.device)
    sc = 0.0 if scale is None else float(scale)
    if window is None:
        rc = attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                      B, Hq, Hkv, Tq, Tk, d, int(bool(causal)), sc, _stream_handle(stream))
        where = "attn_fwd"
    else:
        rc = attn_fwd_window(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                             lse.data_ptr(), B, Hq, Hkv, Tq, Tk, d, int(window), sc,
                             _stream_handle(stream))
        where = "attn_fwd_window"
    if rc != ATTN_OK:
        raise AttnError(rc, where)
    return out, lse


def fwd_host(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None,
             workspace=None, stream=None, device="cuda"):
    """O, LSE from pinned host tensors through attn_fwd_host: q [B,Hq,Tq,d],
    k/v [B,Hkv,Tk,d] in page-locked CPU memory; O and LSE come back in pinned
    CPU tensors, valid once `stream` has been synchronised."""
    import torch

    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check_host_tensor(t, n, 4)
    B, Hq, Tq, d = q.shape
    Bk, Hkv, Tk, dk = k.shape
    if (Bk, dk) != (B, d) or tuple(v.shape) != tuple(k.shape):
        raise ValueError("inconsistent q/k/v shapes")
    if out is None:
        out = torch.empty(q.shape, dtype=torch.bfloat16).pin_memory()
    if lse is None:
        lse = torch.empty((B, Hq, Tq), dtype=torch.float32).pin_memory()
    workspace = _host_workspace(attn_fwd_host_workspace_bytes(B, Hq, Hkv, Tq, Tk, d),
                                workspace, device)
    rc = attn_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                       B, Hq, Hkv, Tq, Tk, d, int(bool(causal)),
                       0.0 if scale is None else float(scale), workspace.data_ptr(),
                       workspace.numel() * workspace.element_size(), _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_host")
    return out, lse


def decode_host(q, k_cache, v_cache, scale: float | None = None, out=None, lse=None,
                workspace=None, stream=None, device="cuda"):
    """O, LSE for one query token per sequence from pinned host tensors
    through attn_decode_host (q [B,Hq,1,d], caches [B,Hkv,Tk,d])."""
    import torch

    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _check_host_tensor(t, n, 4)
    B, Hq, Tq, d = q.shape
    Bk, Hkv, Tk, dk = k_cache.shape
    if Tq != 1 or (Bk, dk) != (B, d) or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("decode expects q [B,Hq,1,d] and caches [B,Hkv,Tk,d]")
    if out is None:
        out = torch.empty(q.shape, dtype=torch.bfloat16).pin_memory()
    if lse is None:
        lse = torch.empty((B, Hq, 1), dtype=torch.float32).pin_memory()
    workspace = _host_workspace(attn_decode_host_workspace_bytes(B, Hq, Hkv, Tk, d),
                                workspace, device)
    rc = attn_decode_host(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), out.data_ptr(),
                          lse.data_ptr(), B, Hq, Hkv, Tk, d,
                          0.0 if scale is None else float(scale), workspace.data_ptr(),
                          workspace.numel() * workspace.element_size(), _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_decode_host")
    return out, lse


def decode_workspace(k_cache, q_heads: int):
    """Allocate the scratch attn_decode needs for this cache shape."""
    import torch

    B, Hkv, Tk, d = k_cache.shape
    n = attn_decode_workspace_bytes(B, q_heads, Hkv, Tk, d)
    if n == 0:
        raise ValueError("invalid decode sizes")
    return torch.empty((n + 15) // 16 * 16, dtype=torch.uint8, device=k_cache.device)


def decode(q, k_cache, v_cache, scale: float | None = None, workspace=None, out=None,
           lse=None, stream=None):
    """O, LSE for one query token per sequence: q [B,Hq,1,d] against the cache."""
    import torch

    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _check_tensor(t, n, 4)
    B, Hq, Tq, d = q.shape
    Bk, Hkv, Tk, dk = k_cache.shape
    if Tq != 1 or (Bk, dk) != (B, d) or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("decode expects q [B,Hq,1,d] and caches [B,Hkv,Tk,d]")
    if workspace is None:
        workspace = decode_workspace(k_cache, Hq)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, 1), dtype=torch.float32, device=q.device)
    rc = attn_decode(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), out.data_ptr(),
                     lse.data_ptr(), B, Hq, Hkv, Tk, d,
                     0.0 if scale is None else float(scale), workspace.data_ptr(),
                     workspace.numel() * workspace.element_size(), _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_decode")
    return out, lse


def decode_paged(q, k_pages, v_pages, block_table, seq_lens, max_seq_len: int | None = None,
                 scale: float | None = None, workspace=None, out=None, lse=None, stream=None):
    """O, LSE for one query token per sequence against a paged cache.

    q [B,Hq,1,d] bf16; k_pages, v_pages [num_pages,Hkv,page_size,d] bf16;
    block_table [B,max_pages] int32 and seq_lens [B] int32, all on the GPU.
    max_seq_len bounds seq_lens (it plans the split along the keys); when
    omitted it is taken to be the table's capacity, max_pages*page_size.
    """
    import torch

    for t, n in ((q, "q"), (k_pages, "k_pages"), (v_pages, "v_pages")):
        _check_tensor(t, n, 4)
    B, Hq, Tq, d = q.shape
    num_pages, Hkv, page_size, dk = k_pages.shape
    if Tq != 1 or dk != d or tuple(v_pages.shape) != tuple(k_pages.shape):
        raise ValueError("decode_paged expects q [B,Hq,1,d] and pages [num_pages,Hkv,page_size,d]")
    for t, n, shape in ((block_table, "block_table", None), (seq_lens, "seq_lens", (B,))):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.int32 or t.device != q.device \
                or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous int32 tensor on {q.device}")
    if block_table.dim() != 2 or block_table.shape[0] != B or tuple(seq_lens.shape) != (B,):
        raise ValueError("block_table must be [B, max_pages] and seq_lens [B]")
    max_pages = block_table.shape[1]
    if max_seq_len is None:
        max_seq_len = max_pages * page_size
    if workspace is None:
        n = attn_decode_workspace_bytes(B, Hq, Hkv, int(max_seq_len), d)
        if n == 0:
            raise ValueError("invalid decode sizes")
        workspace = torch.empty((n + 15) // 16 * 16, dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, 1), dtype=torch.float32, device=q.device)
    rc = attn_decode_paged(q.data_ptr(), k_pages.data_ptr(), v_pages.data_ptr(),
                           block_table.data_ptr(), seq_lens.data_ptr(), out.data_ptr(),
                           lse.data_ptr(), B, Hq, Hkv, d, page_size, num_pages, max_pages,
                           int(max_seq_len), 0.0 if scale is None else float(scale),
                           workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                           _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_decode_paged")
    return out, lse


def fwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, max_seqlen_k: int,
               causal: bool = False, scale: float | None = None, workspace=None, out=None,
               lse=None, stream=None, window: int | None = None):
    """O [total_q,Hq,d], LSE [Hq,total_q] for a packed batch: q [total_q,Hq,d],
    k/v [total_k,Hkv,d] (bf16, token-major), cu_seqlens_q/_k int32 [B+1] on
    the GPU, max_seqlen_q/_k host-side bounds of the lengths.  With `window`
    through attn_fwd_varlen_window (causal, the window inside each sequence)."""
    import torch

    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check_tensor(t, n, 3)
    total_q, Hq, d = q.shape
    total_k, Hkv, dk = k.shape
    if dk != d or tuple(v.shape) != tuple(k.shape):
        raise ValueError("inconsistent q/k/v shapes")
    for t, n in ((cu_seqlens_q, "cu_seqlens_q"), (cu_seqlens_k, "cu_seqlens_k")):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.int32 or t.device != q.device \
                or t.dim() != 1 or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous 1-d int32 tensor on {q.device}")
    if cu_seqlens_q.numel() != cu_seqlens_k.numel() or cu_seqlens_q.numel() < 2:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must both hold B+1 offsets")
    B = cu_seqlens_q.numel() - 1
    if workspace is None:
        n = attn_fwd_varlen_workspace_bytes(B, total_q, int(max_seqlen_q))
        if n == 0:
            raise ValueError("invalid packed-batch sizes")
        workspace = torch.empty(n, dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((Hq, total_q), dtype=torch.float32, device=q.device)
    fn, where = (attn_fwd_varlen, "attn_fwd_varlen") if window is None else \
        (attn_fwd_varlen_window, "attn_fwd_varlen_window")
    rc = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
            cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr(), B, Hq, Hkv, total_q, total_k,
            int(max_seqlen_q), int(max_seqlen_k), d,
            int(bool(causal)) if window is None else int(window),
            0.0 if scale is None else float(scale), workspace.data_ptr(),
            workspace.numel() * workspace.element_size(), _stream_handle(stream))
    if rc != ATTN_OK:
        raise AttnError(rc, where)
    return out, lse


def bwd(q, k, v, o, lse, dout, causal: bool = False, scale: float | None = None,
        workspace=None, dq=None, dk=None, dv=None, stream=None, window: int | None = None):
    """dq, dk, dv of attention through attn_bwd: q/k/v/causal/scale as given
    to `fwd`, (o, lse) what `fwd` returned, dout = dL/dO.  With `window`
    (the same as given to `fwd`) through attn_bwd_window."""
    import torch

    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (dout, "dout")):
        _check_tensor(t, n, 4)
    B, Hq, Tq, d = q.shape
    Bk, Hkv, Tk, dk_ = k.shape
    if (Bk, dk_) != (B, d) or tuple(v.shape) != tuple(k.shape) or o.shape != q.shape \
            or dout.shape != q.shape:
        raise ValueError("inconsistent shapes")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, Hq, Tq) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 [B, Hq, Tq] tensor")
    if workspace is None:
        n = attn_bwd_workspace_bytes(B, Hq, Tq, d)
        if n == 0:
            raise ValueError("invalid backward sizes")
        workspace = torch.empty(n, dtype=torch.uint8, device=q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    sc = 0.0 if scale is None else float(scale)
    ptrs = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
            dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, Hq, Hkv, Tq, Tk, d)
    ws = (workspace.data_ptr(), workspace.numel() * workspace.element_size(),
          _stream_handle(stream))
    if window is None:
        rc, where = attn_bwd(*ptrs, int(bool(causal)), sc, *ws), "attn_bwd"
    else:
        rc, where = attn_bwd_window(*ptrs, int(window), sc, *ws), "attn_bwd_window"
    if rc != ATTN_OK:
        raise AttnError(rc, where)
    return dq, dk, dv


# ------------------------------------------------------------- autograd

def _autograd_function():
    import torch

    class _Attention(torch.autograd.Function):
        """O = attention(q, k, v) through attn_fwd / attn_fwd_window, with the
        gradients of attn_bwd / attn_bwd_window; saves (q, k, v, O, LSE), so
        the backward recomputes the probabilities from the row log-sum-exp
        instead of storing them ("4.2 FlashAttention I", section "The
        backward pass: recomputation instead of storage")."""

        @staticmethod
        def forward(ctx, q, k, v, causal, scale, window):
            o, lse = fwd(q, k, v, causal=causal, scale=scale, window=window)
            ctx.save_for_backward(q, k, v, o, lse)
            ctx.causal, ctx.scale, ctx.window = causal, scale, window
            return o

        @staticmethod
        def backward(ctx, do):
            q, k, v, o, lse = ctx.saved_tensors
            dq, dk, dv = bwd(q, k, v, o, lse, do.contiguous(), causal=ctx.causal,
                             scale=ctx.scale, window=ctx.window)
            return dq, dk, dv, None, None, None

    return _Attention


_ATTENTION = None


def attention(q, k, v, causal: bool = False, scale: float | None = None,
              window: int | None = None):
    """Differentiable attention for bf16 CUDA tensors q [B,Hq,Tq,d] and
    k, v [B,Hkv,Tk,d]: the forward through `fwd`, the backward through `bwd`
    (GQA gradients of a K/V head sum over its query heads).  `window`
    selects the causal sliding window."""
    global _ATTENTION
    if _ATTENTION is None:
        _ATTENTION = _autograd_function()
    return _ATTENTION.apply(q, k, v, bool(causal) or window is not None, scale, window)
