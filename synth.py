"""Seeded synthetic inputs for exact attention forward (prefill and decode).

This module is shared by the tests, the benchmark and the smoke check.  It
draws random tensors and nothing else: it holds none of the attention
arithmetic, and neither the CUDA library nor the oracle imports it.

Recipe (one per workload, fixed here so that both sides of every parity
check receive the same bf16 tensors):

  g = torch.Generator(device).manual_seed(seed)
  Q, then K, then V are drawn in float32 from g, in that order, with the
  workload's distribution (standard normal, or Uniform(-0.8, 0.8) drawn as
  rand * 1.6 - 0.8); Q is multiplied by the workload's q_mult in float32;
  each tensor is then rounded to bf16 (round-to-nearest-even).

Layout: q [B, Hq, Tq, d], k and v [B, Hkv, Tk, d], all contiguous.  For
decode workloads Tq = 1 and k/v are one layer's KV cache.

The generator runs on the device the tensors are made for (torch's Philox
stream on CUDA, its CPU stream on the host), so a workload drawn on CUDA and
one drawn on the CPU with the same seed differ; every check compares two
results computed from one drawn set.
"""
from __future__ import annotations

import dataclasses

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    """One attention problem: shapes, masking and the input distribution."""

    name: str
    B: int
    Hq: int
    Hkv: int
    Tq: int
    Tk: int
    d: int
    causal: bool
    dist: str  # "normal" or "uniform0.8"
    seed: int
    q_mult: float = 1.0
    decode: bool = False

    @property
    def scale(self) -> float:
        return 1.0 / (self.d ** 0.5)

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads the library is specified and measured on.
TINY = Workload("tiny_b1_h4_t128_d32", 1, 4, 4, 128, 128, 32, True, "normal", 0)
TINY_NONCAUSAL = TINY.with_(name="tiny_b1_h4_t128_d32_noncausal", causal=False)
PREFILL_1K = Workload("prefill_b1_h32_t1024_d128_causal", 1, 32, 32, 1024, 1024,
                      128, True, "uniform0.8", 1)
PREFILL_4K = Workload("prefill_b4_h32_t4096_d128_causal", 4, 32, 32, 4096, 4096,
                      128, True, "normal", 2)
LONG_8K_CAUSAL = Workload("long_b1_h32_t8192_d64_causal_q4", 1, 32, 32, 8192, 8192,
                          64, True, "normal", 3, q_mult=4.0)
LONG_8K_FULL = LONG_8K_CAUSAL.with_(name="long_b1_h32_t8192_d64_full_q4",
                                    causal=False)
LONG_8000_CAUSAL = LONG_8K_CAUSAL.with_(name="long_b1_h32_t8000_d64_causal_q4",
                                        Tq=8000, Tk=8000)
LONG_8000_FULL = LONG_8K_CAUSAL.with_(name="long_b1_h32_t8000_d64_full_q4",
                                      Tq=8000, Tk=8000, causal=False)
DECODE_GQA = Workload("decode_b64_hq32_hkv8_tk8192_d128", 64, 32, 8, 1, 8192, 128,
                      False, "normal", 4, decode=True)

# Sliding-window prefill (causal band of WINDOW_KEYS keys); measured beside
# the specified workloads.
WINDOW_KEYS = 1024
WINDOW_8K = Workload("window_b4_h32_t8192_d128_w1024", 4, 32, 32, 8192, 8192, 128, True,
                     "normal", 6)

# Paged-cache decode measured beside the specified workloads: the decode
# workload's shapes with the cache cut into 16-token pages placed in a
# shuffled pool.
PAGED_DECODE = Workload("paged_decode_b64_hq32_hkv8_tk8192_d128_p16", 64, 32, 8, 1, 8192,
                        128, False, "normal", 5, decode=True)
PAGED_PAGE_SIZE = 16

# Packed variable-length prefill measured beside the specified workloads:
# documents of mixed length packed into one batch of VARLEN_TOKENS tokens.
VARLEN_TOKENS = 65536
VARLEN = Workload("varlen_pack65536_h32_d128_causal", 1, 32, 32, 8192, 8192, 128, True,
                  "normal", 7)

ALL = (TINY, TINY_NONCAUSAL, PREFILL_1K, PREFILL_4K, LONG_8K_CAUSAL, LONG_8K_FULL,
       LONG_8000_CAUSAL, LONG_8000_FULL, DECODE_GQA)


def _draw(g: torch.Generator, shape, dist: str, device) -> torch.Tensor:
    if dist == "normal":
        return torch.randn(shape, generator=g, dtype=torch.float32, device=device)
    if dist == "uniform0.8":
        return torch.rand(shape, generator=g, dtype=torch.float32,
                          device=device) * 1.6 - 0.8
    raise ValueError(f"unknown distribution {dist!r}")


def make_inputs(w: Workload, device="cpu"):
    """Draw (q, k, v) as bf16 tensors on `device` following the recipe above."""
    device = torch.device(device)
    g = torch.Generator(device=device).manual_seed(w.seed)
    q = _draw(g, (w.B, w.Hq, w.Tq, w.d), w.dist, device)
    if w.q_mult != 1.0:
        q.mul_(w.q_mult)
    k = _draw(g, (w.B, w.Hkv, w.Tk, w.d), w.dist, device)
    v = _draw(g, (w.B, w.Hkv, w.Tk, w.d), w.dist, device)
    return q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16)


def bf16_bits(t: torch.Tensor):
    """Host numpy uint16 view of a bf16 tensor's bit patterns (for the oracle)."""
    import numpy as np

    t = t.detach().contiguous().cpu()
    return t.view(torch.int16).numpy().view(np.uint16)


def sample_rows(w: Workload, n: int, seed: int = 1234):
    """Seeded (b, h, i) row indices for sampled parity checks.

    Always includes the first and last row of the first and last head, so the
    ragged last query tile and the first key tile are covered.
    """
    g = torch.Generator().manual_seed(seed)
    b = torch.randint(0, w.B, (n,), generator=g)
    h = torch.randint(0, w.Hq, (n,), generator=g)
    i = torch.randint(0, w.Tq, (n,), generator=g)
    fixed_b = torch.tensor([0, 0, w.B - 1, w.B - 1])
    fixed_h = torch.tensor([0, 0, w.Hq - 1, w.Hq - 1])
    fixed_i = torch.tensor([0, w.Tq - 1, 0, w.Tq - 1])
    return (torch.cat([fixed_b, b]).numpy(), torch.cat([fixed_h, h]).numpy(),
            torch.cat([fixed_i, i]).numpy())


def make_paged_inputs(B: int, Hq: int, Hkv: int, d: int, page_size: int, seq_lens,
                      seed: int, device="cpu", spare_pages: int = 0, max_pages=None):
    """Draw a paged decode problem: q [B,Hq,1,d], k_pages and v_pages
    [num_pages,Hkv,page_size,d] (bf16), block_table [B,max_pages] and
    seq_lens [B] (int32).

    Sequence b needs ceil(seq_lens[b]/page_size) pages; the pool holds
    those plus `spare_pages` unused ones.  Which physical page serves which
    (sequence, logical page) is a seeded random permutation (CPU generator,
    seed + 1), so neighbouring logical pages are scattered over the pool.
    Table entries past a sequence's last page are -1 (never read).  q, then
    the K pool, then the V pool are drawn N(0,1) in fp32 on `device` from a
    generator seeded with `seed` and rounded to bf16.
    """
    device = torch.device(device)
    lens = [int(x) for x in seq_lens]
    need = [-(-n // page_size) for n in lens]
    num_pages = sum(need) + spare_pages
    width = max(need) if max_pages is None else max_pages
    perm = torch.randperm(num_pages, generator=torch.Generator().manual_seed(seed + 1))
    table = torch.full((B, width), -1, dtype=torch.int32)
    at = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[at:at + n].to(torch.int32)
        at += n
    g = torch.Generator(device=device).manual_seed(seed)
    q = torch.randn((B, Hq, 1, d), generator=g, dtype=torch.float32, device=device)
    kp = torch.randn((num_pages, Hkv, page_size, d), generator=g, dtype=torch.float32,
                     device=device)
    vp = torch.randn((num_pages, Hkv, page_size, d), generator=g, dtype=torch.float32,
                     device=device)
    return (q.to(torch.bfloat16), kp.to(torch.bfloat16), vp.to(torch.bfloat16),
            table.to(device), torch.tensor(lens, dtype=torch.int32, device=device))


def packed_lengths(total: int, seed: int, mean: float = 2048.0, lo: int = 64,
                   hi: int = 8192):
    """Document lengths for a packed batch: drawn from an exponential
    distribution of the given mean (CPU generator, seeded), clipped to
    [lo, hi], until they fill `total` tokens (the last one is cut to fit)."""
    g = torch.Generator().manual_seed(seed)
    lens, used = [], 0
    while used < total:
        n = int(torch.empty(1).exponential_(1.0 / mean, generator=g).item())
        n = max(lo, min(hi, n), 1)
        n = min(n, total - used)
        lens.append(n)
        used += n
    return lens


def make_varlen_inputs(lens_q, lens_k, Hq: int, Hkv: int, d: int, seed: int, device="cpu",
                       dist: str = "normal", pad_q: int = 0, pad_k: int = 0):
    """Draw a packed batch: q [total_q, Hq, d], k and v [total_k, Hkv, d]
    (bf16, token-major) and int32 offsets cu_q, cu_k of length B+1.  q, then
    k, then v are drawn in fp32 on `device` from a generator seeded with
    `seed`, then rounded to bf16.  pad_q / pad_k add rows after the last
    sequence that belong to no sequence."""
    device = torch.device(device)
    cu_q = [0]
    for n in lens_q:
        cu_q.append(cu_q[-1] + int(n))
    cu_k = [0]
    for n in lens_k:
        cu_k.append(cu_k[-1] + int(n))
    g = torch.Generator(device=device).manual_seed(seed)
    q = _draw(g, (cu_q[-1] + pad_q, Hq, d), dist, device)
    k = _draw(g, (cu_k[-1] + pad_k, Hkv, d), dist, device)
    v = _draw(g, (cu_k[-1] + pad_k, Hkv, d), dist, device)
    return (q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16),
            torch.tensor(cu_q, dtype=torch.int32, device=device),
            torch.tensor(cu_k, dtype=torch.int32, device=device))
