"""Attention backward on the GPU (attn_bwd through the C ABI) against the
fp64 oracle's backward.

The GPU path receives bf16 q, k, v, dO, the bf16 O and fp32 LSE of its own
forward kernel, and returns bf16 gradients; the oracle differentiates the
exact definition on the same bf16 inputs.  Errors are measured relative to
the gradient's own scale (GRAD_TOL_MAX, GRAD_TOL_MEAN, GRAD_ATOL)."""
import numpy as np
import pytest
import torch

import synth
from oracle import oracle as ora
from online_softmax_03_gb300 import binding

pytestmark = pytest.mark.gpu

DEV = "cuda"

# Bound on |GPU - oracle| per gradient tensor: max error <= GRAD_TOL_MAX *
# max|ref| + GRAD_ATOL and mean error <= GRAD_TOL_MEAN * mean|ref| +
# GRAD_ATOL.  The GPU rounds the gradients to bf16 (relative error up to
# 2^-9, about 2^-10 on average), rounds P and dS to bf16 before the dV, dK
# and dQ products, and uses the bf16 O of its forward in D = dO . O.  On
# the cases below the measured errors are about 2.3e-3 of mean|ref| and at
# most 6e-3 of max|ref|; the bounds leave a factor of two to three.  The
# absolute floor covers gradients that vanish exactly (one visible key),
# where the GPU's fp32 rounding leaves residues of order 1e-6.
GRAD_TOL_MAX = 1.5e-2
GRAD_TOL_MEAN = 5e-3
GRAD_ATOL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from online_softmax_03_gb300 import build as cuda_build

    cuda_build.build()
    binding.load_library()
    assert binding.attn_device_status() == binding.ATTN_OK
    yield
    assert binding.attn_device_status() == binding.ATTN_OK


def _case(B, Hq, Hkv, Tq, Tk, d, causal, seed):
    w = synth.Workload(f"bwd_b{B}_h{Hq}_{Hkv}_t{Tq}_{Tk}_d{d}", B, Hq, Hkv, Tq, Tk, d, causal,
                       "normal", seed)
    q, k, v = synth.make_inputs(w, DEV)
    g = torch.Generator(device=DEV).manual_seed(seed + 1000)
    do = torch.randn(q.shape, generator=g, device=DEV, dtype=torch.float32).to(torch.bfloat16)
    return w, q, k, v, do


def _check(name, gpu, ref):
    x = gpu.float().cpu().numpy().astype(np.float64)
    err = np.abs(x - ref)
    scale_max, scale_mean = np.abs(ref).max(), np.abs(ref).mean()
    assert np.isfinite(x).all(), name
    assert err.max() <= GRAD_TOL_MAX * scale_max + GRAD_ATOL, \
        f"{name}: max err {err.max():.3e} vs max|ref| {scale_max:.3e}"
    assert err.mean() <= GRAD_TOL_MEAN * scale_mean + GRAD_ATOL, \
        f"{name}: mean err {err.mean():.3e} vs mean|ref| {scale_mean:.3e}"


@pytest.mark.parametrize("B,Hq,Hkv,Tq,Tk,d,causal", [
    (1, 2, 2, 256, 256, 128, True),
    (1, 4, 2, 200, 300, 64, True),      # GQA, Tq < Tk, ragged tiles
    (2, 2, 1, 130, 130, 32, False),
    (1, 2, 2, 1, 1, 64, True),          # one query, one key
    (1, 3, 3, 700, 700, 128, False),
    (2, 4, 1, 333, 333, 64, True),      # GQA 4
])
def test_backward_against_oracle(B, Hq, Hkv, Tq, Tk, d, causal):
    w, q, k, v, do = _case(B, Hq, Hkv, Tq, Tk, d, causal, seed=Tq + 7 * d)
    o, lse = binding.fwd(q, k, v, causal=causal)
    dq, dk, dv = binding.bwd(q, k, v, o, lse, do, causal=causal)
    torch.cuda.synchronize()
    rq, rk, rv, _, _ = ora.attention_backward(synth.bf16_bits(q), synth.bf16_bits(k),
                                              synth.bf16_bits(v), synth.bf16_bits(do),
                                              causal=causal)
    for name, a, r in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        _check(f"{w.name} {name}", a, r)


def test_backward_long_sequence_sampled_heads():
    """The benchmarked backward workload (B=4, H=32, T=4096, d=128, causal):
    two (batch, head) slices against the oracle (each head's gradients
    depend only on that head)."""
    w, q, k, v, do = _case(4, 32, 32, 4096, 4096, 128, True, seed=2)
    o, lse = binding.fwd(q, k, v, causal=True)
    dq, dk, dv = binding.bwd(q, k, v, o, lse, do, causal=True)
    torch.cuda.synchronize()
    for b, h in ((0, 0), (3, 31)):
        sl = lambda x: x[b:b + 1, h:h + 1]
        rq, rk, rv, _, _ = ora.attention_backward(
            synth.bf16_bits(sl(q)), synth.bf16_bits(sl(k)), synth.bf16_bits(sl(v)),
            synth.bf16_bits(sl(do)), causal=True)
        for name, a, r in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
            _check(f"b{b} h{h} {name}", sl(a), r)


def test_backward_dk_dv_deterministic_dq_close():
    """dK and dV are reduced inside one CTA and repeat bit for bit; dQ is
    summed by atomic reductions in varying order and repeats to rounding."""
    w, q, k, v, do = _case(1, 4, 4, 1000, 1000, 128, True, seed=50)
    o, lse = binding.fwd(q, k, v, causal=True)
    a = binding.bwd(q, k, v, o, lse, do, causal=True)
    b = binding.bwd(q, k, v, o, lse, do, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    assert (a[0].float() - b[0].float()).abs().max().item() <= 1e-2 * a[0].float().abs().max().item()


def test_backward_gradient_invariants():
    """Rows of dS sum to zero, so each head's dK rows sum to ~0 relative to
    their size; each K/V head's dV rows sum to the dO rows of its query
    heads."""
    w, q, k, v, do = _case(1, 4, 2, 512, 512, 64, False, seed=51)
    o, lse = binding.fwd(q, k, v)
    dq, dk, dv = binding.bwd(q, k, v, o, lse, do)
    torch.cuda.synchronize()
    dk_sum = dk.double().sum(dim=2)
    assert dk_sum.abs().max().item() <= 2e-2 * dk.double().abs().sum(dim=2).max().item()
    want = do.double().reshape(1, 2, 2, 512, 64).sum(dim=(2, 3))
    got = dv.double().sum(dim=2)
    assert (got - want).abs().max().item() <= 1e-2 * want.abs().max().item() + 0.05


def test_backward_rejects_bad_arguments():
    w, q, k, v, do = _case(1, 2, 2, 64, 64, 64, True, seed=52)
    o, lse = binding.fwd(q, k, v, causal=True)
    with pytest.raises(binding.AttnError):
        binding.bwd(q, k, v, o, lse, do, causal=True, workspace=torch.empty(16, dtype=torch.uint8,
                                                                             device=DEV))
    with pytest.raises(ValueError):
        binding.bwd(q, k, v, o, lse[:, :, :10], do)


@pytest.mark.parametrize("d,scale", [(32, 0.05), (64, 0.3), (128, 0.02), (128, 0.25)])
def test_backward_explicit_scale(d, scale):
    """A scale other than 1/sqrt(d): the kernels fold -LSE/scale into the
    score product and multiply dK by the scale, so a slip between the two
    conventions shows here and not at the default."""
    w, q, k, v, do = _case(1, 4, 2, 300, 300, d, True, seed=int(scale * 1000) + d)
    o, lse = binding.fwd(q, k, v, causal=True, scale=scale)
    dq, dk, dv = binding.bwd(q, k, v, o, lse, do, causal=True, scale=scale)
    torch.cuda.synchronize()
    rq, rk, rv, _, _ = ora.attention_backward(synth.bf16_bits(q), synth.bf16_bits(k),
                                              synth.bf16_bits(v), synth.bf16_bits(do),
                                              causal=True, scale=scale)
    for name, a, r in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        _check(f"{w.name} scale {scale} {name}", a, r)


def test_backward_d64_long_sequence_sampled_group():
    """The 128-query-step kernel at d = 64 over a long causal sequence with
    GQA: one K/V head's group (its four query heads) against the oracle,
    since dK and dV of a K/V head sum over exactly those query heads."""
    w, q, k, v, do = _case(2, 8, 2, 2048, 2048, 64, True, seed=53)
    o, lse = binding.fwd(q, k, v, causal=True)
    dq, dk, dv = binding.bwd(q, k, v, o, lse, do, causal=True)
    torch.cuda.synchronize()
    b, g = 1, 1
    qs = lambda x: x[b:b + 1, 4 * g:4 * g + 4]
    ks = lambda x: x[b:b + 1, g:g + 1]
    rq, rk, rv, _, _ = ora.attention_backward(
        synth.bf16_bits(qs(q)), synth.bf16_bits(ks(k)), synth.bf16_bits(ks(v)),
        synth.bf16_bits(qs(do)), causal=True)
    _check("d64 long dq", qs(dq), rq)
    _check("d64 long dk", ks(dk), rk)
    _check("d64 long dv", ks(dv), rv)


# --- sliding window ("4.2 FlashAttention I", Exercise 4): attn_bwd_window

@pytest.mark.parametrize("B,Hq,Hkv,Tq,Tk,d,window", [
    (1, 2, 2, 300, 300, 128, 100),
    (1, 4, 2, 200, 333, 64, 129),     # GQA, Tq < Tk, ragged tiles
    (2, 2, 1, 257, 257, 32, 1),       # one key per query: dQ = dK = 0
    (1, 3, 3, 700, 700, 128, 256),
    (2, 4, 1, 333, 333, 64, 2000),    # window past Tk: plain causal
    (1, 2, 2, 1000, 1000, 128, 300),  # key tiles with no query in reach of some tiles
])
def test_window_backward_against_oracle(B, Hq, Hkv, Tq, Tk, d, window):
    w, q, k, v, do = _case(B, Hq, Hkv, Tq, Tk, d, True, seed=Tq + window)
    o, lse = binding.fwd(q, k, v, window=window)
    dq, dk, dv = binding.bwd(q, k, v, o, lse, do, window=window)
    torch.cuda.synchronize()
    rq, rk, rv, _, _ = ora.attention_backward(synth.bf16_bits(q), synth.bf16_bits(k),
                                              synth.bf16_bits(v), synth.bf16_bits(do),
                                              causal=True, window=window)
    for name, a, r in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        _check(f"{w.name} w{window} {name}", a, r)


def test_window_backward_long_sequence_sampled_heads():
    """B=1, H=4, T=4096, d=128, W=1024 (the window row's window over 32 key
    tiles): two heads against the oracle (each head's gradients depend only
    on it)."""
    w, q, k, v, do = _case(1, 4, 4, 4096, 4096, 128, True, seed=57)
    o, lse = binding.fwd(q, k, v, window=1024)
    dq, dk, dv = binding.bwd(q, k, v, o, lse, do, window=1024)
    torch.cuda.synchronize()
    for h in (0, 3):
        sl = lambda x: x[:, h:h + 1]
        rq, rk, rv, _, _ = ora.attention_backward(
            synth.bf16_bits(sl(q)), synth.bf16_bits(sl(k)), synth.bf16_bits(sl(v)),
            synth.bf16_bits(sl(do)), causal=True, window=1024)
        for name, a, r in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
            _check(f"window long h{h} {name}", sl(a), r)


def test_window_backward_at_least_tk_is_the_causal_backward():
    """With window >= Tk every key tile visits the same query tiles with the
    same masks as the causal backward: dK and dV repeat bit for bit, dQ to
    the rounding of its reduction order."""
    w, q, k, v, do = _case(1, 4, 2, 640, 640, 128, True, seed=58)
    o, lse = binding.fwd(q, k, v, causal=True)
    a = binding.bwd(q, k, v, o, lse, do, causal=True)
    b = binding.bwd(q, k, v, o, lse, do, window=640)
    torch.cuda.synchronize()
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    assert (a[0].float() - b[0].float()).abs().max().item() <= 1e-2 * a[0].float().abs().max().item()


def test_window_backward_rejects_bad_windows():
    w, q, k, v, do = _case(1, 2, 2, 64, 64, 64, True, seed=59)
    o, lse = binding.fwd(q, k, v, causal=True)
    for bad in (0, -3):
        with pytest.raises(binding.AttnError):
            binding.bwd(q, k, v, o, lse, do, window=bad)


@pytest.mark.parametrize("causal,window", [(False, None), (True, None), (True, 100)])
def test_autograd_attention_matches_the_oracle(causal, window):
    """binding.attention as a torch autograd op: a loss's gradients through
    it equal the oracle's backward for dO = dLoss/dO."""
    w, q, k, v, do = _case(1, 4, 2, 300, 300, 64, causal, seed=60 + (window or 0))
    qg, kg, vg = (x.clone().requires_grad_(True) for x in (q, k, v))
    o = binding.attention(qg, kg, vg, causal=causal, window=window)
    (o.float() * do.float()).sum().backward()
    torch.cuda.synchronize()
    rq, rk, rv, ro, _ = ora.attention_backward(synth.bf16_bits(q), synth.bf16_bits(k),
                                               synth.bf16_bits(v), synth.bf16_bits(do),
                                               causal=causal, window=window or 0)
    assert np.abs(o.detach().float().cpu().numpy() - ro).max() <= 2e-2
    for name, a, r in (("dq", qg.grad, rq), ("dk", kg.grad, rk), ("dv", vg.grad, rv)):
        _check(f"autograd {name}", a, r)
