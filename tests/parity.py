"""Shared helpers for GPU-vs-oracle parity checks.

Tolerances (bf16 inputs and outputs, fp32 LSE) against the fp64 oracle:
max |dO| <= 2e-2, mean |dO| <= 2e-3, max |dLSE| <= 1e-3.
"""
from __future__ import annotations

import json
import os

import numpy as np

import synth
from oracle import oracle as ora

TOL_MAX_O = 2e-2
TOL_MEAN_O = 2e-3
TOL_MAX_LSE = 1e-3


def errors(o_gpu, lse_gpu, o_ref, lse_ref):
    o = o_gpu.float().cpu().numpy().astype(np.float64)
    lse = lse_gpu.float().cpu().numpy().astype(np.float64)
    do = np.abs(o - o_ref)
    dl = np.abs(lse - lse_ref)
    return do.max(), do.mean(), dl.max()


def assert_close(o_gpu, lse_gpu, o_ref, lse_ref, what="", lse_rel=0.0):
    """lse_rel adds lse_rel * |LSE| to the LSE bound.  Only stress cases far
    outside the specified workloads use it: an fp32 LSE of magnitude ~1e4
    has a spacing of ~1e-3, so an absolute 1e-3 bound cannot hold there."""
    mo, mean_o, _ = errors(o_gpu, lse_gpu, o_ref, lse_ref)
    lse = lse_gpu.float().cpu().numpy().astype(np.float64)
    dl = np.abs(lse - lse_ref)
    ml = dl.max()
    assert np.isfinite(mo) and np.isfinite(ml), what
    assert mo <= TOL_MAX_O, f"{what}: max|dO| = {mo:.3e}"
    assert mean_o <= TOL_MEAN_O, f"{what}: mean|dO| = {mean_o:.3e}"
    bound = TOL_MAX_LSE + lse_rel * np.abs(lse_ref)
    _report(what, mo, mean_o, ml, lse.size)
    assert np.all(dl <= bound), f"{what}: max|dLSE| = {ml:.3e}"
    return mo, mean_o, ml


def _report(what, mo, mean_o, ml, rows):
    """Append the measured errors to the JSON-lines file named by
    ATTN_PARITY_REPORT (unset: nothing is written)."""
    path = os.environ.get("ATTN_PARITY_REPORT")
    if not path:
        return
    with open(path, "a") as f:
        f.write(json.dumps({"case": what, "rows": int(rows), "max_abs_dO": float(mo),
                            "mean_abs_dO": float(mean_o), "max_abs_dLSE": float(ml)}) + "\n")


def oracle_full(q, k, v, causal, scale):
    o, lse, _ = ora.attention_dense(synth.bf16_bits(q), synth.bf16_bits(k),
                                    synth.bf16_bits(v), causal=causal, scale=scale)
    return o, lse


def oracle_rows(q, k, v, causal, scale, rb, rh, ri):
    return ora.attention_rows(synth.bf16_bits(q), synth.bf16_bits(k), synth.bf16_bits(v),
                              rb, rh, ri, causal=causal, scale=scale)
