"""Benchmark: exact attention forward on GB300.

One step = one pass of the whole path over one batch of synthetic input:
  1. causal prefill, B=4, H=32, T=4096, d=128 (attn_fwd, tensor cores), then
  2. GQA decode, B=64, Hq=32, Hkv=8, Tk=8192, d=128 (attn_decode: split + combine).

Printed (rank 0, one JSON line):
  value     prefill TFLOP/s (causal FLOPs = 2*B*H*T^2*d), summed over ranks
  decode    decode HBM GB/s (K+V+q+o+lse bytes), with its own roofline
  e2e       the same metrics through the host-buffer entry points
            (attn_fwd_host / attn_decode_host) on pinned host buffers: the
            host->device inputs and device->host outputs inside the timed
            region, overlapped with the kernels across chunks of the batch
  roofline  prefill kernel: achieved TFLOP/s vs the measured bf16 peak
  cpu_baseline  the fp64 oracle timed on the host cores on a bounded sample

`--impl reference` times the fp64 CPU oracle instead (the only reference that
exists for this path), on the same metric and workload, one bounded sample
per step.  Under torchrun only rank 0 runs it.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402
from online_softmax_03_gb300 import accounting as acct  # noqa: E402

METRIC = "attn fwd TFLOP/s (causal-adjusted) & % bf16 peak; decode HBM GB/s & % of 8TB/s"
PREFILL = synth.PREFILL_4K
DECODE = synth.DECODE_GQA
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def source_sha(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "online_softmax_03_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


PREFILL_SOURCES = ("ptx.cuh", "prefill_kernel.cuh", "prefill.cu")
BACKWARD_SOURCES = ("ptx.cuh", "backward_kernel.cuh", "backward.cu")
DECODE_SOURCES = ("ptx.cuh", "decode_kernel.cuh", "decode.cu")


def ncu_traffic(kernel_key, sha):
    """DRAM bytes per launch recorded from an ncu capture, or None when the
    kernel source changed since the capture."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(kernel_key)
    if not e or e.get("source_sha") != sha:
        return None
    return e["dram_bytes_per_launch"]


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons in the background."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu_index), "-lms", "100"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        self.proc.wait(timeout=10)
        self.file.flush()
        self.file.seek(0)
        rows = [r.split(",") for r in self.file.read().strip().splitlines() if r.strip()]
        os.unlink(self.file.name)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm, mx, reasons = [], [], set()
        for r in rows:
            r = [x.strip() for x in r]
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except (ValueError, IndexError):
                continue
            for n, val in zip(names, r[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ------------------------------------------------------------------ CPU legs

def oracle_prefill_sample(q, k, v, n_heads):
    """Time the fp64 oracle on the first n_heads heads of batch 0 (prefill)."""
    from oracle import oracle as ora

    qs, ks, vs = (synth.bf16_bits(t[:1, :n_heads]) for t in (q, k, v))
    t0 = time.perf_counter()
    ora.attention_dense(qs, ks, vs, causal=PREFILL.causal, scale=PREFILL.scale)
    dt = time.perf_counter() - t0
    flops = acct.attention_flops(1, n_heads, PREFILL.Tq, PREFILL.Tk, PREFILL.d, PREFILL.causal)
    return flops, dt


def oracle_blocked_prefill_sample(q, k, v, n_heads, block=128):
    """Time the oracle's blocked online-softmax forward (the pages' tiled
    algorithm, block x block tiles, whole tiles above the diagonal skipped)
    on the same sample as oracle_prefill_sample."""
    from oracle import oracle as ora

    qs, ks, vs = (synth.bf16_bits(t[:1, :n_heads]) for t in (q, k, v))
    t0 = time.perf_counter()
    ora.attention_blocked(qs, ks, vs, block, block, causal=PREFILL.causal, scale=PREFILL.scale)
    dt = time.perf_counter() - t0
    flops = acct.attention_flops(1, n_heads, PREFILL.Tq, PREFILL.Tk, PREFILL.d, PREFILL.causal)
    return flops, dt


def oracle_decode_sample(q, k, v, n_batch):
    from oracle import oracle as ora

    qs, ks, vs = (synth.bf16_bits(t[:n_batch]) for t in (q, k, v))
    t0 = time.perf_counter()
    ora.attention_dense(qs, ks, vs, causal=False, scale=DECODE.scale)
    dt = time.perf_counter() - t0
    nbytes = acct.decode_bytes(n_batch, DECODE.Hq, DECODE.Hkv, DECODE.Tk, DECODE.d)
    return nbytes, dt


def omp_threads():
    try:
        return int(os.environ.get("OMP_NUM_THREADS", "")) or os.cpu_count()
    except ValueError:
        return os.cpu_count()


PREFILL_SAMPLE_HEADS = 16
DECODE_SAMPLE_BATCH = 8


def cpu_baseline(qp, kp, vp, qd, kd, vd):
    flops, dt = oracle_prefill_sample(qp, kp, vp, PREFILL_SAMPLE_HEADS)
    bflops, dtb = oracle_blocked_prefill_sample(qp, kp, vp, PREFILL_SAMPLE_HEADS)
    nbytes, dtd = oracle_decode_sample(qd, kd, vd, DECODE_SAMPLE_BATCH)
    return {
        "value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": omp_threads(),
        "kind": "oracle",
        "sample": (f"fp64 dense oracle on {PREFILL_SAMPLE_HEADS} of {PREFILL.B * PREFILL.Hq} "
                   f"heads of the prefill workload ({dt:.2f} s)"),
        "blocked": {"value": bflops / dtb / 1e12, "unit": "TFLOP/s",
                    "sample": (f"fp64 blocked online-softmax oracle (128 x 128 tiles) on the "
                               f"same {PREFILL_SAMPLE_HEADS} heads ({dtb:.2f} s)")},
        "decode": {"value": nbytes / dtd / 1e9, "unit": "GB/s",
                   "sample": (f"fp64 dense oracle on {DECODE_SAMPLE_BATCH} of {DECODE.B} "
                              f"sequences of the decode workload ({dtd:.2f} s)")},
    }


# ------------------------------------------------------- multi-rank timing

def aggregate_ranks(local: dict, world: int, device) -> dict:
    """Max over ranks of every timing in `local` (each rank runs a full
    replica, so the slowest rank bounds the whole job)."""
    if world == 1:
        return dict(local)
    import torch
    import torch.distributed as dist

    keys = sorted(local)
    t = torch.tensor([float(local[k]) for k in keys], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return {k: float(x) for k, x in zip(keys, t.tolist())}


def whole_job_rate(units_per_rank: float, seconds_max: float, world: int) -> float:
    """Units processed by all ranks divided by the slowest rank's time."""
    return world * units_per_rank / seconds_max


# ------------------------------------------------------------------ GPU arm

CONFIG_ROWS = (
    ("config1_tiny_causal", synth.TINY),
    ("config1_tiny_full", synth.TINY_NONCAUSAL),
    ("config2_prefill_1k_causal", synth.PREFILL_1K),
    ("config4_t8192_causal", synth.LONG_8K_CAUSAL),
    ("config4_t8192_full", synth.LONG_8K_FULL),
    ("config4_t8000_causal", synth.LONG_8000_CAUSAL),
    ("config4_t8000_full", synth.LONG_8000_FULL),
)
FLUSH_BYTES = 256 << 20  # twice the L2


def time_cold(fn, n, flush, stream):
    """Device time (ms) of each of n launches of fn, every launch preceded by
    an L2 flush that is not timed; the flush also covers the host's work of
    the next call, so the events bracket the kernels alone."""
    import torch

    for _ in range(3):
        flush()
        fn()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n)]
    for a, b in ev:
        flush()
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def time_config_rows(dev, stream, peak_burst):
    """Configurations 1, 2 and 4 of the specification: per-launch device time
    (p10/p50/p90 over 50 launches, each after an L2 flush), TFLOP/s with the
    causal half, and the fraction of the measured burst bf16 peak."""
    import torch

    from online_softmax_03_gb300 import binding

    flush_buf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    rows = {}
    for key, w in CONFIG_ROWS:
        q, k, v = synth.make_inputs(w, dev)
        o = torch.empty_like(q)
        lse = torch.empty((w.B, w.Hq, w.Tq), dtype=torch.float32, device=dev)
        ms = time_cold(lambda: binding.fwd(q, k, v, causal=w.causal, scale=w.scale, out=o,
                                           lse=lse),
                       50, flush_buf.zero_, stream)
        flops = acct.attention_flops(w.B, w.Hq, w.Tq, w.Tk, w.d, w.causal)
        p10, p50, p90 = percentiles(ms)
        rows[key] = {
            "workload": w.name,
            "ms_p10_p50_p90": [p10, p50, p90],
            "tflops": round(flops / (p50 / 1e3) / 1e12, 2),
            "frac_of_burst_peak": round(flops / (p50 / 1e3) / 1e12 / peak_burst, 4),
            "flops_per_launch": flops,
            "traffic": ncu_traffic(f"prefill_fwd_kernel<{w.d}>/{w.name}",
                                   source_sha(*PREFILL_SOURCES)),
        }
        del q, k, v, o, lse
    del flush_buf
    return {"rows": rows,
            "timing": ("50 launches each, every launch after an untimed 256 MB write that "
                       "flushes L2; CUDA events around each launch; median reported"),
            "kernel": "prefill_fwd_kernel<d> (d = 32, 128, 64)"}


def pick_peak(peaks, timed_s, clk):
    """The bf16 denominator for a kernel timed in this run: the burst figure
    when the timed region is short (< 1 s) or the SM clock stayed at its
    maximum, else the sustained one (measured over seconds under the power
    cap)."""
    at_max = (clk.get("sm_mhz") is not None and clk.get("sm_max_mhz")
              and clk["sm_mhz"] >= 0.97 * clk["sm_max_mhz"])
    if timed_s < 1.0 or at_max:
        why = (f"timed region {timed_s:.3f} s" + (", median SM clock at its maximum"
                                                  if at_max else ""))
        return peaks["bf16_tflops"], "bf16_tflops (burst)", why
    return (peaks["bf16_tflops_sustained"], "bf16_tflops_sustained",
            f"timed region {timed_s:.3f} s with the SM clock below its maximum")


def percentiles(ms):
    """10th, 50th and 90th percentile of this rank's per-launch times (ms)."""
    xs = sorted(ms)
    pick = lambda f: xs[min(len(xs) - 1, int(f * (len(xs) - 1) + 0.5))]
    return [round(pick(0.1), 4), round(pick(0.5), 4), round(pick(0.9), 4)]


def run_ours(args, rank, world, local_rank):
    import torch

    from online_softmax_03_gb300 import binding
    from online_softmax_03_gb300 import build as cuda_build

    cuda_build.build()
    binding.load_library()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    peaks, peak_src = load_peaks()

    qp, kp, vp = synth.make_inputs(PREFILL, dev)
    qd, kd, vd = synth.make_inputs(DECODE, dev)
    op = torch.empty_like(qp)
    lp = torch.empty((PREFILL.B, PREFILL.Hq, PREFILL.Tq), dtype=torch.float32, device=dev)
    od = torch.empty_like(qd)
    ld = torch.empty((DECODE.B, DECODE.Hq, 1), dtype=torch.float32, device=dev)
    ws = binding.decode_workspace(kd, DECODE.Hq)
    stream = torch.cuda.current_stream()

    def step():
        binding.fwd(qp, kp, vp, causal=True, out=op, lse=lp)
        binding.decode(qd, kd, vd, workspace=ws, out=od, lse=ld)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_start.record(stream)
    for i in range(K):
        ev[i][0].record(stream)
        binding.fwd(qp, kp, vp, causal=True, out=op, lse=lp)
        ev[i][1].record(stream)
        binding.decode(qd, kd, vd, workspace=ws, out=od, lse=ld)
        ev[i][2].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    total_ms = t_start.elapsed_time(t_end)
    pre_ms = [e[0].elapsed_time(e[1]) for e in ev]
    dec_ms = [e[1].elapsed_time(e[2]) for e in ev]

    # ---- end to end through the host-buffer entry points with pinned buffers
    E = max(3, min(args.e2e_steps, K))
    hq, hk, hv = (t.cpu().pin_memory() for t in (qp, kp, vp))
    hqd, hkd, hvd = (t.cpu().pin_memory() for t in (qd, kd, vd))
    ho, hl = torch.empty_like(op, device="cpu").pin_memory(), torch.empty_like(lp, device="cpu").pin_memory()
    hod, hld = torch.empty_like(od, device="cpu").pin_memory(), torch.empty_like(ld, device="cpu").pin_memory()
    eve = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(E + 1)]
    # attn_fwd_host / attn_decode_host copy the inputs in, run the kernels and
    # copy the outputs back, overlapped across chunks of the batch; their
    # device workspaces hold the device copies
    P, Dc = PREFILL, DECODE
    ws_pre = torch.empty(binding.attn_fwd_host_workspace_bytes(P.B, P.Hq, P.Hkv, P.Tq, P.Tk, P.d),
                         dtype=torch.uint8, device="cuda")
    ws_dec = torch.empty(binding.attn_decode_host_workspace_bytes(Dc.B, Dc.Hq, Dc.Hkv, Dc.Tk,
                                                                  Dc.d),
                         dtype=torch.uint8, device="cuda")

    def e2e_step(i):
        eve[i][0].record(stream)
        binding.fwd_host(hq, hk, hv, causal=True, out=ho, lse=hl, workspace=ws_pre,
                         stream=stream)
        eve[i][1].record(stream)
        binding.decode_host(hqd, hkd, hvd, out=hod, lse=hld, workspace=ws_dec, stream=stream)
        eve[i][2].record(stream)

    e2e_step(E)  # warm-up of the copy path
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    for i in range(E):
        e2e_step(i)
    torch.cuda.synchronize()
    e2e_pre_ms = sum(eve[i][0].elapsed_time(eve[i][1]) for i in range(E)) / E
    e2e_dec_ms = sum(eve[i][1].elapsed_time(eve[i][2]) for i in range(E)) / E

    pre_flops = acct.attention_flops(PREFILL.B, PREFILL.Hq, PREFILL.Tq, PREFILL.Tk, PREFILL.d,
                                     PREFILL.causal)
    dec_bytes = acct.decode_bytes(DECODE.B, DECODE.Hq, DECODE.Hkv, DECODE.Tk, DECODE.d)
    def time_alone(fn, n):
        """Average device time of n back-to-back launches of fn (ms)."""
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    # ---- the other specified configurations, each timed per launch after an
    # L2 flush (their inputs, 0.1-100 MB, would otherwise stay in the 129 MB L2)
    config_rows = None
    if not args.no_extra_rows:
        config_rows = time_config_rows(dev, stream, peaks["bf16_tflops"])

    # ---- rows beyond the specified step, each timed alone after it
    win_ms = paged_ms = varlen_ms = bwd_ms = bwd_win_ms = None
    varlen_flops = varlen_docs = 0
    if not args.no_extra_rows:
        # sliding-window prefill, then its backward (dO drawn like the inputs)
        WW = synth.WINDOW_8K
        qw, kw, vw = synth.make_inputs(WW, dev)
        ow = torch.empty_like(qw)
        lw = torch.empty(qw.shape[:3], dtype=torch.float32, device=dev)
        win_ms = time_alone(
            lambda: binding.fwd(qw, kw, vw, window=synth.WINDOW_KEYS, out=ow, lse=lw), 30)
        wdo = torch.randn(qw.shape, generator=torch.Generator(device=dev).manual_seed(1003),
                          device=dev, dtype=torch.float32).to(torch.bfloat16)
        wws = torch.empty(binding.attn_bwd_workspace_bytes(WW.B, WW.Hq, WW.Tq, WW.d),
                          dtype=torch.uint8, device=dev)
        wdq, wdk, wdv = torch.empty_like(qw), torch.empty_like(kw), torch.empty_like(vw)
        bwd_win_ms = time_alone(
            lambda: binding.bwd(qw, kw, vw, ow, lw, wdo, window=synth.WINDOW_KEYS, workspace=wws,
                                dq=wdq, dk=wdk, dv=wdv), 20)
        del qw, kw, vw, ow, lw, wdo, wws, wdq, wdk, wdv
        # decode against a paged cache (16-token pages, shuffled pool)
        pw = synth.PAGED_DECODE
        pq, pk, pv, ptab, plen = synth.make_paged_inputs(
            pw.B, pw.Hq, pw.Hkv, pw.d, synth.PAGED_PAGE_SIZE, [pw.Tk] * pw.B, pw.seed, dev)
        pws = torch.empty(binding.attn_decode_workspace_bytes(pw.B, pw.Hq, pw.Hkv, pw.Tk, pw.d),
                          dtype=torch.uint8, device=dev)
        po, pl = torch.empty_like(pq), torch.empty((pw.B, pw.Hq, 1), dtype=torch.float32,
                                                   device=dev)
        paged_ms = time_alone(
            lambda: binding.decode_paged(pq, pk, pv, ptab, plen, max_seq_len=pw.Tk,
                                         scale=pw.scale, workspace=pws, out=po, lse=pl), 100)
        del pq, pk, pv, ptab, plen, pws, po, pl
        # packed variable-length prefill (documents of mixed length)
        vw = synth.VARLEN
        vlens = synth.packed_lengths(synth.VARLEN_TOKENS, vw.seed)
        vq, vk, vv, vcq, vck = synth.make_varlen_inputs(vlens, vlens, vw.Hq, vw.Hkv, vw.d,
                                                        vw.seed, dev)
        vo = torch.empty_like(vq)
        vl = torch.empty((vw.Hq, vq.shape[0]), dtype=torch.float32, device=dev)
        vws = torch.empty(binding.attn_fwd_varlen_workspace_bytes(len(vlens), vq.shape[0],
                                                                  max(vlens)),
                          dtype=torch.uint8, device=dev)
        varlen_ms = time_alone(
            lambda: binding.fwd_varlen(vq, vk, vv, vcq, vck, max(vlens), max(vlens),
                                       causal=True, scale=vw.scale, workspace=vws, out=vo,
                                       lse=vl), 30)
        varlen_flops = acct.varlen_flops(vlens, vlens, vw.Hq, vw.d, True)
        varlen_docs = len(vlens)
        del vq, vk, vv, vcq, vck, vo, vl, vws
        # backward of the bench prefill (dO drawn like the inputs)
        gdo = torch.randn(qp.shape, generator=torch.Generator(device=dev).manual_seed(1002),
                          device=dev, dtype=torch.float32).to(torch.bfloat16)
        binding.fwd(qp, kp, vp, causal=True, out=op, lse=lp)
        bws = torch.empty(binding.attn_bwd_workspace_bytes(PREFILL.B, PREFILL.Hq, PREFILL.Tq,
                                                           PREFILL.d),
                          dtype=torch.uint8, device=dev)
        gdq, gdk, gdv = torch.empty_like(qp), torch.empty_like(kp), torch.empty_like(vp)
        bwd_ms = time_alone(
            lambda: binding.bwd(qp, kp, vp, op, lp, gdo, causal=True, workspace=bws, dq=gdq,
                                dk=gdk, dv=gdv), 20)
        del gdo, bws, gdq, gdk, gdv

    agg = aggregate_ranks(
        {"pre_s": sum(pre_ms) / 1e3, "dec_s": sum(dec_ms) / 1e3, "total_ms": total_ms,
         "e2e_pre_ms": e2e_pre_ms, "e2e_dec_ms": e2e_dec_ms},
        world, dev)
    pre_s, dec_s, total_ms = agg["pre_s"], agg["dec_s"], agg["total_ms"]
    e2e_pre_ms, e2e_dec_ms = agg["e2e_pre_ms"], agg["e2e_dec_ms"]

    pre_tflops = whole_job_rate(K * pre_flops, pre_s, world) / 1e12
    dec_gbs = whole_job_rate(K * dec_bytes, dec_s, world) / 1e9
    per_launch_tflops = pre_flops / (pre_s / K) / 1e12
    per_launch_gbs = dec_bytes / (dec_s / K) / 1e9
    peak_tf, peak_key, peak_why = pick_peak(peaks, total_ms / 1e3, clk)
    peak_bw = peaks["hbm_gbs"]
    h2d_pre = sum(t.numel() * t.element_size() for t in (qp, kp, vp))
    d2h_pre = op.numel() * 2 + lp.numel() * 4
    h2d_dec = sum(t.numel() * t.element_size() for t in (qd, kd, vd))
    d2h_dec = od.numel() * 2 + ld.numel() * 4

    paged_bytes = acct.paged_decode_bytes(
        synth.PAGED_DECODE.B, synth.PAGED_DECODE.Hq, synth.PAGED_DECODE.Hkv,
        [synth.PAGED_DECODE.Tk] * synth.PAGED_DECODE.B, synth.PAGED_DECODE.d,
        synth.PAGED_PAGE_SIZE)

    if rank != 0:
        return
    result = {
        "metric": METRIC,
        "value": round(pre_tflops, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(total_ms / K, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": workload_config(world),
        "prefill_ms": round(pre_s * 1e3 / K, 4),
        "prefill_ms_p10_p50_p90": percentiles(pre_ms),
        "roofline": {
            "kernel": "prefill_fwd_kernel<128>",
            "bound": "tensor",
            "achieved": round(per_launch_tflops, 2),
            "peak": peak_tf,
            "unit": "TFLOP/s",
            "frac": round(per_launch_tflops / peak_tf, 4),
            "peak_source": f"{peak_src} {peak_key}: {peak_why}",
            "frac_of_sustained_peak": round(per_launch_tflops / peaks["bf16_tflops_sustained"],
                                            4),
            "traffic": ncu_traffic("prefill_fwd_kernel<128>/" + PREFILL.name,
                                   source_sha(*PREFILL_SOURCES)),
            "algorithmic_flops_per_launch": pre_flops,
        },
        "decode": {
            "value": round(dec_gbs, 1),
            "unit": "GB/s",
            "ms": round(dec_s * 1e3 / K, 4),
            "ms_p10_p50_p90": percentiles(dec_ms),
            "frac_of_8TBs": round(per_launch_gbs / 8000.0, 4),
            "roofline": {
                "kernel": "decode_split_kernel<128,4> + decode_combine_kernel<128>",
                "bound": "hbm",
                "achieved": round(per_launch_gbs, 1),
                "peak": peak_bw,
                "unit": "GB/s",
                "frac": round(per_launch_gbs / peak_bw, 4),
                "peak_source": f"{peak_src} hbm_gbs",
                "traffic": ncu_traffic("decode_split_kernel<128,4>/" + DECODE.name,
                                       source_sha(*DECODE_SOURCES)),
                "algorithmic_bytes_per_launch": dec_bytes,
            },
            "e2e": {"value": round(whole_job_rate(dec_bytes, e2e_dec_ms / 1e3, world) / 1e9, 1),
                    "unit": "GB/s", "h2d_bytes_per_step": h2d_dec,
                    "d2h_bytes_per_step": d2h_dec},
        },
        "e2e": {
            "value": round(whole_job_rate(pre_flops, e2e_pre_ms / 1e3, world) / 1e12, 2),
            "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d_pre,
            "d2h_bytes_per_step": d2h_pre,
            "steps": E,
            "note": "prefill leg; the decode leg's e2e is under decode.e2e",
        },
        "window": None if win_ms is None else {
            "workload": synth.WINDOW_8K.name,
            "window_keys": synth.WINDOW_KEYS,
            "value": round(acct.window_flops(synth.WINDOW_8K.B, synth.WINDOW_8K.Hq,
                                             synth.WINDOW_8K.Tq, synth.WINDOW_8K.Tk,
                                             synth.WINDOW_8K.d, synth.WINDOW_KEYS)
                           / (win_ms / 1e3) / 1e12, 2),
            "unit": "TFLOP/s (4*d per visible pair)",
            "ms": round(win_ms, 4),
            "traffic": ncu_traffic("prefill_fwd_kernel<128,window>/" + synth.WINDOW_8K.name,
                                   source_sha(*PREFILL_SOURCES)),
            "frac_of_burst_peak": round(acct.window_flops(
                synth.WINDOW_8K.B, synth.WINDOW_8K.Hq, synth.WINDOW_8K.Tq, synth.WINDOW_8K.Tk,
                synth.WINDOW_8K.d, synth.WINDOW_KEYS) / (win_ms / 1e3) / 1e12
                / peaks["bf16_tflops"], 4),
        },
        "paged_decode": None if paged_ms is None else {
            "workload": synth.PAGED_DECODE.name,
            "page_size": synth.PAGED_PAGE_SIZE,
            "value": round(paged_bytes / (paged_ms / 1e3) / 1e9, 1),
            "unit": "GB/s",
            "ms": round(paged_ms, 4),
            "frac_of_measured_hbm": round(paged_bytes / (paged_ms / 1e3) / 1e9 / peak_bw, 4),
            "algorithmic_bytes_per_launch": paged_bytes,
            "traffic": ncu_traffic("decode_split_kernel<128,4,paged>/" + synth.PAGED_DECODE.name,
                                   source_sha(*DECODE_SOURCES)),
        },
        "varlen": None if varlen_ms is None else {
            "workload": synth.VARLEN.name,
            "documents": varlen_docs,
            "value": round(varlen_flops / (varlen_ms / 1e3) / 1e12, 2),
            "unit": "TFLOP/s (4*d per visible pair)",
            "ms": round(varlen_ms, 4),
            "frac_of_burst_peak": round(varlen_flops / (varlen_ms / 1e3) / 1e12
                                        / peaks["bf16_tflops"], 4),
            "launches": "planning kernel + prefill kernel",
            "traffic": ncu_traffic("prefill_fwd_kernel<128,varlen>/" + synth.VARLEN.name,
                                   source_sha(*PREFILL_SOURCES)),
        },
        "backward": None if bwd_ms is None else {
            "workload": PREFILL.name,
            "value": round(acct.backward_flops(PREFILL.B, PREFILL.Hq, PREFILL.Tq, PREFILL.Tk,
                                               PREFILL.d, True) / (bwd_ms / 1e3) / 1e12, 2),
            "unit": "TFLOP/s (5 products, causal half)",
            "ms": round(bwd_ms, 4),
            "frac_of_burst_peak": round(acct.backward_flops(
                PREFILL.B, PREFILL.Hq, PREFILL.Tq, PREFILL.Tk, PREFILL.d, True)
                / (bwd_ms / 1e3) / 1e12 / peaks["bf16_tflops"], 4),
            "launches": "prep + backward kernel + dQ conversion",
            "dq_reduction": {
                "bound": "fp32 reductions into the dQ accumulator (L2)",
                "bytes_per_call": acct.backward_dq_reduction_bytes(
                    PREFILL.B, PREFILL.Hq, PREFILL.Tq, PREFILL.Tk, PREFILL.d, True),
                "achieved_tb_s_whole_call": round(acct.backward_dq_reduction_bytes(
                    PREFILL.B, PREFILL.Hq, PREFILL.Tq, PREFILL.Tk, PREFILL.d, True)
                    / (bwd_ms / 1e3) / 1e12, 3),
            },
            "traffic_main_kernel": ncu_traffic("attn_bwd_bm128_kernel/" + PREFILL.name,
                                               source_sha(*BACKWARD_SOURCES)),
        },
        "backward_window": None if bwd_win_ms is None else {
            "workload": synth.WINDOW_8K.name,
            "window_keys": synth.WINDOW_KEYS,
            "value": round(2.5 * acct.window_flops(
                synth.WINDOW_8K.B, synth.WINDOW_8K.Hq, synth.WINDOW_8K.Tq, synth.WINDOW_8K.Tk,
                synth.WINDOW_8K.d, synth.WINDOW_KEYS) / (bwd_win_ms / 1e3) / 1e12, 2),
            "unit": "TFLOP/s (5 products over the visible pairs, 2.5 x the window forward count)",
            "ms": round(bwd_win_ms, 4),
            "launches": "prep + backward kernel + dQ conversion",
            "dq_reduction_bytes_per_call": acct.backward_dq_reduction_bytes(
                synth.WINDOW_8K.B, synth.WINDOW_8K.Hq, synth.WINDOW_8K.Tq, synth.WINDOW_8K.Tk,
                synth.WINDOW_8K.d, True, window=synth.WINDOW_KEYS),
            "traffic_main_kernel": ncu_traffic("attn_bwd_bm128_kernel/" + synth.WINDOW_8K.name,
                                               source_sha(*BACKWARD_SOURCES)),
        },
        "configs": config_rows,
        "gpu_launches": K * 3,
        "clocks": clk,
    }
    if world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(qp, kp, vp, qd, kd, vd)
    print(json.dumps(result), flush=True)


# --------------------------------------------------------- reference arm

def _reference_rows(n, T, heads, offset):
    """n (h, i) rows spread evenly over the heads and the causal row range."""
    import numpy as np

    idx = (np.arange(n, dtype=np.int64) * 7919 + offset) % (heads * T)
    return np.zeros(n, np.int32), (idx // T).astype(np.int32), (idx % T).astype(np.int32)


def workload_config(world):
    """The workload both arms report (the reference arm times a bounded
    sample of it, described in its cpu_baseline)."""
    return {
        "workload": f"{PREFILL.name} + {DECODE.name}",
        "prefill": {"B": PREFILL.B, "Hq": PREFILL.Hq, "Hkv": PREFILL.Hkv, "Tq": PREFILL.Tq,
                    "Tk": PREFILL.Tk, "d": PREFILL.d, "causal": PREFILL.causal,
                    "dist": PREFILL.dist, "seed": PREFILL.seed},
        "decode": {"B": DECODE.B, "Hq": DECODE.Hq, "Hkv": DECODE.Hkv, "Tq": 1,
                   "Tk": DECODE.Tk, "d": DECODE.d, "causal": False,
                   "dist": DECODE.dist, "seed": DECODE.seed},
        "l2": "no flush: inputs exceed the 129 MB L2 (prefill q+k+v 403 MB, decode cache 2.1 GB)",
        "parallelism": f"replicas x{world} (each rank runs the full workload)",
    }


def run_reference(args, rank, world):
    """Time the fp64 oracle (the only reference for this path) on the host
    cores: each step evaluates a bounded, evenly spread sample of rows of the
    causal prefill workload; FLOPs count 4*d per visible (row, key) pair."""
    from oracle import oracle as ora

    if rank != 0:
        return
    heads = 4
    w = PREFILL.with_(B=1, Hq=heads, Hkv=heads)
    q, k, v = (synth.bf16_bits(t) for t in synth.make_inputs(w, "cpu"))
    budget = min(2.0, 150.0 / (args.steps + args.warmup))

    def one(n, offset):
        rb, rh, ri = _reference_rows(n, w.Tq, heads, offset)
        t0 = time.perf_counter()
        ora.attention_rows(q, k, v, rb, rh, ri, causal=True, scale=w.scale)
        dt = time.perf_counter() - t0
        flops = float(4 * w.d * (ri.astype("int64") + 1).sum())
        return flops, dt

    f, dt = one(256, 0)
    n_rows = int(max(32, min(heads * w.Tq, 256 * budget / max(dt, 1e-6))))
    flops_total, t_total = 0.0, 0.0
    for step in range(args.warmup + args.steps):
        flops, dt = one(n_rows, step * 104729)
        if step >= args.warmup:
            flops_total += flops
            t_total += dt
    value = flops_total / t_total / 1e12
    sample = (f"each step: fp64 oracle on {n_rows} rows spread over {heads} causal heads "
              f"of the prefill workload (T=4096, d=128); inputs drawn on the CPU")
    result = {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": t_total * 1e3 / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": workload_config(world),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": omp_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(result), flush=True)


PROFILE_WORKLOADS = {w.name: w for w in synth.ALL + (synth.WINDOW_8K, synth.PAGED_DECODE,
                                                     synth.VARLEN)}


def run_profile(args):
    """Profiling case: `--launches` launches of one workload's kernels and
    nothing else, so that an ncu capture (-k, -s, -c) runs in a process that
    holds only that workload's tensors.  Prints one line naming what ran; it
    is not a bench line."""
    import torch

    from online_softmax_03_gb300 import binding
    from online_softmax_03_gb300 import build as cuda_build

    cuda_build.build()
    binding.load_library()
    name = args.profile
    backward = name.endswith(":bwd")
    w = PROFILE_WORKLOADS[name[:-4] if backward else name]
    dev = torch.device("cuda", 0)
    if w is synth.PAGED_DECODE:
        pq, pk, pv, tab, lens = synth.make_paged_inputs(
            w.B, w.Hq, w.Hkv, w.d, synth.PAGED_PAGE_SIZE, [w.Tk] * w.B, w.seed, dev)
        fn = lambda: binding.decode_paged(pq, pk, pv, tab, lens, max_seq_len=w.Tk,  # noqa
                                          scale=w.scale)
    elif w is synth.VARLEN:
        lens = synth.packed_lengths(synth.VARLEN_TOKENS, w.seed)
        vq, vk, vv, cq, ck = synth.make_varlen_inputs(lens, lens, w.Hq, w.Hkv, w.d, w.seed, dev)
        fn = lambda: binding.fwd_varlen(vq, vk, vv, cq, ck, max(lens), max(lens),  # noqa
                                        causal=True, scale=w.scale)
    if w is synth.PAGED_DECODE or w is synth.VARLEN:
        for _ in range(args.launches):
            fn()
        torch.cuda.synchronize()
        assert binding.attn_device_status() == binding.ATTN_OK
        print(json.dumps({"profile": name, "launches": args.launches,
                          "device_bytes": torch.cuda.max_memory_allocated()}), flush=True)
        return
    q, k, v = synth.make_inputs(w, dev)
    if w.decode:
        ws = binding.decode_workspace(k, w.Hq)
        o, lse = torch.empty_like(q), torch.empty((w.B, w.Hq, 1), dtype=torch.float32, device=dev)
        fn = lambda: binding.decode(q, k, v, workspace=ws, out=o, lse=lse)  # noqa: E731
    else:
        window = synth.WINDOW_KEYS if w is synth.WINDOW_8K else None
        o, lse = binding.fwd(q, k, v, causal=w.causal, scale=w.scale, window=window)
        fn = lambda: binding.fwd(q, k, v, causal=w.causal, scale=w.scale, window=window,  # noqa
                                 out=o, lse=lse)
        if backward:
            do = torch.randn(q.shape, generator=torch.Generator(device=dev).manual_seed(1002),
                             device=dev, dtype=torch.float32).to(torch.bfloat16)
            bws = torch.empty(binding.attn_bwd_workspace_bytes(w.B, w.Hq, w.Tq, w.d),
                              dtype=torch.uint8, device=dev)
            dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
            fn = lambda: binding.bwd(q, k, v, o, lse, do, causal=w.causal, scale=w.scale,  # noqa
                                     window=window, workspace=bws, dq=dq, dk=dk, dv=dv)
    for _ in range(args.launches):
        fn()
    torch.cuda.synchronize()
    assert binding.attn_device_status() == binding.ATTN_OK
    print(json.dumps({"profile": name, "launches": args.launches,
                      "device_bytes": torch.cuda.max_memory_allocated()}), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra-rows", action="store_true",
                    help="skip the separately timed rows beyond the specified step")
    ap.add_argument("--profile", choices=sorted(PROFILE_WORKLOADS) +
                    sorted(n + ":bwd" for n in PROFILE_WORKLOADS
                           if "decode" not in n and "varlen" not in n),
                    help="run only this workload's kernels (for ncu captures); "
                         "NAME:bwd runs the backward")
    ap.add_argument("--launches", type=int, default=3)
    args = ap.parse_args()
    if args.profile:
        run_profile(args)
        return
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus:
        print(f"warning: --gpus {args.gpus} but WORLD_SIZE={world}", file=sys.stderr)
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch

        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch

            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
