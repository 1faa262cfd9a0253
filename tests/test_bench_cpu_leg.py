"""bench.py's CPU leg on this host: the oracle's dense and blocked forwards
time the same slice of the prefill workload (one head here) and report the
same algorithmic FLOPs (no GPU)."""
import bench
import synth


def test_dense_and_blocked_oracle_samples_report_the_same_work():
    w = synth.PREFILL_4K.with_(B=1, Hq=1, Hkv=1)
    q, k, v = synth.make_inputs(w, "cpu")
    flops, dt = bench.oracle_prefill_sample(q, k, v, 1)
    bflops, dtb = bench.oracle_blocked_prefill_sample(q, k, v, 1)
    assert flops == bflops == 2 * 4096 * 4096 * 128  # causal half of 4*T^2*d, one head
    assert dt > 0 and dtb > 0
