"""attn_fwd_host / attn_decode_host: attention from and to pinned host memory,
copies and kernels overlapped across chunks of (batch, K/V head) slices.

The forward's rows must match a single device attn_fwd call bit for bit on
every chunk plan (one chunk, whole batches per chunk, runs of K/V heads of
one batch, uneven runs); the decode, whose key splits depend on how many
sequences a launch holds, must agree with attn_decode to rounding and with
the oracle within the parity bounds."""
import numpy as np
import pytest
import torch

import synth
from oracle import oracle as ora
from online_softmax_03_gb300 import binding
from parity import assert_close

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from online_softmax_03_gb300 import build as cuda_build

    cuda_build.build()
    binding.load_library()
    assert binding.attn_device_status() == binding.ATTN_OK
    yield
    assert binding.attn_device_status() == binding.ATTN_OK


def _pinned(*ts):
    return [t.cpu().pin_memory() for t in ts]


# Problem sizes against the 16 MB chunk target: 1 chunk; 2 chunks of 4
# whole batches; 2 chunks of 2 K/V heads of one batch; 12 uneven runs of
# 3, 3 and 2 K/V heads over 4 batches; ragged Tq < Tk in one chunk.
@pytest.mark.parametrize("B,Hq,Hkv,Tq,Tk,d,causal", [
    (1, 4, 2, 300, 300, 64, True),
    (8, 4, 4, 2048, 2048, 64, False),
    (1, 16, 4, 4096, 4096, 128, True),
    (4, 32, 8, 2048, 2048, 128, True),
    (3, 6, 3, 1000, 1500, 128, True),
    (2, 8, 8, 777, 777, 32, False),
])
def test_fwd_host_matches_device_call_bit_for_bit(B, Hq, Hkv, Tq, Tk, d, causal):
    w = synth.Workload("host", B, Hq, Hkv, Tq, Tk, d, causal, "normal", Tq + d + B)
    q, k, v = synth.make_inputs(w, DEV)
    o_dev, l_dev = binding.fwd(q, k, v, causal=causal)
    hq, hk, hv = _pinned(q, k, v)
    o_h, l_h = binding.fwd_host(hq, hk, hv, causal=causal)
    torch.cuda.synchronize()
    assert torch.equal(o_h.view(torch.int16), o_dev.cpu().view(torch.int16))
    assert torch.equal(l_h, l_dev.cpu())


def test_fwd_host_against_oracle_with_explicit_scale():
    w = synth.Workload("host_oracle", 2, 4, 2, 200, 333, 64, True, "normal", 31)
    q, k, v = synth.make_inputs(w, DEV)
    hq, hk, hv = _pinned(q, k, v)
    o, lse = binding.fwd_host(hq, hk, hv, causal=True, scale=0.2)
    torch.cuda.synchronize()
    o_ref, lse_ref, _ = ora.attention_dense(synth.bf16_bits(q), synth.bf16_bits(k),
                                            synth.bf16_bits(v), causal=True, scale=0.2)
    assert_close(o, lse, o_ref, lse_ref, "fwd_host scale 0.2")


def test_fwd_host_honours_the_stream_and_reuses_buffers():
    """Work on a side stream: the outputs are complete once that stream is
    synchronised, and a second call into the same buffers overwrites them."""
    w = synth.Workload("host_stream", 2, 8, 2, 2048, 2048, 128, True, "normal", 32)
    q, k, v = synth.make_inputs(w, DEV)
    o_dev, l_dev = binding.fwd(q, k, v, causal=True)
    hq, hk, hv = _pinned(q, k, v)
    out = torch.full(q.shape, 7.0, dtype=torch.bfloat16).pin_memory()
    lse = torch.full((2, 8, 2048), -1.0).pin_memory()
    ws = torch.empty(binding.attn_fwd_host_workspace_bytes(2, 8, 2, 2048, 2048, 128),
                     dtype=torch.uint8, device=DEV)
    s = torch.cuda.Stream()
    for _ in range(2):
        binding.fwd_host(hq, hk, hv, causal=True, out=out, lse=lse, workspace=ws, stream=s)
        s.synchronize()
        assert torch.equal(out.view(torch.int16), o_dev.cpu().view(torch.int16))
        assert torch.equal(lse, l_dev.cpu())
        out.fill_(0.0)


@pytest.mark.parametrize("B,Hq,Hkv,Tk,d", [
    (3, 8, 2, 500, 128),      # one chunk
    (64, 32, 8, 1024, 128),   # 16 chunks of 4 whole sequences
    (2, 16, 4, 16384, 128),   # runs of K/V heads of one sequence
    (5, 12, 2, 3000, 64),
])
def test_decode_host_matches_device_call_and_oracle(B, Hq, Hkv, Tk, d):
    w = synth.Workload("host_dec", B, Hq, Hkv, 1, Tk, d, False, "normal", B + Tk)
    q, k, v = synth.make_inputs(w, DEV)
    o_dev, l_dev = binding.decode(q, k, v)
    hq, hk, hv = _pinned(q, k, v)
    o_h, l_h = binding.decode_host(hq, hk, hv)
    torch.cuda.synchronize()
    # to rounding against the single device call
    assert (o_h.float() - o_dev.cpu().float()).abs().max().item() <= 1e-2
    assert (l_h - l_dev.cpu()).abs().max().item() <= 1e-4
    # and within the parity bounds against the oracle, on up to 8 sequences
    nb = min(B, 8)
    o_ref, lse_ref, _ = ora.attention_dense(synth.bf16_bits(q[:nb]), synth.bf16_bits(k[:nb]),
                                            synth.bf16_bits(v[:nb]), causal=False)
    assert_close(o_h[:nb], l_h[:nb], o_ref, lse_ref, f"decode_host b{B} tk{Tk}")


def test_host_entry_points_reject_a_short_workspace():
    x = torch.zeros(1, 2, 128, 64, dtype=torch.bfloat16).pin_memory()
    with pytest.raises(binding.AttnError):
        binding.fwd_host(x, x, x, workspace=torch.empty(256, dtype=torch.uint8, device=DEV))
    q = torch.zeros(1, 2, 1, 64, dtype=torch.bfloat16).pin_memory()
    with pytest.raises(binding.AttnError):
        binding.decode_host(q, x, x, workspace=torch.empty(256, dtype=torch.uint8, device=DEV))
