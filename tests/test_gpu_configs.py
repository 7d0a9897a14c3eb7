"""The full-size workloads on the GPU, in the launch configuration the benchmark times.

The oracle evaluates sampled channels one by one (channels are independent, so
a sample is the same computation restricted to those channels); invariants that
hold at any size are checked on every channel.
"""
import numpy as np
import pytest
import torch

from _gpu import assert_rms_close, cpu_channels, oracle_prefill, run_prefill, sample_channels
from selective_state_space_prefill_gb300 import binding as ssm
from selective_state_space_prefill_gb300.inputs import make_mixer_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL = 2e-3


def _slice_call(inp, lo, hi, out, cso, sso, L=None, cs=None, ss=None):
    sl = slice(lo, hi)
    t = slice(0, L)
    return ssm.prefill(inp.x[:, t, sl], inp.z[:, t, sl], inp.dt[:, t, sl], inp.B[:, t].contiguous() if L else inp.B,
                       inp.C[:, t].contiguous() if L else inp.C, inp.A[sl].contiguous(), inp.D[sl].contiguous(),
                       inp.dt_bias[sl].contiguous(), inp.conv_w[sl].contiguous(), inp.conv_b[sl].contiguous(),
                       conv_state_in=cs, ssm_state_in=ss, out=out, conv_state_out=cso, ssm_state_out=sso)


def test_mamba130m_layer_sampled():
    """Mamba-130M-like layer: batch 4, L 2048, d_inner 1536, bf16, prefill only."""
    inp = make_mixer_inputs(4, 2048, 1536, dtype=torch.bfloat16, seed=0, device=DEV)
    out, cs, ss = run_prefill(inp)
    torch.cuda.synchronize()
    idx = sample_channels(1536, 48, seed=1)
    ref = oracle_prefill(cpu_channels(inp, idx))
    ix = torch.as_tensor(idx, device=DEV)
    assert_rms_close(out.index_select(2, ix), ref["out"], TOL, "out")
    assert_rms_close(ss.index_select(1, ix), ref["ssm_state"], TOL, "ssm_state")
    assert np.array_equal(cs.index_select(2, ix).cpu().double().numpy(), ref["conv_state"])
    assert torch.isfinite(out).all()


def test_falcon_mamba_slices_bit_exact_then_decode():
    """Falcon-Mamba-7B-like: 4 slices of 2048 of d_inner 8192, L 16384, bit-exact vs the unsplit run;
    then 512 decode steps from one slice's cached state against the oracle."""
    Dfull, S, L, steps = 8192, 2048, 16384, 512
    inp = make_mixer_inputs(1, L + steps, Dfull, dtype=torch.bfloat16, seed=0, device=DEV)
    pre = inp.token_slice(0, L)
    full_out, full_cs, full_ss = run_prefill(pre)
    out = torch.empty_like(full_out)
    cso = torch.empty_like(full_cs)
    sso = torch.empty_like(full_ss)
    for s in range(4):
        sl = slice(S * s, S * (s + 1))
        _slice_call(pre, S * s, S * (s + 1), out[..., sl], cso[:, :, sl], sso[:, sl])
    torch.cuda.synchronize()
    assert torch.equal(out, full_out), "slice outputs differ from the unsplit run"
    assert torch.equal(sso, full_ss) and torch.equal(cso, full_cs), "slice states differ"

    # oracle on sampled channels of slice 1, over all L + steps tokens
    lo = S
    idx = lo + sample_channels(S, 16, seed=2)
    ref = oracle_prefill(cpu_channels(inp, idx))
    ix = torch.as_tensor(idx, device=DEV)
    assert_rms_close(full_out.index_select(2, ix), ref["out"][:, :L], TOL, "prefill out")

    # decode from the slice's cached state (views into the full state buffers)
    sl = slice(lo, lo + S)
    cs, ss = cso[:, :, sl], sso[:, sl]
    A, D, dtb, w, b = (getattr(inp, k)[sl].contiguous() for k in ("A", "D", "dt_bias", "conv_w", "conv_b"))
    outs = []
    for t in range(L, L + steps):
        outs.append(ssm.decode_step(inp.x[:, t, sl], inp.z[:, t, sl], inp.dt[:, t, sl], inp.B[:, t], inp.C[:, t],
                                    A, D, dtb, w, b, cs, ss))
    torch.cuda.synchronize()
    dec = torch.stack(outs, 1)                        # [1, steps, S]
    assert_rms_close(dec.index_select(2, ix - lo), ref["out"][:, L:], TOL, "decode out")
    assert_rms_close(ss.index_select(1, ix - lo), ref["ssm_state"], TOL, "decode state")
    assert ssm.device_status() == 0


def test_zamba_long_context_sampled_and_cached():
    """Zamba-7B-like: d_inner 7168, L 65536 prefill; and 49152 prefill + 16384 decode steps vs the full prefill."""
    D, L, L1 = 7168, 65536, 49152
    inp = make_mixer_inputs(1, L, D, dtype=torch.bfloat16, seed=0, device=DEV)
    out, cs, ss = run_prefill(inp)
    torch.cuda.synchronize()
    idx = sample_channels(D, 24, seed=3)
    ix = torch.as_tensor(idx, device=DEV)
    ref = oracle_prefill(cpu_channels(inp, idx))
    assert_rms_close(out.index_select(2, ix), ref["out"], TOL, "long prefill out")
    assert_rms_close(ss.index_select(1, ix), ref["ssm_state"], TOL, "long prefill state")

    part = inp.token_slice(0, L1)
    _, pcs, pss = run_prefill(part)
    dec = torch.empty(1, L - L1, D, device=DEV)
    for i, t in enumerate(range(L1, L)):
        ssm.decode_step(inp.x[:, t], inp.z[:, t], inp.dt[:, t], inp.B[:, t], inp.C[:, t], inp.A, inp.D,
                        inp.dt_bias, inp.conv_w, inp.conv_b, pcs, pss, out=dec[:, i])
    torch.cuda.synchronize()
    assert_rms_close(dec.index_select(2, ix), ref["out"][:, L1:], TOL, "cached decode out")
    assert_rms_close(pss.index_select(1, ix), ref["ssm_state"], TOL, "cached decode state")
    # every channel: decode continuation vs the one-call prefill (both GPU, compared on the GPU)
    ref_all = out[:, L1:].double()
    err = (dec.double() - ref_all).abs().max().item()
    rms = ref_all.pow(2).mean().sqrt().item()
    assert err <= TOL * rms, f"decode vs prefill, all channels: {err:.3e} > {TOL} * {rms:.3e}"
    assert torch.equal(pcs, cs)
