"""ssm_decode_step on the GPU against the fp64 oracle (cached-state decode, batched over requests)."""
import numpy as np
import pytest
import torch

import oracle
from _gpu import assert_parity, assert_rel_close, assert_rms_close, oracle_prefill, run_prefill
from selective_state_space_prefill_gb300 import binding as ssm
from selective_state_space_prefill_gb300.inputs import (make_decode_inputs, make_mixer_inputs,
                                                        make_mixer_params, make_states)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _oracle_step(tok, par, cs, ss):
    return oracle.decode_step(tok["x"], tok["z"], tok["dt"], tok["B"], tok["C"], par["A"], par["D"],
                              par["dt_bias"], par["conv_w"], par["conv_b"], cs, ss)


def _gpu_step(tok, par, cs, ss, slot=None, out_dtype=torch.float32):
    return ssm.decode_step(tok["x"], tok["z"], tok["dt"], tok["B"], tok["C"], par["A"], par["D"],
                           par["dt_bias"], par["conv_w"], par["conv_b"], cs, ss, state_slot=slot,
                           out_dtype=out_dtype)


@pytest.mark.parametrize("batch", [1, 8, 64, 256])
def test_decode_from_random_states(batch):
    """The decode sweep: batch 1/8/64/256, d_inner 8192, fp32 cached states ~ N(0,1), bf16 tokens."""
    D = 8192
    par = make_mixer_params(D, seed=1)
    tok = make_decode_inputs(batch, D, seed=batch)
    cs, ss = make_states(batch, D, seed=batch + 1)
    ref = _oracle_step(tok, par, cs, ss)
    gpar = {k: v.to(DEV) for k, v in par.items()}
    gtok = {k: v.to(DEV) for k, v in tok.items()}
    gcs, gss = cs.to(DEV), ss.to(DEV)
    out = _gpu_step(gtok, gpar, gcs, gss)
    torch.cuda.synchronize()
    assert_rms_close(out, ref["out"], 2e-3, "out")
    assert_rms_close(gss, ref["ssm_state"], 2e-3, "ssm_state")
    assert np.array_equal(gcs.cpu().double().numpy(), ref["conv_state"])
    assert ssm.device_status() == 0


def test_decode_fp32_tokens_and_bf16_out():
    D = 64
    par = make_mixer_params(D, seed=2)
    tok = make_decode_inputs(5, D, dtype=torch.float32, seed=3)
    cs, ss = make_states(5, D, seed=4)
    ref = _oracle_step(tok, par, cs, ss)
    gcs, gss = cs.to(DEV), ss.to(DEV)
    out = _gpu_step({k: v.to(DEV) for k, v in tok.items()}, {k: v.to(DEV) for k, v in par.items()}, gcs, gss)
    assert_rel_close(out, ref["out"], 1e-5, "fp32 out")
    assert_rel_close(gss, ref["ssm_state"], 1e-5, "fp32 state")
    gcs2, gss2 = cs.to(DEV), ss.to(DEV)
    outb = _gpu_step({k: v.to(DEV) for k, v in tok.items()}, {k: v.to(DEV) for k, v in par.items()}, gcs2, gss2,
                     out_dtype=torch.bfloat16)
    assert torch.equal(outb, out.to(torch.bfloat16))


def test_decode_state_slots():
    """Requests name their cache slots; other slots stay bit-identical."""
    D, n_slots, batch = 96, 10, 4
    par = make_mixer_params(D, seed=5)
    tok = make_decode_inputs(batch, D, seed=6)
    cs, ss = make_states(n_slots, D, seed=7)
    slots = torch.tensor([7, 2, 9, 0], dtype=torch.int32)
    ref = _oracle_step(tok, par, cs[slots.long()], ss[slots.long()])
    gcs, gss = cs.to(DEV), ss.to(DEV)
    out = _gpu_step({k: v.to(DEV) for k, v in tok.items()}, {k: v.to(DEV) for k, v in par.items()},
                    gcs, gss, slot=slots.to(DEV))
    torch.cuda.synchronize()
    assert_rms_close(out, ref["out"], 2e-3, "slot out")
    assert_rms_close(gss[slots.long().to(DEV)], ref["ssm_state"], 2e-3, "slot state")
    untouched = [i for i in range(n_slots) if i not in slots.tolist()]
    assert torch.equal(gss[untouched].cpu(), ss[untouched])
    assert torch.equal(gcs[untouched].cpu(), cs[untouched])


def test_decode_bad_slot_is_reported_not_faulting():
    """An out-of-range slot index skips that request and sets SSM_DEV_BAD_SLOT."""
    D = 32
    par = {k: v.to(DEV) for k, v in make_mixer_params(D, seed=8).items()}
    tok = {k: v.to(DEV) for k, v in make_decode_inputs(2, D, seed=9).items()}
    cs, ss = (t.to(DEV) for t in make_states(2, D, seed=10))
    before = ss.clone()
    ssm.device_status(clear=True)
    out = torch.full((2, D), 123.0, device=DEV)
    ssm.decode_step(tok["x"], tok["z"], tok["dt"], tok["B"], tok["C"], par["A"], par["D"], par["dt_bias"],
                    par["conv_w"], par["conv_b"], cs, ss, state_slot=torch.tensor([1, 5], dtype=torch.int32,
                                                                                    device=DEV), out=out)
    st = ssm.device_status(clear=True)
    assert st & ssm.DEV_BAD_SLOT
    assert torch.equal(out[1], torch.full((D,), 123.0, device=DEV))   # skipped request untouched
    assert not torch.equal(ss[1], before[1])                           # slot 1 was updated
    assert torch.equal(ss[0], before[0])
    assert ssm.device_status() == 0


@pytest.mark.parametrize("dtype,tol", [(torch.float32, 1e-5), (torch.bfloat16, 2e-3)])
def test_prefill_then_decode_equals_prefill(dtype, tol):
    """The tiny mixer: prefill 192 tokens, then 64 single-token decode steps, vs prefill of all 256."""
    L1, L2, D = 192, 64, 64
    inp = make_mixer_inputs(1, L1 + L2, D, dtype=dtype, seed=0)
    ref = oracle_prefill(inp)
    g = inp.to(DEV)
    _, cs, ss = run_prefill(inp.token_slice(0, L1).to(DEV))
    xs, zs, dts = (getattr(g, k).transpose(0, 1).contiguous() for k in ("x", "z", "dt"))
    Bs, Cs = (getattr(g, k).transpose(0, 1).contiguous() for k in ("B", "C"))
    outs = []
    for t in range(L1, L1 + L2):
        outs.append(ssm.decode_step(xs[t], zs[t], dts[t], Bs[t], Cs[t], g.A, g.D, g.dt_bias, g.conv_w,
                                    g.conv_b, cs, ss))
    torch.cuda.synchronize()
    assert_parity(torch.stack(outs, 1), ref["out"][:, L1:], dtype, "decode tail")
    assert_parity(ss, ref["ssm_state"], dtype, "final ssm_state")
    assert np.array_equal(cs.cpu().double().numpy(), ref["conv_state"])


# ---------------------------------------------------------------- multi-token blocks
@pytest.mark.parametrize("T", [1, 2, 5, 16])
@pytest.mark.parametrize("dtype,tol", [(torch.bfloat16, 2e-3), (torch.float32, 1e-5)])
def test_decode_tokens_matches_oracle(T, dtype, tol):
    """T tokens per request from random cached states = the oracle's prefill of those tokens from the states."""
    batch, D = 3, 96
    inp = make_mixer_inputs(batch, T, D, dtype=dtype, seed=100 + T)
    cs, ss = make_states(batch, D, seed=200 + T)
    ref = oracle_prefill(inp, cs, ss)
    g = inp.to(DEV)
    gcs, gss = cs.to(DEV), ss.to(DEV)
    out = ssm.decode_tokens(g.x, g.z, g.dt, g.B, g.C, g.A, g.D, g.dt_bias, g.conv_w, g.conv_b, gcs, gss)
    torch.cuda.synchronize()
    assert out.shape == (batch, T, D)
    assert_parity(out, ref["out"], dtype, "block out")
    assert_parity(gss, ref["ssm_state"], dtype, "block state")
    assert np.array_equal(gcs.cpu().double().numpy(), ref["conv_state"])


def test_decode_tokens_one_token_equals_decode_step():
    D = 128
    par = {k: v.to(DEV) for k, v in make_mixer_params(D, seed=11).items()}
    tok = {k: v.to(DEV) for k, v in make_decode_inputs(4, D, seed=12).items()}
    cs, ss = (t.to(DEV) for t in make_states(4, D, seed=13))
    cs2, ss2 = cs.clone(), ss.clone()
    o1 = _gpu_step(tok, par, cs, ss)
    o2 = ssm.decode_tokens(tok["x"][:, None], tok["z"][:, None], tok["dt"][:, None], tok["B"][:, None].contiguous(),
                           tok["C"][:, None].contiguous(), par["A"], par["D"], par["dt_bias"], par["conv_w"],
                           par["conv_b"], cs2, ss2)
    assert torch.equal(o1, o2[:, 0]) and torch.equal(ss, ss2) and torch.equal(cs, cs2)


def test_decode_tokens_slots_and_prefill_continuation():
    """Prefill 40 tokens into slots 3 and 1, then an 8-token block per request through the slots,
    against the oracle's 48-token prefill."""
    D, L1, T = 64, 40, 8
    inp = make_mixer_inputs(2, L1 + T, D, dtype=torch.bfloat16, seed=21)
    ref = oracle_prefill(inp)
    g = inp.to(DEV)
    _, cs, ss = run_prefill(inp.token_slice(0, L1).to(DEV))
    conv = torch.zeros(5, 3, D, device=DEV)
    ssm_s = torch.zeros(5, D, 16, device=DEV)
    slots = torch.tensor([3, 1], dtype=torch.int32, device=DEV)
    conv[slots.long()] = cs
    ssm_s[slots.long()] = ss
    blk = inp.token_slice(L1, L1 + T).to(DEV)
    out = ssm.decode_tokens(blk.x, blk.z, blk.dt, blk.B, blk.C, g.A, g.D, g.dt_bias, g.conv_w, g.conv_b, conv, ssm_s,
                            state_slot=slots)
    torch.cuda.synchronize()
    assert_rms_close(out, ref["out"][:, L1:], 2e-3, "block after prefill")
    assert_rms_close(ssm_s[slots.long()], ref["ssm_state"], 2e-3, "slot states")
    assert torch.equal(conv[0], torch.zeros(3, D, device=DEV)) and torch.equal(ssm_s[2], torch.zeros(D, 16, device=DEV))


def test_decode_tokens_longest_block():
    """The largest block the ABI accepts, 4096 tokens per request, against the oracle."""
    batch, T, D = 2, 4096, 32
    inp = make_mixer_inputs(batch, T, D, dtype=torch.bfloat16, seed=41)
    cs, ss = make_states(batch, D, seed=42)
    ref = oracle_prefill(inp, cs, ss)
    g = inp.to(DEV)
    gcs, gss = cs.to(DEV), ss.to(DEV)
    out = ssm.decode_tokens(g.x, g.z, g.dt, g.B, g.C, g.A, g.D, g.dt_bias, g.conv_w, g.conv_b, gcs, gss)
    torch.cuda.synchronize()
    assert_parity(out, ref["out"], torch.bfloat16, "4096-token block out")
    assert_parity(gss, ref["ssm_state"], torch.bfloat16, "4096-token block state")
    assert np.array_equal(gcs.cpu().double().numpy(), ref["conv_state"])
