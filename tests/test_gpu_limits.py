"""Largest sizes the ABI accepts, where a 32-bit index would overflow.

* a prefill whose [B, L, D] tensors hold more than 2^31 elements (the last batch row
  crosses element 2^31), checked against the oracle on sampled channels;
* q8 over n = 2^31 + 77 elements, checked block by block at both ends and around 2^31;
* decode and prefill at the largest batch, 65535.
"""
import numpy as np
import pytest
import torch

import oracle
from _gpu import assert_rms_close, cpu_channels, half_ulp_bf16, oracle_prefill, sample_channels
from selective_state_space_prefill_gb300 import binding as ssm
from selective_state_space_prefill_gb300.inputs import make_decode_inputs, make_mixer_inputs, make_mixer_params, \
    make_partials, make_states

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _free():
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def test_prefill_tensors_beyond_2e31_elements():
    B, L, D = 4, 65600, 8192
    assert (B - 1) * L * D < 2 ** 31 < B * L * D
    inp = make_mixer_inputs(B, L, D, dtype=torch.bfloat16, seed=5, device=DEV)
    out, cs, ss = ssm.prefill(inp.x, inp.z, inp.dt, inp.B, inp.C, inp.A, inp.D, inp.dt_bias, inp.conv_w, inp.conv_b,
                              out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert ssm.device_status() == 0
    idx = sample_channels(D, 8, seed=4)
    ref = oracle_prefill(cpu_channels(inp, idx))
    ix = torch.as_tensor(idx, device=DEV)
    got = out.index_select(2, ix).float()
    # the last row (elements past 2^31) and the first, at the bf16-out bar
    for b in (B - 1, 0):
        assert_rms_close(got[b], ref["out"][b], 2e-3, f"row {b} out", extra=half_ulp_bf16(ref["out"][b]))
    assert_rms_close(ss.index_select(1, ix), ref["ssm_state"], 2e-3, "ssm_state")
    assert np.array_equal(cs.index_select(2, ix).cpu().double().numpy(), ref["conv_state"])
    del inp, out, cs, ss
    _free()


def test_q8_beyond_2e31_elements():
    n = 2 ** 31 + 77
    parts = make_partials(2, (n,), dtype=torch.bfloat16, seed=9, device=DEV)
    out, sums, scales = ssm.q8_reduce(parts, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    nblk = (n + 127) // 128
    assert scales.numel() == nblk
    for j0, j1 in ((0, 4), (2 ** 24 - 3, 2 ** 24 + 3), (nblk - 4, nblk)):   # 2^24 blocks = element 2^31
        lo, hi = 128 * j0, min(n, 128 * j1)
        ref = oracle.q8_reduce([p[lo:hi].cpu() for p in parts])
        assert np.array_equal(sums[lo:hi].cpu().numpy(), ref["sums"]), (j0, j1)
        assert np.array_equal(scales[j0:j1].cpu().numpy(), ref["scales"]), (j0, j1)
        assert np.array_equal(out[lo:hi].cpu().view(torch.int16).numpy().view(np.uint16), ref["out_bf16"]), (j0, j1)
    del parts, out, sums, scales
    _free()


def test_largest_batch_decode_and_prefill():
    batch, D = 65535, 8
    par = {k: v.to(DEV) for k, v in make_mixer_params(D, seed=2).items()}
    tok = {k: v.to(DEV) for k, v in make_decode_inputs(batch, D, seed=3).items()}
    cs, ss = (t.to(DEV) for t in make_states(batch, D, seed=4))
    cs0, ss0 = cs.cpu(), ss.cpu()
    out = ssm.decode_step(tok["x"], tok["z"], tok["dt"], tok["B"], tok["C"], par["A"], par["D"], par["dt_bias"],
                          par["conv_w"], par["conv_b"], cs, ss)
    torch.cuda.synchronize()
    rows = np.array([0, 1, 12345, 40000, batch - 2, batch - 1])
    from selective_state_space_prefill_gb300.inputs import MixerInputs
    r = torch.as_tensor(rows)
    one = MixerInputs(x=tok["x"].cpu()[r][:, None], z=tok["z"].cpu()[r][:, None], dt=tok["dt"].cpu()[r][:, None],
                      B=tok["B"].cpu()[r][:, None], C=tok["C"].cpu()[r][:, None],
                      **{k: v.cpu() for k, v in par.items()})
    ref = oracle_prefill(one, cs0[r], ss0[r])
    assert_rms_close(out.cpu()[r], ref["out"][:, 0], 2e-3, "decode out")
    assert_rms_close(ss.cpu()[r], ref["ssm_state"], 2e-3, "decode state")
    # prefill of 3 tokens over all 65535 rows (grid y at its limit)
    inp = make_mixer_inputs(batch, 3, D, dtype=torch.bfloat16, seed=6, device=DEV)
    pout, _, pss = ssm.prefill(inp.x, inp.z, inp.dt, inp.B, inp.C, inp.A, inp.D, inp.dt_bias, inp.conv_w, inp.conv_b)
    torch.cuda.synchronize()
    sub = MixerInputs(**{k: (getattr(inp, k).cpu()[r] if k in ("x", "z", "dt", "B", "C") else getattr(inp, k).cpu())
                         for k in inp.__dataclass_fields__})
    pref = oracle_prefill(sub)
    assert_rms_close(pout.cpu()[r], pref["out"], 2e-3, "prefill out")
    assert_rms_close(pss.cpu()[r], pref["ssm_state"], 2e-3, "prefill state")
    assert ssm.device_status() == 0
    _free()
