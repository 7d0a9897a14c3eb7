"""ssm_prefill_segmented on the GPU.

The rows are cut into segments that run in parallel; a carry pass composes the
per-segment pairs (decay product, state from zero) into each segment's start state.
Checked against the fp64 oracle at the tolerances of ssm_prefill, for bit-exact
channel-slice invariance at a fixed seg_len, and for equality with ssm_prefill when
the row is a single segment.
"""
import zlib

import numpy as np
import pytest
import torch

from _gpu import assert_parity, assert_rel_close, assert_rms_close, cpu_channels, oracle_prefill, sample_channels
from selective_state_space_prefill_gb300 import binding as ssm
from selective_state_space_prefill_gb300.inputs import make_decode_inputs, make_mixer_inputs, make_states

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run(inp, seg_len, cs=None, ss=None, workspace=None, sl=slice(None)):
    return ssm.prefill(inp.x[..., sl], inp.z[..., sl], inp.dt[..., sl], inp.B, inp.C, inp.A[sl].contiguous(),
                       inp.D[sl].contiguous(), inp.dt_bias[sl].contiguous(), inp.conv_w[sl].contiguous(),
                       inp.conv_b[sl].contiguous(), conv_state_in=cs, ssm_state_in=ss, seg_len=seg_len,
                       workspace=workspace)


CASES = [
    # name, batch, L, d_inner, dtype, seg_len, input states
    ("fp32_5seg_ragged", 2, 300, 40, torch.float32, 64, False),
    ("fp32_4seg_states", 1, 1000, 64, torch.float32, 256, True),
    ("bf16_tail_of_2", 3, 130, 32, torch.bfloat16, 128, True),
    ("bf16_32seg_states", 1, 2048, 96, torch.bfloat16, 64, True),
    ("fp32_tail_of_1", 2, 65, 16, torch.float32, 64, True),
]


@pytest.mark.parametrize("name,batch,L,D,dtype,seg,states", CASES, ids=[c[0] for c in CASES])
def test_segmented_matches_oracle(name, batch, L, D, dtype, seg, states):
    inp = make_mixer_inputs(batch, L, D, dtype=dtype, seed=zlib.crc32(name.encode()) % 1000)
    cs = ss = None
    if states:
        cs, ss = make_states(batch, D, seed=11)
    out, cso, sso = _run(inp.to(DEV), seg, None if cs is None else cs.to(DEV), None if ss is None else ss.to(DEV))
    torch.cuda.synchronize()
    ref = oracle_prefill(inp, cs, ss)
    assert_parity(out, ref["out"], dtype, "out")
    assert_parity(sso, ref["ssm_state"], dtype, "ssm_state")
    assert np.array_equal(cso.cpu().double().numpy(), ref["conv_state"]), "conv_state must be exact"
    assert ssm.device_status() == 0


def test_single_segment_is_prefill_bit_exact():
    """seg_len >= L runs exactly ssm_prefill (no workspace, same kernel, same bits)."""
    inp = make_mixer_inputs(2, 333, 64, dtype=torch.bfloat16, seed=3).to(DEV)
    cs, ss = (t.to(DEV) for t in make_states(2, 64, seed=5))
    a = ssm.prefill(inp.x, inp.z, inp.dt, inp.B, inp.C, inp.A, inp.D, inp.dt_bias, inp.conv_w, inp.conv_b,
                    conv_state_in=cs, ssm_state_in=ss)
    b = _run(inp, 384, cs, ss)
    for u, v in zip(a, b):
        assert torch.equal(u, v)


def test_segmented_slice_invariance_bit_exact():
    """At a fixed seg_len each channel's result is bit-identical in any channel slice."""
    D, seg = 256, 128
    inp = make_mixer_inputs(1, 1111, D, dtype=torch.bfloat16, seed=13).to(DEV)
    full, cfull, sfull = _run(inp, seg)
    for lo, hi in ((0, 64), (64, 128), (128, 200), (200, 256)):
        o, c, s = _run(inp, seg, sl=slice(lo, hi))
        assert torch.equal(o, full[..., lo:hi]), (lo, hi)
        assert torch.equal(s, sfull[:, lo:hi]), (lo, hi)
        assert torch.equal(c, cfull[:, :, lo:hi]), (lo, hi)


def test_segmented_workspace_reused():
    """One caller workspace serves consecutive calls (its contents on entry do not matter)."""
    inp = make_mixer_inputs(2, 700, 64, dtype=torch.float32, seed=23).to(DEV)
    need = ssm.prefill_workspace_bytes(2, 700, 64, 128)
    assert need == (6 - 1) * 2 * 64 * 128
    ws = torch.full((need,), 0x7f, device=DEV, dtype=torch.uint8)     # garbage (large floats)
    first = _run(inp, 128, workspace=ws)
    second = _run(inp, 128, workspace=ws)
    fresh = _run(inp, 128)
    for u, v, w in zip(first, second, fresh):
        assert torch.equal(u, v) and torch.equal(u, w)
    ref = oracle_prefill(inp.to("cpu"))
    assert_rel_close(first[0], ref["out"], 1e-5, "out")


def test_segmented_then_decode_continues():
    """The segmented prefill's final states are the cache decode continues from."""
    L, D = 900, 64
    inp = make_mixer_inputs(2, L + 3, D, dtype=torch.bfloat16, seed=29)
    g = inp.to(DEV)
    _, cs, ss = _run(g.token_slice(0, L), 192)
    outs = []
    for t in range(L, L + 3):
        tok = g.token_slice(t, t + 1)
        outs.append(ssm.decode_step(tok.x[:, 0], tok.z[:, 0], tok.dt[:, 0], tok.B[:, 0].contiguous(),
                                    tok.C[:, 0].contiguous(), g.A, g.D, g.dt_bias, g.conv_w, g.conv_b, cs, ss))
    torch.cuda.synchronize()
    ref = oracle_prefill(inp)
    assert_rms_close(torch.stack(outs, 1), ref["out"][:, L:], 2e-3, "decode after segmented prefill")
    assert_rms_close(ss, ref["ssm_state"], 2e-3, "state")


@pytest.mark.parametrize("L,D", [(16384, 2048), (2048, 1536)])
def test_batch1_layers_sampled(L, D):
    """Batch-1 rows (the Falcon-Mamba-like slice and a Mamba-130M-like layer) with the
    segment length the binding suggests for this GPU; sampled channels against the oracle."""
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    seg = ssm.suggest_seg_len(1, L, D, n_sm)
    assert seg is not None and seg < L
    inp = make_mixer_inputs(1, L, D, dtype=torch.bfloat16, seed=0, device=DEV)
    out, cs, ss = _run(inp, seg)
    torch.cuda.synchronize()
    idx = sample_channels(D, 16, seed=2)
    ref = oracle_prefill(cpu_channels(inp, idx))
    ix = torch.as_tensor(idx, device=DEV)
    assert_rms_close(out.index_select(2, ix), ref["out"], 2e-3, "out")
    assert_rms_close(ss.index_select(1, ix), ref["ssm_state"], 2e-3, "ssm_state")
    assert np.array_equal(cs.index_select(2, ix).cpu().double().numpy(), ref["conv_state"])
    assert torch.isfinite(out).all() and ssm.device_status() == 0


def test_segmented_bf16_output():
    """Segments with a bf16 output: the bf16-out bar (2e-3 RMS plus half a bf16 ulp)."""
    from _gpu import half_ulp_bf16
    inp = make_mixer_inputs(2, 777, 64, dtype=torch.bfloat16, seed=31)
    g = inp.to(DEV)
    out, _, sso = ssm.prefill(g.x, g.z, g.dt, g.B, g.C, g.A, g.D, g.dt_bias, g.conv_w, g.conv_b,
                              out_dtype=torch.bfloat16, seg_len=192)
    torch.cuda.synchronize()
    ref = oracle_prefill(inp)
    assert out.dtype == torch.bfloat16
    assert_rms_close(out.float(), ref["out"], 2e-3, "bf16 out", extra=half_ulp_bf16(ref["out"]))
    assert_rms_close(sso, ref["ssm_state"], 2e-3, "ssm_state")
