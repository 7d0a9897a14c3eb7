"""ssm_prefill_segmented_noalloc through the C ABI, for callers that cannot allocate.

Some callers cannot allocate device memory when they call: a plugin inside a host
program that owns every allocation on the GPU, or a serving loop that must not call
cudaMalloc after start-up (it can synchronize the device and fail under memory
pressure).  This entry point keeps the segment scratch in a fixed array inside the
library instead of a caller workspace.  Its output must equal that of
ssm_prefill_segmented, the entry point that takes a workspace, within the parity
tolerances, on consecutive calls that share the array.

This file is named so that pytest collects it last.
"""
import pytest
import torch

from _gpu import assert_parity, cpu_channels, oracle_prefill, sample_channels
from selective_state_space_prefill_gb300 import binding as ssm
from selective_state_space_prefill_gb300.inputs import make_mixer_inputs, make_states

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _prefill(inp, seg_len, cs=None, ss=None, noalloc=False):
    return ssm.prefill(inp.x, inp.z, inp.dt, inp.B, inp.C, inp.A, inp.D, inp.dt_bias, inp.conv_w, inp.conv_b,
                       conv_state_in=cs, ssm_state_in=ss, seg_len=seg_len, noalloc=noalloc)


def test_noalloc_matches_workspace_entry_on_consecutive_calls():
    # two calls in a row on one shared array: a batch-1 bf16 row in 4 segments, then a
    # different shape (fp32, two rows, cached input states, 5 segments with a ragged tail)
    cases = [(1, 2048, 1536, torch.bfloat16, 512, False), (2, 300, 64, torch.float32, 64, True)]
    for batch, L, D, dtype, seg, states in cases:
        need = ssm.prefill_workspace_bytes(batch, L, D, seg)
        assert 0 < need <= ssm.NOALLOC_SCRATCH_BYTES
        inp = make_mixer_inputs(batch, L, D, dtype=dtype, seed=L).to(DEV)
        cs = ss = None
        if states:
            cs, ss = (t.to(DEV) for t in make_states(batch, D, seed=3))
        ref = _prefill(inp, seg, cs, ss)                      # caller workspace
        got = _prefill(inp, seg, cs, ss, noalloc=True)        # fixed array in the library
        torch.cuda.synchronize()
        for g, r, what in zip(got, ref, ("out", "conv_state", "ssm_state")):
            assert_parity(g, r.cpu().double().numpy(), dtype, f"noalloc {what} (L={L})")
            assert torch.equal(g, r), f"noalloc {what} differs from the workspace entry (L={L})"
    assert ssm.device_status() == 0


def test_noalloc_against_the_oracle():
    """The entry point checked directly against the fp64 oracle, not only through the workspace
    entry: a batch-1 bf16 row in 4 segments (sampled channels, the 2e-3 RMS bar) and an fp32 pair
    of rows from cached states in 5 segments with a ragged tail (every channel, the fp32 bar)."""
    for batch, L, D, dtype, seg, states in [(1, 2048, 1536, torch.bfloat16, 512, False),
                                            (2, 300, 64, torch.float32, 64, True)]:
        inp = make_mixer_inputs(batch, L, D, dtype=dtype, seed=L + 7)
        cs = ss = None
        if states:
            cs, ss = make_states(batch, D, seed=5)
        g = inp.to(DEV)
        out, cso, sso = _prefill(g, seg, None if cs is None else cs.to(DEV), None if ss is None else ss.to(DEV),
                                 noalloc=True)
        torch.cuda.synchronize()
        ch = sample_channels(D, 40) if D > 64 else list(range(D))
        ix = torch.as_tensor(ch, device=DEV, dtype=torch.long)
        ref = oracle_prefill(cpu_channels(inp, ch), None if cs is None else cs[:, :, ch],
                             None if ss is None else ss[:, ch])
        assert_parity(out.index_select(2, ix), ref["out"], dtype, f"noalloc out vs oracle (L={L})")
        assert_parity(sso.index_select(1, ix), ref["ssm_state"], dtype, f"noalloc ssm_state vs oracle (L={L})")
        assert torch.equal(cso.index_select(2, ix).cpu().double(), torch.as_tensor(ref["conv_state"])), \
            f"noalloc conv_state vs oracle (L={L})"
    assert ssm.device_status() == 0


def test_noalloc_rejects_requests_beyond_the_array():
    # batch 1, d_inner 8192: 5 segments need 4 x 8192 x 128 B = 4 MiB, exactly the array, and are
    # allowed; 6 segments need 5 MiB and are refused on the host, before anything is launched
    inp = make_mixer_inputs(1, 64 * 6, 8192, dtype=torch.bfloat16, seed=1).to(DEV)
    assert ssm.prefill_workspace_bytes(1, 64 * 6, 8192, 64) > ssm.NOALLOC_SCRATCH_BYTES
    with pytest.raises(ssm.SSMError) as e:
        _prefill(inp, 64, noalloc=True)
    assert e.value.code == -1 and "fixed array holds" in str(e.value)
    assert ssm.prefill_workspace_bytes(1, 64 * 5, 8192, 64) == ssm.NOALLOC_SCRATCH_BYTES
    out, _, _ = _prefill(inp.token_slice(0, 64 * 5), 64, noalloc=True)
    ref, _, _ = _prefill(inp.token_slice(0, 64 * 5), 64)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
