"""ssd_prefill and ssd_decode_step (the SSD, Mamba-2-style mixer) on the GPU against the fp64 oracle.

Tolerances are the mixer's bf16-input bar: max |gpu - oracle| <= 2e-3 * RMS(oracle) per output
tensor (out and ssm_state); the conv state is copied raw inputs and must match exactly.  The
tensor-core products carry bf16 hi + lo operand pairs (16 significant bits), so the measured
error sits far below that bar; each test also reports it.
"""
import numpy as np
import pytest
import torch

import oracle
from _gpu import assert_rms_close, half_ulp_bf16
from selective_state_space_prefill_gb300 import binding as ssm
from selective_state_space_prefill_gb300.inputs import make_ssd_inputs, make_ssd_states

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL = 2e-3


def _oracle(inp, cs=None, ss=None, heads=None, threads=None):
    return oracle.ssd_prefill(inp.xBC, inp.z, inp.dt, inp.conv_w, inp.conv_b, inp.A, inp.D, inp.dt_bias,
                              inp.n_heads, inp.head_dim, inp.n_groups, inp.d_state, conv_state_in=cs,
                              ssm_state_in=ss, heads=heads, n_threads=threads)


def _gpu(inp, cs=None, ss=None, out_dtype=torch.float32):
    g = inp.to(DEV)
    return ssm.ssd_prefill(g.xBC, g.z, g.dt, g.conv_w, g.conv_b, g.A, g.D, g.dt_bias, g.n_heads, g.n_groups,
                           conv_state_in=None if cs is None else cs.to(DEV),
                           ssm_state_in=None if ss is None else ss.to(DEV), out_dtype=out_dtype)


def _check(got, ref, what, out_bf16=False):
    out, cso, sso = got
    torch.cuda.synchronize()
    extra = half_ulp_bf16(ref["out"]) if out_bf16 else None
    e_out = assert_rms_close(out, ref["out"], TOL, f"{what} out", extra=extra)
    e_st = assert_rms_close(sso, ref["ssm_state"], TOL, f"{what} ssm_state")
    assert np.array_equal(cso.cpu().double().numpy(), ref["conv_state"]), f"{what} conv_state"
    return e_out, e_st


@pytest.mark.parametrize("L", [1, 5, 127, 128, 129, 300])
def test_ssd_prefill_lengths(L):
    """Chunk edges and ragged tails: one token, less than a chunk, exactly one, one past it, 2.3 chunks."""
    inp = make_ssd_inputs(2, L, 4, n_groups=2, seed=L)
    e = _check(_gpu(inp), _oracle(inp), f"L={L}")
    print(f"L={L}: max err / rms  out {e[0]:.2e}  state {e[1]:.2e}")


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_ssd_prefill_from_states(out_dtype):
    """Input conv and SSM states (a prefill continuing from a cache), fp32 and bf16 outputs."""
    inp = make_ssd_inputs(2, 260, 6, n_groups=3, seed=11)
    g = torch.Generator().manual_seed(12)
    inp.conv_b = torch.randn(inp.channels, generator=g) * 0.3
    inp.D = torch.randn(inp.n_heads, generator=g)
    cs, ss = make_ssd_states(2, 6, 64, 64, inp.channels, seed=13)
    e = _check(_gpu(inp, cs, ss, out_dtype), _oracle(inp, cs, ss), "states", out_dtype == torch.bfloat16)
    print(f"from states ({out_dtype}): out {e[0]:.2e} state {e[1]:.2e}")


def test_ssd_prefill_caching_chain():
    """prefill(L1) on the GPU, then prefill(L2) from its states = oracle prefill(L1 + L2)."""
    inp = make_ssd_inputs(1, 400, 4, n_groups=1, seed=21)
    ref = _oracle(inp)
    o1, c1, s1 = _gpu(inp.token_slice(0, 150))
    o2, c2, s2 = _gpu(inp.token_slice(150, 400), c1, s1)
    torch.cuda.synchronize()
    out = torch.cat([o1, o2], 1)
    assert_rms_close(out, ref["out"], TOL, "chain out")
    assert_rms_close(s2, ref["ssm_state"], TOL, "chain state")
    assert np.array_equal(c2.cpu().double().numpy(), ref["conv_state"])


def test_ssd_head_subset_bit_exact():
    """Heads never exchange data: running a subset of the heads (with the shared B and C
    channels) gives exactly the same bits as those heads of the full run."""
    H, G = 8, 2
    inp = make_ssd_inputs(2, 200, H, n_groups=G, seed=31)
    full = _gpu(inp)
    # heads 2..5 form groups 0 (heads 2, 3) and 1 (heads 4, 5) of the 2-group layout: a run of
    # 4 heads with the same 2 groups
    sub = make_ssd_inputs(2, 200, 4, n_groups=G, seed=31)
    hp = 64
    x = inp.xBC[..., 2 * hp:6 * hp]
    sub.xBC = torch.cat([x, inp.xBC[..., H * hp:]], -1).contiguous()
    sub.z = inp.z[..., 2 * hp:6 * hp].contiguous()
    sub.dt = inp.dt[..., 2:6].contiguous()
    sub.A, sub.D, sub.dt_bias = inp.A[2:6].contiguous(), inp.D[2:6].contiguous(), inp.dt_bias[2:6].contiguous()
    sub.conv_w = torch.cat([inp.conv_w[2 * hp:6 * hp], inp.conv_w[H * hp:]]).contiguous()
    sub.conv_b = torch.cat([inp.conv_b[2 * hp:6 * hp], inp.conv_b[H * hp:]]).contiguous()
    part = _gpu(sub)
    torch.cuda.synchronize()
    assert torch.equal(part[0], full[0][..., 2 * hp:6 * hp])
    assert torch.equal(part[2], full[2][:, 2:6])


def test_ssd_layer_sampled():
    """The Zamba2-2.7B-like layer (batch 4 x 2048 tokens, 80 heads of 64, d_state 64, one group):
    every output of three heads against the oracle."""
    inp = make_ssd_inputs(4, 2048, 80, n_groups=1, seed=0)
    out, cso, sso = _gpu(inp)
    torch.cuda.synchronize()
    heads = [0, 37, 79]
    ref = _oracle(inp, heads=heads)
    cols = np.concatenate([np.arange(h * 64, h * 64 + 64) for h in heads])
    assert_rms_close(out[..., cols], ref["out"][..., cols], TOL, "layer out")
    assert_rms_close(sso[:, heads], ref["ssm_state"][:, heads], TOL, "layer state")


def _oracle_decode(inp, cs, ss):
    """One decode step is the recurrence body for one token: the oracle prefill of L = 1 from the states."""
    return _oracle(inp, cs, ss)


@pytest.mark.parametrize("batch,in_dtype", [(1, torch.bfloat16), (8, torch.bfloat16), (3, torch.float32)])
def test_ssd_decode_from_random_states(batch, in_dtype):
    H, G = 8, 2
    inp = make_ssd_inputs(batch, 1, H, n_groups=G, dtype=in_dtype, seed=40 + batch)
    cs, ss = make_ssd_states(batch, H, 64, 64, inp.channels, seed=41 + batch)
    ref = _oracle_decode(inp, cs, ss)
    g = inp.to(DEV)
    gcs, gss = cs.to(DEV), ss.to(DEV)
    out = ssm.ssd_decode_step(g.xBC[:, 0].contiguous(), g.z[:, 0].contiguous(), g.dt[:, 0].contiguous(),
                              g.conv_w, g.conv_b, g.A, g.D, g.dt_bias, H, G, gcs, gss)
    torch.cuda.synchronize()
    tol = TOL if in_dtype == torch.bfloat16 else 1e-5
    assert_rms_close(out, ref["out"][:, 0], tol, "decode out")
    assert_rms_close(gss, ref["ssm_state"], tol, "decode state")
    assert np.array_equal(gcs.cpu().double().numpy(), ref["conv_state"])


def test_ssd_prefill_then_decode():
    """The state-caching claim for the SSD mixer: GPU prefill of 170 tokens, then 30 GPU decode
    steps from its states, equals the oracle's prefill of all 200 tokens."""
    H, G = 4, 1
    inp = make_ssd_inputs(2, 200, H, n_groups=G, seed=51)
    ref = _oracle(inp)
    g = inp.to(DEV)
    o, cs, ss = ssm.ssd_prefill(g.xBC[:, :170], g.z[:, :170], g.dt[:, :170], g.conv_w, g.conv_b, g.A, g.D,
                                g.dt_bias, H, G)
    outs = [o]
    for t in range(170, 200):
        outs.append(ssm.ssd_decode_step(g.xBC[:, t].contiguous(), g.z[:, t].contiguous(), g.dt[:, t].contiguous(),
                                        g.conv_w, g.conv_b, g.A, g.D, g.dt_bias, H, G, cs, ss)[:, None])
    torch.cuda.synchronize()
    assert_rms_close(torch.cat(outs, 1), ref["out"], TOL, "prefill+decode out")
    assert_rms_close(ss, ref["ssm_state"], TOL, "prefill+decode state")
    assert np.array_equal(cs.cpu().double().numpy(), ref["conv_state"])


def test_ssd_decode_slots():
    """Requests address their cached states through state_slot; other slots are untouched."""
    H, G, n_slots = 4, 2, 6
    inp = make_ssd_inputs(3, 1, H, n_groups=G, seed=61)
    cs, ss = make_ssd_states(n_slots, H, 64, 64, inp.channels, seed=62)
    slots = [4, 0, 2]
    ref = _oracle_decode(inp, cs[slots], ss[slots])
    g = inp.to(DEV)
    gcs, gss = cs.to(DEV), ss.to(DEV)
    out = ssm.ssd_decode_step(g.xBC[:, 0].contiguous(), g.z[:, 0].contiguous(), g.dt[:, 0].contiguous(),
                              g.conv_w, g.conv_b, g.A, g.D, g.dt_bias, H, G, gcs, gss,
                              state_slot=torch.tensor(slots, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    assert_rms_close(out, ref["out"][:, 0], TOL, "slot out")
    assert_rms_close(gss[slots], ref["ssm_state"], TOL, "slot state")
    for s in (1, 3, 5):
        assert torch.equal(gss[s].cpu(), ss[s]) and torch.equal(gcs[s].cpu(), cs[s])


def test_ssd_long_row():
    """A long row (547 chunks, ragged end): the on-chip state carried through every chunk stays
    within the bar against the oracle, output and final state."""
    inp = make_ssd_inputs(1, 70000, 2, n_groups=1, seed=71)
    out, cso, sso = _gpu(inp)
    torch.cuda.synchronize()
    ref = _oracle(inp)
    e_out = assert_rms_close(out, ref["out"], TOL, "long row out")
    e_st = assert_rms_close(sso, ref["ssm_state"], TOL, "long row state")
    assert np.array_equal(cso.cpu().double().numpy(), ref["conv_state"])
    print(f"long row: out {e_out:.2e} state {e_st:.2e}")


def test_ssd_short_prefills_chain():
    """Prefills shorter than the conv window (2 tokens, then 1) splice the incoming conv state into
    the outgoing one; a chain 2 + 1 + 200 equals one prefill of 203 tokens."""
    inp = make_ssd_inputs(2, 203, 4, n_groups=2, seed=81)
    ref = _oracle(inp)
    o1, c1, s1 = _gpu(inp.token_slice(0, 2))
    o2, c2, s2 = _gpu(inp.token_slice(2, 3), c1, s1)
    o3, c3, s3 = _gpu(inp.token_slice(3, 203), c2, s2)
    torch.cuda.synchronize()
    assert_rms_close(torch.cat([o1, o2, o3], 1), ref["out"], TOL, "short chain out")
    assert_rms_close(s3, ref["ssm_state"], TOL, "short chain state")
    assert np.array_equal(c3.cpu().double().numpy(), ref["conv_state"])


def _batch_row(inp, b):
    kw = inp._kw()
    for k in inp._TOKENS:
        kw[k] = kw[k][b:b + 1].contiguous()
    return type(inp)(**kw)


@pytest.mark.parametrize("batch,H,G,L,out_dtype", [(2, 80, 1, 300, torch.float32), (3, 64, 2, 1000, torch.float32),
                                                    (5, 40, 4, 129, torch.float32), (4, 80, 1, 2048, torch.float32),
                                                    (2, 96, 2, 777, torch.bfloat16)])
def test_ssd_rows_cut_between_ctas_bit_exact(batch, H, G, L, out_dtype):
    """More (batch row, head) pairs than CTAs the GPU holds at once: the launch splits the chunks
    of all rows evenly over one CTA per SM, and a row cut between two CTAs hands its state from
    one to the other through the workspace.  The result is bit-identical to running each batch
    row alone (one CTA per head, nothing cut), from input states; heads on both sides of the
    cuts match the oracle."""
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    assert batch * H > n_sm and H <= n_sm, "the case must cut rows and its batch rows alone must not"
    inp = make_ssd_inputs(batch, L, H, n_groups=G, seed=batch * 1000 + L)
    cs, ss = make_ssd_states(batch, H, 64, 64, inp.channels, seed=batch + L)
    out, cso, sso = _gpu(inp, cs, ss, out_dtype)
    for b in range(batch):
        o1, c1, s1 = _gpu(_batch_row(inp, b), cs[b:b + 1], ss[b:b + 1], out_dtype)
        torch.cuda.synchronize()
        assert torch.equal(o1, out[b:b + 1]), f"row {b}: out differs from the cut launch"
        assert torch.equal(s1, sso[b:b + 1]), f"row {b}: ssm_state differs from the cut launch"
        assert torch.equal(c1, cso[b:b + 1]), f"row {b}: conv_state differs from the cut launch"
    assert ssm.device_status() == 0
    if L <= 1000:
        heads = [0, H // 2, H - 1]
        ref = _oracle(inp, cs, ss, heads=heads)
        cols = np.concatenate([np.arange(h * 64, h * 64 + 64) for h in heads])
        extra = half_ulp_bf16(ref["out"][..., cols]) if out_dtype == torch.bfloat16 else None
        assert_rms_close(out[..., cols], ref["out"][..., cols], TOL, "cut rows out", extra=extra)
        assert_rms_close(sso[:, heads], ref["ssm_state"][:, heads], TOL, "cut rows state")


def test_ssd_cut_rows_inside_a_cuda_graph():
    """The cut-rows launch (cooperative, one CTA per SM) captured in a CUDA graph and replayed:
    every replay gives the bits of the direct call (the pre-pass clears the hand-off flags each
    time, so a replay never sees the previous replay's flags)."""
    batch, L, H, G = 2, 1000, 80, 1
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    assert batch * H > n_sm
    inp = make_ssd_inputs(batch, L, H, n_groups=G, seed=91).to(DEV)
    ws = torch.empty(ssm.ssd_prefill_workspace_bytes(batch, L, H, G), device=DEV, dtype=torch.uint8)
    out = torch.empty(batch, L, 64 * H, device=DEV)
    cso = torch.empty(batch, 3, inp.channels, device=DEV)
    sso = torch.empty(batch, H, 64, 64, device=DEV)
    args = (inp.xBC, inp.z, inp.dt, inp.conv_w, inp.conv_b, inp.A, inp.D, inp.dt_bias, H, G)
    ref = [t.clone() for t in ssm.ssd_prefill(*args, workspace=ws)]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        ssm.ssd_prefill(*args, out=out, conv_state_out=cso, ssm_state_out=sso, workspace=ws, stream=s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        ssm.ssd_prefill(*args, out=out, conv_state_out=cso, ssm_state_out=sso, workspace=ws, stream=s)
    for _ in range(3):
        out.zero_()
        sso.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, ref[0]) and torch.equal(cso, ref[1]) and torch.equal(sso, ref[2])
    assert ssm.device_status() == 0


def _head_range(inp, h0, h1):
    """Heads [h0, h1) of a one-group layout with the shared B and C channels: a run of its own."""
    hp, H = 64, inp.n_heads
    sub = make_ssd_inputs(inp.xBC.shape[0], inp.xBC.shape[1], h1 - h0, n_groups=1, seed=0)
    sub.xBC = torch.cat([inp.xBC[..., h0 * hp:h1 * hp], inp.xBC[..., H * hp:]], -1).contiguous()
    sub.z = inp.z[..., h0 * hp:h1 * hp].contiguous()
    sub.dt = inp.dt[..., h0:h1].contiguous()
    sub.A, sub.D, sub.dt_bias = (t[h0:h1].contiguous() for t in (inp.A, inp.D, inp.dt_bias))
    sub.conv_w = torch.cat([inp.conv_w[h0 * hp:h1 * hp], inp.conv_w[H * hp:]]).contiguous()
    sub.conv_b = torch.cat([inp.conv_b[h0 * hp:h1 * hp], inp.conv_b[H * hp:]]).contiguous()
    return sub


def test_ssd_cuts_inside_one_batch_row_bit_exact():
    """Batch 1 with 200 heads: more pairs than CTAs, so heads of the same row are cut between CTAs.
    The output equals, bit for bit, two uncut runs of 100 heads each (heads never exchange data),
    and sampled heads match the oracle."""
    H, L = 200, 300
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    assert H > n_sm and H // 2 <= n_sm
    inp = make_ssd_inputs(1, L, H, n_groups=1, seed=101)
    out, cso, sso = _gpu(inp)
    torch.cuda.synchronize()
    for h0, h1 in ((0, H // 2), (H // 2, H)):
        o, c, s = _gpu(_head_range(inp, h0, h1))
        torch.cuda.synchronize()
        assert torch.equal(o, out[..., 64 * h0:64 * h1]), f"heads {h0}-{h1}: out"
        assert torch.equal(s, sso[:, h0:h1]), f"heads {h0}-{h1}: ssm_state"
        assert torch.equal(c[..., :64 * (h1 - h0)], cso[..., 64 * h0:64 * h1]), f"heads {h0}-{h1}: conv_state"
    heads = [0, 99, 100, 151, 152, 199]
    ref = _oracle(inp, heads=heads)
    cols = np.concatenate([np.arange(h * 64, h * 64 + 64) for h in heads])
    assert_rms_close(out[..., cols], ref["out"][..., cols], TOL, "one-row cuts out")
    assert_rms_close(sso[:, heads], ref["ssm_state"][:, heads], TOL, "one-row cuts state")
    assert ssm.device_status() == 0


def test_ssd_prefill_one_group_per_head():
    """G = H: every head has its own B and C channels."""
    inp = make_ssd_inputs(2, 300, 4, n_groups=4, seed=111)
    e = _check(_gpu(inp), _oracle(inp), "G = H")
    print(f"G = H: out {e[0]:.2e} state {e[1]:.2e}")


def test_ssd_prompt_full_size_sampled():
    """The Zamba2-7B-like batch-1 prompt the bench times (16384 tokens, 112 heads of 64, one group):
    every output and the final state of three heads against the oracle."""
    inp = make_ssd_inputs(1, 16384, 112, n_groups=1, seed=0)
    out, cso, sso = _gpu(inp)
    torch.cuda.synchronize()
    heads = [0, 57, 111]
    ref = _oracle(inp, heads=heads)
    cols = np.concatenate([np.arange(h * 64, h * 64 + 64) for h in heads])
    e_out = assert_rms_close(out[..., cols], ref["out"][..., cols], TOL, "prompt out")
    e_st = assert_rms_close(sso[:, heads], ref["ssm_state"][:, heads], TOL, "prompt state")
    print(f"prompt 1 x 16384 x 112: out {e_out:.2e} state {e_st:.2e}")
