"""Failure reporting without a fault, and writes confined to the output buffers.

* An in-kernel wait that runs out (a barrier phase that nothing completes) is reported
  through the device status word; the kernel returns, and the context stays usable.
* Canaries: every output of every call sits inside a larger buffer filled with a sentinel;
  after the call the guard bands are untouched and the output itself is fully written.
"""
import time

import numpy as np
import pytest
import torch

from _gpu import assert_rms_close, oracle_prefill
from selective_state_space_prefill_gb300 import binding as ssm
from selective_state_space_prefill_gb300.inputs import (make_decode_inputs, make_mixer_inputs, make_mixer_params,
                                                         make_out_proj_inputs, make_partials, make_states)

pytestmark = pytest.mark.gpu
DEV = "cuda"
GUARD = 4096


def test_expired_wait_is_reported_and_the_context_survives():
    ssm.device_status(clear=True)
    t0 = time.perf_counter()
    ssm.selftest_expire_wait(50000)                     # 50 ms
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 >= 0.045
    assert ssm.device_status(clear=True) == ssm.DEV_WAIT_TIMEOUT
    inp = make_mixer_inputs(1, 100, 32, dtype=torch.bfloat16, seed=3)
    g = inp.to(DEV)
    out, _, _ = ssm.prefill(g.x, g.z, g.dt, g.B, g.C, g.A, g.D, g.dt_bias, g.conv_w, g.conv_b)
    torch.cuda.synchronize()
    assert_rms_close(out, oracle_prefill(inp)["out"], 2e-3, "prefill after the expired wait")
    assert ssm.device_status() == 0


class Guarded:
    """A view of `n` elements in the middle of a buffer whose every element holds `fill`."""

    def __init__(self, shape, dtype, fill):
        n = int(np.prod(shape))
        self.buf = torch.full((GUARD + n + GUARD,), fill, device=DEV, dtype=dtype)
        self.view = self.buf[GUARD:GUARD + n].view(*shape)
        self.fill = fill

    def check(self, what):
        torch.cuda.synchronize()
        b = self.buf.cpu()
        sentinel = torch.full((GUARD,), self.fill, dtype=b.dtype)
        same = (lambda x: torch.equal(x, sentinel)) if not b.dtype.is_floating_point else \
            (lambda x: torch.equal(x.view(torch.int16 if b.dtype == torch.bfloat16 else torch.int32),
                                   sentinel.view(torch.int16 if b.dtype == torch.bfloat16 else torch.int32)))
        assert same(b[:GUARD]) and same(b[-GUARD:]), f"{what}: a guard band was written"
        body = b[GUARD:-GUARD]
        if b.dtype.is_floating_point:
            assert not torch.isnan(body.float()).any(), f"{what}: part of the output was not written"
        else:
            assert not (body == self.fill).all(), f"{what}: the output was not written"


def test_prefill_and_segmented_prefill_write_only_their_outputs():
    batch, L, D = 2, 300, 64
    inp = make_mixer_inputs(batch, L, D, dtype=torch.bfloat16, seed=5).to(DEV)
    for seg in (None, 64):
        for out_dtype in (torch.float32, torch.bfloat16):
            out = Guarded((batch, L, D), out_dtype, float("nan"))
            cs = Guarded((batch, 3, D), torch.float32, float("nan"))
            ss = Guarded((batch, D, 16), torch.float32, float("nan"))
            ws = None
            if seg:
                need = ssm.prefill_workspace_bytes(batch, L, D, seg)
                wsb = Guarded((need // 4,), torch.float32, float("nan"))
                ws = wsb.view.view(torch.uint8)
            ssm.prefill(inp.x, inp.z, inp.dt, inp.B, inp.C, inp.A, inp.D, inp.dt_bias, inp.conv_w, inp.conv_b,
                        out=out.view, conv_state_out=cs.view, ssm_state_out=ss.view, seg_len=seg, workspace=ws)
            for g, w in ((out, "out"), (cs, "conv_state_out"), (ss, "ssm_state_out")):
                g.check(f"prefill seg={seg} {out_dtype} {w}")
            if seg:
                wsb.check("segment workspace")


def test_decode_and_decode_tokens_write_only_their_outputs():
    batch, D, T = 5, 96, 3
    par = {k: v.to(DEV) for k, v in make_mixer_params(D, seed=1).items()}
    tok = {k: v.to(DEV) for k, v in make_decode_inputs(batch, D, seed=2).items()}
    cs0, ss0 = make_states(batch, D, seed=3)
    cs = Guarded((batch, 3, D), torch.float32, 0.0)
    ss = Guarded((batch, D, 16), torch.float32, 0.0)
    cs.view.copy_(cs0.to(DEV))
    ss.view.copy_(ss0.to(DEV))
    cs.fill = ss.fill = 0.0
    out = Guarded((batch, D), torch.float32, float("nan"))
    ssm.decode_step(tok["x"], tok["z"], tok["dt"], tok["B"], tok["C"], par["A"], par["D"], par["dt_bias"],
                    par["conv_w"], par["conv_b"], cs.view, ss.view, out=out.view)
    out.check("decode out")
    for g, w in ((cs, "conv_state"), (ss, "ssm_state")):
        torch.cuda.synchronize()
        b = g.buf.cpu()
        assert not b[:GUARD].any() and not b[-GUARD:].any(), f"decode {w}: a guard band was written"
    blk = make_mixer_inputs(batch, T, D, dtype=torch.bfloat16, seed=4).to(DEV)
    outT = Guarded((batch, T, D), torch.bfloat16, float("nan"))
    ssm.decode_tokens(blk.x, blk.z, blk.dt, blk.B, blk.C, par["A"], par["D"], par["dt_bias"], par["conv_w"],
                      par["conv_b"], cs.view, ss.view, out=outT.view)
    outT.check("decode_tokens out")


def test_q8_and_out_proj_write_only_their_outputs():
    n = 4096 * 3 + 77
    parts = [p.to(DEV) for p in make_partials(3, (n,), dtype=torch.bfloat16, seed=7)]
    out = Guarded((n,), torch.bfloat16, float("nan"))
    sums = Guarded((n,), torch.int32, 0x5A5A5A5A)
    scales = Guarded(((n + 127) // 128,), torch.float32, float("nan"))
    ssm.q8_reduce(parts, out=out.view, sums=sums.view, scales=scales.view)
    out.check("q8 out")
    sums.check("q8 sums")
    scales.check("q8 scales")
    M, N, K = 300, 640, 200
    y, W = make_out_proj_inputs(M, K, N, seed=8, device=DEV)
    for out_dtype in (torch.bfloat16, torch.float32):
        o = Guarded((M, N), out_dtype, float("nan"))
        a = Guarded((M * N // 128,), torch.float32, float("nan"))
        ssm.out_proj_partial(y, W, out=o.view, block_amax=a.view)
        o.check(f"out_proj {out_dtype}")
        a.check("out_proj block maxima")


def test_q8_halves_write_only_their_outputs():
    n = 128 * 37 + 77                         # a short last block and a ragged last lane group
    parts = [p.to(DEV) for p in make_partials(2, (n,), dtype=torch.bfloat16, seed=9)]
    nblk = (n + 127) // 128
    amax = Guarded((nblk,), torch.float32, float("nan"))
    ssm.q8_block_absmax(parts[0], out=amax.view)
    amax.check("q8_block_absmax")
    shared = torch.maximum(amax.view, ssm.q8_block_absmax(parts[1]))
    codes, scales = [], None
    for p in parts:
        c = Guarded((n,), torch.int8, 0x5A)
        sc = Guarded((nblk,), torch.float32, float("nan"))
        ssm.q8_quantize_shared(p, shared, codes=c.view, scales=sc.view)
        c.check("q8_quantize_shared codes")
        sc.check("q8_quantize_shared scales")
        codes.append(c.view)
        scales = sc.view
    for out_dtype in (torch.bfloat16, torch.float32):
        out = Guarded((n,), out_dtype, float("nan"))
        sums = Guarded((n,), torch.int32, 0x5A5A5A5A)
        ssm.q8_sum_dequant(codes, scales, out=out.view, sums=sums.view)
        out.check(f"q8_sum_dequant {out_dtype} out")
        sums.check("q8_sum_dequant sums")


def _guards_intact(g, what):
    """Only the guard bands, bit for bit (the body may keep the sentinel in places)."""
    torch.cuda.synchronize()
    b = g.buf.cpu()
    sentinel = torch.full((GUARD,), g.fill, dtype=b.dtype)
    if b.dtype.is_floating_point:
        bits = torch.int16 if b.element_size() == 2 else torch.int32
        b, sentinel = b.view(bits), sentinel.view(bits)
    assert torch.equal(b[:GUARD], sentinel) and torch.equal(b[-GUARD:], sentinel), \
        f"{what}: a guard band was written"


def test_ssd_prefill_writes_only_its_outputs():
    from selective_state_space_prefill_gb300.inputs import make_ssd_inputs
    batch, L, H, G = 2, 300, 4, 2
    inp = make_ssd_inputs(batch, L, H, n_groups=G, seed=7).to(DEV)
    need = ssm.ssd_prefill_workspace_bytes(batch, L, H, G)
    for out_dtype in (torch.float32, torch.bfloat16):
        out = Guarded((batch, L, 64 * H), out_dtype, float("nan"))
        cs = Guarded((batch, 3, inp.channels), torch.float32, float("nan"))
        ss = Guarded((batch, H, 64, 64), torch.float32, float("nan"))
        ws = Guarded((need // 4,), torch.float32, float("nan"))
        ssm.ssd_prefill(inp.xBC, inp.z, inp.dt, inp.conv_w, inp.conv_b, inp.A, inp.D, inp.dt_bias, H, G,
                        out=out.view, conv_state_out=cs.view, ssm_state_out=ss.view,
                        workspace=ws.view.view(torch.uint8))
        for g, w in ((out, "out"), (cs, "conv_state_out"), (ss, "ssm_state_out")):
            g.check(f"ssd_prefill {out_dtype} {w}")
        # the workspace's token padding of the transposed planes is never written: guards only
        _guards_intact(ws, f"ssd_prefill {out_dtype} workspace")


def test_ssd_decode_writes_only_its_outputs():
    from selective_state_space_prefill_gb300.inputs import make_ssd_inputs, make_ssd_states
    batch, H, G, n_slots = 3, 4, 2, 5
    inp = make_ssd_inputs(batch, 1, H, n_groups=G, seed=8).to(DEV)
    cs0, ss0 = make_ssd_states(n_slots, H, 64, 64, inp.channels, seed=9)
    fill = 12345.0
    cs = Guarded(tuple(cs0.shape), torch.float32, fill)
    ss = Guarded(tuple(ss0.shape), torch.float32, fill)
    cs.view.copy_(cs0.to(DEV))
    ss.view.copy_(ss0.to(DEV))
    out = Guarded((batch, 64 * H), torch.float32, float("nan"))
    slots = torch.tensor([4, 0, 2], dtype=torch.int32, device=DEV)
    ssm.ssd_decode_step(inp.xBC[:, 0].contiguous(), inp.z[:, 0].contiguous(), inp.dt[:, 0].contiguous(),
                        inp.conv_w, inp.conv_b, inp.A, inp.D, inp.dt_bias, H, G, cs.view, ss.view,
                        state_slot=slots, out=out.view)
    out.check("ssd_decode_step out")
    _guards_intact(cs, "ssd_decode_step conv_state")
    _guards_intact(ss, "ssd_decode_step ssm_state")
    for s in (1, 3):
        assert torch.equal(cs.view[s].cpu(), cs0[s]) and torch.equal(ss.view[s].cpu(), ss0[s])
