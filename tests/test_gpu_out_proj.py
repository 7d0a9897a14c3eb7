"""ssm_out_proj_partial on the tensor cores against the fp64 oracle.

Bound per element: |gpu - oracle| <= 4 K 2^-24 sum_k |y_mk| |W_nk| (fp32 accumulation of
exact bf16 products in any order), plus half a bf16 ulp of the value for bf16 output.
The block maxima are checked bit for bit against the stored partial and within the same
bound against the oracle's.
"""
import numpy as np
import pytest
import torch

import oracle
from _gpu import half_ulp_bf16
from selective_state_space_prefill_gb300 import binding as ssm
from selective_state_space_prefill_gb300.inputs import make_out_proj_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _bound(ref, K, out_dtype):
    b = 4 * K * 2.0 ** -24 * ref["absdot"]
    if out_dtype == torch.bfloat16:
        b = b + half_ulp_bf16(ref["out"]) * (1 + 2.0 ** -7)
    return b


def _check(y, W, out, amax, ref, out_dtype, rows=None):
    K = y.shape[1]
    got = out.float().cpu().double().numpy()
    r_out, r_abs = ref["out"], ref["absdot"]
    if rows is not None:
        got = got[rows]
    bound = _bound(dict(out=r_out, absdot=r_abs), K, out_dtype)
    err = np.abs(got - r_out)
    assert np.all(err <= bound), f"max err/bound {float((err / np.maximum(bound, 1e-300)).max()):.3g}"
    if amax is not None and rows is None:
        M, N = out.shape
        stored = np.abs(out.float().cpu().numpy()).reshape(-1, 128).max(1)
        assert np.array_equal(amax.cpu().numpy(), stored), "block maxima of the stored partial"
        bb = bound.reshape(-1, 128).max(1)
        assert np.all(np.abs(amax.cpu().double().numpy() - ref["amax"]) <= bb), "block maxima vs oracle"


@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (256, 768, 1536), (300, 640, 200), (64, 128, 8)])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_out_proj_matches_oracle(M, N, K, out_dtype):
    y, W = make_out_proj_inputs(M, K, N, seed=M + N + K)
    out, amax = ssm.out_proj_partial(y.to(DEV), W.to(DEV), out_dtype=out_dtype)
    torch.cuda.synchronize()
    ref = oracle.out_proj(y, W)
    _check(y, W, out, amax, ref, out_dtype)
    assert ssm.device_status() == 0


def test_out_proj_strided_views():
    """y, W and out as column slices of wider row-major buffers (row strides > row lengths)."""
    M, N, K = 200, 384, 320
    yb, Wb = make_out_proj_inputs(M, K + 64, N + 128, seed=5)
    y, W = yb[:, 32:32 + K], Wb[:N, 16:16 + K]
    obuf = torch.full((M, N + 256), float("nan"), device=DEV, dtype=torch.float32)
    out = obuf[:, 128:128 + N]
    _, amax = ssm.out_proj_partial(yb.to(DEV)[:, 32:32 + K], Wb.to(DEV)[:N, 16:16 + K], out=out)
    torch.cuda.synchronize()
    ref = oracle.out_proj(y.contiguous(), W.contiguous())
    _check(y, W, out, amax, ref, torch.float32)
    assert torch.isnan(obuf[:, :128]).all() and torch.isnan(obuf[:, 128 + N:]).all()


def test_out_proj_falcon_slice_sampled_and_q8():
    """The Falcon-Mamba-like rank (M 16384 tokens, K 2048 channels of 8192, N 4096): sampled rows
    against the oracle; then two ranks' partials reduce through q8 with the shared scale that
    the maximum of their block maxima gives."""
    M, N, K = 16384, 4096, 2048
    y, W = make_out_proj_inputs(M, K, N, seed=0, device=DEV)
    out, amax = ssm.out_proj_partial(y, W)
    torch.cuda.synchronize()
    rows = np.array([0, 1, 127, 128, 5000, M - 129, M - 1])
    ref = oracle.out_proj(y[torch.as_tensor(rows, device=DEV)].cpu(), W.cpu())
    _check(y, W, out, None, ref, torch.bfloat16, rows=rows)
    stored = out.float().abs().reshape(-1, 128).amax(1)
    assert torch.equal(amax, stored)
    y2, _ = make_out_proj_inputs(M, K, N, seed=1, device=DEV)
    out2, amax2 = ssm.out_proj_partial(y2, W)
    _, _, scales = ssm.q8_reduce([out, out2])
    torch.cuda.synchronize()
    shared = torch.maximum(amax, amax2).cpu().numpy()
    expect = np.where(shared > 0, shared / np.float32(127.0), np.float32(0.0)).astype(np.float32)   # IEEE fp32 division
    assert np.array_equal(scales.cpu().numpy(), expect)


def test_out_proj_wide_tiles_ragged():
    """Enough tiles for the 256-column path, with a ragged M, a half-filled last N tile and a
    ragged K; sampled rows against the oracle, block maxima against the stored partial."""
    M, N, K = 128 * 152 + 77, 640, 200
    y, W = make_out_proj_inputs(M, K, N, seed=11, device=DEV)
    for out_dtype in (torch.bfloat16, torch.float32):
        out, amax = ssm.out_proj_partial(y, W, out_dtype=out_dtype)
        torch.cuda.synchronize()
        rows = np.array([0, 129, 9000, M - 78, M - 77, M - 1])
        ref = oracle.out_proj(y[torch.as_tensor(rows, device=DEV)].cpu(), W.cpu())
        _check(y, W, out, None, ref, out_dtype, rows=rows)
        assert torch.equal(amax, out.float().abs().reshape(-1, 128).amax(1))
