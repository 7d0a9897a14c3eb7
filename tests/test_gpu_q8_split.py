"""The rank-local halves of the 8-bit all-reduce on the GPU (q8_block_absmax,
q8_quantize_shared, q8_sum_dequant): each bit-exact against the oracle, and composed
(the ranks' block maxima combined by max) bit-exact against q8_reduce_partials."""
import numpy as np
import pytest
import torch

import oracle
from _pins import read_q8_cases
from selective_state_space_prefill_gb300 import binding as ssm
from selective_state_space_prefill_gb300.inputs import make_out_proj_inputs, make_partials

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _bits(t):
    return t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16).reshape(-1)


def _split_on_gpu(parts, out_dtype=torch.float32, amax_list=None):
    """The composition a tensor-parallel all-reduce runs, with every rank on this GPU."""
    g = [p.to(DEV) for p in parts]
    if amax_list is None:
        amax_list = [ssm.q8_block_absmax(p) for p in g]
    shared = torch.stack(amax_list).amax(0)                    # the MAX all-reduce
    q = [ssm.q8_quantize_shared(p, shared) for p in g]
    codes = [c for c, _ in q]                                  # the all-gather of codes
    out, sums = ssm.q8_sum_dequant(codes, q[0][1], out_dtype=out_dtype)
    torch.cuda.synchronize()
    return out, sums, q, shared


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("n", [1, 127, 128, 129, 4096 + 77])
def test_each_half_matches_the_oracle(dtype, n):
    parts = make_partials(3, (n,), dtype=dtype, seed=n + 5)
    g = [p.to(DEV) for p in parts]
    amax = [ssm.q8_block_absmax(p) for p in g]
    torch.cuda.synchronize()
    ref_amax = [oracle.q8_block_absmax(p) for p in parts]
    for a, r in zip(amax, ref_amax):
        assert np.array_equal(a.cpu().numpy(), r), "block maxima"
    shared = torch.stack(amax).amax(0)
    ref_shared = np.max(np.stack(ref_amax), 0)
    for p, pg in zip(parts, g):
        codes, scales = ssm.q8_quantize_shared(pg, shared)
        torch.cuda.synchronize()
        r = oracle.q8_quantize_shared(p, ref_shared)
        assert np.array_equal(codes.cpu().numpy().reshape(-1), r["codes"]), "codes"
        assert np.array_equal(scales.cpu().numpy(), r["scales"]), "scales"
    codes = [ssm.q8_quantize_shared(pg, shared)[0] for pg in g]
    scales = ssm.q8_quantize_shared(g[0], shared)[1]
    ref = oracle.q8_sum_dequant([c.cpu().numpy() for c in codes], scales.cpu().numpy())
    for out_dtype in (torch.float32, torch.bfloat16):
        out, sums = ssm.q8_sum_dequant(codes, scales, out_dtype=out_dtype)
        torch.cuda.synchronize()
        assert np.array_equal(sums.cpu().numpy(), ref["sums"]), "sums"
        if out_dtype == torch.bfloat16:
            assert np.array_equal(_bits(out), ref["out_bf16"]), "bf16 out"
        else:
            assert np.array_equal(out.cpu().numpy().reshape(-1), ref["out_f32"]), "f32 out"


@pytest.mark.parametrize("P", [1, 2, 4, 8])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_composition_equals_the_local_reduction(P, out_dtype):
    """P ranks' partials [256, 1, 4096] (the decode/reduction sweep's largest batch), ragged too."""
    for shape in ((256, 1, 4096), (4096 + 77,)):
        parts = make_partials(P, shape, dtype=torch.bfloat16, seed=P * 31 + len(shape))
        out, sums, q, _ = _split_on_gpu(parts, out_dtype)
        fout, fsums, fscales = ssm.q8_reduce([p.to(DEV) for p in parts], out_dtype=out_dtype)
        torch.cuda.synchronize()
        assert torch.equal(sums, fsums), "sums"
        assert torch.equal(q[0][1], fscales), "scales"
        assert torch.equal(out.reshape(-1), fout.reshape(-1)), "out"
        ref = oracle.q8_reduce(parts)
        assert np.array_equal(sums.cpu().numpy(), ref["sums"])


def test_hand_cases_through_the_halves():
    """The hand-derived cases; their blocks (3 or 4 elements) are padded to the kernels' 128
    with zeros, which leaves every block maximum unchanged."""
    for case in read_q8_cases():
        blk = case["block"]
        for dtype in (torch.float32, torch.bfloat16):
            parts = []
            for p in case["p"]:
                q = torch.zeros(128 * ((len(p) + blk - 1) // blk), dtype=dtype)
                for j in range(0, len(p), blk):
                    seg = torch.from_numpy(p[j:j + blk]).to(dtype)
                    q[128 * (j // blk):128 * (j // blk) + seg.numel()] = seg
                parts.append(q)
            out, sums, q, _ = _split_on_gpu(parts)
            keep = np.concatenate([np.arange(128 * j, 128 * j + blk) for j in range(len(case["scales"]))])
            keep = keep[:len(case["sums"])]
            assert np.array_equal(sums.cpu().numpy()[keep], case["sums"]), case["name"]
            assert np.array_equal(q[0][1].cpu().numpy(), case["scales"]), case["name"]
            if "out" in case:
                assert np.array_equal(out.cpu().numpy()[keep], case["out"]), case["name"]


def test_fed_by_the_out_proj_block_maxima():
    """Two tensor-parallel ranks of a Mamba-130M-like layer (M 8192 tokens, N 768, each rank
    K 768 of the 1536 channels): the partials and block maxima come from ssm_out_proj_partial,
    the shared maxima are their maximum, and the halves reproduce q8_reduce_partials."""
    M, N, K = 8192, 768, 1536
    y, W = make_out_proj_inputs(M, K, N, seed=3, device=DEV)
    ranks = [ssm.out_proj_partial(y[:, r * 768:(r + 1) * 768], W[:, r * 768:(r + 1) * 768]) for r in range(2)]
    parts = [o for o, _ in ranks]
    out, sums, q, shared = _split_on_gpu(parts, torch.bfloat16, amax_list=[a for _, a in ranks])
    fout, fsums, fscales = ssm.q8_reduce(parts, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert torch.equal(sums, fsums) and torch.equal(q[0][1], fscales) and torch.equal(out, fout)
    # the kernel's own block maxima of the stored partials are the same numbers
    assert torch.equal(torch.stack([ssm.q8_block_absmax(p) for p in parts]).amax(0), shared)


def test_nonfinite_blocks_as_the_local_reduction():
    """A NaN is ignored by the maxima and coded 0; a block holding an infinity gets scale
    +inf, codes 0 and NaN outputs -- as q8_reduce_partials documents; other blocks exact."""
    parts = make_partials(3, (128 * 6,), dtype=torch.bfloat16, seed=19)
    parts[1][128 + 5] = float("nan")
    parts[0][384 + 9] = float("inf")
    out, sums, q, _ = _split_on_gpu(parts)
    fout, fsums, fscales = ssm.q8_reduce([p.to(DEV) for p in parts], out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(sums, fsums) and torch.equal(q[0][1], fscales)
    o, fo = out.cpu().numpy(), fout.cpu().numpy()
    assert np.array_equal(np.isnan(o), np.isnan(fo)) and np.array_equal(o[~np.isnan(o)], fo[~np.isnan(fo)])
    assert np.isposinf(q[0][1][3].item()) and np.isnan(o[384:512]).all()
    assert ssm.device_status() == 0


def test_tp_all_reduce_runs_the_kernels():
    """tp.q8_all_reduce with the libssm kernels on a one-rank NCCL group on this GPU: the
    collectives are identities, so the result is the one-partial reduction bit for bit."""
    import socket

    import torch.distributed as dist

    from selective_state_space_prefill_gb300 import tp
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1)
    try:
        x = make_partials(1, (4, 1, 4096 + 64), dtype=torch.bfloat16, seed=41)[0].to(DEV)
        out, sums, scales = tp.q8_all_reduce(x, out_dtype=torch.float32)
        fout, fsums, fscales = ssm.q8_reduce([x], out_dtype=torch.float32)
        torch.cuda.synchronize()
        assert torch.equal(out.reshape(-1), fout.reshape(-1)) and torch.equal(sums, fsums)
        assert torch.equal(scales, fscales)
    finally:
        dist.destroy_process_group()
