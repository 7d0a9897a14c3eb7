"""q8_reduce_partials on the GPU: integer sums and scales bit-exact against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from _pins import read_q8_cases
from selective_state_space_prefill_gb300 import binding as ssm
from selective_state_space_prefill_gb300.inputs import make_partials

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _bits(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def _check(parts, out_dtype):
    ref = oracle.q8_reduce(parts)
    out, sums, scales = ssm.q8_reduce([p.to(DEV) for p in parts], out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert np.array_equal(sums.cpu().numpy(), ref["sums"]), "integer sums"
    assert np.array_equal(scales.cpu().numpy(), ref["scales"]), "scales"
    if out_dtype == torch.bfloat16:
        assert np.array_equal(_bits(out.reshape(-1)), ref["out_bf16"]), "bf16 out"
    else:
        assert np.array_equal(out.reshape(-1).cpu().numpy(), ref["out_f32"]), "f32 out"
    # per-block bound |out - sum_p x_p| <= P * scale / 2 (+ fp32 rounding)
    xs = np.stack([p.float().reshape(-1).numpy().astype(np.float64) for p in parts])
    n = xs.shape[1]
    scale = np.repeat(ref["scales"].astype(np.float64), 128)[:n]
    slack = 4 * 2.0 ** -24 * np.abs(xs).sum(0) + 2.0 ** -24 * np.abs(ref["out_f32"])
    assert np.all(np.abs(ref["out_f32"] - xs.sum(0)) <= len(parts) * scale / 2 + slack)


@pytest.mark.parametrize("batch", [1, 8, 64, 256])
def test_q8_sweep(batch):
    """P = 4 bf16 partial buffers [batch, 1, 4096], per-128 absmax scales."""
    _check(make_partials(4, (batch, 1, 4096), dtype=torch.bfloat16, seed=batch), torch.bfloat16)


@pytest.mark.parametrize("P", [1, 2, 3, 8])
@pytest.mark.parametrize("n", [1, 5, 127, 129, 4096 + 77])
def test_q8_ragged_and_P(P, n):
    _check(make_partials(P, (n,), dtype=torch.bfloat16, seed=P * 1000 + n), torch.float32)


def test_q8_fp32_partials_and_zero_blocks():
    parts = make_partials(3, (1000,), dtype=torch.float32, seed=11)
    for p in parts:
        p[128:256] = 0.0   # one all-zero block
        p[900:] = 0.0      # a zero tail block
    _check(parts, torch.float32)
    _check(parts, torch.bfloat16)


def test_q8_hand_cases_on_gpu():
    for case in read_q8_cases():
        for dtype in (torch.float32, torch.bfloat16):
            parts = [torch.from_numpy(p).to(dtype).to(DEV) for p in case["p"]]
            if case["block"] != 128:
                # the kernel's block is 128: pad each case block to 128 with zeros (amax unchanged)
                padded = []
                for p in parts:
                    q = torch.zeros(128 * ((p.numel() + case["block"] - 1) // case["block"]), dtype=dtype, device=DEV)
                    for j in range(0, p.numel(), case["block"]):
                        seg = p[j:j + case["block"]]
                        q[128 * (j // case["block"]):128 * (j // case["block"]) + seg.numel()] = seg
                    padded.append(q)
                parts = padded
            out, sums, scales = ssm.q8_reduce(parts, out_dtype=torch.float32)
            s = sums.cpu().numpy()
            blocks = [s[128 * j:128 * j + case["block"]] for j in range(len(case["scales"]))]
            got = np.concatenate(blocks)[:len(case["sums"])]
            assert np.array_equal(got, case["sums"]), case["name"]
            assert np.array_equal(scales.cpu().numpy(), case["scales"]), case["name"]


def _tie_blocks(n_blocks, seed):
    """Blocks of bf16 values in which fl(x * inv) is a half-integer although the exact
    product x * inv is not: round-half-even must act on the ROUNDED product (a fused
    multiply-add would round the exact product instead and miss the tie)."""
    rng = np.random.default_rng(seed)
    blocks, n_ties = [], 0
    odd = (2 * np.arange(127) + 1) / 254.0
    while len(blocks) < n_blocks:
        amax = torch.tensor(rng.uniform(0.5, 8.0)).to(torch.bfloat16).float().numpy().astype(np.float32)
        inv = np.float32(np.float32(127.0) / amax)
        cand = torch.from_numpy((amax * odd * rng.choice([-1, 1], odd.size)).astype(np.float32))
        cand = cand.to(torch.bfloat16).float().numpy()
        t = (cand * inv).astype(np.float32)                       # fp32 product, rounded
        exact = cand.astype(np.float64) * np.float64(inv)
        tie = (np.abs(t - np.trunc(t)) == 0.5) & (exact != t.astype(np.float64))
        if not tie.any():
            continue
        vals = np.zeros(128, np.float32)
        vals[0] = amax
        k = min(int(tie.sum()), 127)
        vals[1:1 + k] = cand[tie][:k]
        n_ties += k
        blocks.append(vals)
    return np.concatenate(blocks), n_ties


def test_q8_ties_of_the_rounded_product():
    """Half-integer products that only appear after fp32 rounding, one and several partials."""
    x, n_ties = _tie_blocks(256, seed=3)
    assert n_ties >= 256
    p0 = torch.from_numpy(x).to(torch.bfloat16)
    _check([p0], torch.float32)
    _check([p0, torch.zeros_like(p0), p0.neg()], torch.bfloat16)
    _check([p0.float()], torch.float32)


def test_q8_nonfinite_blocks_leave_the_others_exact():
    """Inputs outside the method: a NaN element contributes code 0; a block holding an
    infinity gets scale +inf, codes 0 and NaN outputs.  Every other block is unaffected."""
    for dtype in (torch.bfloat16, torch.float32):
        parts = make_partials(3, (128 * 8,), dtype=dtype, seed=17)
        parts[1][128 + 5] = float("nan")        # block 1: one NaN
        parts[0][384 + 9] = float("inf")        # block 3: +inf
        parts[2][640 + 1] = float("-inf")       # block 5: -inf and a NaN
        parts[0][640 + 2] = float("nan")
        out, sums, scales = ssm.q8_reduce([p.to(DEV) for p in parts], out_dtype=torch.float32)
        torch.cuda.synchronize()
        s, sc, o = sums.cpu().numpy(), scales.cpu().numpy(), out.cpu().numpy()
        finite = [0, 2, 4, 6, 7]
        ref = oracle.q8_reduce([p.reshape(8, 128)[finite].reshape(-1) for p in parts])
        got = np.concatenate([s[128 * j:128 * j + 128] for j in finite])
        assert np.array_equal(got, ref["sums"])
        assert np.array_equal(sc[finite], ref["scales"])
        # block 1: the maximum ignores the NaN, whose code is 0
        clean = [p.clone() for p in parts]
        clean[1][128 + 5] = 0.0
        ref1 = oracle.q8_reduce([c[128:256] for c in clean])
        assert np.array_equal(s[128:256], ref1["sums"]) and sc[1] == ref1["scales"][0]
        for j in (3, 5):
            assert np.isposinf(sc[j]) and not s[128 * j:128 * j + 128].any()
            assert np.isnan(o[128 * j:128 * j + 128]).all()
