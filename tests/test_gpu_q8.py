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
