"""Evidence for the reading of "1e-5 relative" with all-fp32 inputs.

The mixer is evaluated here in plain sequential float32 -- the formulas token by token
(causal width-4 conv, SiLU, softplus(dt + dt_bias), h = exp(delta A) h + delta u B,
y = C.h + D u, out = y SiLU(z)), numpy float32 ufuncs, no reordering beyond vectorising over
independent (batch, channel) rows -- and compared with the fp64 oracle on the 24 seeds of the
GPU's fp32 seed sweep (2 rows x 700 tokens x 64 channels).

Outputs of the mixer are heavy-tailed (products of Gaussians summed over a decaying state):
the largest elements reach tens of times the tensor's RMS.  There a bound of 1e-5 x RMS asks
for about one float32 ulp of the element, which the plain float32 evaluation itself misses on
some seeds, while it holds 1e-5 x max(|ref|, RMS) -- the per-element reading -- on every one.
So the per-element reading is the one an fp32 implementation of these formulas can meet.
"""
import numpy as np
import torch

import oracle
from selective_state_space_prefill_gb300.inputs import make_mixer_inputs

SEEDS = range(20, 44)


def plain_fp32_mixer(inp):
    f = np.float32
    x, z, dt = (getattr(inp, k).numpy().astype(f) for k in ("x", "z", "dt"))
    Bm, Cm = inp.B.numpy().astype(f), inp.C.numpy().astype(f)
    A, D, bias = inp.A.numpy().astype(f), inp.D.numpy().astype(f), inp.dt_bias.numpy().astype(f)
    w, cb = inp.conv_w.numpy().astype(f), inp.conv_b.numpy().astype(f)
    batch, L, d = x.shape
    n_state = A.shape[1]
    h = np.zeros((batch, d, n_state), f)
    prev = np.zeros((batch, 3, d), f)          # x[t-3], x[t-2], x[t-1]
    out = np.zeros((batch, L, d), f)
    one = f(1)
    for t in range(L):
        xt = x[:, t]
        xc = cb + w[:, 0] * prev[:, 0]
        xc = xc + w[:, 1] * prev[:, 1]
        xc = xc + w[:, 2] * prev[:, 2]
        xc = xc + w[:, 3] * xt
        prev = np.stack([prev[:, 1], prev[:, 2], xt], 1)
        u = xc / (one + np.exp(-xc))
        v = dt[:, t] + bias
        delta = np.where(v > 20, v, np.log1p(np.exp(np.minimum(v, f(20)))))
        h = np.exp(delta[:, :, None] * A[None]) * h + (delta * u)[:, :, None] * Bm[:, t][:, None, :]
        y = np.zeros((batch, d), f)
        for n in range(n_state):
            y = y + Cm[:, t, n][:, None] * h[:, :, n]
        out[:, t] = (y + D * u) * (z[:, t] / (one + np.exp(-z[:, t])))
    return out, h


def _errors(got, ref):
    err = np.abs(got.astype(np.float64) - ref)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    return float(err.max() / rms), float(np.max(err / np.maximum(np.abs(ref), rms)))


def test_plain_fp32_misses_the_rms_bar_and_holds_the_per_element_bar():
    worst_rms, worst_el = {}, {}
    for seed in SEEDS:
        inp = make_mixer_inputs(2, 700, 64, dtype=torch.float32, seed=seed)
        out, h = plain_fp32_mixer(inp)
        ref = oracle.prefill(inp.x, inp.z, inp.dt, inp.B, inp.C, inp.A, inp.D, inp.dt_bias, inp.conv_w,
                             inp.conv_b)
        for got, r, what in ((out, ref["out"], "out"), (h, ref["ssm_state"], "state")):
            e_rms, e_el = _errors(got, r)
            worst_rms[(seed, what)] = e_rms
            worst_el[(seed, what)] = e_el
    # the RMS-relative reading: the plain float32 evaluation itself fails it on some seed
    k = max(worst_rms, key=worst_rms.get)
    assert worst_rms[k] > 1e-5, f"plain fp32 stays within 1e-5 x RMS everywhere (worst {worst_rms[k]:.2e} at {k})"
    # the per-element reading (RMS floor near zero crossings): held on every seed and output
    k = max(worst_el, key=worst_el.get)
    assert worst_el[k] <= 1e-5, f"plain fp32 misses the per-element bar: {worst_el[k]:.2e} at {k}"
