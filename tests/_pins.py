"""Pins that tie the fp64 oracle to facts other than itself.

Each pin takes an oracle library handle (``oracle.oracle.load()`` or a mutated
copy) and raises AssertionError when the oracle disagrees with:

* closed forms of the recurrence (A = 0 gives a prefix sum, constant a and b give
  a geometric series, C = 0 leaves only the skip and gate),
* an O(L^2) brute force that unrolls h_t = sum_s (prod_{r>s} a_r) b_s with explicit
  products and evaluates the causal conv as a Toeplitz matrix product,
* the state-caching invariant (prefill then decode = longer prefill) and channel-
  slice independence from the pages' Methodology 2 and 3,
* hand-derived cases of the 8-bit reduction (tests/golden/q8_hand_cases.txt) and
  its per-block error bound,
* an independent fp64 matrix product and closed forms (identity, rank one) for the
  output-projection partial.

The same pins run against deliberately broken copies of the oracle source in
``test_oracle_mutations.py``; each planted mistake must fail at least one pin.
"""
from __future__ import annotations

from pathlib import Path

import numpy as np
import torch
from scipy.special import expit

import oracle.oracle as orc
from selective_state_space_prefill_gb300.inputs import (log_expm1, make_mixer_inputs, make_partials,
                                                         make_ssd_inputs)

GOLDEN = Path(__file__).resolve().parent / "golden"


# ----------------------------------------------------------------- helpers
def _np64(t):
    return t.detach().cpu().double().numpy() if isinstance(t, torch.Tensor) else np.asarray(t, np.float64)


def _close(got, ref, rel=1e-12, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, f"{what}: shape {got.shape} vs {ref.shape}"
    scale = max(1.0, float(np.max(np.abs(ref))) if ref.size else 1.0)
    err = float(np.max(np.abs(got - ref))) if ref.size else 0.0
    assert err <= rel * scale, f"{what}: max|err| {err:.3e} > {rel:.1e} * {scale:.3e}"


def _run_prefill(lib, inp, cs=None, ss=None, **kw):
    return orc.prefill(inp.x, inp.z, inp.dt, inp.B, inp.C, inp.A, inp.D, inp.dt_bias,
                       inp.conv_w, inp.conv_b, conv_state_in=cs, ssm_state_in=ss, n_threads=2,
                       lib=lib, **kw)


def brute_force_prefill(inp, cs=None, ss=None):
    """Independent O(L^2) evaluation of one prefill in float64.

    conv: xc = T_d @ [conv_state_in ; x] with T_d the banded Toeplitz matrix of
    conv_w[d]; u = xc * expit(xc); delta = logaddexp(0, dt + dt_bias);
    h_t = (prod_{r<=t} a_r) h_0 + sum_{s<=t} (prod_{s<r<=t} a_r) b_s with
    a_r = exp(delta_r A), b_s = delta_s B_s u_s; y = C h + D u; out = y z expit(z).
    """
    x, z, dt, B, C = (_np64(getattr(inp, k)) for k in ("x", "z", "dt", "B", "C"))
    A, D, dtb, w, cb = (_np64(getattr(inp, k)) for k in ("A", "D", "dt_bias", "conv_w", "conv_b"))
    batch, L, Dn = x.shape
    N, W = A.shape[1], w.shape[1]
    cs = np.zeros((batch, W - 1, Dn)) if cs is None else _np64(cs)
    ss = np.zeros((batch, Dn, N)) if ss is None else _np64(ss)
    out = np.zeros((batch, L, Dn))
    h_last = np.zeros((batch, Dn, N))
    for b in range(batch):
        xe = np.concatenate([cs[b], x[b]], 0)  # [(W-1)+L, Dn], oldest first
        for d in range(Dn):
            T = np.zeros((L, L + W - 1))
            for t in range(L):
                T[t, t:t + W] = w[d]
            xc = T @ xe[:, d] + cb[d]
            u = xc * expit(xc)
            delta = np.logaddexp(0.0, dt[b, :, d] + dtb[d])
            a = np.exp(delta[:, None] * A[d][None, :])  # [L, N]
            bb = (delta * u)[:, None] * B[b]  # [L, N]
            for t in range(L):
                h = np.prod(a[:t + 1], axis=0) * ss[b, d]
                for s in range(t + 1):
                    h = h + np.prod(a[s + 1:t + 1], axis=0) * bb[s]
                y = float(np.dot(C[b, t], h)) + D[d] * u[t]
                out[b, t, d] = y * z[b, t, d] * expit(z[b, t, d])
                if t == L - 1:
                    h_last[b, d] = h
            if L == 0:
                h_last[b, d] = ss[b, d]
    xe_all = np.concatenate([cs, x], 1)
    conv_last = xe_all[:, xe_all.shape[1] - (W - 1):, :]
    return dict(out=out, conv_state=conv_last, ssm_state=h_last)


# ----------------------------------------------------------------- mixer pins
def pin_brute_force(lib, dtype=torch.float32, seed=1, L=13, batch=2, Dn=5):
    """Random tiny problem with input states vs the O(L^2) brute force."""
    inp = make_mixer_inputs(batch, L, Dn, dtype=dtype, seed=seed)
    g = torch.Generator().manual_seed(seed + 1)
    inp.conv_b = torch.randn(Dn, generator=g) * 0.3
    inp.D = torch.randn(Dn, generator=g)
    inp.A = -torch.rand(Dn, 16, generator=g) * 2.0
    cs = torch.randn(batch, 3, Dn, generator=g, dtype=torch.float64)
    ss = torch.randn(batch, Dn, 16, generator=g, dtype=torch.float64)
    got = _run_prefill(lib, inp, cs, ss)
    ref = brute_force_prefill(inp, cs, ss)
    for k in ("out", "ssm_state", "conv_state"):
        _close(got[k], ref[k], 1e-12, f"brute force {k}")


def pin_brute_force_bf16(lib):
    pin_brute_force(lib, dtype=torch.bfloat16, seed=3, L=9, batch=1, Dn=4)


def pin_short_sequence(lib):
    """L = 2 < W - 1: the output conv state mixes the input state and the new tokens."""
    pin_brute_force(lib, seed=5, L=2, batch=1, Dn=3)


def pin_prefix_sum_A_zero(lib, L=40, Dn=6):
    """A = 0: a_t = 1, so h_t = h_0 + sum_{s<=t} delta_s B_s u_s (a running sum).

    With conv_w = (0, 0, 0, 1), conv_b = 0: u = x expit(x).  With dt = 0 and
    dt_bias = log(expm1(v)): delta = softplus(dt_bias).
    """
    inp = make_mixer_inputs(1, L, Dn, dtype=torch.float32, seed=11)
    inp.A = torch.zeros(Dn, 16)
    inp.conv_w = torch.tensor([[0.0, 0.0, 0.0, 1.0]]).repeat(Dn, 1)
    inp.dt = torch.zeros_like(inp.dt)
    inp.D = torch.full((Dn,), 0.75)
    g = torch.Generator().manual_seed(12)
    ss = torch.randn(1, Dn, 16, generator=g, dtype=torch.float64)
    got = _run_prefill(lib, inp, None, ss)
    x, z, B, C = (_np64(getattr(inp, k))[0] for k in ("x", "z", "B", "C"))
    delta = np.logaddexp(0.0, _np64(inp.dt_bias))  # [Dn]
    u = x * expit(x)  # [L, Dn]
    incr = delta[None, :, None] * u[:, :, None] * B[:, None, :]  # [L, Dn, N]
    h = _np64(ss)[0][None] + np.cumsum(incr, axis=0)
    y = np.einsum("tn,tdn->td", C, h) + 0.75 * u
    _close(got["ssm_state"][0], h[-1], 1e-12, "prefix-sum state")
    _close(got["out"][0], y * z * expit(z), 1e-12, "prefix-sum out")


def pin_geometric_series(lib, L=64, Dn=4):
    """Constant a and b: h_t = a^(t+1) h_0 + b (1 - a^(t+1)) / (1 - a)."""
    inp = make_mixer_inputs(1, L, Dn, dtype=torch.float32, seed=21)
    c = torch.tensor([0.8, -1.3, 2.0, 0.4])[:Dn]
    w3 = torch.tensor([0.9, 0.5, -0.7, 1.1])[:Dn]
    inp.x = c[None, None, :].expand(1, L, Dn).contiguous()
    inp.conv_w = torch.zeros(Dn, 4)
    inp.conv_w[:, 3] = w3
    inp.conv_b = torch.zeros(Dn)
    inp.dt = torch.zeros(1, L, Dn)
    inp.dt_bias = torch.tensor([-1.0, 0.3, -2.5, 0.0])[:Dn]
    Bn = torch.randn(16, generator=torch.Generator().manual_seed(22))
    inp.B = Bn[None, None, :].expand(1, L, 16).contiguous()
    ss = torch.randn(1, Dn, 16, generator=torch.Generator().manual_seed(23), dtype=torch.float64)
    got = _run_prefill(lib, inp, None, ss)
    xc = _np64(c) * _np64(w3)
    u = xc * expit(xc)
    delta = np.logaddexp(0.0, _np64(inp.dt_bias))
    A = _np64(inp.A)
    a = np.exp(delta[:, None] * A)  # [Dn, N]
    b = (delta * u)[:, None] * _np64(Bn)[None, :]
    t = np.arange(1, L + 1)[:, None, None]
    h = a[None] ** t * _np64(ss)[0][None] + b[None] * (1 - a[None] ** t) / (1 - a[None])
    C = _np64(inp.C)[0]
    z = _np64(inp.z)[0]
    y = np.einsum("tn,tdn->td", C, h) + _np64(inp.D)[None, :] * u[None, :]
    _close(got["ssm_state"][0], h[-1], 1e-12, "geometric state")
    _close(got["out"][0], y * z * expit(z), 1e-11, "geometric out")


def pin_C_zero_skip_gate(lib, L=33, Dn=7):
    """C = 0: out = D u SiLU(z) with u from the Toeplitz conv (states in)."""
    inp = make_mixer_inputs(2, L, Dn, dtype=torch.float32, seed=31)
    inp.C = torch.zeros_like(inp.C)
    g = torch.Generator().manual_seed(32)
    inp.D = torch.randn(Dn, generator=g)
    inp.conv_b = torch.randn(Dn, generator=g)
    cs = torch.randn(2, 3, Dn, generator=g, dtype=torch.float64)
    got = _run_prefill(lib, inp, cs, None)
    x, z, w = _np64(inp.x), _np64(inp.z), _np64(inp.conv_w)
    xe = np.concatenate([_np64(cs), x], 1)
    xc = sum(w[None, None, :, k] * xe[:, k:k + L, :] for k in range(4)) + _np64(inp.conv_b)
    u = xc * expit(xc)
    _close(got["out"], _np64(inp.D) * u * z * expit(z), 1e-12, "C = 0")
    _close(got["conv_state"], xe[:, L:, :], 0.0, "conv state")


def pin_softplus_ln2(lib, L=8, Dn=3):
    """dt = dt_bias = 0: delta = ln 2 exactly; with A = 0, B = 1 the state is ln2 * sum u."""
    inp = make_mixer_inputs(1, L, Dn, dtype=torch.float32, seed=41)
    inp.dt = torch.zeros_like(inp.dt)
    inp.dt_bias = torch.zeros(Dn)
    inp.A = torch.zeros(Dn, 16)
    inp.B = torch.ones_like(inp.B)
    inp.conv_w = torch.tensor([[0.0, 0.0, 0.0, 1.0]]).repeat(Dn, 1)
    got = _run_prefill(lib, inp)
    x = _np64(inp.x)[0]
    u = x * expit(x)
    _close(got["ssm_state"][0], np.repeat((np.log(2.0) * u.sum(0))[:, None], 16, 1), 1e-13, "ln2")


def pin_dt_bias_is_softplus_inverse(lib, Dn=16):
    """dt = 0 with dt_bias = log(expm1(u)): delta = softplus(dt_bias) = u, up to the fp32 rounding of
    dt_bias (times the slope sigmoid(dt_bias) ~ u).  A = 0, B = 1, x = 1 and the current-token tap only
    leave h = delta * SiLU(1) after one token."""
    u = torch.exp(torch.linspace(np.log(1e-3), np.log(1e-1), Dn, dtype=torch.float64))
    inp = make_mixer_inputs(1, 1, Dn, dtype=torch.float32, seed=43)
    inp.x = torch.ones_like(inp.x)
    inp.dt = torch.zeros_like(inp.dt)
    inp.dt_bias = log_expm1(u).float()
    inp.A = torch.zeros(Dn, 16)
    inp.B = torch.ones_like(inp.B)
    inp.conv_w = torch.tensor([[0.0, 0.0, 0.0, 1.0]]).repeat(Dn, 1)
    inp.conv_b = torch.zeros(Dn)
    got = _run_prefill(lib, inp)
    delta = got["ssm_state"][0][:, 0] / expit(1.0)
    b64 = log_expm1(u).numpy()
    slack = np.abs(inp.dt_bias.double().numpy() - b64) * expit(b64) * 1.01 + 1e-15
    assert np.all(np.abs(delta - u.numpy()) <= slack + 1e-13 * u.numpy()), (delta, u)

def pin_state_caching(lib, L1=21, L2=11, Dn=6, dtype=torch.float32):
    """Methodology 3: prefill(L1) then L2 decode steps equals prefill(L1 + L2)."""
    inp = make_mixer_inputs(2, L1 + L2, Dn, dtype=dtype, seed=51)
    full = _run_prefill(lib, inp)
    part = _run_prefill(lib, inp.token_slice(0, L1))
    cs, ss = part["conv_state"], part["ssm_state"]
    outs = []
    for t in range(L1, L1 + L2):
        step = orc.decode_step(inp.x[:, t], inp.z[:, t], inp.dt[:, t], inp.B[:, t], inp.C[:, t],
                               inp.A, inp.D, inp.dt_bias, inp.conv_w, inp.conv_b, cs, ss, lib=lib)
        cs, ss = step["conv_state"], step["ssm_state"]
        outs.append(step["out"])
    _close(part["out"], full["out"][:, :L1], 0.0, "prefix of prefill")
    _close(np.stack(outs, 1), full["out"][:, L1:], 1e-12, "decode tail")
    _close(ss, full["ssm_state"], 1e-12, "decode ssm_state")
    _close(cs, full["conv_state"], 0.0, "decode conv_state")
    # and prefill resumed from the cached states (chunked prefill)
    rest = _run_prefill(lib, inp.token_slice(L1, L1 + L2), part["conv_state"], part["ssm_state"])
    _close(rest["out"], full["out"][:, L1:], 1e-12, "resumed prefill")
    _close(rest["ssm_state"], full["ssm_state"], 1e-12, "resumed ssm_state")


def pin_decode_matches_brute(lib, Dn=9):
    """One decode step from random states equals the brute force over one token."""
    inp = make_mixer_inputs(3, 1, Dn, dtype=torch.bfloat16, seed=61)
    g = torch.Generator().manual_seed(62)
    cs = torch.randn(3, 3, Dn, generator=g, dtype=torch.float64)
    ss = torch.randn(3, Dn, 16, generator=g, dtype=torch.float64)
    step = orc.decode_step(inp.x[:, 0], inp.z[:, 0], inp.dt[:, 0], inp.B[:, 0], inp.C[:, 0],
                           inp.A, inp.D, inp.dt_bias, inp.conv_w, inp.conv_b, cs, ss, lib=lib)
    ref = brute_force_prefill(inp, cs, ss)
    _close(step["out"], ref["out"][:, 0], 1e-12, "decode out")
    _close(step["ssm_state"], ref["ssm_state"], 1e-12, "decode state")
    _close(step["conv_state"], ref["conv_state"], 0.0, "decode conv state")


def pin_split_invariance(lib, L=24, Dn=16):
    """Methodology 2: channels split into slices and run alone equal the unsplit run."""
    inp = make_mixer_inputs(2, L, Dn, dtype=torch.bfloat16, seed=71)
    full = _run_prefill(lib, inp)
    for lo, hi in ((0, 4), (4, 12), (12, 16)):
        part = _run_prefill(lib, inp, channels=list(range(lo, hi)))
        assert np.array_equal(part["out"], full["out"][..., lo:hi]), "split out"
        assert np.array_equal(part["ssm_state"], full["ssm_state"][:, lo:hi]), "split state"


def pin_scan_sequential(lib):
    """a = 1 gives a running sum; constant (a, b) gives the geometric series."""
    rng = np.random.default_rng(81)
    b = rng.standard_normal(50)
    _close(orc.scan_sequential(np.ones(50), b, 0.5, lib=lib), 0.5 + np.cumsum(b), 1e-13, "cumsum")
    a = 0.93
    t = np.arange(1, 51)
    ref = a ** t * 2.0 + 0.3 * (1 - a ** t) / (1 - a)
    _close(orc.scan_sequential(np.full(50, a), np.full(50, 0.3), 2.0, lib=lib), ref, 1e-13, "geom")


def pin_scan_chunked(lib):
    """The chunked associative scan equals the sequential scan for any chunk size."""
    rng = np.random.default_rng(91)
    L = 300
    a = rng.uniform(0.0, 1.0, L)
    b = rng.standard_normal(L)
    seq = orc.scan_sequential(a, b, -0.7, lib=lib)
    for chunk in (1, 7, 64, 299, 300, 1000):
        _close(orc.scan_chunked(a, b, -0.7, chunk, lib=lib), seq, 1e-12, f"chunk {chunk}")


# ----------------------------------------------------------------- q8 pins
def read_q8_cases(path=GOLDEN / "q8_hand_cases.txt"):
    cases, cur = [], None
    for raw in Path(path).read_text().splitlines():
        line = raw.split("#", 1)[0].strip()
        if not line:
            continue
        head, *rest = line.split()
        if head == "case":
            kv = dict(item.split("=") for item in rest[1:])
            cur = dict(name=rest[0], block=int(kv["block"]), P=int(kv["P"]), p=[])
        elif head == "p":
            cur["p"].append(np.array([float(v) for v in rest], np.float32))
        elif head == "sums":
            cur["sums"] = np.array([int(v) for v in rest], np.int32)
        elif head == "scales":
            cur["scales"] = np.array([float.fromhex(v) for v in rest], np.float32)
        elif head == "out":
            cur["out"] = np.array([float(v) for v in rest], np.float32)
        elif head == "end":
            assert len(cur["p"]) == cur["P"]
            cases.append(cur)
            cur = None
    return cases


def pin_q8_hand_cases(lib):
    for case in read_q8_cases():
        for dtype in (torch.float32, torch.bfloat16):
            parts = [torch.from_numpy(p).to(dtype) for p in case["p"]]
            r = orc.q8_reduce(parts, case["block"], lib=lib)
            assert np.array_equal(r["sums"], case["sums"]), (case["name"], r["sums"])
            assert np.array_equal(r["scales"], case["scales"]), (case["name"], r["scales"])
            if "out" in case:
                assert np.array_equal(r["out_f32"], case["out"]), (case["name"], r["out_f32"])


def pin_q8_bounds(lib, P=4, n=4096 + 77, block=128):
    """|out - sum_p x_p| <= P * scale / 2 per block (plus fp32 rounding); P = 1 round trip."""
    parts = make_partials(P, (n,), dtype=torch.bfloat16, seed=101)
    r = orc.q8_reduce(parts, block, lib=lib)
    xs = np.stack([p.float().numpy().astype(np.float64) for p in parts])
    exact = xs.sum(0)
    scale = np.repeat(r["scales"].astype(np.float64), block)[:n]
    amax = np.maximum.reduceat(np.abs(xs).max(0), np.arange(0, n, block))
    assert np.array_equal(r["scales"], (amax.astype(np.float32) / np.float32(127.0))), "scale"
    slack = 4 * 2.0 ** -24 * np.abs(xs).sum(0) + 2.0 ** -24 * np.abs(r["out_f32"])
    assert np.all(np.abs(r["out_f32"] - exact) <= P * scale / 2 + slack), "P*scale/2 bound"
    assert np.all(np.abs(r["sums"]) <= 127 * P)
    one = orc.q8_reduce(parts[:1], block, lib=lib)
    s1 = np.repeat(one["scales"].astype(np.float64), block)[:n]
    assert np.all(np.abs(one["out_f32"] - xs[0]) <= s1 / 2 + 4 * 2.0 ** -24 * np.abs(xs[0])), "P=1"
    bf = torch.from_numpy(r["out_f32"]).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(r["out_bf16"], bf), "bf16 rounding of the output"



def _split_reduce(parts, block, lib):
    """The rank-local halves composed: max of the ranks' block maxima, codes, sum."""
    amax = np.max(np.stack([orc.q8_block_absmax(p, block, lib=lib) for p in parts]), 0)
    q = [orc.q8_quantize_shared(p, amax, block, lib=lib) for p in parts]
    for r in q[1:]:
        assert np.array_equal(r["scales"], q[0]["scales"]), "ranks disagree on the shared scale"
    s = orc.q8_sum_dequant([r["codes"] for r in q], q[0]["scales"], block, lib=lib)
    return s, q


def pin_q8_split_hand_cases(lib):
    """The hand-derived cases (golden file) through the rank-local halves."""
    for case in read_q8_cases():
        for dtype in (torch.float32, torch.bfloat16):
            parts = [torch.from_numpy(p).to(dtype) for p in case["p"]]
            s, q = _split_reduce(parts, case["block"], lib)
            assert np.array_equal(s["sums"], case["sums"]), (case["name"], s["sums"])
            assert np.array_equal(q[0]["scales"], case["scales"]), (case["name"], q[0]["scales"])
            if "out" in case:
                assert np.array_equal(s["out_f32"], case["out"]), (case["name"], s["out_f32"])


def pin_q8_split_composes_to_reduce(lib):
    """Block maxima combined by max, shared-scale codes and their sum equal the local
    reduction bit for bit (sums, scales, fp32 and bf16 outputs), for ragged lengths."""
    for P, n, dtype, seed in ((1, 300, torch.float32, 7), (3, 128 * 9 + 5, torch.bfloat16, 8),
                              (4, 4096, torch.bfloat16, 9), (8, 1000, torch.float32, 10)):
        parts = make_partials(P, (n,), dtype=dtype, seed=seed)
        ref = orc.q8_reduce(parts, 128, lib=lib)
        s, q = _split_reduce(parts, 128, lib)
        assert np.array_equal(s["sums"], ref["sums"]), (P, n, "sums")
        assert np.array_equal(q[0]["scales"], ref["scales"]), (P, n, "scales")
        assert np.array_equal(s["out_f32"], ref["out_f32"]), (P, n, "out")
        assert np.array_equal(s["out_bf16"], ref["out_bf16"]), (P, n, "bf16 out")


def pin_q8_split_round_trip(lib, n=128 * 5 + 33):
    """Independent checks of each half: the block maxima are numpy's; every code lies in
    [-127, 127] and dequantizes within half a scale of its value; a block of zeros gives
    zero codes and scale; one code buffer dequantizes to code * scale."""
    x = make_partials(1, (n,), dtype=torch.float32, seed=11)[0]
    x[128:256] = 0.0
    xs = x.numpy().astype(np.float64)
    amax = orc.q8_block_absmax(x, 128, lib=lib)
    ref = np.array([np.abs(xs[j:j + 128]).max() for j in range(0, n, 128)], np.float32)
    assert np.array_equal(amax, ref), "block maxima"
    q = orc.q8_quantize_shared(x, amax, 128, lib=lib)
    c = q["codes"].astype(np.int64)
    sc = np.repeat(q["scales"].astype(np.float64), 128)[:n]
    assert np.all(np.abs(c) <= 127)
    assert np.all(np.abs(c * sc - xs) <= sc / 2 + 4 * 2.0 ** -24 * np.abs(xs)), "half-scale round trip"
    assert q["scales"][1] == 0.0 and not np.any(c[128:256]), "zero block"
    assert np.array_equal(q["scales"], (amax / np.float32(127.0)).astype(np.float32)), "scale"
    s = orc.q8_sum_dequant([q["codes"]], q["scales"], 128, lib=lib)
    assert np.array_equal(s["sums"], q["codes"].astype(np.int32))
    assert np.array_equal(s["out_f32"], (q["codes"].astype(np.float32) * np.repeat(q["scales"], 128)[:n]))


def pin_out_proj_vs_matmul(lib):
    """The partial equals an independent fp64 matrix product of the widened inputs; absdot is
    |y| |W|^T; the block maxima are those of the row-major partial, the last block short."""
    g = torch.Generator().manual_seed(7)
    for dtype in (torch.bfloat16, torch.float32):
        y = torch.randn(33, 70, generator=g).to(dtype)
        W = torch.randn(21, 70, generator=g).to(dtype)
        r = orc.out_proj(y, W, lib=lib)
        yd, wd = _np64(y), _np64(W)
        ref = yd @ wd.T
        _close(r["out"], ref, 1e-12, "out_proj vs matmul")
        _close(r["absdot"], np.abs(yd) @ np.abs(wd).T, 1e-12, "absdot")
        flat = np.abs(ref).reshape(-1)
        blocks = [flat[i:i + 128].max() for i in range(0, flat.size, 128)]
        assert r["amax"].shape == (len(blocks),) and flat.size % 128 != 0
        _close(r["amax"], np.array(blocks), 1e-12, "block amax")


def pin_out_proj_identity_and_rank_one(lib):
    """W = I returns y exactly; rank-one y and W give the closed form u_m p_n (v . q)."""
    y = torch.randn(9, 16, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    r = orc.out_proj(y, torch.eye(16).to(torch.bfloat16), lib=lib)
    assert np.array_equal(r["out"], _np64(y)), "identity"
    u = np.array([1, -2, 3, 0.5, -4], np.float64)
    v = np.array([2, -1, 0.25, 3, 1, -2, 0.5], np.float64)
    pn = np.array([-1, 2, 0.5], np.float64)
    q = np.array([1, 1, -3, 0.5, 2, -1, 4], np.float64)
    yy = torch.from_numpy(np.outer(u, v)).to(torch.bfloat16)   # small dyadic values: exact in bf16
    WW = torch.from_numpy(np.outer(pn, q)).to(torch.bfloat16)
    r = orc.out_proj(yy, WW, lib=lib)
    assert np.array_equal(r["out"], np.outer(u, pn) * float(v @ q)), "rank one"

# ----------------------------------------------------------------- SSD (Mamba-2-style) pins
def _ssd_run(lib, inp, cs=None, ss=None, **kw):
    return orc.ssd_prefill(inp.xBC, inp.z, inp.dt, inp.conv_w, inp.conv_b, inp.A, inp.D, inp.dt_bias,
                           inp.n_heads, inp.head_dim, inp.n_groups, inp.d_state,
                           conv_state_in=cs, ssm_state_in=ss, n_threads=2, lib=lib, **kw)


def _ssd_conv_silu(inp, cs):
    """u[b, t, c] = SiLU(conv_b[c] + sum_k conv_w[c, k] xe[b, t + k, c]) over xe = [cs ; xBC]."""
    x = _np64(inp.xBC)
    w, cb = _np64(inp.conv_w), _np64(inp.conv_b)
    batch, L, Cx = x.shape
    W = w.shape[1]
    xe = np.concatenate([cs, x], 1)
    xc = np.broadcast_to(cb, (batch, L, Cx)).copy()
    for k in range(W):
        xc += w[:, k][None, None, :] * xe[:, k:k + L, :]
    return xc * expit(xc), xe


def ssd_matrix_form(inp, cs=None, ss=None, chunk=None):
    """The SSD mixer evaluated through its quadratic ("dual") matrix form, in float64.

    Per batch row and head h (group g = h // (H // G)), with u = SiLU(conv(xBC)):
      delta_t = logaddexp(0, dt_t + dt_bias_h), s_t = sum_{r <= t} delta_r A_h,
      M[i, j] = exp(s_i - s_j) (C_i . B_j) for j <= i, else 0,
      Y = M @ (delta[:, None] x) + exp(s)[:, None] (C @ S0^T) + D_h x,
      S_L = exp(s_L) S0 + (x * w[:, None])^T B with w_j = exp(s_L - s_j) delta_j,
      out = Y * z * expit(z).
    With ``chunk`` the same form is applied chunk by chunk, the state carried between chunks
    (the chunked algorithm the GPU kernel follows).  Nothing here steps a recurrence token by token.
    """
    H, P, G, N = inp.n_heads, inp.head_dim, inp.n_groups, inp.d_state
    z, dt = _np64(inp.z), _np64(inp.dt)
    A, D, dtb = _np64(inp.A), _np64(inp.D), _np64(inp.dt_bias)
    batch, L, Cx = inp.xBC.shape
    W = inp.conv_w.shape[1]
    cs = np.zeros((batch, W - 1, Cx)) if cs is None else _np64(cs)
    ss = np.zeros((batch, H, P, N)) if ss is None else _np64(ss)
    u, xe = _ssd_conv_silu(inp, cs)
    out = np.zeros((batch, L, H * P))
    s_last = np.zeros((batch, H, P, N))
    Q = L if not chunk else chunk
    for b in range(batch):
        for h in range(H):
            g = h // (H // G)
            xh = u[b, :, h * P:(h + 1) * P]
            Bg = u[b, :, H * P + g * N:H * P + (g + 1) * N]
            Cg = u[b, :, H * P + G * N + g * N:H * P + G * N + (g + 1) * N]
            delta = np.logaddexp(0.0, dt[b, :, h] + dtb[h])
            S = ss[b, h].copy()
            for t0 in range(0, L, max(Q, 1)):
                t1 = min(L, t0 + Q)
                dl, xc, Bc, Cc = delta[t0:t1], xh[t0:t1], Bg[t0:t1], Cg[t0:t1]
                sc = np.cumsum(dl * A[h])
                diff = sc[:, None] - sc[None, :]
                M = np.where(np.tril(np.ones((t1 - t0, t1 - t0), bool)), np.exp(np.minimum(diff, 0.0)), 0.0)
                M = M * (Cc @ Bc.T)
                Y = M @ (dl[:, None] * xc) + np.exp(sc)[:, None] * (Cc @ S.T) + D[h] * xc
                out[b, t0:t1, h * P:(h + 1) * P] = Y * z[b, t0:t1, h * P:(h + 1) * P] * expit(
                    z[b, t0:t1, h * P:(h + 1) * P])
                w = np.exp(sc[-1] - sc) * dl
                S = np.exp(sc[-1]) * S + (xc * w[:, None]).T @ Bc
            s_last[b, h] = S
    return dict(out=out, conv_state=xe[:, xe.shape[1] - (W - 1):, :], ssm_state=s_last)


def _ssd_tiny(seed, dtype=torch.float32, batch=2, L=13, H=4, P=3, G=2, N=5):
    inp = make_ssd_inputs(batch, L, H, P, G, N, dtype=dtype, seed=seed)
    g = torch.Generator().manual_seed(seed + 11)
    inp.conv_b = torch.randn(inp.channels, generator=g) * 0.3
    inp.D = torch.randn(H, generator=g)
    cs = torch.randn(batch, 3, inp.channels, generator=g, dtype=torch.float64)
    ss = torch.randn(batch, H, P, N, generator=g, dtype=torch.float64)
    return inp, cs, ss


def pin_ssd_matrix_form(lib):
    """Random tiny SSD problems (fp32 and bf16, with input states) against the quadratic form."""
    for seed, dtype in ((21, torch.float32), (22, torch.bfloat16)):
        inp, cs, ss = _ssd_tiny(seed, dtype)
        got = _ssd_run(lib, inp, cs, ss)
        ref = ssd_matrix_form(inp, cs, ss)
        for k in ("out", "ssm_state", "conv_state"):
            _close(got[k], ref[k], 1e-12, f"SSD matrix form {k} ({dtype})")


def pin_ssd_chunked_state_passing(lib):
    """The chunk-by-chunk form with the state carried across chunks equals the oracle for
    chunk sizes 1, 4, 7 and L (and a ragged last chunk)."""
    inp, cs, ss = _ssd_tiny(23, batch=1, L=17, H=2, P=4, G=1, N=6)
    got = _ssd_run(lib, inp, cs, ss)
    for q in (1, 4, 7, 17):
        ref = ssd_matrix_form(inp, cs, ss, chunk=q)
        for k in ("out", "ssm_state"):
            _close(got[k], ref[k], 1e-12, f"SSD chunk {q} {k}")


def pin_ssd_state_caching(lib, L1=11, L2=9):
    """Prefill of L1 tokens, then of L2 more from the returned states, equals one prefill of L1 + L2."""
    inp, cs, ss = _ssd_tiny(24, batch=2, L=L1 + L2, H=4, P=3, G=2, N=4)
    full = _ssd_run(lib, inp, cs, ss)
    first = _ssd_run(lib, inp.token_slice(0, L1), cs, ss)
    second = _ssd_run(lib, inp.token_slice(L1, L1 + L2), first["conv_state"], first["ssm_state"])
    _close(np.concatenate([first["out"], second["out"]], 1), full["out"], 1e-12, "SSD caching out")
    _close(second["ssm_state"], full["ssm_state"], 1e-12, "SSD caching ssm_state")
    _close(second["conv_state"], full["conv_state"], 0.0, "SSD caching conv_state")


def pin_ssd_reduces_to_mamba1(lib, L=15, H=6, N=5):
    """With one position per head (P = 1), one group and identity convs on the B and C
    channels, the SSD mixer is the selective-scan mixer with A[d, n] = A[h] for every n and
    B, C replaced by SiLU(B), SiLU(C): the two oracles must agree (fp32 rounding of the
    SiLU'd B and C handed to the selective-scan oracle is the only difference)."""
    inp = make_ssd_inputs(1, L, H, 1, 1, N, dtype=torch.float32, seed=25)
    w = inp.conv_w.clone()
    w[H:] = torch.tensor([0.0, 0.0, 0.0, 1.0])
    inp.conv_w = w
    got = _ssd_run(lib, inp)
    xBC = _np64(inp.xBC)
    Bs = torch.from_numpy(xBC[..., H:H + N] * expit(xBC[..., H:H + N])).float()
    Cs = torch.from_numpy(xBC[..., H + N:] * expit(xBC[..., H + N:])).float()
    m1 = orc.prefill(inp.xBC[..., :H].contiguous(), inp.z, inp.dt, Bs, Cs,
                     inp.A[:, None].expand(H, N).contiguous(), inp.D, inp.dt_bias,
                     inp.conv_w[:H].contiguous(), inp.conv_b[:H].contiguous(), n_threads=2)
    _close(got["out"], m1["out"], 1e-6, "SSD vs selective scan out")
    _close(got["ssm_state"][..., 0, :], m1["ssm_state"], 1e-6, "SSD vs selective scan state")


def pin_ssd_heads_subset(lib):
    """Evaluating a subset of heads gives exactly those heads of the full run (and NaN elsewhere)."""
    inp, cs, ss = _ssd_tiny(26, batch=2, L=10, H=6, P=2, G=3, N=3)
    full = _ssd_run(lib, inp, cs, ss)
    part = _ssd_run(lib, inp, cs, ss, heads=[4, 1])
    P = inp.head_dim
    for h in (1, 4):
        assert np.array_equal(part["out"][..., h * P:(h + 1) * P], full["out"][..., h * P:(h + 1) * P])
        assert np.array_equal(part["ssm_state"][:, h], full["ssm_state"][:, h])
    assert np.isnan(part["out"][..., 0]).all()
    HP, N, G = inp.n_heads * P, inp.d_state, inp.n_groups
    for g in (0, 2):                      # the groups of heads 1 and 4 (two heads per group)
        for base in (HP + g * N, HP + G * N + g * N):
            assert np.array_equal(part["conv_state"][..., base:base + N], full["conv_state"][..., base:base + N])
    assert np.isnan(part["conv_state"][..., HP + N:HP + 2 * N]).all()


SSD_PINS = [pin_ssd_matrix_form, pin_ssd_chunked_state_passing, pin_ssd_state_caching,
            pin_ssd_reduces_to_mamba1, pin_ssd_heads_subset]

MIXER_PINS = [pin_brute_force, pin_brute_force_bf16, pin_short_sequence, pin_prefix_sum_A_zero,
              pin_geometric_series, pin_C_zero_skip_gate, pin_softplus_ln2, pin_dt_bias_is_softplus_inverse,
              pin_state_caching,
              pin_decode_matches_brute, pin_split_invariance]
SCAN_PINS = [pin_scan_sequential, pin_scan_chunked]
Q8_PINS = [pin_q8_hand_cases, pin_q8_bounds, pin_q8_split_hand_cases, pin_q8_split_composes_to_reduce,
           pin_q8_split_round_trip]
OUT_PROJ_PINS = [pin_out_proj_vs_matmul, pin_out_proj_identity_and_rank_one]
ALL_PINS = MIXER_PINS + SCAN_PINS + Q8_PINS + OUT_PROJ_PINS + SSD_PINS
