"""Shared helpers for the GPU parity tests (CUDA path through the C ABI vs the fp64 oracle)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from selective_state_space_prefill_gb300 import binding as ssm
from selective_state_space_prefill_gb300.inputs import MixerInputs

# Tolerances.  bf16 token inputs (fp32 state): max |gpu - oracle| <= 2e-3 * RMS(oracle) per
# output tensor.  All-fp32 inputs: |gpu - oracle| <= 1e-5 * max(|oracle|, RMS(oracle)) per element.
TOL_BF16 = 2e-3
TOL_F32 = 1e-5


def tol_for(dtype) -> float:
    return TOL_BF16 if dtype == torch.bfloat16 else TOL_F32


def assert_rms_close(got, ref, tol, what="", extra=None):
    got = np.asarray(got.detach().cpu().double().numpy() if isinstance(got, torch.Tensor) else got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, f"{what}: shape {got.shape} vs {ref.shape}"
    err = np.abs(got - ref)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    bound = tol * rms + (0.0 if extra is None else extra)
    worst = float(np.max(err - bound)) if np.ndim(bound) else float(np.max(err)) - bound
    assert worst <= 0.0, f"{what}: max|err| {float(np.max(err)):.3e} vs tol {tol:g} * rms {rms:.3e}"
    return float(np.max(err)) / max(rms, 1e-300)


def assert_rel_close(got, ref, tol, what=""):
    """Per-element relative error with an RMS floor: |err_i| <= tol * max(|ref_i|, RMS(ref)).
    The reading of "1e-5 relative" for all-fp32 inputs: relative error of each element, and
    near a zero crossing (where relative error has no meaning) the tensor's RMS instead."""
    got = np.asarray(got.detach().cpu().double().numpy() if isinstance(got, torch.Tensor) else got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, f"{what}: shape {got.shape} vs {ref.shape}"
    rms = float(np.sqrt(np.mean(ref ** 2)))
    scale = np.maximum(np.abs(ref), rms)
    rel = np.abs(got - ref) / np.maximum(scale, 1e-300)
    k = int(np.argmax(rel))
    assert rel.flat[k] <= tol, (f"{what}: error {float(np.abs(got - ref).flat[k]):.3e} at |ref| "
                                f"{float(np.abs(ref).flat[k]):.3e} (rms {rms:.3e}) is {float(rel.flat[k]):.3e} > {tol:g}")
    return float(rel.flat[k])


def assert_parity(got, ref, dtype, what=""):
    """The parity bar by input precision: bf16 inputs max|err| <= 2e-3 * RMS; fp32 inputs
    relative error <= 1e-5 per element with an RMS floor."""
    if dtype == torch.bfloat16:
        return assert_rms_close(got, ref, TOL_BF16, what)
    return assert_rel_close(got, ref, TOL_F32, what)


def half_ulp_bf16(ref):
    """Half a bfloat16 ulp of |ref| (the rounding a bf16 output adds)."""
    a = np.abs(np.asarray(ref, np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return 0.5 * 2.0 ** (e - 7)


def run_prefill(inp: MixerInputs, cs=None, ss=None, out_dtype=torch.float32):
    return ssm.prefill(inp.x, inp.z, inp.dt, inp.B, inp.C, inp.A, inp.D, inp.dt_bias, inp.conv_w,
                       inp.conv_b, conv_state_in=cs, ssm_state_in=ss, out_dtype=out_dtype)


def cpu_channels(inp: MixerInputs, idx) -> MixerInputs:
    """The given channels of (possibly device-resident) inputs, gathered then moved to the CPU."""
    ix = torch.as_tensor(idx, device=inp.x.device, dtype=torch.long)
    kw = {}
    for k in ("x", "z", "dt"):
        kw[k] = getattr(inp, k).index_select(2, ix).cpu().contiguous()
    for k in ("B", "C"):
        kw[k] = getattr(inp, k).cpu().contiguous()
    for k in ("A", "D", "dt_bias", "conv_w", "conv_b"):
        kw[k] = getattr(inp, k).index_select(0, ix).cpu().contiguous()
    return MixerInputs(**kw)


def oracle_prefill(inp: MixerInputs, cs=None, ss=None, threads=None):
    """Oracle on CPU copies of `inp`; states are CPU float64 (or fp32 widened)."""
    return oracle.prefill(inp.x, inp.z, inp.dt, inp.B, inp.C, inp.A, inp.D, inp.dt_bias, inp.conv_w,
                          inp.conv_b, conv_state_in=cs, ssm_state_in=ss, n_threads=threads)


def sample_channels(d_inner: int, k: int, seed: int = 0) -> np.ndarray:
    """k channels spread over [0, d_inner): both ends, every 32-channel group edge kind, random rest."""
    rng = np.random.default_rng(seed)
    fixed = [0, 1, 31, 32, d_inner - 1, d_inner - 32, d_inner // 2]
    rest = rng.choice(d_inner, size=max(0, k - len(fixed)), replace=False)
    return np.unique(np.clip(np.concatenate([fixed, rest]), 0, d_inner - 1))
