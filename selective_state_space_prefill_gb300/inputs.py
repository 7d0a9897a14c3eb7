"""Seeded synthetic inputs for the selective-SSM mixer.

This module only draws random numbers and lays them out; it holds none of the
mixer's arithmetic, so both the CUDA path and the CPU oracle can be fed from it
without sharing any computation.

Distributions (one recipe for every workload, following the tiny-mixer recipe
that the other workloads reuse):

* x, z, dt ~ N(0, 1), shape [batch, L, d_inner]
* B, C ~ N(0, 1), shape [batch, L, d_state], shared by every channel
* dt_bias[d] = log(expm1(u_d)) with u_d ~ LogUniform[1e-3, 1e-1], so that
  softplus(0 + dt_bias[d]) = u_d (the usual Mamba initialisation of the step size)
* A[d, n] = -(n + 1), D[d] = 1, conv_w ~ U(-0.5, 0.5) [d_inner, d_conv], conv_b = 0
* cached states (decode workloads) ~ N(0, 1) in fp32
* q8 partial buffers ~ N(0, 1)

Draws come from one ``torch.Generator`` seeded with ``seed`` in a fixed order,
on the device given, then cast (round-to-nearest-even) to the input dtype.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

__all__ = [
    "MixerInputs",
    "make_mixer_inputs",
    "make_mixer_params",
    "make_decode_inputs",
    "make_states",
    "make_partials",
    "log_expm1",
    "SSDInputs",
    "make_ssd_inputs",
    "make_ssd_states",
]


def log_expm1(u: torch.Tensor) -> torch.Tensor:
    """log(expm1(u)) evaluated stably in float64 (u + log(-expm1(-u)))."""
    u = u.double()
    return u + torch.log(-torch.expm1(-u))


@dataclass
class MixerInputs:
    """Token inputs [batch, L, ...] plus per-channel parameters."""

    x: torch.Tensor
    z: torch.Tensor
    dt: torch.Tensor
    B: torch.Tensor
    C: torch.Tensor
    A: torch.Tensor
    D: torch.Tensor
    dt_bias: torch.Tensor
    conv_w: torch.Tensor
    conv_b: torch.Tensor

    def to(self, device) -> "MixerInputs":
        return MixerInputs(**{k: getattr(self, k).to(device) for k in self.__dataclass_fields__})

    def token_slice(self, t0: int, t1: int) -> "MixerInputs":
        """Tokens [t0, t1) of every [batch, L, ...] tensor (contiguous copies)."""
        kw = {k: getattr(self, k) for k in self.__dataclass_fields__}
        for k in ("x", "z", "dt", "B", "C"):
            kw[k] = kw[k][:, t0:t1].contiguous()
        return MixerInputs(**kw)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def make_mixer_params(d_inner: int, d_state: int = 16, d_conv: int = 4, seed: int = 0,
                      device="cpu") -> dict:
    """Per-channel parameters A, D, dt_bias, conv_w, conv_b (all fp32)."""
    g = _gen(seed + 7919, device)
    lo, hi = math.log(1e-3), math.log(1e-1)
    u = torch.exp(torch.rand(d_inner, generator=g, device=device, dtype=torch.float64) * (hi - lo) + lo)
    dt_bias = log_expm1(u).float()
    conv_w = (torch.rand(d_inner, d_conv, generator=g, device=device) - 0.5).float().contiguous()
    conv_b = torch.zeros(d_inner, device=device, dtype=torch.float32)
    n = torch.arange(d_state, device=device, dtype=torch.float32)
    A = (-(n + 1.0)).expand(d_inner, d_state).contiguous()
    D = torch.ones(d_inner, device=device, dtype=torch.float32)
    return dict(A=A, D=D, dt_bias=dt_bias, conv_w=conv_w, conv_b=conv_b)


def make_mixer_inputs(batch: int, seqlen: int, d_inner: int, d_state: int = 16, d_conv: int = 4,
                      dtype: torch.dtype = torch.bfloat16, seed: int = 0, device="cpu") -> MixerInputs:
    """Token tensors x, z, dt [batch, L, d_inner] and B, C [batch, L, d_state]."""
    g = _gen(seed, device)

    def normal(*shape):
        return torch.randn(*shape, generator=g, device=device, dtype=torch.float32).to(dtype)

    x = normal(batch, seqlen, d_inner)
    z = normal(batch, seqlen, d_inner)
    dt = normal(batch, seqlen, d_inner)
    B = normal(batch, seqlen, d_state)
    C = normal(batch, seqlen, d_state)
    return MixerInputs(x=x, z=z, dt=dt, B=B, C=C,
                       **make_mixer_params(d_inner, d_state, d_conv, seed, device))


def make_decode_inputs(batch: int, d_inner: int, d_state: int = 16, dtype=torch.bfloat16,
                       seed: int = 0, device="cpu") -> dict:
    """One token per request: x, z, dt [batch, d_inner]; B, C [batch, d_state]."""
    g = _gen(seed + 104729, device)

    def normal(*shape):
        return torch.randn(*shape, generator=g, device=device, dtype=torch.float32).to(dtype)

    return dict(x=normal(batch, d_inner), z=normal(batch, d_inner), dt=normal(batch, d_inner),
                B=normal(batch, d_state), C=normal(batch, d_state))


def make_states(batch: int, d_inner: int, d_state: int = 16, d_conv: int = 4, seed: int = 0,
                device="cpu") -> tuple[torch.Tensor, torch.Tensor]:
    """Cached fp32 states ~ N(0,1): conv_state [batch, d_conv-1, d_inner], ssm_state [batch, d_inner, d_state]."""
    g = _gen(seed + 15485863, device)
    conv_state = torch.randn(batch, d_conv - 1, d_inner, generator=g, device=device, dtype=torch.float32)
    ssm_state = torch.randn(batch, d_inner, d_state, generator=g, device=device, dtype=torch.float32)
    return conv_state, ssm_state


def make_partials(P: int, shape, dtype=torch.bfloat16, seed: int = 0, device="cpu") -> list[torch.Tensor]:
    """P partial-output buffers of the given shape, ~ N(0, 1)."""
    g = _gen(seed + 32452843, device)
    return [torch.randn(*shape, generator=g, device=device, dtype=torch.float32).to(dtype)
            for _ in range(P)]


def make_out_proj_inputs(M: int, K: int, N: int, dtype=torch.bfloat16, seed: int = 0,
                         device="cpu") -> tuple[torch.Tensor, torch.Tensor]:
    """One rank's out_proj operands: the mixer output of its channel slice y [M, K] ~ N(0, 1)
    and the matching weight columns W [N, K] ~ N(0, 1/K) (the usual fan-in scale)."""
    g = _gen(seed + 15485863, device)
    y = torch.randn(M, K, generator=g, device=device, dtype=torch.float32).to(dtype)
    W = (torch.randn(N, K, generator=g, device=device, dtype=torch.float32) / K ** 0.5).to(dtype)
    return y, W


@dataclass
class SSDInputs:
    """Inputs of the SSD (Mamba-2-style) mixer.

    xBC [batch, L, H*P + 2*G*N] holds the pre-conv channels x (head-major), then B and C
    of each group; z [batch, L, H*P]; dt [batch, L, H]; per-head A, D, dt_bias [H];
    per-channel conv_w [Cx, d_conv] and conv_b [Cx].
    """

    xBC: torch.Tensor
    z: torch.Tensor
    dt: torch.Tensor
    A: torch.Tensor
    D: torch.Tensor
    dt_bias: torch.Tensor
    conv_w: torch.Tensor
    conv_b: torch.Tensor
    n_heads: int
    head_dim: int
    n_groups: int
    d_state: int

    _TENSORS = ("xBC", "z", "dt", "A", "D", "dt_bias", "conv_w", "conv_b")
    _TOKENS = ("xBC", "z", "dt")

    def _kw(self):
        return {k: getattr(self, k) for k in self.__dataclass_fields__}

    def to(self, device) -> "SSDInputs":
        kw = self._kw()
        for k in self._TENSORS:
            kw[k] = kw[k].to(device)
        return SSDInputs(**kw)

    def token_slice(self, t0: int, t1: int) -> "SSDInputs":
        kw = self._kw()
        for k in self._TOKENS:
            kw[k] = kw[k][:, t0:t1].contiguous()
        return SSDInputs(**kw)

    @property
    def channels(self) -> int:
        return self.n_heads * self.head_dim + 2 * self.n_groups * self.d_state


def make_ssd_inputs(batch: int, seqlen: int, n_heads: int, head_dim: int = 64, n_groups: int = 1,
                    d_state: int = 64, d_conv: int = 4, dtype: torch.dtype = torch.bfloat16,
                    seed: int = 0, device="cpu") -> SSDInputs:
    """Seeded SSD inputs: xBC, z, dt ~ N(0, 1); dt_bias = log(expm1(u_h)) with u_h ~
    LogUniform[1e-3, 1e-1] per head; A[h] = -U[1, 16] (the usual Mamba-2 initialisation of
    A = -exp(A_log)); D = 1; conv_w ~ U(-0.5, 0.5); conv_b = 0."""
    g = _gen(seed + 49979687, device)
    HP = n_heads * head_dim
    Cx = HP + 2 * n_groups * d_state

    def normal(*shape):
        return torch.randn(*shape, generator=g, device=device, dtype=torch.float32).to(dtype)

    xBC = normal(batch, seqlen, Cx)
    z = normal(batch, seqlen, HP)
    dt = normal(batch, seqlen, n_heads)
    lo, hi = math.log(1e-3), math.log(1e-1)
    u = torch.exp(torch.rand(n_heads, generator=g, device=device, dtype=torch.float64) * (hi - lo) + lo)
    dt_bias = log_expm1(u).float()
    A = -(1.0 + 15.0 * torch.rand(n_heads, generator=g, device=device, dtype=torch.float32))
    conv_w = (torch.rand(Cx, d_conv, generator=g, device=device) - 0.5).float().contiguous()
    return SSDInputs(xBC=xBC, z=z, dt=dt, A=A.contiguous(),
                     D=torch.ones(n_heads, device=device, dtype=torch.float32), dt_bias=dt_bias,
                     conv_w=conv_w, conv_b=torch.zeros(Cx, device=device, dtype=torch.float32),
                     n_heads=n_heads, head_dim=head_dim, n_groups=n_groups, d_state=d_state)


def make_ssd_states(batch: int, n_heads: int, head_dim: int, d_state: int, channels: int,
                    d_conv: int = 4, seed: int = 0, device="cpu") -> tuple[torch.Tensor, torch.Tensor]:
    """Cached fp32 SSD states ~ N(0, 1): conv_state [batch, d_conv-1, channels] and
    ssm_state [batch, n_heads, head_dim, d_state]."""
    g = _gen(seed + 67867967, device)
    conv_state = torch.randn(batch, d_conv - 1, channels, generator=g, device=device, dtype=torch.float32)
    ssm_state = torch.randn(batch, n_heads, head_dim, d_state, generator=g, device=device, dtype=torch.float32)
    return conv_state, ssm_state
