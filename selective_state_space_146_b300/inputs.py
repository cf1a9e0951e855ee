"""Seeded synthetic inputs shaped like the layers the Mamba pages describe.

This module holds the workload table and the random-input recipes only: it
draws numbers and lays them out, and computes none of the scan itself.  The
CUDA path and the fp64 oracle both take their inputs from here.

Recipe (every workload):
  * one CPU ``torch.Generator`` per tensor, seeded ``seed * 1000 + k`` with a
    fixed tensor index k (u=0, delta=1, z=2, B=3, C=4, D=5, dt=6, A=7, x=8,
    dt0=9, dout=10);
  * normal draws are float32, then rounded to bfloat16 (round to nearest
    even) for bfloat16 workloads; the oracle reads the rounded values;
  * selective scan: u, z, B, C ~ N(0, 1); delta_raw ~ N(0, 0.1^2); B, C
    either shared per batch row or one per group of channels (same draws,
    one more dimension);
    A[d, n] = -(n + 1) (S4D-real); D ~ N(0, 1);
    delta_bias[d] = log(expm1(dt_d)) so that softplus(delta_bias) = dt_d, with
    dt_d log-uniform in [dt_min, dt_max];
  * backward: the incoming gradient dout of y ~ N(0, 1), shaped like y;
  * SSD: x, B, C ~ N(0, 1); A_h = -exp(U[log 1, log 16]); D_h ~ N(0, 1);
    dt = softplus(N(0, 0.1^2) + log(expm1(dt0_h))), dt0_h log-uniform in
    [1e-3, 1e-1], computed in float64 and then rounded to the input dtype
    (the SSD entry point takes an already positive dt).

No dataset is read: these tensors stand in for the activations of the
language-model layers named on the pages (Mamba-130M, Mamba-2.8B, Mamba-2).
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch

_IDX = dict(u=0, delta=1, z=2, B=3, C=4, D=5, dt=6, A=7, x=8, dt0=9, dout=10)


@dataclass(frozen=True)
class SelectiveConfig:
    name: str
    batch: int
    d_inner: int
    d_state: int
    seqlen: int
    dtype: str  # "f32" or "bf16"
    gate: bool = True
    skip: bool = True
    bias: bool = True
    softplus: bool = True
    dt_min: float = 1e-3
    dt_max: float = 1e-1
    last_state: bool = True

    @property
    def channel_steps(self) -> int:
        return self.batch * self.d_inner * self.seqlen


@dataclass(frozen=True)
class SSDConfig:
    name: str
    batch: int
    seqlen: int
    nheads: int
    headdim: int
    d_state: int
    ngroups: int
    chunk: int
    dtype: str
    skip: bool = True
    last_state: bool = True

    @property
    def channel_steps(self) -> int:
        return self.batch * self.seqlen * self.nheads * self.headdim


# The five workloads: a tiny fp32 case, two Mamba-1 layer shapes, a long
# context case and a Mamba-2 SSD layer.
WORKLOADS = {
    "tiny_f32": SelectiveConfig("tiny_f32", 1, 64, 16, 256, "f32"),
    "mamba130m_layer": SelectiveConfig("mamba130m_layer", 8, 1536, 16, 2048, "bf16"),
    "mamba2p8b_layer": SelectiveConfig("mamba2p8b_layer", 4, 5120, 16, 8192, "bf16"),
    "long_context": SelectiveConfig("long_context", 1, 2048, 16, 262144, "bf16", gate=False,
                                    dt_min=1e-4, dt_max=1e-1),
    "mamba2_ssd": SSDConfig("mamba2_ssd", 4, 8192, 64, 64, 128, 1, 256, "bf16"),
}


_DEVICE = "cpu"  # where the generators draw; see on_device()


def _gen(seed: int, k: str) -> torch.Generator:
    return torch.Generator(device=_DEVICE).manual_seed(seed * 1000 + _IDX[k])


class on_device:
    """Draw with generators on another device (e.g. "cuda") inside this block.

    The recipe is the same; the values differ from the CPU draws, so this is
    for timing runs only -- parity tests use the CPU draws the oracle reads.
    """

    def __init__(self, device):
        self.device = str(device)

    def __enter__(self):
        global _DEVICE
        self._old, _DEVICE = _DEVICE, self.device
        return self

    def __exit__(self, *exc):
        global _DEVICE
        _DEVICE = self._old


def _tdtype(dtype: str):
    return {"f32": torch.float32, "bf16": torch.bfloat16}[dtype]


def _normal(shape, seed, k, std=1.0):
    t = torch.randn(*shape, generator=_gen(seed, k), dtype=torch.float32, device=_DEVICE)
    if std != 1.0:
        t.mul_(std)
    return t


def _log_uniform(n, lo, hi, seed, k):
    r = torch.rand(n, generator=_gen(seed, k), dtype=torch.float64, device=_DEVICE)
    return torch.exp(math.log(lo) + r * (math.log(hi) - math.log(lo)))


def selective_inputs(batch, d_inner, d_state, seqlen, dtype="bf16", *, gate=True, skip=True,
                     bias=True, dt_min=1e-3, dt_max=1e-1, groups=None, seed=0):
    """Inputs of one selective-scan call, as CPU tensors.

    Returns a dict with u, delta (raw, before bias and softplus), z, A, B, C,
    D, delta_bias; z / D / delta_bias are None when switched off.
    Layouts: u, delta, z (batch, d_inner, seqlen); A (d_inner, d_state) f32;
    B, C (batch, d_state, seqlen), or (batch, groups, d_state, seqlen) when
    `groups` is given (one B, C per group of d_inner / groups channels);
    D, delta_bias (d_inner,) f32.
    """
    td = _tdtype(dtype)
    shp = (batch, d_inner, seqlen)
    bc = (batch, d_state, seqlen) if groups is None else (batch, groups, d_state, seqlen)
    out = {
        "u": _normal(shp, seed, "u").to(td),
        "delta": _normal(shp, seed, "delta", 0.1).to(td),
        "z": _normal(shp, seed, "z").to(td) if gate else None,
        "B": _normal(bc, seed, "B").to(td),
        "C": _normal(bc, seed, "C").to(td),
        "D": _normal((d_inner,), seed, "D") if skip else None,
        "A": -(torch.arange(d_state, dtype=torch.float32, device=_DEVICE) + 1.0)
        .expand(d_inner, d_state).contiguous(),
    }
    if bias:
        dt = _log_uniform(d_inner, dt_min, dt_max, seed, "dt")
        out["delta_bias"] = torch.log(torch.expm1(dt)).to(torch.float32)
    else:
        out["delta_bias"] = None
    return out


def grad_output(shape, dtype="bf16", seed=0):
    """The incoming gradient of a scan's output (stands in for the gradient
    the layers above would send back), as a CPU tensor."""
    return _normal(tuple(shape), seed, "dout").to(_tdtype(dtype))


def workload_selective_inputs(cfg: SelectiveConfig, seed=0):
    return selective_inputs(cfg.batch, cfg.d_inner, cfg.d_state, cfg.seqlen, cfg.dtype,
                            gate=cfg.gate, skip=cfg.skip, bias=cfg.bias, dt_min=cfg.dt_min,
                            dt_max=cfg.dt_max, seed=seed)


def ssd_inputs(batch, seqlen, nheads, headdim, d_state, ngroups=1, dtype="bf16", *, skip=True,
               seed=0):
    """Inputs of one SSD call, as CPU tensors.

    Layouts: x (batch, seqlen, nheads, headdim); dt (batch, seqlen, nheads);
    A_head (nheads,) f32; B, C (batch, seqlen, ngroups, d_state); D (nheads,) f32.
    """
    td = _tdtype(dtype)
    dt0 = _log_uniform(nheads, 1e-3, 1e-1, seed, "dt0")  # per-head target step
    bias = torch.log(torch.expm1(dt0))
    raw = _normal((batch, seqlen, nheads), seed, "dt", 0.1).double() + bias
    dt = torch.nn.functional.softplus(raw)  # the recipe's positive step, fp64
    r = torch.rand(nheads, generator=_gen(seed, "A"), dtype=torch.float64, device=_DEVICE)
    A_head = -torch.exp(r * math.log(16.0))
    return {
        "x": _normal((batch, seqlen, nheads, headdim), seed, "x").to(td),
        "dt": dt.to(torch.float32).to(td),
        "A_head": A_head.to(torch.float32),
        "B": _normal((batch, seqlen, ngroups, d_state), seed, "B").to(td),
        "C": _normal((batch, seqlen, ngroups, d_state), seed, "C").to(td),
        "D": _normal((nheads,), seed, "D") if skip else None,
    }


def workload_ssd_inputs(cfg: SSDConfig, seed=0):
    return ssd_inputs(cfg.batch, cfg.seqlen, cfg.nheads, cfg.headdim, cfg.d_state, cfg.ngroups,
                      cfg.dtype, skip=cfg.skip, seed=seed)


def sample_units(total: int, k: int, seed: int = 0) -> np.ndarray:
    """k distinct unit indices in [0, total), always including the first and last."""
    rng = np.random.default_rng(seed + 12345)
    k = min(k, total)
    pick = set([0, total - 1]) if total > 1 else {0}
    while len(pick) < k:
        pick.add(int(rng.integers(0, total)))
    return np.array(sorted(pick), dtype=np.int64)
