"""Seeded synthetic inputs for the low-rank bottleneck sublayer.

This module only draws random numbers and shapes them. It holds none of the
method's arithmetic, so both the CUDA path and the fp64 oracle can consume its
arrays without sharing any computation.

Recipe (the pages train LLaMA-2-family models on an unnamed corpus; no dataset
or trained weights are available, so seeded synthetic tensors of the same
shapes stand in for them):

* activations ``x`` and upstream gradients ``G`` ~ N(0, 1);
* RMSNorm gain ``g`` = 1 + N(0, 0.1) (0.1 is the standard deviation);
* each low-rank pair: ``A`` [r, d_in] ~ N(0, 1/d_in), ``B`` [d_out, r] ~ N(0, 1/r)
  (N(0, 1/fan_in) for both factors);
* draws are fp32 from one ``torch.Generator`` per case, in a fixed order (x, g,
  then each pair's A and B, then gradients / targets), and are then rounded once
  to the case's storage dtype.  Both sides read the rounded values; the oracle
  widens them exactly to fp64.  Parity cases draw on the CPU; timing-only
  workloads may draw on the GPU (``device=``), which gives other values of the
  same distribution.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional

import torch

__all__ = [
    "MlpShape",
    "ProjShape",
    "make_mlp_case",
    "make_proj_case",
    "make_stack_case",
    "MLP_TINY_F32",
    "MLP_BLOCK_BF16",
    "ATTN_PROJ_BF16",
    "STACK_BF16",
    "sweep_shapes",
    "EXTREMES",
    "make_extreme_mlp_case",
    "make_extreme_proj_case",
]


@dataclasses.dataclass(frozen=True)
class MlpShape:
    """One low-rank SwiGLU MLP block: tokens T, model width d, MLP width f, rank r."""

    T: int
    d: int
    f: int
    r: int
    dtype: str = "bf16"  # "bf16" or "f32"
    eps: float = 1e-6


@dataclasses.dataclass(frozen=True)
class ProjShape:
    """A group of ``group`` low-rank pairs that read the same input [T, d_in]."""

    T: int
    d_in: int
    d_out: int
    r: int
    group: int
    norm: bool = True
    dtype: str = "bf16"
    eps: float = 1e-6


# Workloads named by what they are.
MLP_TINY_F32 = MlpShape(T=2 * 64, d=256, f=688, r=64, dtype="f32")
MLP_BLOCK_BF16 = MlpShape(T=8 * 2048, d=2048, f=5632, r=512, dtype="bf16")
ATTN_PROJ_BF16 = ProjShape(T=4 * 4096, d_in=4096, d_out=4096, r=1024, group=3, norm=True)
ATTN_OPROJ_BF16 = ProjShape(T=4 * 4096, d_in=4096, d_out=4096, r=1024, group=1, norm=False)
STACK_BF16 = dict(blocks=24, shape=MLP_BLOCK_BF16)


def sweep_shapes() -> List[ProjShape]:
    """The 144-shape grouped GEMM-pair sweep: d x r x T x group size (no norm, d_out = d)."""
    out = []
    for d in (2048, 4096, 5120, 8192):
        for r in (d // 8, d // 4, d // 2):
            for T in (2048, 8192, 32768, 65536):
                for gs in (1, 2, 3):
                    out.append(ProjShape(T=T, d_in=d, d_out=d, r=r, group=gs, norm=False))
    return out


def _torch_dtype(name: str) -> torch.dtype:
    if name == "bf16":
        return torch.bfloat16
    if name == "f32":
        return torch.float32
    raise ValueError(f"unknown dtype {name!r}")


def _normal(gen: torch.Generator, shape, std: float, mean: float = 0.0) -> torch.Tensor:
    t = torch.randn(*shape, generator=gen, dtype=torch.float32, device=gen.device)
    if std != 1.0:
        t = t * std
    if mean != 0.0:
        t = t + mean
    return t


def _pair(gen: torch.Generator, r: int, d_in: int, d_out: int, dt: torch.dtype):
    A = _normal(gen, (r, d_in), d_in ** -0.5).to(dt)
    B = _normal(gen, (d_out, r), r ** -0.5).to(dt)
    return A, B


def make_mlp_case(shape: MlpShape, seed: int = 0, with_grad: bool = True, device: str = "cpu") -> Dict[str, torch.Tensor]:
    """Host tensors for one MLP block: x, g, A/B of gate, up, down, and upstream grad G."""
    dt = _torch_dtype(shape.dtype)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    c: Dict[str, torch.Tensor] = {}
    c["x"] = _normal(gen, (shape.T, shape.d), 1.0).to(dt)
    c["g"] = _normal(gen, (shape.d,), 0.1, mean=1.0).to(dt)
    c["A_gate"], c["B_gate"] = _pair(gen, shape.r, shape.d, shape.f, dt)
    c["A_up"], c["B_up"] = _pair(gen, shape.r, shape.d, shape.f, dt)
    c["A_down"], c["B_down"] = _pair(gen, shape.r, shape.f, shape.d, dt)
    if with_grad:
        c["G"] = _normal(gen, (shape.T, shape.d), 1.0).to(dt)
    return c


@dataclasses.dataclass(frozen=True)
class BlockShape:
    """One low-rank transformer block: b sequences of s tokens, H heads of dh (d = H*dh),
    attention rank ra, MLP width f and rank rm; bf16."""
    b: int
    s: int
    H: int
    dh: int
    f: int
    ra: int
    rm: int
    eps: float = 1e-6

    @property
    def T(self) -> int:
        return self.b * self.s

    @property
    def d(self) -> int:
        return self.H * self.dh


# LLaMA-7B-class widths (d 4096, f 11008) on 8 x 2048 tokens, ranks d/4.
BLOCK_7B = BlockShape(b=8, s=2048, H=32, dh=128, f=11008, ra=1024, rm=1024)


def make_block_case(shape: BlockShape, seed: int = 0, device: str = "cpu") -> Dict[str, torch.Tensor]:
    """Host tensors for one transformer block (bf16): x, g_attn, A/B of q, k, v, o, g_mlp,
    A/B of gate, up, down, and the upstream grad G."""
    dt = torch.bfloat16
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    d = shape.d
    c: Dict[str, torch.Tensor] = {}
    c["x"] = _normal(gen, (shape.T, d), 1.0).to(dt)
    c["g_attn"] = _normal(gen, (d,), 0.1, mean=1.0).to(dt)
    for n in "qkvo":
        c[f"A_{n}"], c[f"B_{n}"] = _pair(gen, shape.ra, d, d, dt)
    c["g_mlp"] = _normal(gen, (d,), 0.1, mean=1.0).to(dt)
    c["A_gate"], c["B_gate"] = _pair(gen, shape.rm, d, shape.f, dt)
    c["A_up"], c["B_up"] = _pair(gen, shape.rm, d, shape.f, dt)
    c["A_down"], c["B_down"] = _pair(gen, shape.rm, shape.f, d, dt)
    c["G"] = _normal(gen, (shape.T, d), 1.0).to(dt)
    return c


def make_dense_case(shape: MlpShape, seed: int = 0, with_grad: bool = True, device: str = "cpu") -> Dict[str, torch.Tensor]:
    """Host tensors for the dense (full-rank) MLP block of the same d, f: x, g, W_gate, W_up [f, d],
    W_down [d, f] (N(0, 1/fan_in)) and upstream grad G.  shape.r is not used."""
    dt = _torch_dtype(shape.dtype)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    c: Dict[str, torch.Tensor] = {}
    c["x"] = _normal(gen, (shape.T, shape.d), 1.0).to(dt)
    c["g"] = _normal(gen, (shape.d,), 0.1, mean=1.0).to(dt)
    c["W_gate"] = _normal(gen, (shape.f, shape.d), shape.d ** -0.5).to(dt)
    c["W_up"] = _normal(gen, (shape.f, shape.d), shape.d ** -0.5).to(dt)
    c["W_down"] = _normal(gen, (shape.d, shape.f), shape.f ** -0.5).to(dt)
    if with_grad:
        c["G"] = _normal(gen, (shape.T, shape.d), 1.0).to(dt)
    return c


def make_proj_case(shape: ProjShape, seed: int = 0, with_grad: bool = True, device: str = "cpu") -> Dict[str, object]:
    """Host tensors for a projection group: x, optional g, pairs, and one upstream grad per pair."""
    dt = _torch_dtype(shape.dtype)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    c: Dict[str, object] = {}
    c["x"] = _normal(gen, (shape.T, shape.d_in), 1.0).to(dt)
    c["g"] = _normal(gen, (shape.d_in,), 0.1, mean=1.0).to(dt) if shape.norm else None
    As, Bs = [], []
    for _ in range(shape.group):
        A, B = _pair(gen, shape.r, shape.d_in, shape.d_out, dt)
        As.append(A)
        Bs.append(B)
    c["A"], c["B"] = As, Bs
    if with_grad:
        c["G"] = [_normal(gen, (shape.T, shape.d_out), 1.0).to(dt) for _ in range(shape.group)]
    return c


def make_stack_case(shape: MlpShape, blocks: int, seed: int = 0, device: str = "cpu") -> Dict[str, object]:
    """Host tensors for a residual stack of MLP blocks trained against an MSE target."""
    dt = _torch_dtype(shape.dtype)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    c: Dict[str, object] = {}
    c["x"] = _normal(gen, (shape.T, shape.d), 1.0).to(dt)
    layers = []
    for _ in range(blocks):
        L = {"g": _normal(gen, (shape.d,), 0.1, mean=1.0).to(dt)}
        L["A_gate"], L["B_gate"] = _pair(gen, shape.r, shape.d, shape.f, dt)
        L["A_up"], L["B_up"] = _pair(gen, shape.r, shape.d, shape.f, dt)
        L["A_down"], L["B_down"] = _pair(gen, shape.r, shape.f, shape.d, dt)
        layers.append(L)
    c["blocks"] = layers
    c["target"] = _normal(gen, (shape.T, shape.d), 1.0).to(dt)
    return c


def sample_rows(T: int, n: int, seed: int = 1) -> torch.Tensor:
    """A sorted, seeded sample of ``n`` distinct row indices in [0, T) that always holds 0 and T-1."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    if n >= T:
        return torch.arange(T)
    idx = torch.randperm(T, generator=gen)[: n - 2]
    idx = torch.cat([idx, torch.tensor([0, T - 1])]).unique()
    return idx.sort().values


# Inputs at the edges of the arithmetic (same draws as the plain cases, then reshaped):
#   "saturated": the A factors that read the input (gate and up of a block, every A of a group)
#                scaled by 30 and their B factors by 1/30, so their pre-activations u reach
#                |u| ~ 30-130 in both signs (SiLU and SiLU' saturated, e^-u past the fp32 range)
#                while what follows the pair keeps its usual scale.  The scaled pairs are those
#                whose u is computed from the stored input itself: a pre-activation of large
#                scale computed from rounded intermediates carries an absolute error of that
#                scale times the storage precision, which SiLU' (slope 1/2 at 0) turns into
#                relative errors of several percent near u = 0 for any bf16-storing path;
#   "zero_rows": rows 0 and the last of x set to 0 (1/rms = eps^-1/2 = 1000 on a zero row) and row 5
#                scaled by 1e-3 (mean square ~ eps: the eps term decides 1/rms);
#   "big_rows":  rows 1 and 6 of x scaled by 1e3 (sums of squares ~1e9 next to rows of ~1).
EXTREMES = ("saturated", "zero_rows", "big_rows")
_SAT_SCALE = 30.0
_BIG = 1e3


def _reshape_x(x: torch.Tensor, kind: str) -> torch.Tensor:
    x = x.clone()
    T = x.shape[0]
    if kind == "zero_rows":
        tiny = min(5, T - 1)
        x[tiny] = (x[tiny].float() * 1e-3).to(x.dtype)
        x[[0, T - 1]] = 0
    elif kind == "big_rows":
        rows = sorted({min(1, T - 1), min(6, T - 1)})
        x[rows] = (x[rows].float() * _BIG).to(x.dtype)
    return x


def make_extreme_mlp_case(shape: MlpShape, kind: str, seed: int = 0) -> Dict[str, torch.Tensor]:
    """make_mlp_case(shape, seed) reshaped to one of EXTREMES (host tensors, rounded to the dtype)."""
    if kind not in EXTREMES:
        raise ValueError(kind)
    c = make_mlp_case(shape, seed)
    if kind == "saturated":
        for k in ("gate", "up"):
            c["A_" + k] = (c["A_" + k].float() * _SAT_SCALE).to(c["A_" + k].dtype)
            c["B_" + k] = (c["B_" + k].float() / _SAT_SCALE).to(c["B_" + k].dtype)
    else:
        c["x"] = _reshape_x(c["x"], kind)
    return c


def make_extreme_proj_case(shape: ProjShape, kind: str, seed: int = 0) -> Dict[str, object]:
    """make_proj_case(shape, seed) reshaped to one of EXTREMES."""
    if kind not in EXTREMES:
        raise ValueError(kind)
    c = make_proj_case(shape, seed)
    if kind == "saturated":
        c["A"] = [(A.float() * _SAT_SCALE).to(A.dtype) for A in c["A"]]
        c["B"] = [(B.float() / _SAT_SCALE).to(B.dtype) for B in c["B"]]
    else:
        c["x"] = _reshape_x(c["x"], kind)
    return c
