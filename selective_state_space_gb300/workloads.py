"""Seeded synthetic workloads for the SSD forward pass.

This module only draws random inputs; it holds none of the method's
arithmetic.  Both the GPU path and the CPU oracle consume the tensors it
returns, so both sides see exactly the same (already rounded) values.

Shapes follow the benchmark shapes of the cuTile Mamba-2 blog (section
"Mamba-2 forward benchmark": ``Mamba2ProblemSpec(batch_size, num_tokens,
num_groups, num_heads, state_size, head_size, chunk_size, dtype,
state_dtype)``) and five named layer shapes used throughout this library.

Draw order for one workload, from a single CPU ``torch.Generator`` seeded
with the workload seed, every draw in float32 and then cast to the input
dtype: x, B, C, dt (or its pre-activation), A, D, h0, the dt-zero mask.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class Shape:
    name: str
    batch: int
    seqlen: int
    nheads: int
    headdim: int       # H, the per-head value width (x, y)
    dstate: int        # S, the state width (B, C)
    ngroups: int
    chunk: int
    dtype: str         # "f32" or "bf16": dtype of x, dt, B, C and y
    dt_recipe: str     # "loguniform" (exp(U(log 1e-3, log 1e-1))) or "softplus" (softplus(N(-4, 1)))
    a_range: tuple     # A = -U(lo, hi)
    d_recipe: str      # "one" or "normal" (N(1, 0.1))
    h0_recipe: str     # "zeros", "none" or "normal" (N(0, 0.1), float32)
    dt_zero_frac: float
    seed: int

    @property
    def nchunks(self) -> int:
        return (self.seqlen + self.chunk - 1) // self.chunk

    @property
    def tokens(self) -> int:
        return self.batch * self.seqlen


# The five layer shapes, in order, plus the blog's own benchmark shape.
WORKLOADS = [
    Shape("tiny-f32", 1, 256, 4, 64, 64, 1, 64, "f32", "loguniform", (1.0, 16.0), "one", "zeros", 0.0, 0),
    Shape("mamba2-130m-layer", 2, 2048, 24, 64, 128, 1, 256, "bf16", "softplus", (1.0, 16.0), "normal", "none", 0.0, 1),
    Shape("mamba2-2.7b-layer", 4, 4096, 80, 64, 128, 1, 256, "bf16", "softplus", (1.0, 16.0), "normal", "normal", 0.0, 2),
    Shape("long-prefill-64k", 1, 65536, 32, 64, 128, 8, 256, "bf16", "softplus", (1.0, 16.0), "normal", "none", 0.05, 3),
    Shape("wide-state-batched", 32, 1024, 64, 128, 256, 4, 128, "bf16", "loguniform", (0.5, 8.0), "normal", "none", 0.0, 4),
]
BLOG_SHAPE = Shape("blog-b4-l16k", 4, 16384, 8, 64, 128, 1, 128, "bf16", "softplus", (1.0, 16.0), "normal", "none", 0.0, 5)


def by_name(name: str) -> Shape:
    for s in WORKLOADS + [BLOG_SHAPE]:
        if s.name == name:
            return s
    raise KeyError(name)


def custom(batch, seqlen, nheads, headdim, dstate, ngroups, chunk, dtype="bf16", *,
           dt_recipe="softplus", a_range=(1.0, 16.0), d_recipe="normal", h0_recipe="none",
           dt_zero_frac=0.0, seed=0, name="custom") -> Shape:
    return Shape(name, batch, seqlen, nheads, headdim, dstate, ngroups, chunk, dtype, dt_recipe,
                 tuple(a_range), d_recipe, h0_recipe, dt_zero_frac, seed)


def torch_dtype(d: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[d]


@dataclasses.dataclass
class Inputs:
    shape: Shape
    x: torch.Tensor            # [B, L, nh, H]      input dtype
    dt: torch.Tensor           # [B, L, nh]         input dtype
    A: torch.Tensor            # [nh]               float32 (all negative)
    B: torch.Tensor            # [B, L, G, S]       input dtype
    C: torch.Tensor            # [B, L, G, S]       input dtype
    D: torch.Tensor            # [nh]               float32
    h0: Optional[torch.Tensor]  # [B, nh, H, S]     float32 or None

    def tensors(self):
        return dict(x=self.x, dt=self.dt, A=self.A, B=self.B, C=self.C, D=self.D, h0=self.h0)


def make_inputs(shape: Shape, seed: Optional[int] = None, dt_dtype: Optional[str] = None) -> Inputs:
    """Draw one workload on the CPU (deterministic for a given seed).  dt_dtype ("f32" or
    "bf16") overrides the dtype dt is cast to (by default the shape's input dtype)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(shape.seed if seed is None else seed)
    Bsz, L, nh, H, S, G = shape.batch, shape.seqlen, shape.nheads, shape.headdim, shape.dstate, shape.ngroups
    dt_ = torch_dtype(shape.dtype)
    f32 = torch.float32
    x = torch.randn((Bsz, L, nh, H), generator=g, dtype=f32).to(dt_)
    scale = 1.0 / math.sqrt(S)
    Bm = (torch.randn((Bsz, L, G, S), generator=g, dtype=f32) * scale).to(dt_)
    Cm = (torch.randn((Bsz, L, G, S), generator=g, dtype=f32) * scale).to(dt_)
    if shape.dt_recipe == "loguniform":
        u = torch.rand((Bsz, L, nh), generator=g, dtype=f32)
        lo, hi = math.log(1e-3), math.log(1e-1)
        dt = torch.exp(lo + (hi - lo) * u)
    elif shape.dt_recipe == "softplus":
        dt = torch.nn.functional.softplus(torch.randn((Bsz, L, nh), generator=g, dtype=f32) - 4.0)
    else:
        raise ValueError(shape.dt_recipe)
    lo, hi = shape.a_range
    A = -(lo + (hi - lo) * torch.rand((nh,), generator=g, dtype=f32))
    if shape.d_recipe == "one":
        D = torch.ones((nh,), dtype=f32)
    else:
        D = 1.0 + 0.1 * torch.randn((nh,), generator=g, dtype=f32)
    if shape.h0_recipe == "zeros":
        h0 = torch.zeros((Bsz, nh, H, S), dtype=f32)
    elif shape.h0_recipe == "normal":
        h0 = 0.1 * torch.randn((Bsz, nh, H, S), generator=g, dtype=f32)
    else:
        h0 = None
    if shape.dt_zero_frac > 0.0:
        # exactly round(frac * L) token positions per batch row hold their state (dt = 0 for all heads)
        nz = int(round(shape.dt_zero_frac * L))
        for b in range(Bsz):
            idx = torch.randperm(L, generator=g)[:nz]
            dt[b, idx, :] = 0.0
    dt = dt.to(torch_dtype(dt_dtype) if dt_dtype else dt_)
    return Inputs(shape, x.contiguous(), dt.contiguous(), A.contiguous(), Bm.contiguous(),
                  Cm.contiguous(), D.contiguous(), None if h0 is None else h0.contiguous())


@dataclasses.dataclass
class GradInputs:
    dy: torch.Tensor                  # [B, L, nh, H]   input dtype (the gradient of y)
    dh_final: Optional[torch.Tensor]  # [B, nh, H, S]   float32 (the gradient of h_final) or None


def make_grad_inputs(shape: Shape, with_dh_final: bool = True, seed: Optional[int] = None) -> GradInputs:
    """Upstream gradients for the gradient pass, from their own generator (seed + 1000 by
    default): dy ~ N(0, 1) in the input dtype, then dh_final ~ N(0, 0.1) float32."""
    g = torch.Generator(device="cpu")
    g.manual_seed((shape.seed + 1000) if seed is None else seed)
    Bsz, L, nh, H, S = shape.batch, shape.seqlen, shape.nheads, shape.headdim, shape.dstate
    dy = torch.randn((Bsz, L, nh, H), generator=g, dtype=torch.float32).to(torch_dtype(shape.dtype))
    dhf = 0.1 * torch.randn((Bsz, nh, H, S), generator=g, dtype=torch.float32) if with_dh_final else None
    return GradInputs(dy.contiguous(), None if dhf is None else dhf.contiguous())


# ---- Mamba-1 selective scan (S6) workloads ----

@dataclasses.dataclass(frozen=True)
class S6Shape:
    name: str
    batch: int
    seqlen: int
    dim: int           # channels (d_inner)
    dstate: int        # N
    ngroups: int
    dtype: str         # "f32" or "bf16": x, delta, B, C and y
    recipe: str        # "hardway" (the page's create()) or "mamba1" (see make_s6_inputs)
    skip: bool         # D present
    h0: bool
    seed: int

    @property
    def tokens(self) -> int:
        return self.batch * self.seqlen


S6_WORKLOADS = [
    # the timing run of "Mamba: The Hard Way", Part 5: mamba(*create(S=2048, Ba=8, D=1024, N=4))
    S6Shape("s6-hardway-run", 8, 2048, 1024, 4, 1, "f32", "hardway", False, False, 20),
    # a Mamba-1 130M-shaped layer: d_inner 1536, N = 16
    S6Shape("s6-mamba-130m-layer", 8, 2048, 1536, 16, 1, "bf16", "mamba1", True, False, 21),
]


def s6_by_name(name: str) -> S6Shape:
    for s in S6_WORKLOADS:
        if s.name == name:
            return s
    raise KeyError(name)


def s6_custom(batch, seqlen, dim, dstate, ngroups=1, dtype="f32", recipe="mamba1", skip=True, h0=True, seed=0,
              name="s6-custom") -> S6Shape:
    return S6Shape(name, batch, seqlen, dim, dstate, ngroups, dtype, recipe, skip, h0, seed)


@dataclasses.dataclass
class S6Inputs:
    shape: S6Shape
    x: torch.Tensor               # [B, dim, L]      input dtype
    delta: torch.Tensor           # [B, dim, L]      input dtype (positive)
    A: torch.Tensor               # [dim, N]         float32 (negative)
    B: torch.Tensor               # [B, G, N, L]     input dtype
    C: torch.Tensor               # [B, G, N, L]     input dtype
    D: Optional[torch.Tensor]     # [dim]            float32 or None
    h0: Optional[torch.Tensor]    # [B, dim, N]      float32 or None

    def tensors(self):
        return dict(x=self.x, delta=self.delta, A=self.A, B=self.B, C=self.C, D=self.D, h0=self.h0)


def make_s6_inputs(shape: S6Shape, seed: Optional[int] = None) -> S6Inputs:
    """Draw one selective-scan workload on the CPU, in the order x, delta, A, B, C, D, h0.

    "hardway": the page's create(): x ~ U(0, 1), A = -1, B = 0.1, C ~ 0.1 U(0, 1),
    delta ~ 0.1 U(0, 1).  "mamba1": x ~ N(0, 1), delta = exp(U(log 1e-3, log 1e-1)),
    A[d][n] = -(n + 1) U(0.5, 1.5), B, C ~ N(0, 1), D ~ N(1, 0.1), h0 ~ N(0, 0.1)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(shape.seed if seed is None else seed)
    Bsz, L, dim, N, G = shape.batch, shape.seqlen, shape.dim, shape.dstate, shape.ngroups
    f32, dt_ = torch.float32, torch_dtype(shape.dtype)
    if shape.recipe == "hardway":
        x = torch.rand((Bsz, dim, L), generator=g, dtype=f32)
        delta = 0.1 * torch.rand((Bsz, dim, L), generator=g, dtype=f32)
        A = -torch.ones((dim, N), dtype=f32)
        Bm = torch.full((Bsz, G, N, L), 0.1, dtype=f32)
        Cm = 0.1 * torch.rand((Bsz, G, N, L), generator=g, dtype=f32)
    elif shape.recipe == "mamba1":
        x = torch.randn((Bsz, dim, L), generator=g, dtype=f32)
        lo, hi = math.log(1e-3), math.log(1e-1)
        delta = torch.exp(lo + (hi - lo) * torch.rand((Bsz, dim, L), generator=g, dtype=f32))
        A = -(torch.arange(1, N + 1, dtype=f32)[None, :] * (0.5 + torch.rand((dim, N), generator=g, dtype=f32)))
        Bm = torch.randn((Bsz, G, N, L), generator=g, dtype=f32)
        Cm = torch.randn((Bsz, G, N, L), generator=g, dtype=f32)
    else:
        raise ValueError(shape.recipe)
    D = (1.0 + 0.1 * torch.randn((dim,), generator=g, dtype=f32)) if shape.skip else None
    h0 = 0.1 * torch.randn((Bsz, dim, N), generator=g, dtype=f32) if shape.h0 else None
    return S6Inputs(shape, x.to(dt_).contiguous(), delta.to(dt_).contiguous(), A.contiguous(),
                    Bm.to(dt_).contiguous(), Cm.to(dt_).contiguous(), D, h0)
