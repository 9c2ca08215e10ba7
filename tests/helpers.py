"""Shared test helpers: device transfer, error metric, oracle on sampled (batch, head) pairs."""
from __future__ import annotations

import numpy as np
import torch

import oracle

# Acceptance bounds on max|got - ref| / max|ref| (y and h_final):
# float32 inputs (TF32 tensor-core arithmetic allowed) and bfloat16 inputs with float32 accumulation.
TOL = {"f32": 1e-3, "bf16": 2e-2}


def rel_max_err(got, ref) -> float:
    got = got.detach().double().cpu().numpy() if torch.is_tensor(got) else np.asarray(got, dtype=np.float64)
    ref = ref.detach().double().cpu().numpy() if torch.is_tensor(ref) else np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    if ref.size == 0:
        return 0.0
    denom = float(np.max(np.abs(ref)))
    assert np.all(np.isfinite(got)), "non-finite values in the GPU result"
    return float(np.max(np.abs(got - ref))) / max(denom, 1e-30)


def to_dev(inp, device="cuda"):
    t = inp.tensors()
    return {k: (None if v is None else v.to(device)) for k, v in t.items()}


def head_problem(inp, b, h):
    """The (batch b, head h) pair as a one-batch, one-head, one-group problem (pure indexing)."""
    s = inp.shape
    g = h // (s.nheads // s.ngroups)
    sub = dict(x=inp.x[b:b + 1, :, h:h + 1], dt=inp.dt[b:b + 1, :, h:h + 1], A=inp.A[h:h + 1],
               B=inp.B[b:b + 1, :, g:g + 1], C=inp.C[b:b + 1, :, g:g + 1], D=inp.D[h:h + 1],
               h0=None if inp.h0 is None else inp.h0[b:b + 1, h:h + 1])
    return sub


def oracle_pairs(inp, pairs):
    """Sequential oracle for each sampled (b, h): returns {(b, h): (y [L, H], h_final [H, S])}."""
    out = {}
    for b, h in pairs:
        p = head_problem(inp, b, h)
        y, hf = oracle.ssd_fwd_seq(p["x"], p["dt"], p["A"], p["B"], p["C"], p["D"], p["h0"])
        out[(b, h)] = (y[0, :, 0], hf[0, 0])
    return out


def oracle_full(inp):
    t = inp.tensors()
    return oracle.ssd_fwd_seq(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], t["h0"])


def sample_pairs(shape, n_random=3, seed=0):
    rng = np.random.default_rng(seed)
    pairs = {(0, 0), (shape.batch - 1, shape.nheads - 1), (shape.batch // 2, shape.nheads // 2)}
    while len(pairs) < 3 + n_random and len(pairs) < shape.batch * shape.nheads:
        pairs.add((int(rng.integers(shape.batch)), int(rng.integers(shape.nheads))))
    return sorted(pairs)
