"""Shared test helpers: device transfer, error metric, the oracle over a whole problem."""
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


def oracle_full(inp):
    t = inp.tensors()
    return oracle.ssd_fwd_seq(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], t["h0"])
