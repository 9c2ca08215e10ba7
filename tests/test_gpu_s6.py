"""GPU parity of the Mamba-1 selective scan (s6_fwd, through the C ABI) against the CPU oracle.

Small problems: every element of y and h_final.  The two named workloads at
full size: sampled channels, which the oracle computes one by one (a channel's
scan reads only its own x, delta and A row and its group's B, C).  Bounds:
max|got - ref| / max|ref| <= 1e-3 for float32 inputs, <= 2e-2 for bfloat16.
"""
import numpy as np
import pytest
import torch

import oracle
from selective_state_space_gb300 import api, workloads

from .helpers import TOL, rel_max_err

pytestmark = pytest.mark.gpu

SMALL = [
    workloads.s6_custom(2, 128, 4, 4, 1, "f32", recipe="hardway", skip=False, h0=False, seed=50, name="hardway-test"),
    workloads.s6_custom(2, 200, 48, 16, 2, "f32", seed=51, name="f32-g2-ragged"),
    workloads.s6_custom(1, 77, 40, 3, 1, "f32", seed=52, name="f32-n3"),
    workloads.s6_custom(3, 64, 96, 1, 3, "f32", seed=53, name="f32-n1-g3"),
    workloads.s6_custom(2, 300, 64, 32, 1, "f32", seed=54, name="f32-n32"),
    workloads.s6_custom(2, 257, 160, 16, 2, "bf16", seed=55, name="bf16-n16"),
    workloads.s6_custom(1, 1, 33, 8, 1, "bf16", seed=56, name="bf16-one-token"),
]


def run_s6(inp, out_dtype=None):
    d = {k: (None if v is None else v.cuda()) for k, v in inp.tensors().items()}
    y, hf = api.s6_fwd(d["x"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["h0"], out_dtype=out_dtype)
    torch.cuda.synchronize()
    return y, hf


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: s.name)
def test_s6_small_all_elements(shape):
    inp = workloads.make_s6_inputs(shape)
    y, hf = run_s6(inp)
    t = inp.tensors()
    y_ref, hf_ref = oracle.s6_fwd_seq(t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["h0"])
    tol = TOL[shape.dtype]
    assert rel_max_err(y, y_ref) <= tol
    assert rel_max_err(hf, hf_ref) <= tol


def test_s6_float32_output_from_bf16_inputs():
    shape = SMALL[5]
    inp = workloads.make_s6_inputs(shape)
    y, _ = run_s6(inp, out_dtype=torch.float32)
    t = inp.tensors()
    y_ref, _ = oracle.s6_fwd_seq(t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["h0"])
    assert y.dtype == torch.float32 and rel_max_err(y, y_ref) <= 1e-3


def test_s6_empty_sequence_copies_h0():
    shape = workloads.s6_custom(2, 0, 8, 4, 1, "f32", seed=57)
    inp = workloads.make_s6_inputs(shape)
    y, hf = run_s6(inp)
    assert y.numel() == 0 and torch.equal(hf.cpu(), inp.h0)


@pytest.mark.slow
@pytest.mark.parametrize("name", [s.name for s in workloads.S6_WORKLOADS])
def test_s6_full_size_sampled_channels(name):
    shape = workloads.s6_by_name(name)
    inp = workloads.make_s6_inputs(shape)
    y, hf = run_s6(inp)
    t = inp.tensors()
    cpg = shape.dim // shape.ngroups
    rng = np.random.default_rng(0)
    chans = {(0, 0), (shape.batch - 1, shape.dim - 1)} | {(int(rng.integers(shape.batch)), int(rng.integers(shape.dim)))
                                                          for _ in range(6)}
    tol = TOL[shape.dtype]
    for b, d in sorted(chans):
        g = d // cpg
        y_ref, hf_ref = oracle.s6_fwd_seq(t["x"][b:b + 1, d:d + 1], t["delta"][b:b + 1, d:d + 1], t["A"][d:d + 1],
                                          t["B"][b:b + 1, g:g + 1], t["C"][b:b + 1, g:g + 1],
                                          None if t["D"] is None else t["D"][d:d + 1],
                                          None if t["h0"] is None else t["h0"][b:b + 1, d:d + 1])
        assert rel_max_err(y[b:b + 1, d:d + 1], y_ref) <= tol, (b, d)
        assert rel_max_err(hf[b:b + 1, d:d + 1], hf_ref) <= tol, (b, d)
