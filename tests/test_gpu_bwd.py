"""GPU parity of the gradient pass (ssd_bwd, through the C ABI) against the CPU oracle.

Small problems: every element of dx, ddt, dB, dC, dh0 and dA, dD against
``oracle.ssd_bwd_seq``.  The 2.7B-shaped layer at full size: dx, ddt, dh0 of
sampled (batch, head) pairs and dA, dD of sampled heads (the oracle runs those
sequences alone, which gives their exact gradients), and dC through Euler's
identity for C, token by token, which holds at any size.  Bounds: max|got - ref| / max|ref|
<= 1e-3 for float32 inputs, <= 2e-2 for bfloat16 inputs.
"""
import numpy as np
import pytest
import torch

import oracle
from selective_state_space_gb300 import api, workloads

from .helpers import TOL, rel_max_err, to_dev

pytestmark = pytest.mark.gpu

SMALL = [
    workloads.custom(1, 96, 4, 16, 8, 2, 32, "f32", dt_recipe="loguniform", h0_recipe="normal", seed=31,
                     name="f32-small"),
    workloads.custom(2, 77, 6, 8, 16, 3, 16, "f32", h0_recipe="normal", seed=32, name="f32-ragged"),
    workloads.custom(1, 33, 2, 1, 1, 1, 1, "f32", seed=33, name="scalar-T1"),
    workloads.custom(2, 512, 6, 64, 128, 1, 256, "bf16", h0_recipe="normal", seed=34, name="bf16-c1-small"),
    workloads.custom(1, 700, 8, 64, 128, 2, 256, "bf16", dt_zero_frac=0.05, seed=35, name="bf16-ragged-g2"),
    workloads.custom(2, 300, 4, 128, 256, 2, 128, "bf16", dt_recipe="loguniform", a_range=(0.5, 8.0),
                     seed=36, name="bf16-h128-s256-ragged"),
    # many heads per group over few tiles: each group's heads are split into slices
    workloads.custom(1, 128, 80, 64, 128, 1, 64, "bf16", h0_recipe="normal", seed=37, name="bf16-80-heads"),
    workloads.custom(2, 1024, 24, 64, 128, 1, 256, "bf16", seed=38, name="bf16-24-heads"),
]

GRADS = ("dx", "ddt", "dB", "dC", "dh0", "dA", "dD")


def run_bwd(inp, gin):
    d = to_dev(inp)
    dy = gin.dy.cuda()
    dhf = None if gin.dh_final is None else gin.dh_final.cuda()
    out = api.ssd_bwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], dy, inp.shape.chunk, d["h0"], dhf)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: s.name)
def test_bwd_small_all_elements(shape):
    inp = workloads.make_inputs(shape)
    gin = workloads.make_grad_inputs(shape, with_dh_final=shape.seed % 2 == 0)
    got = run_bwd(inp, gin)
    t = inp.tensors()
    ref = oracle.ssd_bwd_seq(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], gin.dy, h0=t["h0"],
                             dh_final=gin.dh_final)
    tol = TOL[shape.dtype]
    for name in GRADS:
        err = rel_max_err(got[name], ref[name])
        assert err <= tol, (shape.name, name, err)


def test_bwd_is_deterministic():
    shape = SMALL[6]
    inp = workloads.make_inputs(shape)
    gin = workloads.make_grad_inputs(shape)
    a, b = run_bwd(inp, gin), run_bwd(inp, gin)
    for name in GRADS:
        assert torch.equal(a[name], b[name]), name


def test_bwd_empty_sequence():
    shape = workloads.custom(2, 0, 4, 16, 8, 2, 32, "f32", h0_recipe="normal", seed=39)
    inp = workloads.make_inputs(shape)
    gin = workloads.make_grad_inputs(shape)
    got = run_bwd(inp, gin)
    assert torch.equal(got["dh0"].cpu(), gin.dh_final)
    assert not got["dA"].any() and not got["dD"].any()


def test_bwd_rejects_unsupported_and_bad_args():
    shape = workloads.custom(1, 64, 2, 16, 8, 1, 512, "f32", seed=40)   # chunk > 256
    inp = workloads.make_inputs(shape)
    gin = workloads.make_grad_inputs(shape)
    with pytest.raises(api._native.SSDError) as ei:
        run_bwd(inp, gin)
    assert ei.value.code == 2
    shape = workloads.custom(1, 64, 2, 16, 8, 1, 32, "f32", seed=41)
    inp = workloads.make_inputs(shape)
    d = to_dev(inp)
    dy = torch.zeros_like(d["x"])
    desc = api.desc_for(d["x"], d["B"], 32)
    ws = torch.empty(api.bwd_workspace_size(desc), dtype=torch.uint8, device="cuda")
    lib = api._native.load()
    import ctypes
    outs = [torch.empty_like(d["x"]), torch.empty_like(d["dt"]), torch.empty(2, device="cuda"),
            torch.empty_like(d["B"]), torch.empty_like(d["C"]), torch.empty(2, device="cuda")]
    # dx aliasing x is refused before any launch
    rc = lib.ssd_bwd(ctypes.byref(desc), d["x"].data_ptr(), d["dt"].data_ptr(), d["A"].data_ptr(),
                     d["B"].data_ptr(), d["C"].data_ptr(), d["D"].data_ptr(), None, dy.data_ptr(), None,
                     d["x"].data_ptr(), outs[1].data_ptr(), outs[2].data_ptr(), outs[3].data_ptr(),
                     outs[4].data_ptr(), outs[5].data_ptr(), None, ws.data_ptr(), ws.numel(), None)
    assert rc == 1
    # a workspace one byte short is refused
    rc = lib.ssd_bwd(ctypes.byref(desc), d["x"].data_ptr(), d["dt"].data_ptr(), d["A"].data_ptr(),
                     d["B"].data_ptr(), d["C"].data_ptr(), d["D"].data_ptr(), None, dy.data_ptr(), None,
                     outs[0].data_ptr(), outs[1].data_ptr(), outs[2].data_ptr(), outs[3].data_ptr(),
                     outs[4].data_ptr(), outs[5].data_ptr(), None, ws.data_ptr(), ws.numel() - 1, None)
    assert rc == 3


@pytest.mark.slow
def test_bwd_full_size_layer_sampled():
    """The 2.7B-shaped layer (B=4, L=4096, nh=80) at full size."""
    shape = workloads.by_name("mamba2-2.7b-layer")
    inp = workloads.make_inputs(shape)
    gin = workloads.make_grad_inputs(shape)
    got = run_bwd(inp, gin)
    t = inp.tensors()
    tol = TOL[shape.dtype]
    for h in (0, 57):
        sub = dict(x=t["x"][:, :, h:h + 1], dt=t["dt"][:, :, h:h + 1], A=t["A"][h:h + 1], B=t["B"], C=t["C"],
                   D=t["D"][h:h + 1], h0=t["h0"][:, h:h + 1])
        ref = oracle.ssd_bwd_seq(sub["x"], sub["dt"], sub["A"], sub["B"], sub["C"], sub["D"],
                                 gin.dy[:, :, h:h + 1], h0=sub["h0"], dh_final=gin.dh_final[:, h:h + 1])
        assert rel_max_err(got["dx"][:, :, h:h + 1], ref["dx"]) <= tol, h
        assert rel_max_err(got["ddt"][:, :, h:h + 1], ref["ddt"]) <= tol, h
        assert rel_max_err(got["dh0"][:, h:h + 1], ref["dh0"]) <= tol, h
        assert abs(got["dA"][h].item() - ref["dA"][0]) <= tol * abs(ref["dA"][0]), h
        assert abs(got["dD"][h].item() - ref["dD"][0]) <= tol * abs(ref["dD"][0]), h
    # Euler's identity for C, token by token (C_t enters y_t only, linearly):
    #   sum_s dC[b,t,g,s] C[b,t,g,s] = sum_{h in g} dy[b,t,h] . (y[b,t,h] - D x[b,t,h]),
    # with y from the forward pass; error bound relative to the largest sum_s |dC C| of a token
    d = to_dev(inp)
    y, _ = api.ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], shape.chunk, d["h0"],
                       out_dtype=torch.float32)
    dy = gin.dy.cuda().double()
    hpg = shape.nheads // shape.ngroups
    per_head = (dy * (y.double() - d["D"].double()[None, None, :, None] * d["x"].double())).sum(-1)
    rhs = per_head.view(shape.batch, shape.seqlen, shape.ngroups, hpg).sum(-1)
    terms = got["dC"].double() * d["C"].double()
    lhs = terms.sum(-1)
    scale = terms.abs().sum(-1).max().item()
    err = (lhs - rhs).abs().max().item()
    assert err <= tol * scale, (err, scale)
