"""The autograd binding's wiring, on the CPU: the two C-ABI calls it makes are replaced by
fakes that return the oracle's results, so the test checks only what the binding itself
does -- which gradient goes to which input, the dtypes, absent h0 and unused outputs.
(On a GPU the same binding runs libssd.so; tests/test_gpu_bwd.py covers the kernels.)
"""
import numpy as np
import pytest
import torch

import oracle
from selective_state_space_gb300 import api, autograd, workloads


def _fake_fwd(x, dt, A, B, C, D, chunk, h0=None, **kw):
    y, hf = oracle.ssd_fwd_seq(x, dt, A, B, C, D, h0)
    return torch.from_numpy(y).to(x.dtype), torch.from_numpy(hf).float()


def _fake_bwd(x, dt, A, B, C, D, dy, chunk, h0=None, dh_final=None, *, want_dh0=True, **kw):
    g = oracle.ssd_bwd_seq(x, dt, A, B, C, D, dy, h0=h0, dh_final=dh_final)
    out = {k: torch.from_numpy(v) for k, v in g.items()}
    out = {"dx": out["dx"].to(x.dtype), "ddt": out["ddt"].to(dt.dtype), "dA": out["dA"].float(),
           "dB": out["dB"].to(B.dtype), "dC": out["dC"].to(C.dtype), "dD": out["dD"].float(),
           "dh0": out["dh0"].float() if want_dh0 else None}
    return out


@pytest.fixture
def fakes(monkeypatch):
    monkeypatch.setattr(api, "ssd_fwd", _fake_fwd)
    monkeypatch.setattr(api, "ssd_bwd", _fake_bwd)


@pytest.mark.parametrize("with_h0", [True, False])
def test_gradients_reach_the_right_inputs(fakes, with_h0):
    shape = workloads.custom(2, 24, 4, 3, 5, 2, 8, "f32", h0_recipe="normal" if with_h0 else "none", seed=61)
    inp = workloads.make_inputs(shape)
    t = {k: (None if v is None else v.clone().requires_grad_()) for k, v in inp.tensors().items()}
    y, hf = autograd.ssd_chunked(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], shape.chunk, t["h0"])
    gy = torch.randn(y.shape, generator=torch.Generator().manual_seed(1))
    gh = torch.randn(hf.shape, generator=torch.Generator().manual_seed(2))
    ((y * gy).sum() + (hf * gh).sum()).backward()
    ref = oracle.ssd_bwd_seq(inp.x, inp.dt, inp.A, inp.B, inp.C, inp.D, gy, h0=inp.h0, dh_final=gh)
    names = {"x": "dx", "dt": "ddt", "A": "dA", "B": "dB", "C": "dC", "D": "dD"}
    if with_h0:
        names["h0"] = "dh0"
    for k, gk in names.items():
        np.testing.assert_allclose(t[k].grad.double().numpy(), ref[gk], rtol=1e-5, atol=1e-6, err_msg=k)
        assert t[k].grad.dtype == t[k].dtype


def test_unused_final_state_means_zero_dh_final(fakes):
    shape = workloads.custom(1, 16, 2, 2, 3, 1, 4, "f32", seed=62)
    inp = workloads.make_inputs(shape)
    t = {k: (None if v is None else v.clone().requires_grad_()) for k, v in inp.tensors().items()}
    y, _ = autograd.ssd_chunked(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], shape.chunk)
    y.sum().backward()
    ref = oracle.ssd_bwd_seq(inp.x, inp.dt, inp.A, inp.B, inp.C, inp.D, np.ones(tuple(y.shape)))
    np.testing.assert_allclose(t["x"].grad.double().numpy(), ref["dx"], rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(t["A"].grad.double().numpy(), ref["dA"], rtol=1e-5, atol=1e-6)
