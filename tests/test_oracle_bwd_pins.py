"""Pins for the oracle's gradients (``oracle.ssd_bwd_seq``), from sources other than itself.

- Central finite differences of the forward oracle, on tiny shapes, for every
  input: the definition of the gradient, evaluated with an error of O(eps^2).
- The scalar case (H = S = 1, two tokens) differentiated by hand.
- dt = 0: the state never moves, and every gradient has a closed form.
- Euler's identity for the parts of the loss that are homogeneous of degree one
  (in (x, h0) jointly, in C, in D, and in B when h0 = 0): sum(g * v) = loss part.
- Split/resume: the gradient of the second half's entering state is the
  gradient the first half receives for its final state.
- The chunked restatement (``oracle.bwd_chunked``) agrees at every chunk size.

Page references:
  [hard]  "Sasha Rush: Mamba: The Hard Way", Part 3 (deriving the derivatives).
  [blog]  NVIDIA developer blog "Accelerating Mamba-2 with High-Performance
          Forward Pass Kernels in NVIDIA CUDA Tile", section "Mamba-2 architecture".
"""
import math

import numpy as np
import pytest

import oracle
from oracle.bwd_chunked import ssd_bwd_chunked
from tests.test_oracle_pins import rand_problem, relerr

NAMES = {"x": "dx", "dt": "ddt", "A": "dA", "Bm": "dB", "Cm": "dC", "D": "dD", "h0": "dh0"}


def problem(seed, batch, L, nh, H, S, G, h0=True, dhf=True):
    rng = np.random.default_rng(seed)
    x, dt, A, Bm, Cm, D, h = rand_problem(rng, batch, L, nh, H, S, G, h0=h0)
    dy = rng.standard_normal((batch, L, nh, H))
    dh_final = rng.standard_normal((batch, nh, H, S)) if dhf else None
    return dict(x=x, dt=dt, A=A, Bm=Bm, Cm=Cm, D=D, h0=h), dy, dh_final


def loss(inp, dy, dh_final):
    y, hf = oracle.ssd_fwd_seq(inp["x"], inp["dt"], inp["A"], inp["Bm"], inp["Cm"], inp["D"], inp["h0"],
                               nthreads=1)
    val = float(np.sum(dy * y))
    if dh_final is not None:
        val += float(np.sum(dh_final * hf))
    return val


def grads(inp, dy, dh_final):
    return oracle.ssd_bwd_seq(inp["x"], inp["dt"], inp["A"], inp["Bm"], inp["Cm"], inp["D"], dy,
                              h0=inp["h0"], dh_final=dh_final)


FD_SHAPES = [
    # batch, L, nh, H, S, G
    (1, 1, 1, 1, 1, 1),
    (1, 5, 2, 2, 3, 1),
    (2, 6, 4, 3, 2, 2),     # groups > 1, two heads per group
    (1, 4, 6, 2, 2, 3),
]


@pytest.mark.parametrize("shape", FD_SHAPES)
def test_bwd_matches_finite_differences(shape):
    """Every gradient equals the central difference of the forward oracle's loss."""
    inp, dy, dhf = problem(11, *shape)
    g = grads(inp, dy, dhf)
    eps = 1e-6
    for name, gname in NAMES.items():
        v = inp[name]
        fd = np.zeros_like(v)
        for idx in np.ndindex(v.shape):
            vp, vm = v.copy(), v.copy()
            vp[idx] += eps
            vm[idx] -= eps
            fd[idx] = (loss({**inp, name: vp}, dy, dhf) - loss({**inp, name: vm}, dy, dhf)) / (2 * eps)
        assert relerr(g[gname], fd) < 1e-6, (shape, gname)


def test_bwd_scalar_case_by_hand():
    """H = S = 1, two tokens, dy = (1, 1), dh_final = 0, written out by hand.

    y0 = c0 (a0 h0 + d0 b0 x0) + D x0,  y1 = c1 (a1 (a0 h0 + d0 b0 x0) + d1 b1 x1) + D x1,
    a_t = exp(A d_t).  Each derivative below is the partial of y0 + y1.
    """
    A, D, h0 = -1.3, 0.7, 0.4
    d0, d1, b0, b1, c0, c1, x0, x1 = 0.2, 0.5, 0.9, -0.6, 1.1, -0.8, 0.3, -1.7
    a0, a1 = math.exp(A * d0), math.exp(A * d1)
    h_0 = a0 * h0 + d0 * b0 * x0
    want = {
        "dx": [c0 * d0 * b0 + c1 * a1 * d0 * b0 + D, c1 * d1 * b1 + D],
        "dB": [c0 * d0 * x0 + c1 * a1 * d0 * x0, c1 * d1 * x1],
        "dC": [h_0, a1 * h_0 + d1 * b1 * x1],
        "dD": [x0 + x1],
        "dh0": [c0 * a0 + c1 * a1 * a0],
        # dt enters through a_t = exp(A dt_t) and through the input weight dt_t b_t
        "ddt": [c0 * (A * a0 * h0 + b0 * x0) + c1 * a1 * (A * a0 * h0 + b0 * x0),
                c1 * (A * a1 * h_0 + b1 * x1)],
        "dA": [c0 * d0 * a0 * h0 + c1 * (d1 * a1 * h_0 + a1 * d0 * a0 * h0)],
    }
    g = oracle.ssd_bwd_seq(np.array([x0, x1]).reshape(1, 2, 1, 1), np.array([d0, d1]).reshape(1, 2, 1),
                           np.array([A]), np.array([b0, b1]).reshape(1, 2, 1, 1),
                           np.array([c0, c1]).reshape(1, 2, 1, 1), np.array([D]),
                           np.ones((1, 2, 1, 1)), h0=np.array([h0]).reshape(1, 1, 1, 1))
    for k, v in want.items():
        np.testing.assert_allclose(g[k].ravel(), v, rtol=1e-14, atol=1e-15, err_msg=k)


def test_bwd_dt_zero_closed_form():
    """dt = 0 everywhere: h_t = h0 for all t, and lam_t = sum_{i >= t} dy_i C_i^T + dh_final."""
    inp, dy, dhf = problem(5, 2, 6, 4, 3, 5, 2)
    inp["dt"] = np.zeros_like(inp["dt"])
    g = grads(inp, dy, dhf)
    hpg = 2
    batch, L, nh, H = dy.shape
    S = inp["Bm"].shape[3]
    dC = np.zeros_like(inp["Cm"])
    ddt = np.zeros_like(inp["dt"])
    dh0 = np.zeros((batch, nh, H, S))
    for b in range(batch):
        for h in range(nh):
            gg = h // hpg
            lam = dhf[b, h].copy()
            for t in range(L - 1, -1, -1):
                lam += np.outer(dy[b, t, h], inp["Cm"][b, t, gg])
                ddt[b, t, h] = (inp["x"][b, t, h] @ lam @ inp["Bm"][b, t, gg]
                                + inp["A"][h] * np.sum(lam * inp["h0"][b, h]))
                dC[b, t, gg] += inp["h0"][b, h].T @ dy[b, t, h]
            dh0[b, h] = lam
    assert relerr(g["dx"], inp["D"][None, None, :, None] * dy) < 1e-14
    assert np.all(g["dB"] == 0) and np.all(g["dA"] == 0)
    assert relerr(g["dC"], dC) < 1e-13
    assert relerr(g["ddt"], ddt) < 1e-13
    assert relerr(g["dh0"], dh0) < 1e-13
    assert relerr(g["dD"], np.einsum("blhp,blhp->h", dy, inp["x"])) < 1e-13


@pytest.mark.parametrize("with_h0", [True, False])
def test_bwd_homogeneity(with_h0):
    """Euler's identity on the degree-one parts of the loss, at a size past the tiny ones."""
    inp, dy, dhf = problem(9, 2, 37, 4, 6, 5, 2, h0=with_h0)
    g = grads(inp, dy, dhf)
    y, hf = oracle.ssd_fwd_seq(inp["x"], inp["dt"], inp["A"], inp["Bm"], inp["Cm"], inp["D"], inp["h0"])
    total = np.sum(dy * y) + np.sum(dhf * hf)
    skip = np.sum(dy * inp["D"][None, None, :, None] * inp["x"])
    # (x, h0) jointly: y and h_final are linear in them
    lhs = np.sum(g["dx"] * inp["x"]) + (np.sum(g["dh0"] * inp["h0"]) if with_h0 else 0.0)
    assert abs(lhs - total) < 1e-12 * max(1.0, abs(total))
    # C: y - D x is linear in C; h_final does not depend on C
    assert abs(np.sum(g["dC"] * inp["Cm"]) - (np.sum(dy * y) - skip)) < 1e-12 * max(1.0, abs(total))
    # D: only the skip term
    assert abs(np.sum(g["dD"] * inp["D"]) - skip) < 1e-12 * max(1.0, abs(skip))
    if not with_h0:  # with h0 = 0 every state is linear in B
        assert abs(np.sum(g["dB"] * inp["Bm"]) - (total - skip)) < 1e-12 * max(1.0, abs(total))


def test_bwd_split_resume():
    """Second half from the first half's h_final; its dh0 is the first half's dh_final."""
    inp, dy, dhf = problem(3, 2, 20, 4, 3, 4, 2)
    full = grads(inp, dy, dhf)
    half = 9
    first = {k: (v[:, :half] if k in ("x", "dt", "Bm", "Cm") else v) for k, v in inp.items()}
    _, hf1 = oracle.ssd_fwd_seq(first["x"], first["dt"], first["A"], first["Bm"], first["Cm"], first["D"],
                                first["h0"])
    second = {k: (v[:, half:] if k in ("x", "dt", "Bm", "Cm") else v) for k, v in inp.items()}
    second["h0"] = hf1
    g2 = grads(second, dy[:, half:], dhf)
    g1 = grads(first, dy[:, :half], g2["dh0"])
    for name in ("dx", "ddt", "dB", "dC"):
        assert relerr(np.concatenate([g1[name], g2[name]], axis=1), full[name]) < 1e-12, name
    for name in ("dA", "dD"):
        assert relerr(g1[name] + g2[name], full[name]) < 1e-12, name
    assert relerr(g1["dh0"], full["dh0"]) < 1e-12


@pytest.mark.parametrize("chunk", [1, 3, 8, 64])
def test_bwd_chunked_form_agrees(chunk):
    """The per-chunk restatement gives the same gradients (ragged last chunk at 3 and 8)."""
    inp, dy, dhf = problem(7, 2, 29, 4, 5, 3, 2)
    a = grads(inp, dy, dhf)
    b = ssd_bwd_chunked(inp["x"], inp["dt"], inp["A"], inp["Bm"], inp["Cm"], inp["D"], dy, chunk,
                        h0=inp["h0"], dh_final=dhf)
    for k in a:
        assert relerr(b[k], a[k]) < 1e-11, (chunk, k)


def test_bwd_empty_sequence():
    """No tokens: h_final = h0, so dh0 = dh_final and every other gradient is zero."""
    inp, dy, dhf = problem(2, 2, 0, 2, 3, 2, 1)
    g = grads(inp, dy, dhf)
    assert np.array_equal(g["dh0"], dhf)
    assert not np.any(g["dA"]) and not np.any(g["dD"])
    assert g["dx"].shape == (2, 0, 2, 3) and g["dB"].shape == (2, 0, 1, 2)
