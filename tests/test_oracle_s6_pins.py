"""Pins for the oracle's Mamba-1 selective scan (``oracle.s6_fwd_seq``), from sources other than itself.

- The worked example printed on the page: discretize(log(0.9)/0.5, -log(0.9), 0.5)
  = (0.9000, 0.0527), read from ``tests/golden/ema_discretize.txt``.
- The EMA loop of the same page (Part 2) as a one-state scan.
- With A[d][n] equal over n, channel d is a Mamba-2 head with H = 1, S = N: the SSD
  oracle (a separate implementation) must give the same y and final state.
- The unrolled sum of the recurrence, term by term, on tiny shapes with G > 1.
- delta = 0 holds the state; the geometric closed form; split/resume; the output is
  the sum of the single-state scans (which fixes the [dim][N] layout of A).

Page reference:
  [hard]  "Sasha Rush: Mamba: The Hard Way", Part 5 (Mamba / S6) and Part 2 (EMA).
"""
import math

import numpy as np
import pytest

import oracle
from tests.test_oracle_pins import read_golden, relerr


def rand_s6(rng, batch, L, dim, N, G, h0=True, skip=True):
    x = rng.standard_normal((batch, dim, L))
    delta = rng.uniform(0.0, 0.4, (batch, dim, L))
    A = -rng.uniform(0.5, 4.0, (dim, N))
    Bm = rng.standard_normal((batch, G, N, L))
    Cm = rng.standard_normal((batch, G, N, L))
    D = rng.standard_normal(dim) if skip else None
    h = 0.3 * rng.standard_normal((batch, dim, N)) if h0 else None
    return x, delta, A, Bm, Cm, D, h


def unrolled_s6(x, delta, A, Bm, Cm, D, h0):
    """y_t = sum_n C_t[n] (exp(A[n] sum_{s<=t} delta_s) h0[n]
                           + sum_{j<=t} exp(A[n] sum_{j<s<=t} delta_s) delta_j B_j[n] x_j) + D x_t."""
    batch, dim, L = x.shape
    G, N = Bm.shape[1], Bm.shape[2]
    cpg = dim // G
    y = np.zeros_like(x)
    for b in range(batch):
        for d in range(dim):
            g = d // cpg
            for t in range(L):
                acc = 0.0
                for n in range(N):
                    a = A[d, n]
                    term = math.exp(a * delta[b, d, :t + 1].sum()) * (0.0 if h0 is None else h0[b, d, n])
                    for j in range(t + 1):
                        term += math.exp(a * delta[b, d, j + 1:t + 1].sum()) * delta[b, d, j] * Bm[b, g, n, j] * x[b, d, j]
                    acc += Cm[b, g, n, t] * term
                y[b, d, t] = acc + (0.0 if D is None else D[d] * x[b, d, t])
    return y


def test_s6_worked_example_printed_values():
    """[hard] Part 5 prints discretize(log(0.9)/0.5, -log(0.9), 0.5) = (0.9000, 0.0527): a one-state scan
    with C = 1 returns abar (h0 = 1, x = 0) and bbar (h0 = 0, x = 1) after one token."""
    g = read_golden("ema_discretize.txt")
    alpha, delta, nd = g["alpha"], g["delta"], int(g["decimals"])
    A = np.array([[math.log(alpha) / delta]])
    one = np.ones((1, 1, 1))
    B1 = np.full((1, 1, 1, 1), -math.log(alpha))
    C1 = np.ones((1, 1, 1, 1))
    y_a, _ = oracle.s6_fwd_seq(0 * one, delta * one, A, B1, C1, h0=one)
    y_b, _ = oracle.s6_fwd_seq(one, delta * one, A, B1, C1)
    assert round(float(y_a[0, 0, 0]), nd) == g["a_bar"]
    assert round(float(y_b[0, 0, 0]), nd) == g["b_bar"]


def test_s6_reduces_to_ema_loop():
    """[hard] Part 2: h = alpha h + (1 - alpha) x, y = h; a one-state scan with exp(delta A) = alpha and
    delta B = 1 - alpha, C = 1."""
    alpha, delta, L = 0.9, 0.5, 64
    xs = np.arange(L, dtype=np.float64)
    h, ema = 0.0, []
    for k in range(L):
        h = alpha * h + (1 - alpha) * xs[k]
        ema.append(h)
    y, hf = oracle.s6_fwd_seq(xs.reshape(1, 1, L), np.full((1, 1, L), delta), np.array([[math.log(alpha) / delta]]),
                              np.full((1, 1, 1, L), (1 - alpha) / delta), np.ones((1, 1, 1, L)))
    assert relerr(y[0, 0], np.array(ema)) < 1e-13
    assert abs(hf[0, 0, 0] - ema[-1]) < 1e-12 * abs(ema[-1])


@pytest.mark.parametrize("G", [1, 2])
def test_s6_equals_ssd_when_A_is_shared_over_states(G):
    """A[d][n] = A_d: channel d is a Mamba-2 head (H = 1, S = N, dt = delta) of the SSD oracle."""
    rng = np.random.default_rng(4)
    batch, L, dim, N = 2, 23, 6, 5
    x, delta, _, Bm, Cm, D, h0 = rand_s6(rng, batch, L, dim, N, G)
    Ad = -rng.uniform(0.5, 4.0, dim)
    A = np.repeat(Ad[:, None], N, axis=1)
    y, hf = oracle.s6_fwd_seq(x, delta, A, Bm, Cm, D, h0)
    # SSD layouts: x [B, L, nh, 1], dt [B, L, nh], B/C [B, L, G, S], h0 [B, nh, 1, S]
    ys, hs = oracle.ssd_fwd_seq(x.transpose(0, 2, 1)[..., None], delta.transpose(0, 2, 1), Ad,
                                Bm.transpose(0, 3, 1, 2), Cm.transpose(0, 3, 1, 2), D, h0[:, :, None, :])
    assert relerr(y, ys[..., 0].transpose(0, 2, 1)) < 1e-13
    assert relerr(hf, hs[:, :, 0, :]) < 1e-13


@pytest.mark.parametrize("shape", [(1, 1, 1, 1, 1), (1, 6, 2, 3, 1), (2, 5, 4, 2, 2), (1, 7, 6, 3, 3)])
def test_s6_unrolled_sum(shape):
    rng = np.random.default_rng(sum(shape))
    batch, L, dim, N, G = shape
    args = rand_s6(rng, batch, L, dim, N, G)
    y, _ = oracle.s6_fwd_seq(*args)
    assert relerr(y, unrolled_s6(*args)) < 1e-12


def test_s6_zero_step_holds_state():
    rng = np.random.default_rng(6)
    x, delta, A, Bm, Cm, D, h0 = rand_s6(rng, 2, 9, 4, 3, 2)
    delta[:] = 0.0
    y, hf = oracle.s6_fwd_seq(x, delta, A, Bm, Cm, D, h0)
    want = np.einsum("bdnt,bdn->bdt", Cm.repeat(2, axis=1), h0) + D[None, :, None] * x
    assert relerr(y, want) < 1e-14
    assert np.array_equal(hf, h0)


def test_s6_geometric_closed_form():
    """Constant delta, A, B, x = 1, C = 1, h0 = 0: h_t = delta B (1 - q^(t+1)) / (1 - q), q = exp(delta A)."""
    L, dl, a, bv = 40, 0.3, -1.7, 0.8
    y, hf = oracle.s6_fwd_seq(np.ones((1, 1, L)), np.full((1, 1, L), dl), np.array([[a]]),
                              np.full((1, 1, 1, L), bv), np.ones((1, 1, 1, L)))
    q = math.exp(dl * a)
    want = np.array([dl * bv * (1 - q ** (t + 1)) / (1 - q) for t in range(L)])
    assert relerr(y[0, 0], want) < 1e-13


def test_s6_split_resume():
    rng = np.random.default_rng(8)
    x, delta, A, Bm, Cm, D, h0 = rand_s6(rng, 2, 30, 4, 3, 2)
    y, hf = oracle.s6_fwd_seq(x, delta, A, Bm, Cm, D, h0)
    y1, h1 = oracle.s6_fwd_seq(x[..., :11], delta[..., :11], A, Bm[..., :11], Cm[..., :11], D, h0)
    y2, h2 = oracle.s6_fwd_seq(x[..., 11:], delta[..., 11:], A, Bm[..., 11:], Cm[..., 11:], D, h1)
    assert relerr(np.concatenate([y1, y2], axis=-1), y) < 1e-13
    assert relerr(h2, hf) < 1e-13


def test_s6_output_is_the_sum_of_single_state_scans():
    """The N states are independent given delta and x: y = sum_n (scan with state n alone)."""
    rng = np.random.default_rng(9)
    x, delta, A, Bm, Cm, _, h0 = rand_s6(rng, 2, 12, 5, 3, 1, skip=False)
    y, hf = oracle.s6_fwd_seq(x, delta, A, Bm, Cm, None, h0)
    parts = [oracle.s6_fwd_seq(x, delta, A[:, n:n + 1], Bm[:, :, n:n + 1], Cm[:, :, n:n + 1], None,
                               h0[:, :, n:n + 1]) for n in range(3)]
    assert relerr(sum(p[0] for p in parts), y) < 1e-13
    assert relerr(np.concatenate([p[1] for p in parts], axis=-1), hf) < 1e-14
