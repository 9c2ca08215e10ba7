"""Pins for the CPU oracle: checks against what the pages and the mathematics fix.

None of these tests re-types the oracle's own loop.  Each pin comes from an
independent source: a worked example printed on a page, a closed form, a
special case that reduces to a textbook computation (causal linear attention,
the exponential moving average), the unrolled sum of the recurrence written
term by term, or invariants (chunk-size invariance, split/resume, decode).

Page references:
  [blog]  NVIDIA developer blog "Accelerating Mamba-2 with High-Performance
          Forward Pass Kernels in NVIDIA CUDA Tile", section "Mamba-2 architecture".
  [hard]  "Mamba: The Hard Way" (Sasha Rush), Parts 2 and 5.
"""
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_problem(rng, batch, L, nh, H, S, G, h0=True, a_lo=0.5, a_hi=4.0, dt_lo=0.01, dt_hi=0.5):
    x = rng.standard_normal((batch, L, nh, H))
    dt = rng.uniform(dt_lo, dt_hi, (batch, L, nh))
    A = -rng.uniform(a_lo, a_hi, nh)
    Bm = rng.standard_normal((batch, L, G, S)) / math.sqrt(S)
    Cm = rng.standard_normal((batch, L, G, S)) / math.sqrt(S)
    D = rng.standard_normal(nh)
    h = 0.3 * rng.standard_normal((batch, nh, H, S)) if h0 else None
    return x, dt, A, Bm, Cm, D, h


def relerr(a, b):
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


TINY_SHAPES = [
    # batch, L, nh, H, S, G, chunk
    (1, 1, 1, 1, 1, 1, 1),
    (1, 7, 1, 1, 1, 1, 3),
    (2, 8, 4, 3, 2, 2, 4),      # groups > 1, 2 heads per group
    (1, 13, 6, 4, 5, 3, 4),     # ragged last chunk
    (2, 16, 2, 2, 3, 1, 16),
    (1, 33, 4, 8, 4, 2, 8),
]


def unrolled(x, dt, A, Bm, Cm, D, h0):
    """Brute force from the unrolled recurrence ([blog], the decayed expansion of h_{t+T}):

        h_t = exp(sum_{s<=t} a_s) h0 + sum_{j<=t} exp(sum_{j<s<=t} a_s) dt_j B_j x_j^T
        y_t = C_t^T h_t + D x_t,  a_s = A dt_s,  group(head) = head // (nh / G)

    evaluated term by term for every t (O(L^2)), with the state stored [p][s].
    """
    batch, L, nh, H = x.shape
    G, S = Bm.shape[2], Bm.shape[3]
    hpg = nh // G
    y = np.zeros_like(x)
    hf = np.zeros((batch, nh, H, S))
    for b in range(batch):
        for h in range(nh):
            g = h // hpg
            a = A[h] * dt[b, :, h]
            for t in range(L):
                state = np.zeros((H, S)) if h0 is None else math.exp(a[: t + 1].sum()) * h0[b, h]
                for j in range(t + 1):
                    w = math.exp(a[j + 1: t + 1].sum())
                    state = state + w * dt[b, j, h] * np.outer(x[b, j, h], Bm[b, j, g])
                y[b, t, h] = state @ Cm[b, t, g] + D[h] * x[b, t, h]
                if t == L - 1:
                    hf[b, h] = state
    return y, hf


@pytest.mark.parametrize("shape", TINY_SHAPES)
def test_bruteforce_unrolled_tiny(shape):
    batch, L, nh, H, S, G, T = shape
    rng = np.random.default_rng(100 + L * 7 + nh)
    x, dt, A, Bm, Cm, D, h0 = rand_problem(rng, batch, L, nh, H, S, G)
    y_ref, hf_ref = unrolled(x, dt, A, Bm, Cm, D, h0)
    y_s, hf_s = oracle.ssd_fwd_seq(x, dt, A, Bm, Cm, D, h0)
    y_c, hf_c = oracle.ssd_fwd_chunked(x, dt, A, Bm, Cm, D, T, h0)
    assert relerr(y_s, y_ref) < 1e-12 and relerr(hf_s, hf_ref) < 1e-12
    assert relerr(y_c, y_ref) < 1e-12 and relerr(hf_c, hf_ref) < 1e-12


@pytest.mark.parametrize("shape", TINY_SHAPES + [(2, 200, 4, 16, 8, 2, 64), (1, 256, 4, 64, 64, 1, 64)])
def test_sequential_equals_chunked(shape):
    batch, L, nh, H, S, G, T = shape
    rng = np.random.default_rng(7 + L)
    x, dt, A, Bm, Cm, D, h0 = rand_problem(rng, batch, L, nh, H, S, G)
    y_s, hf_s = oracle.ssd_fwd_seq(x, dt, A, Bm, Cm, D, h0)
    y_c, hf_c = oracle.ssd_fwd_chunked(x, dt, A, Bm, Cm, D, T, h0)
    assert relerr(y_c, y_s) < 1e-10
    assert relerr(hf_c, hf_s) < 1e-10


def test_chunk_size_invariance():
    rng = np.random.default_rng(11)
    L = 96
    x, dt, A, Bm, Cm, D, h0 = rand_problem(rng, 1, L, 4, 6, 5, 2)
    y_ref, hf_ref = oracle.ssd_fwd_seq(x, dt, A, Bm, Cm, D, h0)
    for T in (1, 2, 5, 16, 64, L, 2 * L):
        y, hf = oracle.ssd_fwd_chunked(x, dt, A, Bm, Cm, D, T, h0)
        assert relerr(y, y_ref) < 1e-10, T
        assert relerr(hf, hf_ref) < 1e-10, T


def test_dt_zero_holds_state():
    """dt = 0 leaves the state unchanged ([blog]: exp(A*0) = 1, no input term)."""
    rng = np.random.default_rng(3)
    x, dt, A, Bm, Cm, D, h0 = rand_problem(rng, 2, 20, 4, 3, 5, 2)
    dt[:] = 0.0
    for fn in (lambda: oracle.ssd_fwd_seq(x, dt, A, Bm, Cm, D, h0),
               lambda: oracle.ssd_fwd_chunked(x, dt, A, Bm, Cm, D, 8, h0)):
        y, hf = fn()
        assert np.array_equal(hf, h0)
        # y_t = C_t^T h0 + D x_t, per head with its group
        hpg = 2
        for h in range(4):
            yh = np.einsum("bts,bps->btp", Cm[:, :, h // hpg], h0[:, h]) + D[h] * x[:, :, h]
            assert relerr(y[:, :, h], yh) < 1e-13


def test_a_zero_is_causal_linear_attention():
    """A = 0 removes the decay: Y = ((C b^T) o M) X + C h0 + D X with b = dt B and
    M the causal mask including the diagonal ([blog], linear-attention form)."""
    rng = np.random.default_rng(5)
    batch, L, nh, H, S, G = 2, 24, 4, 5, 3, 2
    x, dt, A, Bm, Cm, D, h0 = rand_problem(rng, batch, L, nh, H, S, G)
    A[:] = 0.0
    M = np.tril(np.ones((L, L)))
    y_s, hf_s = oracle.ssd_fwd_seq(x, dt, A, Bm, Cm, D, h0)
    y_c, _ = oracle.ssd_fwd_chunked(x, dt, A, Bm, Cm, D, 7, h0)
    for b in range(batch):
        for h in range(nh):
            g = h // (nh // G)
            bt = dt[b, :, h, None] * Bm[b, :, g]            # stacked b_t (L x S)
            Y = ((Cm[b, :, g] @ bt.T) * M) @ x[b, :, h] + Cm[b, :, g] @ h0[b, h].T + D[h] * x[b, :, h]
            assert relerr(y_s[b, :, h], Y) < 1e-12
            assert relerr(y_c[b, :, h], Y) < 1e-12
            # final state: h0 + b^T X  (undecayed jump), stored [p][s]
            assert relerr(hf_s[b, h], h0[b, h] + x[b, :, h].T @ bt) < 1e-12


def test_scalar_geometric_closed_form():
    """S = H = 1, constant inputs, h0 = 0: h_t = dt B x (1 - q^{t+1}) / (1 - q), q = exp(A dt)."""
    L = 50
    Av, dtv, Bv, Cv, Dv, xv = -0.7, 0.3, 1.3, -0.4, 0.25, 2.0
    x = np.full((1, L, 1, 1), xv)
    dt = np.full((1, L, 1), dtv)
    Bm = np.full((1, L, 1, 1), Bv)
    Cm = np.full((1, L, 1, 1), Cv)
    q = math.exp(Av * dtv)
    t = np.arange(L)
    h = dtv * Bv * xv * (1 - q ** (t + 1)) / (1 - q)
    y_ref = Cv * h + Dv * xv
    for T in (1, 4, L):
        y, hf = oracle.ssd_fwd_chunked(x, dt, np.array([Av]), Bm, Cm, np.array([Dv]), T)
        assert relerr(y[0, :, 0, 0], y_ref) < 1e-12
        assert abs(hf[0, 0, 0, 0] - h[-1]) < 1e-12
    y, hf = oracle.ssd_fwd_seq(x, dt, np.array([Av]), Bm, Cm, np.array([Dv]))
    assert relerr(y[0, :, 0, 0], y_ref) < 1e-12


def test_single_step_by_hand():
    """T = 1, S = H = 1: y = C (exp(A dt) h0 + dt B x) + D x."""
    Av, dtv, Bv, Cv, Dv, xv, h0v = -2.0, 0.125, 0.5, 3.0, -1.5, 0.75, 0.4
    expect_h = math.exp(Av * dtv) * h0v + dtv * Bv * xv
    expect_y = Cv * expect_h + Dv * xv
    args = (np.full((1, 1, 1, 1), xv), np.full((1, 1, 1), dtv), np.array([Av]),
            np.full((1, 1, 1, 1), Bv), np.full((1, 1, 1, 1), Cv), np.array([Dv]))
    h0 = np.full((1, 1, 1, 1), h0v)
    for y, hf in (oracle.ssd_fwd_seq(*args, h0), oracle.ssd_fwd_chunked(*args, 1, h0)):
        assert abs(y[0, 0, 0, 0] - expect_y) < 1e-15
        assert abs(hf[0, 0, 0, 0] - expect_h) < 1e-15
    yd, hd = oracle.ssd_step(np.full((1, 1, 1), xv), np.full((1, 1), dtv), np.array([Av]),
                             np.full((1, 1, 1), Bv), np.full((1, 1, 1), Cv), np.array([Dv]), h0)
    assert abs(yd[0, 0, 0] - expect_y) < 1e-15 and abs(hd[0, 0, 0, 0] - expect_h) < 1e-15


def read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = line.split()
                vals[k] = float(v)
    return vals


def test_ema_worked_example_printed_values():
    """[hard] Part 5 prints discretize(log(0.9)/0.5, -log(0.9), 0.5) = (0.9000, 0.0527).

    With S = H = 1, C = 1, D = 0 the oracle's one-step output exposes both
    discretised coefficients: with h0 = 1, x = 0 it returns exp(A dt); with
    h0 = 0, x = 1 it returns dt * B.
    """
    g = read_golden("ema_discretize.txt")
    alpha, delta, nd = g["alpha"], g["delta"], int(g["decimals"])
    A = np.array([math.log(alpha) / delta])
    Bv = -math.log(alpha)
    one = np.ones((1, 1, 1, 1))
    dt = np.full((1, 1, 1), delta)
    y_a, _ = oracle.ssd_fwd_seq(0 * one, dt, A, Bv * one, one, np.zeros(1), h0=one)
    y_b, _ = oracle.ssd_fwd_seq(one, dt, A, Bv * one, one, np.zeros(1))
    assert round(float(y_a[0, 0, 0, 0]), nd) == g["a_bar"]
    assert round(float(y_b[0, 0, 0, 0]), nd) == g["b_bar"]


def test_reduces_to_ema_loop():
    """[hard] Part 2: h = alpha h + (1 - alpha) x; y = h.  An S = H = 1 SSD with
    exp(A dt) = alpha and dt B = 1 - alpha, C = 1, D = 0 is that EMA."""
    alpha, delta, L = 0.9, 0.5, 128
    xs = np.arange(L, dtype=np.float64)
    h, ema = 0.0, []
    for k in range(L):
        h = alpha * h + (1 - alpha) * xs[k]
        ema.append(h)
    A = np.array([math.log(alpha) / delta])
    Bv = (1 - alpha) / delta
    x = xs.reshape(1, L, 1, 1)
    args = (x, np.full((1, L, 1), delta), A, np.full((1, L, 1, 1), Bv), np.ones((1, L, 1, 1)), np.zeros(1))
    for y, hf in (oracle.ssd_fwd_seq(*args), oracle.ssd_fwd_chunked(*args, 16)):
        assert relerr(y[0, :, 0, 0], np.array(ema)) < 1e-12
        assert abs(hf[0, 0, 0, 0] - ema[-1]) < 1e-9


def test_split_resume():
    """Feeding h_final of the first half as h0 of the second half equals one call
    ([blog] section "Kernel 2": the final state can seed the next call)."""
    rng = np.random.default_rng(21)
    x, dt, A, Bm, Cm, D, h0 = rand_problem(rng, 2, 40, 4, 3, 4, 2)
    y, hf = oracle.ssd_fwd_seq(x, dt, A, Bm, Cm, D, h0)
    for cut in (1, 16, 23):
        y1, h1 = oracle.ssd_fwd_chunked(x[:, :cut], dt[:, :cut], A, Bm[:, :cut], Cm[:, :cut], D, 8, h0)
        y2, h2 = oracle.ssd_fwd_chunked(x[:, cut:], dt[:, cut:], A, Bm[:, cut:], Cm[:, cut:], D, 8, h1)
        assert relerr(np.concatenate([y1, y2], axis=1), y) < 1e-12
        assert relerr(h2, hf) < 1e-12


def test_decode_steps_equal_forward():
    rng = np.random.default_rng(8)
    x, dt, A, Bm, Cm, D, h0 = rand_problem(rng, 2, 12, 4, 3, 5, 2)
    y, hf = oracle.ssd_fwd_seq(x, dt, A, Bm, Cm, D, h0)
    h = h0.copy()
    for t in range(x.shape[1]):
        yt, h = oracle.ssd_step(x[:, t], dt[:, t], A, Bm[:, t], Cm[:, t], D, h)
        assert relerr(yt, y[:, t]) < 1e-12
    assert relerr(h, hf) < 1e-12


def test_chunk_intermediates():
    """The chunked form's intermediates against their definitions:
    gcum is the inclusive in-chunk cumsum of A dt (restarting at each chunk);
    h_start[k] is the sequential state after the first k*T tokens;
    h_start[k+1] = exp(G_last,k) h_start[k] + s_local[k]."""
    rng = np.random.default_rng(31)
    batch, L, nh, H, S, G, T = 1, 45, 4, 3, 4, 2, 10
    x, dt, A, Bm, Cm, D, h0 = rand_problem(rng, batch, L, nh, H, S, G)
    y, hf, gc, s_loc, h_st = oracle.ssd_fwd_chunked(x, dt, A, Bm, Cm, D, T, h0, intermediates=True)
    nc = (L + T - 1) // T
    for h in range(nh):
        a = A[h] * dt[0, :, h]
        for k in range(nc):
            seg = a[k * T:(k + 1) * T]
            assert np.allclose(gc[0, h, k * T:(k + 1) * T], np.cumsum(seg), rtol=0, atol=1e-13)
    for k in range(nc):
        if k == 0:
            expect = h0
        else:
            _, expect = oracle.ssd_fwd_seq(x[:, :k * T], dt[:, :k * T], A, Bm[:, :k * T], Cm[:, :k * T], D, h0)
        assert relerr(h_st[:, :, k], expect) < 1e-12
    for k in range(nc):
        last = min(L, (k + 1) * T) - 1
        nxt = hf if k == nc - 1 else h_st[:, :, k + 1]
        decay = np.exp(gc[0, :, last])[None, :, None, None]
        assert relerr(decay * h_st[:, :, k] + s_loc[:, :, k], nxt) < 1e-12


def test_empty_sequence():
    rng = np.random.default_rng(1)
    x, dt, A, Bm, Cm, D, h0 = rand_problem(rng, 1, 0, 2, 3, 4, 1)
    y, hf = oracle.ssd_fwd_seq(x, dt, A, Bm, Cm, D, h0)
    assert y.shape == (1, 0, 2, 3) and np.array_equal(hf, h0)
    y, hf = oracle.ssd_fwd_chunked(x, dt, A, Bm, Cm, D, 4, None)
    assert np.array_equal(hf, np.zeros_like(h0))
