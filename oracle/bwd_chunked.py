"""Gradients of the SSD forward pass in chunked form (second, independent CPU form; float64).

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``.  It restates the reverse
mode of "Sasha Rush: Mamba: The Hard Way", Part 3 (the adjoint is the same scan
run backwards; every coefficient's derivative pairs a forward and a backward
quantity) for the chunked form of the NVIDIA blog "Accelerating Mamba-2 with
High-Performance Forward Pass Kernels in NVIDIA CUDA Tile", section "Mamba-2
architecture".  Natural exp, no log2 scaling.  Its only use is to check
``oracle.ssd_bwd_seq`` against a different order of the same arithmetic.

Per (batch b, head h) and chunk k with tokens i, j (in-chunk G = inclusive
cumsum of a = A dt, G_last its last value, h_in the state entering the chunk,
Lam the gradient of the state leaving it):

  entering-state gradient  u_k = sum_i exp(G_i) dy_i C_i^T
  backwards over chunks    Lam_{k-1} = exp(G_last,k) Lam_k + u_k,  Lam_{nc-1} = dh_final,
                           dh0 = exp(G_last,0) Lam_0 + u_0
  Dec[i, j] = exp(G_i - G_j) for i >= j, else 0;   el_j = exp(G_last - G_j)
  v_j   = sum_i Dec[i,j] (C_i . B_j) dy_i + el_j Lam B_j        dx_j = dt_j v_j + D dy_j
  dB_j += dt_j (sum_i Dec[i,j] (dy_i . x_j) C_i + el_j Lam^T x_j)
  dC_i += exp(G_i) h_in^T dy_i + sum_j Dec[i,j] dt_j (dy_i . x_j) B_j
  M[i, j] = Dec[i,j] (C_i . B_j) dt_j (dy_i . x_j),  N_j = el_j dt_j x_j . (Lam B_j)
  dG_i  = exp(G_i) dy_i . (h_in C_i) + sum_j M[i,j] - sum_i' M[i',i] - N_i
          + [i last] (exp(G_last) <Lam, h_in> + sum_j N_j)
  da_t  = sum_{i >= t} dG_i,   ddt_t = x_t . v_t + A da_t,   dA += dt_t da_t
"""
from __future__ import annotations

import numpy as np

from . import _f64, _shapes, ssd_fwd_chunked


def ssd_bwd_chunked(x, dt, A, Bm, Cm, D, dy, chunk, h0=None, dh_final=None):
    """Same outputs as ``oracle.ssd_bwd_seq``, computed chunk by chunk."""
    x, dt, A, Bm, Cm, D, dy, h0, dh_final = map(_f64, (x, dt, A, Bm, Cm, D, dy, h0, dh_final))
    batch, L, nh, H, S, ng = _shapes(x, Bm)
    hpg = nh // ng
    nc = (L + chunk - 1) // chunk
    out = dict(dx=np.zeros_like(x), ddt=np.zeros_like(dt), dA=np.zeros(nh), dB=np.zeros_like(Bm),
               dC=np.zeros_like(Cm), dD=np.zeros(nh), dh0=np.zeros((batch, nh, H, S)))
    if L == 0:
        if dh_final is not None:
            out["dh0"][:] = dh_final
        return out
    # forward: in-chunk cumsums and the state entering each chunk
    _, _, gcum, _, h_start = ssd_fwd_chunked(x, dt, A, Bm, Cm, D, chunk, h0=h0, intermediates=True)
    for b in range(batch):
        for h in range(nh):
            g = h // hpg
            spans = [(k * chunk, min(L, (k + 1) * chunk)) for k in range(nc)]
            # gradient of each chunk's leaving state, chunk by chunk backwards
            lam = np.zeros((nc, H, S))
            run = np.zeros((H, S)) if dh_final is None else dh_final[b, h].copy()
            for k in range(nc - 1, -1, -1):
                t0, t1 = spans[k]
                G = gcum[b, h, t0:t1]
                lam[k] = run
                u = (dy[b, t0:t1, h].T * np.exp(G)) @ Cm[b, t0:t1, g]
                run = np.exp(G[-1]) * run + u
            out["dh0"][b, h] = run
            for k in range(nc):
                t0, t1 = spans[k]
                n = t1 - t0
                G = gcum[b, h, t0:t1]
                X, Y, dtk = x[b, t0:t1, h], dy[b, t0:t1, h], dt[b, t0:t1, h]
                Bk, Ck = Bm[b, t0:t1, g], Cm[b, t0:t1, g]
                hin, Lam = h_start[b, h, k], lam[k]
                ii, jj = np.meshgrid(np.arange(n), np.arange(n), indexing="ij")
                Dec = np.where(ii >= jj, np.exp(np.where(ii >= jj, G[:, None] - G[None, :], 0.0)), 0.0)
                el = np.exp(G[-1] - G)
                CB = Ck @ Bk.T                       # [i, j] = C_i . B_j
                YX = Y @ X.T                         # [i, j] = dy_i . x_j
                LamB = Bk @ Lam.T                    # [j, p] = (Lam B_j)_p
                v = (Dec * CB).T @ Y + el[:, None] * LamB
                out["dx"][b, t0:t1, h] = dtk[:, None] * v + D[h] * Y
                out["dB"][b, t0:t1, g] += dtk[:, None] * ((Dec * YX).T @ Ck + el[:, None] * (X @ Lam))
                w = Y @ hin                          # [i, s] = (h_in^T dy_i)_s
                out["dC"][b, t0:t1, g] += np.exp(G)[:, None] * w + (Dec * YX * dtk[None, :]) @ Bk
                M = Dec * CB * dtk[None, :] * YX
                N = el * dtk * np.sum(X * LamB, axis=1)
                dG = np.exp(G) * np.sum(w * Ck, axis=1) + M.sum(axis=1) - M.sum(axis=0) - N
                dG[-1] += np.exp(G[-1]) * np.sum(Lam * hin) + N.sum()
                da = np.cumsum(dG[::-1])[::-1]
                out["ddt"][b, t0:t1, h] = np.sum(X * v, axis=1) + A[h] * da
                out["dA"][h] += np.sum(dtk * da)
                out["dD"][h] += np.sum(Y * X)
    return out
