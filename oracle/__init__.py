"""Double-precision CPU oracle for the Mamba-2 SSD forward pass, its gradients and the decode step.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The GPU library never
imports it, and it imports nothing from the GPU library.

The arithmetic lives in ``ssd_oracle.c`` (plain C, ``double``); this module
only builds it with gcc, loads it with ctypes and converts arrays to float64.
Formulas follow the NVIDIA developer blog "Accelerating Mamba-2 with
High-Performance Forward Pass Kernels in NVIDIA CUDA Tile", section
"Mamba-2 architecture" (recurrence, output line, log-space chunk jump and
chunk output).  The gradients follow "Sasha Rush: Mamba: The Hard Way",
Part 3 (the adjoint runs the same scan backwards), applied to that recurrence;
``bwd_chunked`` restates them per chunk as a second, independent form.
``s6_fwd_seq`` is the Mamba-1 selective scan of the same page, Part 5
(discretize, then the per-channel vector recurrence).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssd_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libssd_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ssd_oracle.c into oracle/_build/libssd_oracle.so with gcc."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    # -ffp-contract=off: keep every multiply and add separately rounded, as written.
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
           "-o", tmp, _SRC, "-lpthread", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            D = ctypes.POINTER(ctypes.c_double)
            i64 = ctypes.c_int64
            lib.oracle_ssd_fwd_seq.argtypes = [i64] * 6 + [D] * 9 + [ctypes.c_int]
            lib.oracle_ssd_fwd_seq.restype = ctypes.c_int
            lib.oracle_ssd_fwd_chunked.argtypes = [i64] * 7 + [D] * 12 + [ctypes.c_int]
            lib.oracle_ssd_fwd_chunked.restype = ctypes.c_int
            lib.oracle_ssd_step.argtypes = [i64] * 5 + [D] * 8
            lib.oracle_ssd_step.restype = ctypes.c_int
            lib.oracle_ssd_bwd_seq.argtypes = [i64] * 6 + [D] * 16 + [ctypes.c_int]
            lib.oracle_ssd_bwd_seq.restype = ctypes.c_int
            lib.oracle_s6_fwd_seq.argtypes = [i64] * 5 + [D] * 9
            lib.oracle_s6_fwd_seq.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(a):
    """Any array-like (numpy, torch CPU tensor of any float dtype) -> contiguous float64."""
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor: widen exactly (bf16 -> f32 -> f64 is exact)
        a = a.detach().to("cpu")
        import torch
        a = a.to(torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    if a is None:
        return ctypes.POINTER(ctypes.c_double)()
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def _shapes(x, Bm):
    batch, seqlen, nheads, H = x.shape
    ngroups, S = Bm.shape[2], Bm.shape[3]
    return batch, seqlen, nheads, H, S, ngroups


def ssd_fwd_seq(x, dt, A, Bm, Cm, D, h0=None, nthreads=None):
    """Sequential recurrence.  Returns (y [B,L,nh,H], h_final [B,nh,H,S]) in float64."""
    x, dt, A, Bm, Cm, D, h0 = map(_f64, (x, dt, A, Bm, Cm, D, h0))
    batch, seqlen, nheads, H, S, ngroups = _shapes(x, Bm)
    y = np.zeros((batch, seqlen, nheads, H))
    hf = np.zeros((batch, nheads, H, S))
    rc = _load().oracle_ssd_fwd_seq(batch, seqlen, nheads, H, S, ngroups,
                                    _ptr(x), _ptr(dt), _ptr(A), _ptr(Bm), _ptr(Cm), _ptr(D),
                                    _ptr(h0), _ptr(y), _ptr(hf),
                                    nthreads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_ssd_fwd_seq failed ({rc})")
    return y, hf


def ssd_fwd_chunked(x, dt, A, Bm, Cm, D, chunk, h0=None, nthreads=None, intermediates=False):
    """Chunked form (the blog's jump and chunk-output equations, natural exp).

    Returns (y, h_final) or, with ``intermediates=True``,
    (y, h_final, gcum [B,nh,L], s_local [B,nh,nc,H,S], h_start [B,nh,nc,H,S]).
    ``gcum`` is the in-chunk inclusive cumsum of A*dt in natural-log units.
    """
    x, dt, A, Bm, Cm, D, h0 = map(_f64, (x, dt, A, Bm, Cm, D, h0))
    batch, seqlen, nheads, H, S, ngroups = _shapes(x, Bm)
    nc = (seqlen + chunk - 1) // chunk
    y = np.zeros((batch, seqlen, nheads, H))
    hf = np.zeros((batch, nheads, H, S))
    g = s_loc = h_st = None
    if intermediates:
        g = np.zeros((batch, nheads, seqlen))
        s_loc = np.zeros((batch, nheads, nc, H, S))
        h_st = np.zeros((batch, nheads, nc, H, S))
    rc = _load().oracle_ssd_fwd_chunked(batch, seqlen, nheads, H, S, ngroups, chunk,
                                        _ptr(x), _ptr(dt), _ptr(A), _ptr(Bm), _ptr(Cm), _ptr(D),
                                        _ptr(h0), _ptr(y), _ptr(hf), _ptr(g), _ptr(s_loc),
                                        _ptr(h_st), nthreads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_ssd_fwd_chunked failed ({rc})")
    if intermediates:
        return y, hf, g, s_loc, h_st
    return y, hf


def ssd_step(x, dt, A, Bm, Cm, D, h):
    """One decode step.  x [B,nh,H], dt [B,nh], Bm/Cm [B,G,S], h [B,nh,H,S].

    Returns (y [B,nh,H], h_new [B,nh,H,S]); the input ``h`` is not modified.
    """
    x, dt, A, Bm, Cm, D = map(_f64, (x, dt, A, Bm, Cm, D))
    h = _f64(h).copy()
    batch, nheads, H = x.shape
    ngroups, S = Bm.shape[1], Bm.shape[2]
    y = np.zeros((batch, nheads, H))
    rc = _load().oracle_ssd_step(batch, nheads, H, S, ngroups, _ptr(x), _ptr(dt), _ptr(A),
                                 _ptr(Bm), _ptr(Cm), _ptr(D), _ptr(h), _ptr(y))
    if rc != 0:
        raise ValueError(f"oracle_ssd_step failed ({rc})")
    return y, h


def ssd_bwd_seq(x, dt, A, Bm, Cm, D, dy, h0=None, dh_final=None, nthreads=None):
    """Gradients of sum(dy * y) + sum(dh_final * h_final) (reverse mode of the recurrence).

    Returns a dict of float64 arrays: dx [B,L,nh,H], ddt [B,L,nh], dA [nh], dB, dC
    [B,L,G,S], dD [nh], dh0 [B,nh,H,S] (the gradient of the initial state, zeros or not).
    """
    x, dt, A, Bm, Cm, D, h0, dy, dh_final = map(_f64, (x, dt, A, Bm, Cm, D, h0, dy, dh_final))
    batch, seqlen, nheads, H, S, ngroups = _shapes(x, Bm)
    out = dict(dx=np.zeros_like(x), ddt=np.zeros_like(dt), dA=np.zeros(nheads),
               dB=np.zeros_like(Bm), dC=np.zeros_like(Cm), dD=np.zeros(nheads),
               dh0=np.zeros((batch, nheads, H, S)))
    rc = _load().oracle_ssd_bwd_seq(batch, seqlen, nheads, H, S, ngroups,
                                    _ptr(x), _ptr(dt), _ptr(A), _ptr(Bm), _ptr(Cm), _ptr(D),
                                    _ptr(h0), _ptr(dy), _ptr(dh_final),
                                    _ptr(out["dx"]), _ptr(out["ddt"]), _ptr(out["dA"]),
                                    _ptr(out["dB"]), _ptr(out["dC"]), _ptr(out["dD"]),
                                    _ptr(out["dh0"]), nthreads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_ssd_bwd_seq failed ({rc})")
    return out


def s6_fwd_seq(x, delta, A, Bm, Cm, D=None, h0=None):
    """Mamba-1 selective scan (S6).  x, delta [B, dim, L]; A [dim, N]; Bm, Cm [B, G, N, L];
    D [dim] or None; h0 [B, dim, N] or None.  Returns (y [B, dim, L], h_final [B, dim, N])."""
    x, delta, A, Bm, Cm, D, h0 = map(_f64, (x, delta, A, Bm, Cm, D, h0))
    batch, dim, seqlen = x.shape
    ngroups, N = Bm.shape[1], Bm.shape[2]
    y = np.zeros((batch, dim, seqlen))
    hf = np.zeros((batch, dim, N))
    rc = _load().oracle_s6_fwd_seq(batch, seqlen, dim, N, ngroups, _ptr(x), _ptr(delta), _ptr(A), _ptr(Bm),
                                   _ptr(Cm), _ptr(D), _ptr(h0), _ptr(y), _ptr(hf))
    if rc != 0:
        raise ValueError(f"oracle_s6_fwd_seq failed ({rc})")
    return y, hf
