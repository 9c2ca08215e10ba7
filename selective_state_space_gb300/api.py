"""Thin torch-facing binding of libssd.so: argument marshalling only.

Every function here checks shapes, allocates outputs with torch (device
memory is PyTorch's job) and calls the C ABI of include/ssd.h, which runs
every step of the computation in CUDA kernels.  Tensors must live on a CUDA
device; there is no CPU path.
"""
from __future__ import annotations

import ctypes
from typing import Optional, Sequence

import torch

from . import _native
from ._native import Desc, SSD_BF16, SSD_F32, check

_DT = {torch.float32: SSD_F32, torch.bfloat16: SSD_BF16}


def _dtype_code(t: torch.dtype) -> int:
    if t not in _DT:
        raise TypeError(f"unsupported dtype {t}; use float32 or bfloat16")
    return _DT[t]


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors must be on a CUDA device (no CPU implementation exists)")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def make_desc(batch, seqlen, nheads, headdim, dstate, ngroups, chunk, in_dtype, out_dtype,
              flags: int = 0, dt_dtype: int = 0) -> Desc:
    d = Desc()
    d.batch, d.seqlen, d.nheads, d.headdim = batch, seqlen, nheads, headdim
    d.dstate, d.ngroups, d.chunk = dstate, ngroups, chunk
    d.in_dtype = _dtype_code(in_dtype) if isinstance(in_dtype, torch.dtype) else int(in_dtype)
    d.out_dtype = _dtype_code(out_dtype) if isinstance(out_dtype, torch.dtype) else int(out_dtype)
    d.flags, d.dt_dtype = flags, dt_dtype
    return d


def desc_for(x: torch.Tensor, Bm: torch.Tensor, chunk: int, out_dtype=None, flags: int = 0, dt=None) -> Desc:
    """The descriptor of a forward pass on these tensors; a float32 ``dt`` beside bfloat16
    ``x`` selects SSD_DT_FLOAT32."""
    batch, seqlen, nheads, headdim = x.shape
    ngroups, dstate = Bm.shape[2], Bm.shape[3]
    dt_dtype = (_native.SSD_DT_FLOAT32 if dt is not None and dt.dtype == torch.float32 and x.dtype == torch.bfloat16
                else _native.SSD_DT_AS_INPUTS)
    return make_desc(batch, seqlen, nheads, headdim, dstate, ngroups, chunk, x.dtype,
                     out_dtype or x.dtype, flags, dt_dtype)


def workspace_size(desc: Desc) -> int:
    n = ctypes.c_size_t(0)
    check("ssd_fwd_workspace_size", _native.load().ssd_fwd_workspace_size(ctypes.byref(desc), ctypes.byref(n)))
    return int(n.value)


def uses_tensor_cores(desc: Desc) -> bool:
    v = ctypes.c_int32(0)
    check("ssd_fwd_path", _native.load().ssd_fwd_path(ctypes.byref(desc), ctypes.byref(v)))
    return bool(v.value)


def fwd_plan(desc: Desc) -> dict:
    """How ssd_fwd runs ``desc`` on the current device (ssd_fwd_plan): path, tokens per
    super-chunk and super-chunks per sequence for the first ``split_sequences`` sequences
    and for the rest (``tail_*``), kernel launches and memsets per call."""
    p = _native.Plan()
    check("ssd_fwd_plan", _native.load().ssd_fwd_plan(ctypes.byref(desc), ctypes.byref(p)))
    return {name: (bool(getattr(p, name)) if name == "tensor_cores" else int(getattr(p, name)))
            for name, _ in _native.Plan._fields_}


def alloc_workspace(desc: Desc, device) -> torch.Tensor:
    n = workspace_size(desc)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device)


def ssd_fwd(x, dt, A, B, C, D, chunk: int, h0=None, *, y=None, h_final=None, want_h_final=True,
            workspace=None, out_dtype=None, flags: int = 0, stream=None, events: Sequence = None,
            check_errors: bool = False):
    """Chunked SSD forward.  Returns (y, h_final or None).

    x [B,L,nh,H], dt [B,L,nh], B/C [B,L,G,S] in float32 or bfloat16 (same dtype; dt may
    also be float32 beside bfloat16 x, B, C);
    A, D [nh] float32; h0 [B,nh,H,S] float32 or None.  ``events`` (8 CUDA events)
    selects ssd_fwd_timed, which records them around the four stages.
    ``check_errors`` synchronises and raises if a bounded device wait expired.
    """
    desc = desc_for(x, B, chunk, out_dtype, flags, dt)
    batch, seqlen, nheads, headdim = x.shape
    dstate = B.shape[3]
    if y is None:
        y = torch.empty((batch, seqlen, nheads, headdim), dtype=out_dtype or x.dtype, device=x.device)
    if h_final is None and want_h_final:
        h_final = torch.empty((batch, nheads, headdim, dstate), dtype=torch.float32, device=x.device)
    if workspace is None:
        workspace = alloc_workspace(desc, x.device)
    args = [ctypes.byref(desc), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(h0), _ptr(y),
            _ptr(h_final), _ptr(workspace), workspace.numel(), _stream(stream)]
    lib = _native.load()
    if events is None:
        check("ssd_fwd", lib.ssd_fwd(*args))
    else:
        arr = (ctypes.c_void_p * 8)(*[e.cuda_event for e in events])
        check("ssd_fwd_timed", lib.ssd_fwd_timed(*args, arr))
    if check_errors:
        check("ssd_fwd_check", lib.ssd_fwd_check(_ptr(workspace), _stream(stream)))
    return y, h_final


def host_buffer_size(desc: Desc) -> int:
    n = ctypes.c_size_t(0)
    check("ssd_fwd_host_buffer_size",
          _native.load().ssd_fwd_host_buffer_size(ctypes.byref(desc), ctypes.byref(n)))
    return int(n.value)


def _host_ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if t.is_cuda:
        raise ValueError("ssd_fwd_host takes host tensors")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def ssd_fwd_host(x, dt, A, B, C, D, chunk: int, h0=None, *, y, h_final=None, device_buffer, out_dtype=None,
                 flags: int = 0, stream=None, check_errors: bool = False):
    """Chunked SSD forward on host tensors (ssd_fwd_host): inputs read from, y and h_final
    written to host memory (pinned memory lets the copies overlap the computation);
    ``device_buffer`` is a device tensor of ``host_buffer_size(desc)`` bytes.  Only enqueues
    on ``stream``; synchronise it (or pass ``check_errors``) before reading y."""
    desc = desc_for(x, B, chunk, out_dtype, flags, dt)
    lib = _native.load()
    check("ssd_fwd_host", lib.ssd_fwd_host(ctypes.byref(desc), _host_ptr(x), _host_ptr(dt), _host_ptr(A),
                                           _host_ptr(B), _host_ptr(C), _host_ptr(D), _host_ptr(h0), _host_ptr(y),
                                           _host_ptr(h_final), _ptr(device_buffer), device_buffer.numel(),
                                           _stream(stream)))
    if check_errors:
        check("ssd_fwd_host_check", lib.ssd_fwd_host_check(_ptr(device_buffer), _stream(stream)))
    return y, h_final


def ssd_step(x, dt, A, B, C, D, h, *, y=None, out_dtype=None, stream=None):
    """One decode step.  x [B,nh,H], dt [B,nh], B/C [B,G,S], h [B,nh,H,S] float32 (updated in place).
    Returns y [B,nh,H]."""
    batch, nheads, headdim = x.shape
    ngroups, dstate = B.shape[1], B.shape[2]
    desc = make_desc(batch, 1, nheads, headdim, dstate, ngroups, 1, x.dtype, out_dtype or x.dtype)
    if y is None:
        y = torch.empty((batch, nheads, headdim), dtype=out_dtype or x.dtype, device=x.device)
    check("ssd_step", _native.load().ssd_step(ctypes.byref(desc), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C),
                                              _ptr(D), _ptr(h), _ptr(y), _stream(stream)))
    return y


def bwd_workspace_size(desc: Desc) -> int:
    n = ctypes.c_size_t(0)
    check("ssd_bwd_workspace_size", _native.load().ssd_bwd_workspace_size(ctypes.byref(desc), ctypes.byref(n)))
    return int(n.value)


def ssd_bwd(x, dt, A, B, C, D, dy, chunk: int, h0=None, dh_final=None, *, want_dh0=True, workspace=None,
            stream=None):
    """Gradients of sum(dy * y) + sum(dh_final * h_final) for the forward pass of ``ssd_fwd``.

    Same input layouts as ``ssd_fwd``; dy has the layout and dtype of x (the gradient
    pass needs the output dtype equal to the input dtype).  Returns a dict with dx, ddt,
    dB, dC (the input dtype), dA, dD [nh] float32 and dh0 [B,nh,H,S] float32 (or None).
    """
    desc = desc_for(x, B, chunk, None, 0)
    batch, seqlen, nheads, headdim = x.shape
    dstate = B.shape[3]
    out = {"dx": torch.empty_like(x), "ddt": torch.empty_like(dt), "dB": torch.empty_like(B),
           "dC": torch.empty_like(C), "dA": torch.empty(nheads, dtype=torch.float32, device=x.device),
           "dD": torch.empty(nheads, dtype=torch.float32, device=x.device),
           "dh0": torch.empty((batch, nheads, headdim, dstate), dtype=torch.float32, device=x.device)
           if want_dh0 else None}
    if workspace is None:
        workspace = torch.empty(max(bwd_workspace_size(desc), 256), dtype=torch.uint8, device=x.device)
    check("ssd_bwd", _native.load().ssd_bwd(
        ctypes.byref(desc), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(h0), _ptr(dy),
        _ptr(dh_final), _ptr(out["dx"]), _ptr(out["ddt"]), _ptr(out["dA"]), _ptr(out["dB"]), _ptr(out["dC"]),
        _ptr(out["dD"]), _ptr(out["dh0"]), _ptr(workspace), workspace.numel(), _stream(stream)))
    return out


def s6_fwd(x, delta, A, B, C, D=None, h0=None, *, y=None, want_h_final=True, out_dtype=None, stream=None):
    """Mamba-1 selective scan (S6).  x, delta [B, dim, L] (float32 or bfloat16, same dtype);
    A [dim, N] float32; B, C [B, G, N, L] (input dtype); D [dim] float32 or None;
    h0 [B, dim, N] float32 or None.  Returns (y [B, dim, L], h_final [B, dim, N] or None)."""
    batch, dim, seqlen = x.shape
    ngroups, dstate = B.shape[1], B.shape[2]
    d = _native.S6Desc()
    d.batch, d.seqlen, d.dim, d.dstate, d.ngroups = batch, seqlen, dim, dstate, ngroups
    d.in_dtype = _dtype_code(x.dtype)
    d.out_dtype = _dtype_code(out_dtype or x.dtype)
    d.flags = d.reserved = 0
    if y is None:
        y = torch.empty((batch, dim, seqlen), dtype=out_dtype or x.dtype, device=x.device)
    h_final = torch.empty((batch, dim, dstate), dtype=torch.float32, device=x.device) if want_h_final else None
    check("ssd_s6_fwd", _native.load().ssd_s6_fwd(ctypes.byref(d), _ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                                          _ptr(h0), _ptr(y), _ptr(h_final), _stream(stream)))
    return y, h_final


# ---- the four stages, one call each (intermediate layouts in include/ssd.h) ----

def ssd_chunk_cumsum(dt, A, chunk: int, desc: Desc = None, *, G=None, stream=None):
    batch, seqlen, nheads = dt.shape
    if desc is None:
        desc = make_desc(batch, seqlen, nheads, 1, 1, 1, chunk, dt.dtype, dt.dtype)
    if G is None:
        G = torch.empty((batch, nheads, seqlen), dtype=torch.float32, device=dt.device)
    check("ssd_chunk_cumsum", _native.load().ssd_chunk_cumsum(ctypes.byref(desc), _ptr(dt), _ptr(A), _ptr(G),
                                                              _stream(stream)))
    return G


def ssd_chunk_state(x, dt, B, G, chunk: int, *, s_local=None, flags: int = 0, stream=None):
    desc = desc_for(x, B, chunk, None, flags)
    batch, seqlen, nheads, headdim = x.shape
    nc = (seqlen + chunk - 1) // chunk
    if s_local is None:
        s_local = torch.empty((batch, nheads, nc, headdim, B.shape[3]), dtype=torch.float32, device=x.device)
    check("ssd_chunk_state", _native.load().ssd_chunk_state(ctypes.byref(desc), _ptr(x), _ptr(dt), _ptr(B), _ptr(G),
                                                            _ptr(s_local), _stream(stream)))
    return s_local


def ssd_state_passing(G, s_local, chunk: int, in_dtype, h0=None, *, ngroups: int = 1, h_start=None,
                      want_h_final=True, stream=None):
    batch, nheads, nc, headdim, dstate = s_local.shape
    seqlen = G.shape[2]
    desc = make_desc(batch, seqlen, nheads, headdim, dstate, ngroups, chunk, in_dtype, in_dtype)
    if h_start is None:
        h_start = torch.empty(s_local.shape, dtype=torch.float32, device=s_local.device)
    h_final = torch.empty((batch, nheads, headdim, dstate), dtype=torch.float32,
                          device=s_local.device) if want_h_final else None
    check("ssd_state_passing", _native.load().ssd_state_passing(ctypes.byref(desc), _ptr(G), _ptr(s_local), _ptr(h0),
                                                                _ptr(h_start), _ptr(h_final), _stream(stream)))
    return h_start, h_final


def ssd_chunk_scan(x, dt, B, C, D, G, h_start, chunk: int, *, y=None, out_dtype=None, flags: int = 0,
                   stream=None):
    desc = desc_for(x, B, chunk, out_dtype, flags)
    if y is None:
        y = torch.empty(x.shape, dtype=out_dtype or x.dtype, device=x.device)
    check("ssd_chunk_scan", _native.load().ssd_chunk_scan(ctypes.byref(desc), _ptr(x), _ptr(dt), _ptr(B), _ptr(C),
                                                          _ptr(D), _ptr(G), _ptr(h_start), _ptr(y), _stream(stream)))
    return y
