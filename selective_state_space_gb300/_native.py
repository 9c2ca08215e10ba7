"""ctypes view of libssd.so (include/ssd.h).  Loading fails loudly if the library
is missing: there is no other implementation to fall back to."""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libssd.so")

SSD_F32, SSD_BF16 = 0, 1
SSD_FLAG_FORCE_SIMT = 1
SSD_FLAG_EXPIRE_WAITS = 2   # test hook: every bounded device wait expires at once
SSD_DT_AS_INPUTS, SSD_DT_FLOAT32 = 0, 1   # ssd_desc.dt_dtype
NOALLOC_SCRATCH_BYTES = 32 << 20   # SSD_NOALLOC_SCRATCH_BYTES of include/ssd.h
STATUS = {0: "SSD_OK", 1: "SSD_ERR_INVALID_ARG", 2: "SSD_ERR_UNSUPPORTED", 3: "SSD_ERR_WORKSPACE",
          4: "SSD_ERR_CUDA", 5: "SSD_ERR_TOO_LARGE", 6: "SSD_ERR_TIMEOUT"}

# Every symbol include/ssd.h declares.
EXPORTS = ("ssd_status_string", "ssd_fwd_workspace_size", "ssd_fwd_path", "ssd_fwd_plan", "ssd_fwd", "ssd_fwd_timed",
           "ssd_fwd_check",
           "ssd_step",
           "ssd_chunk_cumsum", "ssd_chunk_state", "ssd_state_passing", "ssd_chunk_scan", "ssd_bwd_workspace_size",
           "ssd_bwd", "ssd_s6_fwd", "ssd_fwd_noalloc", "ssd_fwd_noalloc_check", "ssd_fwd_host_buffer_size",
           "ssd_fwd_host", "ssd_fwd_host_check")


class Desc(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("seqlen", ctypes.c_int64), ("nheads", ctypes.c_int64),
                ("headdim", ctypes.c_int64), ("dstate", ctypes.c_int64), ("ngroups", ctypes.c_int64),
                ("chunk", ctypes.c_int64), ("in_dtype", ctypes.c_int32), ("out_dtype", ctypes.c_int32),
                ("flags", ctypes.c_int32), ("dt_dtype", ctypes.c_int32)]


class S6Desc(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("seqlen", ctypes.c_int64), ("dim", ctypes.c_int64),
                ("dstate", ctypes.c_int64), ("ngroups", ctypes.c_int64), ("in_dtype", ctypes.c_int32),
                ("out_dtype", ctypes.c_int32), ("flags", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class Plan(ctypes.Structure):
    _fields_ = [("tensor_cores", ctypes.c_int32), ("super_tokens", ctypes.c_int32), ("n_super", ctypes.c_int32),
                ("split_sequences", ctypes.c_int32), ("tail_super_tokens", ctypes.c_int32),
                ("tail_n_super", ctypes.c_int32), ("kernel_launches", ctypes.c_int32), ("memsets", ctypes.c_int32)]


class SSDError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__(f"{fn} returned {STATUS.get(code, code)}")
        self.code = code


_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"libssd.so not built ({path}); run selective_state_space_gb300.build.build()")
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        DP = ctypes.POINTER(Desc)
        st = ctypes.c_int
        lib.ssd_status_string.argtypes = [st]
        lib.ssd_status_string.restype = ctypes.c_char_p
        lib.ssd_fwd_workspace_size.argtypes = [DP, ctypes.POINTER(ctypes.c_size_t)]
        lib.ssd_fwd_workspace_size.restype = st
        lib.ssd_fwd_path.argtypes = [DP, ctypes.POINTER(ctypes.c_int32)]
        lib.ssd_fwd_path.restype = st
        lib.ssd_fwd_plan.argtypes = [DP, ctypes.POINTER(Plan)]
        lib.ssd_fwd_plan.restype = st
        lib.ssd_fwd.argtypes = [DP] + [P] * 10 + [ctypes.c_size_t, P]
        lib.ssd_fwd.restype = st
        lib.ssd_fwd_timed.argtypes = [DP] + [P] * 10 + [ctypes.c_size_t, P, ctypes.POINTER(P)]
        lib.ssd_fwd_timed.restype = st
        lib.ssd_step.argtypes = [DP] + [P] * 9
        lib.ssd_step.restype = st
        lib.ssd_chunk_cumsum.argtypes = [DP, P, P, P, P]
        lib.ssd_chunk_cumsum.restype = st
        lib.ssd_chunk_state.argtypes = [DP, P, P, P, P, P, P]
        lib.ssd_chunk_state.restype = st
        lib.ssd_state_passing.argtypes = [DP, P, P, P, P, P, P]
        lib.ssd_state_passing.restype = st
        lib.ssd_chunk_scan.argtypes = [DP] + [P] * 9
        lib.ssd_chunk_scan.restype = st
        lib.ssd_fwd_check.argtypes = [P, P]
        lib.ssd_fwd_check.restype = st
        lib.ssd_fwd_noalloc.argtypes = [DP] + [P] * 9 + [P]
        lib.ssd_fwd_noalloc.restype = st
        lib.ssd_fwd_noalloc_check.argtypes = [P]
        lib.ssd_fwd_noalloc_check.restype = st
        lib.ssd_fwd_host_buffer_size.argtypes = [DP, ctypes.POINTER(ctypes.c_size_t)]
        lib.ssd_fwd_host_buffer_size.restype = st
        lib.ssd_fwd_host.argtypes = [DP] + [P] * 10 + [ctypes.c_size_t, P]
        lib.ssd_fwd_host.restype = st
        lib.ssd_fwd_host_check.argtypes = [P, P]
        lib.ssd_fwd_host_check.restype = st
        lib.ssd_bwd_workspace_size.argtypes = [DP, ctypes.POINTER(ctypes.c_size_t)]
        lib.ssd_bwd_workspace_size.restype = st
        lib.ssd_bwd.argtypes = [DP] + [P] * 17 + [ctypes.c_size_t, P]
        lib.ssd_bwd.restype = st
        lib.ssd_s6_fwd.argtypes = [ctypes.POINTER(S6Desc)] + [P] * 10
        lib.ssd_s6_fwd.restype = st
        _lib = lib
        return lib


def check(fn: str, code: int) -> None:
    if code != 0:
        raise SSDError(fn, code)
