"""The timeout path of the tensor-core forward kernels.

Every wait in those kernels for another warp's work is bounded; when one expires the
kernel records an error bit, every role stops, the copies and MMAs already issued are
waited for, and the CTA retires.  SSD_FLAG_EXPIRE_WAITS makes each such wait that is not
satisfied at once expire, so these tests drive that path on purpose, without a fault: the
call must report SSD_ERR_TIMEOUT through ssd_fwd_check, and the next normal call on the
same stream and workspace must run and match the call made before it.
"""
import ctypes

import pytest
import torch

from selective_state_space_gb300 import _native, api, workloads

from .helpers import TOL, rel_max_err, to_dev

pytestmark = pytest.mark.gpu

SSD_ERR_TIMEOUT = 6

# every tensor-core kernel: the two-head scan with chunk_state (S = 128, H = 64), the one-head
# scan with two C/B stages (H = 128) and with one (S = 256), and a ragged last chunk
CASES = [
    workloads.custom(2, 2048, 8, 64, 128, 1, 256, "bf16", h0_recipe="normal", seed=81, name="to-pair"),
    workloads.custom(1, 1024, 4, 128, 128, 1, 128, "bf16", seed=82, name="to-h128"),
    workloads.custom(1, 1024, 2, 64, 256, 1, 256, "bf16", seed=83, name="to-s256"),
    workloads.custom(1, 1000, 8, 64, 128, 2, 256, "bf16", seed=84, name="to-ragged"),
]


def _fwd(lib, desc, d, y, hf, ws):
    ptr = lambda t: None if t is None else t.data_ptr()
    return lib.ssd_fwd(ctypes.byref(desc), ptr(d["x"]), ptr(d["dt"]), ptr(d["A"]), ptr(d["B"]), ptr(d["C"]),
                       ptr(d["D"]), ptr(d["h0"]), ptr(y), ptr(hf), ptr(ws), ws.numel(),
                       torch.cuda.current_stream().cuda_stream)


def _check(lib, ws):
    return lib.ssd_fwd_check(ws.data_ptr(), torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("shape", CASES, ids=lambda s: s.name)
def test_expired_waits_report_timeout_and_leave_the_context_usable(shape):
    lib = _native.load()
    d = to_dev(workloads.make_inputs(shape))
    desc = api.desc_for(d["x"], d["B"], shape.chunk)
    plan = api.fwd_plan(desc)
    assert plan["tensor_cores"], "the case must run the tensor-core kernels"
    ws = api.alloc_workspace(desc, d["x"].device)
    y_ref = torch.empty_like(d["x"])
    hf_ref = torch.empty((shape.batch, shape.nheads, shape.headdim, shape.dstate), dtype=torch.float32,
                         device="cuda")
    assert _fwd(lib, desc, d, y_ref, hf_ref, ws) == 0 and _check(lib, ws) == 0

    expire = api.desc_for(d["x"], d["B"], shape.chunk, flags=_native.SSD_FLAG_EXPIRE_WAITS)
    y_bad, hf_bad = torch.zeros_like(y_ref), torch.zeros_like(hf_ref)
    assert _fwd(lib, expire, d, y_bad, hf_bad, ws) == 0
    assert _check(lib, ws) == SSD_ERR_TIMEOUT
    torch.cuda.synchronize()

    # the context is still usable: the same call again, on the same workspace
    y, hf = torch.full_like(y_ref, float("nan")), torch.full_like(hf_ref, float("nan"))
    assert _fwd(lib, desc, d, y, hf, ws) == 0 and _check(lib, ws) == 0
    torch.cuda.synchronize()
    if plan["memsets"] == 1:          # no atomics in the plan: the same kernels give the same bits
        assert torch.equal(y, y_ref) and torch.equal(hf, hf_ref)
    else:
        assert rel_max_err(y, y_ref) <= TOL["bf16"] and rel_max_err(hf, hf_ref) <= TOL["bf16"]


def test_expire_flag_is_ignored_by_the_cuda_core_path():
    """The CUDA-core kernels have no waits: the flag changes nothing there."""
    lib = _native.load()
    shape = workloads.custom(1, 512, 4, 64, 128, 1, 128, "bf16", seed=85, name="to-simt")
    d = to_dev(workloads.make_inputs(shape))
    flags = _native.SSD_FLAG_FORCE_SIMT
    y_ref, _ = api.ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], shape.chunk, flags=flags,
                           want_h_final=False, check_errors=True)
    y, _ = api.ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], shape.chunk, want_h_final=False,
                       flags=flags | _native.SSD_FLAG_EXPIRE_WAITS, check_errors=True)
    assert torch.equal(y, y_ref)
