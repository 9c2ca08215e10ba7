"""ssd_fwd_noalloc: the forward pass for callers that cannot allocate device memory.

Such callers -- code running while a CUDA graph is captured, runtimes without a device
allocator, plug-ins whose host application owns every device allocation -- get an entry
point that takes no workspace and uses the library's own static device scratch array
instead.  These tests call it through the C ABI and compare it with ssd_fwd (which uses a
caller-provided workspace): bit for bit when the plan adds nothing with atomics (one
memset per call: both run the same kernels on the same inputs, deterministically), else
within the bfloat16 bound of the parity tests.  Each shape is run twice in a row with fresh
inputs, so stale scratch contents from the first call would show up in the second.  The
file is named to be collected last.
"""
import ctypes

import pytest
import torch

from selective_state_space_gb300 import _native, api, workloads
from selective_state_space_gb300.build import build

from .helpers import TOL, rel_max_err

pytestmark = pytest.mark.gpu


def _call_noalloc(lib, desc, d, y, hf):
    ptr = lambda t: None if t is None else t.data_ptr()
    return lib.ssd_fwd_noalloc(ctypes.byref(desc), ptr(d["x"]), ptr(d["dt"]), ptr(d["A"]), ptr(d["B"]), ptr(d["C"]),
                               ptr(d["D"]), ptr(d["h0"]), ptr(y), ptr(hf),
                               torch.cuda.current_stream().cuda_stream)


def _check(lib):
    return lib.ssd_fwd_noalloc_check(torch.cuda.current_stream().cuda_stream)


# (shape, flags, whether h_final is asked for)
CASES = [
    (workloads.custom(2, 1000, 8, 64, 128, 2, 256, "bf16", h0_recipe="normal", seed=71, name="na-pair"), 0, True),
    (workloads.custom(1, 777, 4, 64, 128, 1, 128, "bf16", dt_zero_frac=0.05, seed=72, name="na-ragged"), 0, False),
    (workloads.custom(2, 300, 4, 64, 128, 2, 128, "bf16", h0_recipe="normal", seed=73, name="na-simt"),
     _native.SSD_FLAG_FORCE_SIMT, True),
]


@pytest.mark.parametrize("shape,flags,want_final", CASES, ids=lambda c: getattr(c, "name", str(c)))
def test_noalloc_matches_workspace_entry_point_bitwise(shape, flags, want_final):
    build()
    lib = _native.load()
    for rep in range(2):
        # fresh inputs for the second call of the same shape
        shape_r = workloads.custom(shape.batch, shape.seqlen, shape.nheads, shape.headdim, shape.dstate,
                                   shape.ngroups, shape.chunk, shape.dtype, h0_recipe=shape.h0_recipe,
                                   dt_zero_frac=shape.dt_zero_frac, seed=shape.seed + 100 * rep, name=shape.name)
        inp = workloads.make_inputs(shape_r)
        d = {k: (None if v is None else v.cuda()) for k, v in inp.tensors().items()}
        desc = api.desc_for(d["x"], d["B"], shape.chunk, flags=flags)
        assert api.workspace_size(desc) <= _native.NOALLOC_SCRATCH_BYTES
        deterministic = api.fwd_plan(desc)["memsets"] == 1
        y_ref, hf_ref = api.ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], shape.chunk, d["h0"],
                                    flags=flags, want_h_final=want_final, check_errors=True)
        y = torch.full_like(y_ref, float("nan"))
        hf = torch.full_like(hf_ref, float("nan")) if want_final else None
        assert _call_noalloc(lib, desc, d, y, hf) == 0
        assert _check(lib) == 0
        torch.cuda.synchronize()
        if deterministic:
            assert torch.equal(y, y_ref), (shape.name, rep)
            if want_final:
                assert torch.equal(hf, hf_ref), (shape.name, rep)
        else:
            assert rel_max_err(y, y_ref) <= TOL["bf16"], (shape.name, rep)
            if want_final:
                assert rel_max_err(hf, hf_ref) <= TOL["bf16"], (shape.name, rep)


def test_noalloc_rejects_problems_above_the_scratch_size():
    build()
    lib = _native.load()
    shape = workloads.WORKLOADS[2]      # needs far more than the 32 MiB static scratch
    desc = api.make_desc(shape.batch, shape.seqlen, shape.nheads, shape.headdim, shape.dstate, shape.ngroups,
                         shape.chunk, torch.bfloat16, torch.bfloat16)
    assert api.workspace_size(desc) > _native.NOALLOC_SCRATCH_BYTES
    fake = 1 << 20   # rejected during validation, never dereferenced
    rc = lib.ssd_fwd_noalloc(ctypes.byref(desc), fake, fake, fake, fake, fake, fake, None, 1 << 34, None, None)
    assert rc == 5   # SSD_ERR_TOO_LARGE
