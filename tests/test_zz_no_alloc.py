"""ssd_fwd_noalloc: the forward pass for callers that cannot allocate device memory.

Such callers (code running during CUDA-graph capture, allocator-less runtimes,
plug-ins whose host application owns every device allocation) get an entry
point that takes no workspace and uses the library's own static device scratch
array instead.  This test calls it through the C ABI and checks it against
ssd_fwd (which uses a caller-provided workspace) on two calls in a row with
different inputs, so stale scratch contents from the first call would show up
in the second.  The file is named to be collected last.
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


def test_noalloc_matches_workspace_entry_point_twice():
    build()
    lib = _native.load()
    shapes = [
        workloads.custom(2, 1000, 8, 64, 128, 2, 256, "bf16", h0_recipe="normal", seed=71, name="na1"),
        workloads.custom(1, 777, 4, 64, 128, 1, 128, "bf16", dt_zero_frac=0.05, seed=72, name="na2"),
    ]
    for shape in shapes:
        inp = workloads.make_inputs(shape)
        d = {k: (None if v is None else v.cuda()) for k, v in inp.tensors().items()}
        desc = api.desc_for(d["x"], d["B"], shape.chunk)
        assert api.workspace_size(desc) <= 32 << 20
        y_ref, hf_ref = api.ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], shape.chunk, d["h0"])
        y = torch.full_like(y_ref, float("nan"))
        hf = torch.full_like(hf_ref, float("nan"))
        assert _call_noalloc(lib, desc, d, y, hf) == 0
        torch.cuda.synchronize()
        assert rel_max_err(y, y_ref) <= TOL["bf16"]
        assert rel_max_err(hf, hf_ref) <= TOL["bf16"]


def test_noalloc_rejects_problems_above_the_scratch_size():
    build()
    lib = _native.load()
    shape = workloads.WORKLOADS[2]      # needs far more than the 32 MiB static scratch
    desc = api.make_desc(shape.batch, shape.seqlen, shape.nheads, shape.headdim, shape.dstate, shape.ngroups,
                         shape.chunk, torch.bfloat16, torch.bfloat16)
    assert api.workspace_size(desc) > 32 << 20
    fake = 1 << 20   # rejected during validation, never dereferenced
    rc = lib.ssd_fwd_noalloc(ctypes.byref(desc), fake, fake, fake, fake, fake, fake, None, 1 << 34, None, None)
    assert rc == 5   # SSD_ERR_TOO_LARGE
