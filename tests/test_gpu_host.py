"""ssd_fwd_host: the forward pass on host buffers, with the batch cut into slices whose copies
overlap the computation.  Compared element by element with the oracle (and with the device
entry point), over slice counts 1 to 4, ragged chunks, with and without h0 / h_final, a float32
dt, the CUDA-core path, the empty sequence, and the timeout report of a slice."""
import pytest
import torch

from selective_state_space_gb300 import _native, api, workloads

from .helpers import TOL, oracle_full, rel_max_err

pytestmark = pytest.mark.gpu

CASES = [
    (workloads.custom(4, 1024, 8, 64, 128, 2, 256, "bf16", h0_recipe="normal", seed=51, name="host-4-slices"), 0, None),
    (workloads.custom(3, 777, 4, 64, 128, 1, 128, "bf16", dt_zero_frac=0.05, seed=52, name="host-ragged-3"), 0, None),
    (workloads.custom(1, 512, 4, 128, 256, 1, 128, "bf16", h0_recipe="normal", seed=53, name="host-1-slice"), 0, None),
    (workloads.custom(2, 300, 4, 64, 128, 2, 128, "bf16", h0_recipe="normal", seed=54, name="host-simt"),
     _native.SSD_FLAG_FORCE_SIMT, None),
    (workloads.custom(2, 1024, 8, 64, 128, 2, 256, "bf16", seed=55, name="host-dt-f32"), 0, "f32"),
    (workloads.custom(2, 96, 4, 16, 32, 2, 32, "f32", h0_recipe="normal", seed=56, name="host-f32"), 0, None),
    (workloads.custom(2, 300, 4, 64, 64, 1, 64, "f32", seed=60, name="host-tf32"), 0, None),
]


def _pinned(t):
    return None if t is None else t.pin_memory()


@pytest.mark.parametrize("want_final", [True, False], ids=["with-final", "no-final"])
@pytest.mark.parametrize("shape,flags,dt_dtype", CASES, ids=lambda c: getattr(c, "name", str(c)))
def test_host_buffers_match_oracle(shape, flags, dt_dtype, want_final):
    inp = workloads.make_inputs(shape, dt_dtype=dt_dtype)
    t = {k: _pinned(v) for k, v in inp.tensors().items()}
    desc = api.desc_for(t["x"], t["B"], shape.chunk, flags=flags, dt=t["dt"])
    buf = torch.empty(api.host_buffer_size(desc), dtype=torch.uint8, device="cuda")
    y = torch.full(t["x"].shape, float("nan"), dtype=t["x"].dtype).pin_memory()
    hf = (torch.full((shape.batch, shape.nheads, shape.headdim, shape.dstate), float("nan")).pin_memory()
          if want_final else None)
    api.ssd_fwd_host(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], shape.chunk, t["h0"], y=y, h_final=hf,
                     device_buffer=buf, flags=flags, check_errors=True)
    y_ref, hf_ref = oracle_full(inp)
    tol = TOL[shape.dtype]
    assert rel_max_err(y, y_ref) <= tol
    if want_final:
        assert rel_max_err(hf, hf_ref) <= tol
    # the device entry point on the same inputs agrees to the same bound
    d = {k: (None if v is None else v.cuda()) for k, v in inp.tensors().items()}
    y_dev, hf_dev = api.ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], shape.chunk, d["h0"], flags=flags,
                                check_errors=True)
    assert rel_max_err(y, y_dev) <= tol


def test_host_buffers_twice_in_a_row_and_the_empty_sequence():
    shape = workloads.custom(4, 512, 8, 64, 128, 2, 256, "bf16", h0_recipe="normal", seed=57, name="host-twice")
    desc = api.make_desc(4, 512, 8, 64, 128, 2, 256, torch.bfloat16, torch.bfloat16)
    buf = torch.empty(api.host_buffer_size(desc), dtype=torch.uint8, device="cuda")
    for seed in (57, 157):                      # fresh inputs the second time: nothing stale is reused
        inp = workloads.make_inputs(shape, seed=seed)
        t = {k: _pinned(v) for k, v in inp.tensors().items()}
        y = torch.empty_like(t["x"]).pin_memory()
        hf = torch.empty((4, 8, 64, 128)).pin_memory()
        api.ssd_fwd_host(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], 256, t["h0"], y=y, h_final=hf,
                         device_buffer=buf, check_errors=True)
        y_ref, hf_ref = oracle_full(inp)
        assert rel_max_err(y, y_ref) <= TOL["bf16"] and rel_max_err(hf, hf_ref) <= TOL["bf16"]
    # L = 0: h_final is h0
    empty = workloads.custom(3, 0, 4, 64, 128, 1, 256, "bf16", h0_recipe="normal", seed=58, name="host-empty")
    inp = workloads.make_inputs(empty)
    t = {k: _pinned(v) for k, v in inp.tensors().items()}
    desc = api.desc_for(t["x"], t["B"], 256)
    buf = torch.empty(max(256, api.host_buffer_size(desc)), dtype=torch.uint8, device="cuda")
    y = torch.empty_like(t["x"]).pin_memory()
    hf = torch.full((3, 4, 64, 128), float("nan")).pin_memory()
    api.ssd_fwd_host(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], 256, t["h0"], y=y, h_final=hf,
                     device_buffer=buf, check_errors=True)
    assert torch.equal(hf, t["h0"])


def test_host_buffers_report_an_expired_wait_of_any_slice():
    shape = workloads.custom(4, 1024, 8, 64, 128, 2, 256, "bf16", seed=59, name="host-timeout")
    inp = workloads.make_inputs(shape)
    t = {k: _pinned(v) for k, v in inp.tensors().items()}
    desc = api.desc_for(t["x"], t["B"], shape.chunk)
    buf = torch.empty(api.host_buffer_size(desc), dtype=torch.uint8, device="cuda")
    y = torch.empty_like(t["x"]).pin_memory()
    lib = _native.load()
    stream = torch.cuda.current_stream()
    api.ssd_fwd_host(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], shape.chunk, y=y, device_buffer=buf,
                     flags=_native.SSD_FLAG_EXPIRE_WAITS)
    assert lib.ssd_fwd_host_check(buf.data_ptr(), stream.cuda_stream) == 6     # SSD_ERR_TIMEOUT
    api.ssd_fwd_host(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], shape.chunk, y=y, device_buffer=buf,
                     check_errors=True)
    y_ref, _ = oracle_full(inp)
    assert rel_max_err(y, y_ref) <= TOL["bf16"]
