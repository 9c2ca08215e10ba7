"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Small problems are compared on every element of y and h_final; the five
full-size layer shapes are compared element by element on sampled
(batch, head) pairs, which the oracle computes one by one, in the same launch
configuration bench.py times.  Bounds: max|got - ref| / max|ref| <= 1e-3 for
float32 inputs and <= 2e-2 for bfloat16 inputs (y and the final state).
"""
import numpy as np
import pytest
import torch

import oracle
from selective_state_space_gb300 import _native, api, workloads
from selective_state_space_gb300._native import SSD_FLAG_FORCE_SIMT

from .helpers import TOL, oracle_full, rel_max_err, to_dev

pytestmark = pytest.mark.gpu

PATHS = {"default": 0, "simt": SSD_FLAG_FORCE_SIMT}


def run_fwd(inp, flags=0, chunk=None):
    d = to_dev(inp)
    y, hf = api.ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], chunk or inp.shape.chunk, d["h0"],
                        flags=flags, check_errors=True)
    torch.cuda.synchronize()
    return y, hf


def tc_path(shape, flags=0):
    desc = api.make_desc(shape.batch, shape.seqlen, shape.nheads, shape.headdim, shape.dstate, shape.ngroups,
                         shape.chunk, workloads.torch_dtype(shape.dtype), workloads.torch_dtype(shape.dtype), flags)
    return api.uses_tensor_cores(desc)


# Shapes the oracle finishes in seconds; several 128-row tiles, several chunks and
# super-chunks, ragged tails, groups > 1, both state widths and both head widths.
SMALL = [
    workloads.WORKLOADS[0],
    workloads.custom(2, 512, 6, 64, 128, 1, 256, "bf16", h0_recipe="normal", seed=11, name="c1-small"),
    workloads.custom(1, 1536, 8, 64, 128, 2, 256, "bf16", dt_zero_frac=0.05, seed=12, name="c3-small"),
    workloads.custom(1, 700, 8, 64, 128, 2, 256, "bf16", dt_zero_frac=0.05, seed=12, name="c3-ragged"),
    workloads.custom(2, 384, 4, 128, 256, 2, 128, "bf16", dt_recipe="loguniform", a_range=(0.5, 8.0),
                     seed=13, name="c4-small"),
    workloads.custom(2, 300, 4, 128, 256, 2, 128, "bf16", dt_recipe="loguniform", a_range=(0.5, 8.0),
                     seed=13, name="c4-ragged"),
    workloads.custom(1, 640, 4, 64, 128, 1, 128, "bf16", h0_recipe="normal", seed=14, name="blog-small"),
    workloads.custom(1, 256, 2, 128, 128, 1, 256, "bf16", seed=17, name="h128-s128"),
    workloads.custom(1, 256, 2, 64, 256, 1, 128, "bf16", seed=18, name="h64-s256"),
    # three heads per group: the one-head-per-CTA scan kernel at S = 128, H = 64
    workloads.custom(2, 512, 6, 64, 128, 2, 256, "bf16", h0_recipe="normal", seed=19, name="odd-hpg"),
    # ragged lengths on the tensor-core path: a last chunk of 76 tokens (one short sub-chunk),
    # and a long sequence cut into super-chunks whose last chunk holds 64 tokens
    workloads.custom(2, 1100, 6, 64, 128, 1, 256, "bf16", h0_recipe="normal", seed=26, name="tc-ragged-76"),
    workloads.custom(1, 8000, 8, 64, 128, 2, 256, "bf16", seed=27, name="tc-ragged-super"),
    # L not a multiple of 4: chunk_state loads G and dt per thread (rows are not 16-byte aligned)
    workloads.custom(1, 3001, 4, 64, 128, 1, 128, "bf16", h0_recipe="normal", seed=28, name="tc-ragged-odd"),
    workloads.custom(2, 77, 6, 8, 16, 3, 16, "f32", h0_recipe="normal", seed=15, name="odd-f32"),
    workloads.custom(1, 33, 2, 1, 1, 1, 1, "f32", seed=16, name="scalar-T1"),
    # float32 inputs that take the kind::tf32 tensor-core kernel (H = 64, S = 64 or 128): ragged,
    # several sub-chunks, chunks shorter and longer than its 128-token sub-chunk, G > 1, dt = 0
    workloads.custom(2, 300, 4, 64, 64, 2, 64, "f32", h0_recipe="normal", seed=17, name="tf32-ragged"),
    workloads.custom(1, 520, 2, 64, 128, 1, 32, "f32", seed=18, name="tf32-s128"),
    workloads.custom(2, 384, 4, 64, 64, 1, 256, "f32", dt_zero_frac=0.1, h0_recipe="normal", seed=19,
                     name="tf32-hold"),
]


def test_tensor_core_path_selected_for_bf16_layer_shapes():
    for shape in workloads.WORKLOADS[1:] + [workloads.BLOG_SHAPE]:
        assert tc_path(shape), shape.name
        assert not tc_path(shape, SSD_FLAG_FORCE_SIMT)
    assert tc_path(workloads.WORKLOADS[0])       # float32 inputs of H = 64, S <= 128: kind::tf32
    assert not tc_path(workloads.WORKLOADS[0], SSD_FLAG_FORCE_SIMT)
    assert not tc_path(workloads.custom(1, 64, 2, 8, 16, 1, 16, "f32", name="f32-narrow"))
    # lengths that are not a multiple of the chunk stay on the tensor cores
    for shape in SMALL:
        if shape.name in ("c3-ragged", "c4-ragged", "tc-ragged-76", "tc-ragged-super", "tc-ragged-odd"):
            assert tc_path(shape), shape.name


@pytest.mark.parametrize("path", sorted(PATHS))
@pytest.mark.parametrize("shape", SMALL, ids=lambda s: s.name)
def test_fwd_small_all_elements(shape, path):
    inp = workloads.make_inputs(shape)
    y_ref, hf_ref = oracle_full(inp)
    y, hf = run_fwd(inp, PATHS[path])
    tol = TOL[shape.dtype]
    assert rel_max_err(y, y_ref) <= tol
    assert rel_max_err(hf, hf_ref) <= tol


@pytest.mark.parametrize("shape", workloads.WORKLOADS + [workloads.BLOG_SHAPE], ids=lambda s: s.name)
def test_fwd_full_size_all_elements(shape):
    """Every element of y and h_final at full size, in the launch configuration the bench
    times (the same plan: whole, cut and tail sequences, split-slice atomics), against the
    sequential oracle over the whole problem (a few seconds of the host's cores at most)."""
    inp = workloads.make_inputs(shape)
    y, hf = run_fwd(inp)
    y_ref, hf_ref = oracle_full(inp)
    tol = TOL[shape.dtype]
    assert rel_max_err(y, y_ref) <= tol
    assert rel_max_err(hf, hf_ref) <= tol


STAGE_SHAPES = [
    workloads.custom(2, 768, 4, 64, 128, 2, 256, "bf16", h0_recipe="normal", seed=21, name="stages-t256"),
    workloads.custom(1, 512, 2, 128, 256, 1, 128, "bf16", dt_recipe="loguniform", a_range=(0.5, 8.0),
                     h0_recipe="normal", seed=22, name="stages-wide"),
    workloads.custom(2, 640, 4, 64, 128, 2, 256, "bf16", h0_recipe="normal", seed=23, name="stages-ragged"),
]


@pytest.mark.parametrize("path", sorted(PATHS))
@pytest.mark.parametrize("shape", STAGE_SHAPES, ids=lambda s: s.name)
def test_stages_against_oracle_intermediates(shape, path):
    """Each stage of the pipeline on its own, against the oracle's chunked-form intermediates."""
    flags = PATHS[path]
    inp = workloads.make_inputs(shape)
    t = inp.tensors()
    y_ref, hf_ref, g_ref, s_ref, hs_ref = oracle.ssd_fwd_chunked(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"],
                                                                 shape.chunk, t["h0"], intermediates=True)
    d = to_dev(inp)
    T = shape.chunk
    G = api.ssd_chunk_cumsum(d["dt"], d["A"], T)
    torch.cuda.synchronize()
    # G holds log2(e) * cumsum; compare in natural-log units
    assert rel_max_err(G.double() * np.log(2.0), g_ref) <= 1e-5
    s_loc = api.ssd_chunk_state(d["x"], d["dt"], d["B"], G, T, flags=flags)
    torch.cuda.synchronize()
    assert rel_max_err(s_loc, s_ref) <= TOL["bf16"]
    h_start, h_final = api.ssd_state_passing(G, s_loc, T, torch.bfloat16, d["h0"], ngroups=shape.ngroups)
    torch.cuda.synchronize()
    assert rel_max_err(h_start, hs_ref) <= TOL["bf16"]
    assert rel_max_err(h_final, hf_ref) <= TOL["bf16"]
    # chunk_scan alone, fed the oracle's chunk-start states
    hs_dev = torch.from_numpy(hs_ref).float().cuda()
    y = api.ssd_chunk_scan(d["x"], d["dt"], d["B"], d["C"], d["D"], G, hs_dev, T, flags=flags)
    torch.cuda.synchronize()
    assert rel_max_err(y, y_ref) <= TOL["bf16"]


# dt in float32 beside bfloat16 x, B, C (SSD_DT_FLOAT32): the two-head scan with staged
# chunk_state (L a multiple of 4), and a ragged one-head shape whose chunk_state loads dt per
# thread (from the cumsum's bfloat16 copy)
DT_F32_SHAPES = [
    workloads.custom(2, 1024, 8, 64, 128, 2, 256, "bf16", h0_recipe="normal", seed=41, name="dtf32-pair"),
    workloads.custom(1, 1001, 4, 128, 128, 1, 128, "bf16", dt_zero_frac=0.05, seed=42, name="dtf32-ragged-h128"),
]


@pytest.mark.parametrize("path", sorted(PATHS))
@pytest.mark.parametrize("shape", DT_F32_SHAPES, ids=lambda s: s.name)
def test_fwd_float32_dt_beside_bfloat16_inputs(shape, path):
    inp = workloads.make_inputs(shape, dt_dtype="f32")
    assert inp.dt.dtype == torch.float32 and inp.x.dtype == torch.bfloat16
    d = to_dev(inp)
    desc = api.desc_for(d["x"], d["B"], shape.chunk, flags=PATHS[path], dt=d["dt"])
    assert desc.dt_dtype == _native.SSD_DT_FLOAT32
    y_ref, hf_ref = oracle_full(inp)          # the oracle sees the same float32 dt
    y, hf = run_fwd(inp, PATHS[path])
    assert rel_max_err(y, y_ref) <= TOL["bf16"]
    assert rel_max_err(hf, hf_ref) <= TOL["bf16"]
    # the cumsum runs on the float32 dt: G to 1e-5 of the oracle's in-chunk cumsum
    t = inp.tensors()
    _, _, g_ref, _, _ = oracle.ssd_fwd_chunked(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], shape.chunk,
                                               t["h0"], intermediates=True)
    G = api.ssd_chunk_cumsum(d["dt"], d["A"], shape.chunk)
    torch.cuda.synchronize()
    assert rel_max_err(G.double() * np.log(2.0), g_ref) <= 1e-5


@pytest.mark.parametrize("chunk", [16, 32, 64, 128, 256])
def test_chunk_size_invariance(chunk):
    shape = workloads.custom(1, 512, 4, 64, 128, 1, chunk, "bf16", h0_recipe="normal", seed=31)
    inp = workloads.make_inputs(shape)
    y_ref, hf_ref = oracle_full(inp)
    y, hf = run_fwd(inp)
    assert rel_max_err(y, y_ref) <= TOL["bf16"]
    assert rel_max_err(hf, hf_ref) <= TOL["bf16"]


def test_split_resume_on_gpu():
    shape = workloads.custom(2, 1024, 4, 64, 128, 1, 256, "bf16", h0_recipe="normal", seed=41)
    inp = workloads.make_inputs(shape)
    d = to_dev(inp)
    y, hf = api.ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], 256, d["h0"])
    cut = 512
    sl = lambda k, a, b: d[k][:, a:b].contiguous()
    y1, h1 = api.ssd_fwd(sl("x", 0, cut), sl("dt", 0, cut), d["A"], sl("B", 0, cut), sl("C", 0, cut), d["D"], 256,
                         d["h0"])
    y2, h2 = api.ssd_fwd(sl("x", cut, None), sl("dt", cut, None), d["A"], sl("B", cut, None), sl("C", cut, None),
                         d["D"], 256, h1)
    torch.cuda.synchronize()
    assert rel_max_err(torch.cat([y1, y2], 1), y) <= 1e-2
    assert rel_max_err(h2, hf) <= 1e-3


def test_empty_and_degenerate_sizes():
    dev = "cuda"
    # L = 0: nothing to scan, h_final = h0
    x = torch.zeros((2, 0, 4, 8), dtype=torch.bfloat16, device=dev)
    dt = torch.zeros((2, 0, 4), dtype=torch.bfloat16, device=dev)
    Bm = torch.zeros((2, 0, 2, 16), dtype=torch.bfloat16, device=dev)
    A = -torch.ones(4, device=dev)
    D = torch.ones(4, device=dev)
    h0 = torch.randn((2, 4, 8, 16), device=dev)
    y, hf = api.ssd_fwd(x, dt, A, Bm, Bm, D, 64, h0)
    torch.cuda.synchronize()
    assert y.shape == (2, 0, 4, 8) and torch.equal(hf, h0)
    y, hf = api.ssd_fwd(x, dt, A, Bm, Bm, D, 64, None)
    torch.cuda.synchronize()
    assert torch.count_nonzero(hf) == 0
    # batch = 0
    x = torch.zeros((0, 16, 4, 8), dtype=torch.bfloat16, device=dev)
    y, hf = api.ssd_fwd(x, torch.zeros((0, 16, 4), dtype=torch.bfloat16, device=dev), A,
                        torch.zeros((0, 16, 2, 16), dtype=torch.bfloat16, device=dev),
                        torch.zeros((0, 16, 2, 16), dtype=torch.bfloat16, device=dev), D, 8, None)
    assert y.numel() == 0 and hf.numel() == 0
    # L = 1 and dt = 0 everywhere (state held exactly)
    shape = workloads.custom(1, 1, 4, 64, 128, 1, 256, "bf16", h0_recipe="normal", seed=51)
    inp = workloads.make_inputs(shape)
    y_ref, hf_ref = oracle_full(inp)
    y, hf = run_fwd(inp)
    assert rel_max_err(y, y_ref) <= TOL["bf16"] and rel_max_err(hf, hf_ref) <= TOL["bf16"]
    inp.dt.zero_()
    y, hf = run_fwd(inp)
    assert torch.equal(hf.cpu(), inp.h0)


def test_decode_step_matches_oracle_and_forward():
    shape = workloads.custom(2, 24, 8, 64, 128, 2, 8, "bf16", h0_recipe="normal", seed=61)
    inp = workloads.make_inputs(shape)
    d = to_dev(inp)
    h = d["h0"].clone()
    h_ref = inp.h0.double().numpy()
    ys = []
    for t in range(shape.seqlen):
        args = [d["x"][:, t].contiguous(), d["dt"][:, t].contiguous(), d["A"], d["B"][:, t].contiguous(),
                d["C"][:, t].contiguous(), d["D"]]
        yt = api.ssd_step(*args, h)
        y_or, h_ref = oracle.ssd_step(inp.x[:, t], inp.dt[:, t], inp.A, inp.B[:, t], inp.C[:, t], inp.D, h_ref)
        torch.cuda.synchronize()
        assert rel_max_err(yt, y_or) <= TOL["bf16"]
        ys.append(yt)
    assert rel_max_err(h, h_ref) <= 1e-4   # the state stays float32 end to end
    y_fwd, hf = run_fwd(inp)
    assert rel_max_err(torch.stack(ys, 1), y_fwd.float()) <= TOL["bf16"]
    assert rel_max_err(h, hf) <= 1e-3


def test_decode_step_f32_large_batch():
    shape = workloads.custom(64, 1, 16, 64, 128, 4, 1, "f32", h0_recipe="normal", seed=62)
    inp = workloads.make_inputs(shape)
    d = to_dev(inp)
    h = d["h0"].clone()
    y = api.ssd_step(d["x"][:, 0].contiguous(), d["dt"][:, 0].contiguous(), d["A"], d["B"][:, 0].contiguous(),
                     d["C"][:, 0].contiguous(), d["D"], h)
    y_or, h_or = oracle.ssd_step(inp.x[:, 0], inp.dt[:, 0], inp.A, inp.B[:, 0], inp.C[:, 0], inp.D, inp.h0)
    torch.cuda.synchronize()
    assert rel_max_err(y, y_or) <= 1e-5 and rel_max_err(h, h_or) <= 1e-5


@pytest.mark.parametrize("dt_hot", [0.24, 1.0], ids=["decay-2^83-per-block", "decay-2^346-per-block"])
def test_fast_decay_blocks(dt_hot):
    """Runs of tokens whose 16-token blocks decay by 2^83 and 2^346 (dt = 0.24 and 1 with A
    near -16): the scan's factored decays must stay finite (no factor above 1 may be formed
    from a block's decay) and the masked entries must stay exactly zero."""
    shape = workloads.custom(2, 768, 4, 64, 128, 1, 256, "bf16", a_range=(14.0, 16.0), h0_recipe="normal",
                             seed=21, name="fast-decay")
    inp = workloads.make_inputs(shape)
    dt = inp.dt.float()
    dt[:, 100:180, :] = dt_hot          # spans two sub-chunks and a chunk boundary's neighbourhood
    dt[1, 300:310, 1] = dt_hot
    inp.dt = dt.to(inp.dt.dtype).contiguous()
    assert tc_path(shape)
    y_ref, hf_ref = oracle_full(inp)
    y, hf = run_fwd(inp)
    assert rel_max_err(y, y_ref) <= TOL["bf16"]
    assert rel_max_err(hf, hf_ref) <= TOL["bf16"]


@pytest.mark.parametrize("shape", [
    workloads.custom(2, 1024, 6, 64, 128, 1, 256, "bf16", h0_recipe="normal", seed=22, name="pair-h0"),
    workloads.custom(1, 2048, 4, 64, 128, 2, 128, "bf16", seed=23, name="pair-g2"),
    workloads.custom(2, 512, 6, 64, 128, 2, 256, "bf16", h0_recipe="normal", seed=24, name="single-hpg3"),
], ids=lambda s: s.name)
def test_without_final_state(shape):
    """Without h_final the scan skips the state update of each sequence's last sub-chunk:
    y must not change (bit for bit), on both tensor-core scan kernels."""
    inp = workloads.make_inputs(shape)
    d = to_dev(inp)
    y1, hf = api.ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], shape.chunk, d["h0"], check_errors=True)
    y2, none = api.ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], shape.chunk, d["h0"],
                           want_h_final=False, check_errors=True)
    torch.cuda.synchronize()
    assert none is None
    assert torch.equal(y1, y2)
    y_ref, hf_ref = oracle_full(inp)
    assert rel_max_err(y1, y_ref) <= TOL["bf16"]
    assert rel_max_err(hf, hf_ref) <= TOL["bf16"]


def test_plan_cuts_a_tail_for_the_pair_scan():
    """A layer whose head pairs leave a nearly empty last wave of scan CTAs: the plan cuts the
    last pairs into short super-chunks (chunk_state and state_passing for those sequences only),
    and the result still matches the oracle everywhere, and on each part at the cut."""
    shape = workloads.custom(4, 2048, 80, 64, 128, 1, 256, "bf16", h0_recipe="normal", seed=25, name="tail-cut")
    inp = workloads.make_inputs(shape)
    d = to_dev(inp)
    plan = api.fwd_plan(api.desc_for(d["x"], d["B"], shape.chunk))
    nseq = shape.batch * shape.nheads
    if plan["split_sequences"] >= nseq:
        pytest.skip("this GPU's SM count leaves no nearly empty last wave for this shape")
    assert plan["split_sequences"] % 2 == 0
    y, hf = run_fwd(inp)
    y_ref, hf_ref = oracle_full(inp)
    assert rel_max_err(y, y_ref) <= TOL["bf16"]
    assert rel_max_err(hf, hf_ref) <= TOL["bf16"]
    # and each part on its own: the last whole sequence and the first cut one
    split = plan["split_sequences"]
    for bh in (split - 1, split):
        b, h = divmod(bh, shape.nheads)
        assert rel_max_err(y[b, :, h], y_ref[b, :, h]) <= TOL["bf16"], (b, h)
        assert rel_max_err(hf[b, h], hf_ref[b, h]) <= TOL["bf16"], (b, h)
