"""Host-side checks of libssd.so that need no GPU: the library loads, exports every
symbol include/ssd.h declares, and rejects bad arguments before launching anything.

The invalid-argument calls below return during validation, before any CUDA
call; the pointers passed are never dereferenced.
"""
import ctypes
import os
import re

import pytest

from selective_state_space_gb300 import _native
from selective_state_space_gb300.build import build

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "ssd.h")


@pytest.fixture(scope="module")
def lib():
    build()
    return _native.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(ssd_\w+)\s*\(", text, flags=re.M)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 10
    assert sorted(names) == sorted(_native.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code in range(7):
        s = lib.ssd_status_string(code).decode()
        assert s.startswith(_native.STATUS[code])
    assert lib.ssd_status_string(99).decode() == "unknown ssd_status"


def desc(**kw):
    d = _native.Desc()
    base = dict(batch=2, seqlen=512, nheads=8, headdim=64, dstate=128, ngroups=2, chunk=256,
                in_dtype=_native.SSD_BF16, out_dtype=_native.SSD_BF16, flags=0, dt_dtype=0)
    base.update(kw)
    for k, v in base.items():
        setattr(d, k, v)
    return d


def ws_size(lib, d):
    n = ctypes.c_size_t(0)
    rc = lib.ssd_fwd_workspace_size(ctypes.byref(d), ctypes.byref(n))
    return rc, n.value


def test_workspace_size_arithmetic(lib):
    rc, n = ws_size(lib, desc())
    assert rc == 0
    B, L, nh, H, S, T = 2, 512, 8, 64, 128, 256
    nc = (L + T - 1) // T
    al = lambda v: (v + 255) // 256 * 256
    # error word + G + local states + chunk-start states (float32)
    assert n == 256 + 2 * al(4 * B * nh * L) + 2 * al(4 * B * nh * nc * H * S)
    rc, n = ws_size(lib, desc(seqlen=0))
    assert rc == 0 and n == 0
    rc, n = ws_size(lib, desc(seqlen=513))   # ragged: one more chunk
    assert rc == 0 and n > ws_size(lib, desc())[1]


@pytest.mark.parametrize("bad,code", [
    (dict(ngroups=3), 1), (dict(nheads=-1), 1), (dict(headdim=0), 1), (dict(dstate=0), 1),
    (dict(chunk=0), 1), (dict(seqlen=-5), 1), (dict(in_dtype=7), 1), (dict(out_dtype=-1), 1),
    (dict(flags=1 << 8), 1), (dict(dt_dtype=2), 1), (dict(dt_dtype=-1), 1),
    (dict(dstate=257), 2), (dict(headdim=2048), 2), (dict(chunk=4096), 2),
])
def test_bad_descriptors_rejected(lib, bad, code):
    rc, _ = ws_size(lib, desc(**bad))
    assert rc == code
    d = desc(**bad)
    fake = 1 << 20     # 256-byte aligned, never dereferenced
    rc = lib.ssd_fwd(ctypes.byref(d), fake, fake, fake, fake, fake, fake, None, fake * 2, None, fake * 4,
                     1 << 40, None)
    assert rc == code


def test_null_and_misaligned_pointers_rejected(lib):
    d = desc()
    a = 1 << 20
    args = [a, a, a, a, a, a, None, 1 << 30, None, 1 << 34, 1 << 40, None]
    for i in (0, 1, 2, 3, 4, 5, 7):      # required pointers
        bad = list(args)
        bad[i] = None
        assert lib.ssd_fwd(ctypes.byref(d), *bad) == 1, i
    bad = list(args)
    bad[0] = a + 2                        # x not 16-byte aligned
    assert lib.ssd_fwd(ctypes.byref(d), *bad) == 1
    bad = list(args)
    bad[7] = a                            # y overlaps x
    assert lib.ssd_fwd(ctypes.byref(d), *bad) == 1
    bad = list(args)
    bad[9] = None                         # no workspace
    assert lib.ssd_fwd(ctypes.byref(d), *bad) == 3
    bad = list(args)
    bad[10] = 1024                        # workspace too small
    assert lib.ssd_fwd(ctypes.byref(d), *bad) == 3
    bad = list(args)
    bad[9] = (1 << 34) + 128              # workspace misaligned
    assert lib.ssd_fwd(ctypes.byref(d), *bad) == 3


def test_step_and_stage_validation(lib):
    d = desc(ngroups=3)
    a = 1 << 20
    assert lib.ssd_step(ctypes.byref(d), a, a, a, a, a, a, a, a, None) == 1
    assert lib.ssd_chunk_cumsum(ctypes.byref(d), a, a, a, None) == 1
    d = desc()
    assert lib.ssd_step(ctypes.byref(d), None, a, a, a, a, a, a, a, None) == 1
    assert lib.ssd_chunk_state(ctypes.byref(d), a, a, a, a, None, None) == 1
    assert lib.ssd_chunk_scan(ctypes.byref(d), a, a, a, a, a, a, a, None, None) == 1
    assert lib.ssd_state_passing(ctypes.byref(d), a, a, None, a, None, None) == 1   # s_local overlaps h_start
    iv = ctypes.c_int32(-1)
    assert lib.ssd_fwd_path(ctypes.byref(d), ctypes.byref(iv)) == 0 and iv.value in (0, 1)
    assert lib.ssd_fwd_path(ctypes.byref(d), None) == 1


def test_fwd_plan_is_consistent(lib):
    """ssd_fwd_plan: host-side query; the plan must be self-consistent for every path."""
    P = _native.Plan
    # bf16 layer shape on the tensor-core path: nc = 16 chunks of 256 tokens
    d = desc(batch=4, seqlen=4096, nheads=80, headdim=64, dstate=128, ngroups=1, chunk=256,
             in_dtype=_native.SSD_BF16, out_dtype=_native.SSD_BF16)
    p = P()
    assert lib.ssd_fwd_plan(ctypes.byref(d), ctypes.byref(p)) == 0
    assert p.tensor_cores == 1
    nc, nseq, L, T = 16, 4 * 80, 4096, 256
    for tokens, nsup in ((p.super_tokens, p.n_super), (p.tail_super_tokens, p.tail_n_super)):
        assert tokens % T == 0 and T <= tokens <= L          # whole chunks
        assert nsup == -(-L // tokens) and 1 <= nsup <= nc
    assert 0 < p.split_sequences <= nseq
    # the split falls on a whole chunk_state head group (4 heads of one group here)
    assert p.split_sequences % 4 == 0
    parts = [(p.split_sequences, p.n_super), (nseq - p.split_sequences, p.tail_n_super)]
    assert p.kernel_launches == 2 + sum(2 for n, ns in parts if n > 0 and ns > 1)
    assert 1 <= p.memsets <= 3
    # the same shape asks for the same plan
    q = P()
    assert lib.ssd_fwd_plan(ctypes.byref(d), ctypes.byref(q)) == 0 and bytes(q) == bytes(p)
    # forced CUDA-core path: one chunk per super-chunk, four stages, no split
    d.flags = 1
    assert lib.ssd_fwd_plan(ctypes.byref(d), ctypes.byref(p)) == 0
    assert (p.tensor_cores, p.super_tokens, p.n_super, p.kernel_launches, p.memsets) == (0, T, nc, 4, 1)
    assert (p.split_sequences, p.tail_super_tokens, p.tail_n_super) == (nseq, T, nc)
    # float32 inputs of H = 64, S <= 128: one kind::tf32 launch walking every sequence whole
    d = desc(in_dtype=_native.SSD_F32, out_dtype=_native.SSD_F32, dstate=64, chunk=64)
    assert lib.ssd_fwd_plan(ctypes.byref(d), ctypes.byref(p)) == 0
    assert (p.tensor_cores, p.n_super, p.super_tokens, p.kernel_launches, p.memsets) == (1, 1, 512, 1, 1)
    d.flags = 1
    assert lib.ssd_fwd_plan(ctypes.byref(d), ctypes.byref(p)) == 0 and p.tensor_cores == 0
    # empty sequence: nothing launched
    d = desc(seqlen=0)
    assert lib.ssd_fwd_plan(ctypes.byref(d), ctypes.byref(p)) == 0 and p.kernel_launches == 0
    assert lib.ssd_fwd_plan(ctypes.byref(d), None) == 1


def test_timed_variant_requires_events(lib):
    d = desc()
    a = 1 << 20
    assert lib.ssd_fwd_timed(ctypes.byref(d), a, a, a, a, a, a, None, 1 << 30, None, 1 << 34, 1 << 40, None,
                             None) == 1


# ---- gradient pass and selective scan: host-side validation (nothing is launched) ----

def bwd_ws(lib, d):
    n = ctypes.c_size_t(0)
    rc = lib.ssd_bwd_workspace_size(ctypes.byref(d), ctypes.byref(n))
    return rc, n.value


def test_bwd_workspace_size(lib):
    B, L, nh, H, S, G, T = 2, 512, 8, 64, 128, 2, 256
    rc, n = bwd_ws(lib, desc())
    assert rc == 0
    nc = (L + T - 1) // T
    al = lambda v: (v + 255) // 256 * 256
    # G, the entering states and their gradients, six per-token arrays, two partial sums (>= 1 slice)
    fixed = 7 * al(4 * B * nh * L) + 2 * al(4 * B * nh * nc * H * S)
    part = al(4 * B * L * G * S)
    assert n >= fixed + 2 * part and (n - fixed) % (2 * 256) == 0
    slices = (n - fixed) // 2 // 4 // (B * L * G * S)
    assert 1 <= slices <= nh // G
    assert bwd_ws(lib, desc(seqlen=0)) == (0, 0)
    assert bwd_ws(lib, desc(seqlen=513))[1] > n
    for bad in (dict(chunk=512), dict(headdim=256), dict(out_dtype=_native.SSD_F32)):
        assert bwd_ws(lib, desc(**bad))[0] == 2, bad
    assert bwd_ws(lib, desc(ngroups=3))[0] == 1
    assert lib.ssd_bwd_workspace_size(ctypes.byref(desc()), None) == 1


def test_bwd_argument_validation(lib):
    d = desc()
    rc, need = bwd_ws(lib, d)
    a = 1 << 20
    ws = 1 << 40
    # x, dt, A, B, C, D, h0, dy, dh_final, dx, ddt, dA, dB, dC, dD, dh0, workspace, bytes, stream
    args = [a, a + (1 << 24), a + (2 << 24), a + (3 << 24), a + (4 << 24), a + (5 << 24), None, a + (6 << 24), None,
            1 << 32, (1 << 32) + (1 << 28), (1 << 32) + (2 << 28), (1 << 32) + (3 << 28), (1 << 32) + (4 << 28),
            (1 << 32) + (5 << 28), None, ws, need, None]
    for i in (0, 1, 2, 3, 4, 5, 7, 9, 10, 11, 12, 13, 14):   # required pointers
        bad = list(args)
        bad[i] = None
        assert lib.ssd_bwd(ctypes.byref(d), *bad) == 1, i
    bad = list(args)
    bad[0] = a + 1                                              # x misaligned for bf16
    assert lib.ssd_bwd(ctypes.byref(d), *bad) == 1
    bad = list(args)
    bad[9] = args[7]                                            # dx aliases dy
    assert lib.ssd_bwd(ctypes.byref(d), *bad) == 1
    bad = list(args)
    bad[13] = args[12]                                          # dC aliases dB
    assert lib.ssd_bwd(ctypes.byref(d), *bad) == 1
    bad = list(args)
    bad[17] = need - 1                                          # workspace one byte short
    assert lib.ssd_bwd(ctypes.byref(d), *bad) == 3
    bad = list(args)
    bad[16] = ws + 128                                          # workspace misaligned
    assert lib.ssd_bwd(ctypes.byref(d), *bad) == 3
    d = desc(chunk=512)
    assert lib.ssd_bwd(ctypes.byref(d), *args) == 2


def s6desc(**kw):
    d = _native.S6Desc()
    base = dict(batch=2, seqlen=256, dim=64, dstate=16, ngroups=1, in_dtype=_native.SSD_BF16,
                out_dtype=_native.SSD_BF16, flags=0, reserved=0)
    base.update(kw)
    for k, v in base.items():
        setattr(d, k, v)
    return d


@pytest.mark.parametrize("bad,code", [
    (dict(dstate=0), 1), (dict(ngroups=3), 1), (dict(batch=-1), 1), (dict(in_dtype=5), 1), (dict(flags=1), 1),
    (dict(reserved=2), 1), (dict(dstate=33), 2), (dict(batch=70000), 2),
])
def test_s6_bad_descriptors_rejected(lib, bad, code):
    d = s6desc(**bad)
    a = 1 << 20
    assert lib.ssd_s6_fwd(ctypes.byref(d), a, a, a, a, a, None, None, 1 << 30, None, None) == code


def test_s6_argument_validation(lib):
    d = s6desc()
    a = 1 << 20
    args = [a, a + (1 << 24), a + (2 << 24), a + (3 << 24), a + (4 << 24), None, None, 1 << 30, None, None]
    for i in (0, 1, 2, 3, 4, 7):
        bad = list(args)
        bad[i] = None
        assert lib.ssd_s6_fwd(ctypes.byref(d), *bad) == 1, i
    bad = list(args)
    bad[7] = args[0]                                            # y aliases x
    assert lib.ssd_s6_fwd(ctypes.byref(d), *bad) == 1
    bad = list(args)
    bad[1] = args[1] + 1                                        # delta misaligned
    assert lib.ssd_s6_fwd(ctypes.byref(d), *bad) == 1
    assert lib.ssd_s6_fwd(None, *args) == 1
    # nothing to do: no batch rows, or no tokens and no final state requested
    assert lib.ssd_s6_fwd(ctypes.byref(s6desc(batch=0)), *args) == 0
    assert lib.ssd_s6_fwd(ctypes.byref(s6desc(seqlen=0)), *args) == 0


def test_float32_dt_beside_bfloat16_inputs(lib):
    """SSD_DT_FLOAT32: the forward pass takes it (its workspace grows by a bfloat16 copy of dt);
    the entry points that read dt directly after the cumsum refuse it."""
    base, f32dt = desc(), desc(dt_dtype=_native.SSD_DT_FLOAT32)
    nb, nf = ctypes.c_size_t(0), ctypes.c_size_t(0)
    assert lib.ssd_fwd_workspace_size(ctypes.byref(base), ctypes.byref(nb)) == 0
    assert lib.ssd_fwd_workspace_size(ctypes.byref(f32dt), ctypes.byref(nf)) == 0
    copy = 2 * 512 * 8 * 2                      # B * L * nh bfloat16
    assert nf.value - nb.value == (copy + 255) // 256 * 256
    p = _native.Plan()
    assert lib.ssd_fwd_plan(ctypes.byref(f32dt), ctypes.byref(p)) == 0 and p.tensor_cores == 1
    fake = 1 << 20   # refused before any pointer is used
    assert lib.ssd_step(ctypes.byref(f32dt), fake, fake, fake, fake, fake, fake, fake, fake, None) == 2
    assert lib.ssd_bwd_workspace_size(ctypes.byref(f32dt), ctypes.byref(nb)) == 2
    assert lib.ssd_chunk_state(ctypes.byref(f32dt), fake, fake, fake, fake, fake, None) == 2
    assert lib.ssd_chunk_scan(ctypes.byref(f32dt), fake, fake, fake, fake, fake, fake, fake, fake, None) == 2
    # with float32 inputs the field changes nothing
    f = desc(in_dtype=_native.SSD_F32, out_dtype=_native.SSD_F32)
    g = desc(in_dtype=_native.SSD_F32, out_dtype=_native.SSD_F32, dt_dtype=_native.SSD_DT_FLOAT32)
    assert lib.ssd_fwd_workspace_size(ctypes.byref(f), ctypes.byref(nb)) == 0
    assert lib.ssd_fwd_workspace_size(ctypes.byref(g), ctypes.byref(nf)) == 0 and nb.value == nf.value


def test_tail_super_chunks_hold_two_chunks(lib):
    """A plan that cuts the sequences of a nearly empty last wave into short super-chunks gives
    them at least two chunks when the whole sequences' super-chunks are longer: a scan CTA's
    start-up costs about two 128-token periods.  Host-side query (the SM count of the device, or
    148 without one): with 80 heads of 64 x 128 and 256-token chunks, 160 head pairs leave a
    short last wave on a GB300-sized part."""
    P = _native.Plan
    for seqlen in (1024, 2048, 4096):
        d = desc(batch=4, seqlen=seqlen, nheads=80, headdim=64, dstate=128, ngroups=1, chunk=256,
                 in_dtype=_native.SSD_BF16, out_dtype=_native.SSD_BF16)
        p = P()
        assert lib.ssd_fwd_plan(ctypes.byref(d), ctypes.byref(p)) == 0
        if p.split_sequences == 4 * 80 or p.super_tokens <= 2 * 256:
            continue                                   # no tail cut on this device, or nothing longer
        assert p.tail_super_tokens >= 2 * 256, (seqlen, p.tail_super_tokens)
        assert p.tail_super_tokens % 256 == 0 and p.tail_n_super * p.tail_super_tokens >= seqlen


def test_sizes_that_would_wrap_are_refused(lib):
    """A problem whose arrays would need 2^62 bytes or more is refused (SSD_ERR_UNSUPPORTED)
    before any size is formed: a wrapped workspace size would let the kernels write past a
    buffer sized from it."""
    n = ctypes.c_size_t(0)
    huge = desc(batch=65535, seqlen=1 << 38, nheads=8, headdim=64, dstate=128, ngroups=1, chunk=256,
                in_dtype=_native.SSD_BF16, out_dtype=_native.SSD_BF16)
    assert lib.ssd_fwd_workspace_size(ctypes.byref(huge), ctypes.byref(n)) == 2
    assert lib.ssd_fwd_host_buffer_size(ctypes.byref(huge), ctypes.byref(n)) == 2
    assert lib.ssd_bwd_workspace_size(ctypes.byref(huge), ctypes.byref(n)) == 2
    p = _native.Plan()
    assert lib.ssd_fwd_plan(ctypes.byref(huge), ctypes.byref(p)) == 2
    s6 = _native.S6Desc(batch=65535, seqlen=1 << 40, dim=1 << 20, dstate=16, ngroups=1,
                        in_dtype=_native.SSD_BF16, out_dtype=_native.SSD_BF16, flags=0, reserved=0)
    fake = 1 << 20    # refused during validation, never dereferenced
    assert lib.ssd_s6_fwd(ctypes.byref(s6), fake, fake, fake, fake, fake, None, None, fake, None, None) == 2
    # sequence indices are 32-bit in the kernels: B * nh of 2^31 or more is refused
    many = desc(batch=65535, seqlen=1, nheads=65535, headdim=1, dstate=1, ngroups=1, chunk=1)
    assert lib.ssd_fwd_workspace_size(ctypes.byref(many), ctypes.byref(n)) == 2
    # a large but representable problem still gets a size
    big = desc(batch=64, seqlen=1 << 20, nheads=8, headdim=64, dstate=128, ngroups=1, chunk=256,
               in_dtype=_native.SSD_BF16, out_dtype=_native.SSD_BF16)
    assert lib.ssd_fwd_workspace_size(ctypes.byref(big), ctypes.byref(n)) == 0 and n.value > 0


def test_host_buffer_size(lib):
    """ssd_fwd_host_buffer_size: host-side query; grows with the batch, covers the device path's
    workspace for one slice, and rejects what ssd_fwd rejects."""
    n1, n4, nw = ctypes.c_size_t(0), ctypes.c_size_t(0), ctypes.c_size_t(0)
    d1, d4 = desc(batch=1), desc(batch=4)
    assert lib.ssd_fwd_host_buffer_size(ctypes.byref(d1), ctypes.byref(n1)) == 0
    assert lib.ssd_fwd_host_buffer_size(ctypes.byref(d4), ctypes.byref(n4)) == 0
    assert lib.ssd_fwd_workspace_size(ctypes.byref(d1), ctypes.byref(nw)) == 0
    x_bytes = 512 * 8 * 64 * 2
    assert n1.value >= nw.value + 2 * x_bytes          # the slice's workspace, x and y at least
    assert n4.value >= 4 * 2 * x_bytes + nw.value       # four one-row slices and one slice's workspace
    assert lib.ssd_fwd_host_buffer_size(ctypes.byref(desc(ngroups=3)), ctypes.byref(n1)) == 1
    assert lib.ssd_fwd_host_buffer_size(ctypes.byref(d1), None) == 1
    # a buffer that is too short is refused before anything is enqueued
    fake = 1 << 20
    assert lib.ssd_fwd_host(ctypes.byref(d1), fake, fake, fake, fake, fake, fake, None, fake, None, 1 << 21, 16,
                            None) == 3

