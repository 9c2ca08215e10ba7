"""The selective-scan kernel's own source, compiled for the CPU and checked against the oracle.

tests/emu holds a stand-in for the CUDA features the kernel uses: a block's threads become host
threads, __syncthreads a barrier, its dynamic shared memory one static array (blocks run one after
another).  The kernel is taken from csrc/s6_scan.cu as it stands, up to its launcher, with the
special-function exp2 replaced by exp2f.  This checks the kernel's control flow and indexing -- the
tiles and the short last tile, the groups of eight tokens, the (B_n, B_n+1, C_n, C_n+1) staging of
pairs of states, channels split over four lanes, partial blocks of channels, groups -- on every CPU
run; the GPU parity tests (tests/test_gpu_s6.py) check the arithmetic as the GPU runs it.
"""
import os
import re
import shutil
import subprocess

import numpy as np
import pytest

import oracle
from selective_state_space_gb300 import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
EMU = os.path.join(ROOT, "tests", "emu")
KERNEL = os.path.join(ROOT, "selective_state_space_gb300", "csrc", "s6_scan.cu")


@pytest.fixture(scope="module")
def emu_binary(tmp_path_factory):
    if shutil.which("g++") is None:
        pytest.skip("g++ is not installed")
    src = open(KERNEL).read()
    head, sep, _ = src.partition("template <typename Tin, typename Tout, int NS>\ncudaError_t s6_launch_t")
    assert sep, "the launcher marker moved: update this test"
    n_smem = head.count("extern __shared__ float4 s6_smem[];")
    head = head.replace("extern __shared__ float4 s6_smem[];", "float4 *s6_smem = emu_smem();")
    head, n_ex2 = re.subn(r'asm\("ex2\.approx\.ftz\.f32 %0, %1;" : "=f"\(r\) : "f"\(v\)\);', "r = exp2f(v);", head)
    assert n_smem == 1 and n_ex2 == 1, "the kernel's shared memory or exp2 changed form: update this test"
    tmp = tmp_path_factory.mktemp("s6emu")
    (tmp / "s6_kernel.inc").write_text(head + "\n}  // namespace\n}  // namespace ssd\n")
    exe = tmp / "s6_emu"
    r = subprocess.run(["g++", "-std=c++20", "-O1", "-pthread", "-Wno-unknown-pragmas", "-I", EMU, "-I", str(tmp),
                        os.path.join(EMU, "s6_main.cpp"), "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-3000:]
    return exe, tmp


def _run(emu, shape):
    exe, tmp = emu
    inp = workloads.make_s6_inputs(shape)
    t = {k: (None if v is None else v.float().numpy()) for k, v in inp.tensors().items()}
    B, L, dim, N, G = shape.batch, shape.seqlen, shape.dim, shape.dstate, shape.ngroups
    hdr = np.array([B, L, dim, N, G, t["D"] is not None, t["h0"] is not None], dtype=np.int64)
    path_in, path_out = tmp / f"{shape.name}.in", tmp / f"{shape.name}.out"
    with open(path_in, "wb") as f:
        f.write(hdr.tobytes())
        for k in ("x", "delta", "A", "B", "C", "D", "h0"):
            if t[k] is not None:
                f.write(np.ascontiguousarray(t[k], dtype=np.float32).tobytes())
    r = subprocess.run([str(exe), str(path_in), str(path_out)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, (r.returncode, r.stderr[-2000:])
    out = np.fromfile(path_out, dtype=np.float32)
    y, hf = out[: B * dim * L].reshape(B, dim, L), out[B * dim * L:].reshape(B, dim, N)
    y_ref, hf_ref = oracle.s6_fwd_seq(t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["h0"])
    return y, hf, y_ref, hf_ref


def _rel(a, ref):
    return float(np.abs(a - ref).max() / max(np.abs(ref).max(), 1e-30))


# (batch, seqlen, dim, N, groups): one to eight states per lane, odd N, a short last tile and a
# sequence shorter than a tile, channel blocks that are not full (dim / G = 40 channels of 32 per
# block), several groups, with and without D and h0
CASES = [
    (2, 150, 80, 4, 2, True, True),
    (2, 150, 80, 3, 2, False, True),
    (1, 192, 64, 8, 1, True, False),
    (2, 70, 48, 7, 3, True, True),
    (1, 128, 40, 16, 1, True, True),
    (2, 7, 80, 13, 2, True, True),
    (1, 100, 32, 32, 1, False, False),
    (1, 64, 36, 20, 2, True, True),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "b{}-l{}-d{}-n{}-g{}".format(*c[:5]))
def test_s6_kernel_source_on_cpu_matches_oracle(emu_binary, case):
    B, L, dim, N, G, skip, h0 = case
    shape = workloads.s6_custom(B, L, dim, N, G, "f32", "mamba1", skip, h0, seed=1000 + N + L,
                                name="emu-b{}-l{}-d{}-n{}-g{}".format(B, L, dim, N, G))
    y, hf, y_ref, hf_ref = _run(emu_binary, shape)
    # float32 arithmetic against the double oracle over up to 192 steps of the recurrence
    assert _rel(y, y_ref) < 1e-5, _rel(y, y_ref)
    assert _rel(hf, hf_ref) < 1e-5, _rel(hf, hf_ref)
