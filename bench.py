"""Benchmark of the chunked SSD forward pass on GB300 (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one ssd_fwd call (all four stages: chunk_cumsum, chunk_state,
state_passing, chunk_scan) over one batch of seeded synthetic inputs already
resident in HBM.  The headline workload is the Mamba-2-2.7B-shaped layer
(B=4, L=4096, 80 heads, H=64, S=128, chunk 256, bf16 inputs, float32 state).
Its inputs and outputs (367 MB) are larger than the 129 MB L2, so no L2 flush
is done between steps.

The default line also carries ``second_workload``: the long-context prefill
(B=1, L=65536, 32 heads, 8 B/C groups) timed the same way in the same run.

Under torchrun (N > 1) every rank runs its own replica of the workload
(independent problems, no collective on the data path); value = tokens of all
ranks / max-over-ranks time.  ``--impl reference`` times the CPU oracle on a
bounded sample of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from selective_state_space_gb300 import workloads  # noqa: E402

METRIC = "ssd_fwd_tokens_per_s"
UNIT = "tokens/s"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
STAGES = ("chunk_cumsum", "chunk_state", "state_passing", "chunk_scan")
KERNEL_SOURCES = {  # the files that hold each kernel (for the traffic record's freshness check)
    "chunk_cumsum": ["ssd_simt.cu"], "state_passing": ["ssd_simt.cu"],
    "chunk_state": ["ssd_tc.cu", "sm100_ptx.cuh"],
    "chunk_scan": ["ssd_tc.cu", "sm100_ptx.cuh"],
}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return PEAKS_FALLBACK, "fallback"


def esize(dtype: str) -> int:
    return 2 if dtype == "bf16" else 4


def stage_bytes(s: workloads.Shape, plan: dict):
    """Bytes per launch of each stage as the library runs it (``plan`` is ssd_fwd_plan), with
    the intermediates it moves counted: G, the float32 dt copy, the super-chunk states and the
    super-chunk-start states, all float32; 0 for a stage that does not launch.  A plan cuts the
    sequences ((batch, head) pairs) in two parts; chunk_state and state_passing run per part and
    their bytes are summed.  Also the whole-step compulsory I/O ("step": each input read once,
    each output written once, intermediates excluded)."""
    e = esize(s.dtype)
    Bsz, L, nh, H, S, G, T, nc = s.batch, s.seqlen, s.nheads, s.headdim, s.dstate, s.ngroups, s.chunk, s.nchunks
    x = Bsz * L * nh * H * e
    dt = Bsz * L * nh * e
    bc = Bsz * L * G * S * e
    g = Bsz * nh * L * 4
    state = Bsz * nh * H * S * 4                       # one float32 state per (batch, head)
    hs = H * S * 4                                     # one float32 state of one sequence
    h0 = state if s.h0_recipe != "none" else 0
    y = Bsz * L * nh * H * e
    ad = 2 * nh * 4
    step = x + dt + 2 * bc + ad + h0 + y + state
    nseq, hpg = Bsz * nh, nh // G
    split = plan["split_sequences"]
    parts = [(0, split, plan["super_tokens"], plan["n_super"]),
             (split, nseq - split, plan["tail_super_tokens"], plan["tail_n_super"])]
    cs = sp = carried = 0.0
    if plan["tensor_cores"]:
        parts = [(lo, n, tok // T, nsup) for lo, n, tok, nsup in parts]
    else:
        parts = [(0, nseq, 1, nc)]
    # the cumsum writes the float32 copy of dt only for the sequences chunk_state reads
    dtT_seqs = sum(n for lo, n, R, nsup in parts if n > 0 and nsup > 1) if plan["tensor_cores"] else 0
    for lo, n, R, nsup in parts:
        if n == 0:
            continue
        # super-chunks whose state chunk_state produces: all but the last on the tensor-core
        # path (the scan carries the last one itself), every chunk on the CUDA-core path
        nm = nsup - 1 if plan["tensor_cores"] else nc
        carried += n * (nsup - 1) * hs if plan["tensor_cores"] else 0
        if nm == 0:
            continue
        frac = min(nm * R * T, L) / L                  # share of each sequence chunk_state reads
        pairs = len({(bh // nh, (bh % nh) // hpg) for bh in range(lo, lo + n)})   # (batch, group) pairs read
        per_seq = L * (H * e + e + 4)                  # x, dt and G of one sequence
        cs += frac * (n * per_seq + pairs * L * S * e) + n * nm * hs
        sp += 2 * n * nm * hs + n * nc * 4 + (n * hs if h0 else 0)
    out = {
        "chunk_cumsum": dt + nh * 4 + g + dtT_seqs * L * 4,   # + the float32 copy of dt
        "chunk_state": cs,
        "state_passing": sp,
        "chunk_scan": x + dt + 2 * bc + g + h0 + carried + nh * 4 + y + state,
        "step": step,
    }
    if not plan["tensor_cores"]:
        out["state_passing"] += state                  # the CUDA-core path writes h_final there
        out["chunk_scan"] += nc * state - state - h0   # reads every chunk-start state, not h0 or h_final
    return out


def alg_flops(s: workloads.Shape) -> float:
    """Algorithmic flops of one forward pass: per (batch, chunk), per head
    2TSH (chunk state) + 2TSH (C h^T) + 2 T(T+1)/2 H (causal intra-chunk product)
    + 2SH (state pass), plus per group 2 T(T+1)/2 S (C B^T, lower triangle)."""
    T, S, H = s.chunk, s.dstate, s.headdim
    per_head = 4 * T * S * H + T * (T + 1) * H + 2 * S * H
    per_group = T * (T + 1) * S
    return float(s.batch * s.nchunks * (s.nheads * per_head + s.ngroups * per_group))


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"ssd_bench_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return None
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "", 1).isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "", 1).isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def traffic_record(stage: str, shape_name: str):
    """DRAM bytes per launch from a committed ncu summary, if the kernel source is
    unchanged since the capture (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    ent = rec.get(shape_name, {}).get(stage)
    if not ent:
        return None
    h = hashlib.sha256()
    for fn in KERNEL_SOURCES[stage]:
        with open(os.path.join(ROOT, "selective_state_space_gb300", "csrc", fn), "rb") as f:
            h.update(f.read())
    if ent.get("source_sha256") != h.hexdigest():
        return None
    return ent.get("dram_bytes_per_launch")


def _head_windows(s, width):
    """(batch, lo, hi) head windows whose heads keep their B/C group mapping when
    cut out as a sub-problem: inside one group, or whole groups."""
    hpg = s.nheads // s.ngroups
    if hpg >= width:
        step = width
    else:
        step = max(1, width // hpg) * hpg
    for b in range(s.batch):
        lo = 0
        while lo < s.nheads:
            hi = min(s.nheads, lo + step)
            if hpg >= width:     # stay inside one group
                hi = min(hi, (lo // hpg + 1) * hpg)
            yield b, lo, hi
            lo = hi


def cpu_model() -> str:
    """The host CPU's model name, as lscpu or /proc/cpuinfo reports it."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def cpu_baseline(inp, budget_s: float):
    """The oracle as it stands, timed on a bounded sample of (batch, head) pairs at
    full sequence length, with every core this process may use."""
    import oracle
    s = inp.shape
    cores = oracle.default_threads()
    hpg = s.nheads // s.ngroups
    windows = list(_head_windows(s, cores))
    done, rounds, t0 = 0, 0, time.perf_counter()
    while True:   # cycle over the windows (repeating the workload if it is small) until the budget is spent
        b, lo, hi = windows[rounds % len(windows)]
        glo, ghi = lo // hpg, (hi - 1) // hpg + 1
        oracle.ssd_fwd_seq(inp.x[b:b + 1, :, lo:hi], inp.dt[b:b + 1, :, lo:hi], inp.A[lo:hi],
                           inp.B[b:b + 1, :, glo:ghi], inp.C[b:b + 1, :, glo:ghi], inp.D[lo:hi],
                           None if inp.h0 is None else inp.h0[b:b + 1, lo:hi], nthreads=cores)
        done += hi - lo
        rounds += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    el = time.perf_counter() - t0
    tokens_equiv = done * s.seqlen / s.nheads      # (batch, head) pairs -> whole-workload tokens
    return {"value": tokens_equiv / el, "unit": UNIT, "cores": cores, "model": cpu_model(), "kind": "oracle",
            "sample": f"{done} (batch, head) pairs (workload has {s.batch * s.nheads}) at full length L={s.seqlen}, "
                      f"sequential float64 recurrence, {el:.1f} s; tokens/s scaled to the whole workload"}


def run_reference(args, shape):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    inp = workloads.make_inputs(shape)
    import oracle
    oracle.build()
    per_step = max(1.0, args.ref_step_s)
    vals = []
    for i in range(args.warmup + args.steps):
        r = cpu_baseline(inp, per_step)
        if i >= args.warmup:
            vals.append(r)
    tok = statistics.median(v["value"] for v in vals)
    line = {"impl": "reference", "metric": METRIC, "value": tok, "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": shape.tokens / tok * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_of(shape),
            "cpu_baseline": {"value": tok, "unit": UNIT, "cores": vals[0]["cores"], "kind": "oracle",
                             "sample": vals[0]["sample"]},
            "e2e": {"value": tok, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


L2_BYTES = 129 * 10**6


def max_over_ranks(ms: float, dist, device) -> float:
    """The slowest rank's time: each rank contributes its own, every rank receives the maximum
    (a no-op on one process)."""
    if dist is None:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world: int, units_per_rank: float, ms: float) -> float:
    """Units per second of the whole job: every rank processes its own units in `ms` (the max over ranks)."""
    return world * units_per_rank / (ms * 1e-3)


def needs_l2_flush(shape) -> bool:
    """Steps whose compulsory I/O is under twice the L2 could run partly from L2 on
    back-to-back steps; those are timed one step at a time with an L2 flush between."""
    return step_io_bytes(shape) < 2 * L2_BYTES


def step_io_bytes(shape) -> int:
    e = esize(shape.dtype)
    Bsz, L, nh, H, S, G = shape.batch, shape.seqlen, shape.nheads, shape.headdim, shape.dstate, shape.ngroups
    state = Bsz * nh * H * S * 4
    return (2 * Bsz * L * nh * H * e + Bsz * L * nh * e + 2 * Bsz * L * G * S * e + 2 * nh * 4
            + (state if shape.h0_recipe != "none" else 0) + state)


def config_of(shape):
    l2 = ("flushed between steps: each step timed alone after writing a 512 MB buffer" if needs_l2_flush(shape)
          else "no flush: compulsory I/O per step exceeds twice the 129 MB L2")
    return {"workload": shape.name, "batch": shape.batch, "seqlen": shape.seqlen, "nheads": shape.nheads,
            "headdim": shape.headdim, "dstate": shape.dstate, "ngroups": shape.ngroups, "chunk": shape.chunk,
            "input_dtype": shape.dtype, "state_dtype": "f32", "l2": l2}


DECODE_METRIC = "ssd_step_tokens_per_s"


def parse_decode(name: str):
    """decode-<layer workload>-b<batch>: single-token decode steps of that layer's heads at that batch."""
    if not name.startswith("decode-") or "-b" not in name:
        return None
    layer, batch = name[len("decode-"):].rsplit("-b", 1)
    base = workloads.by_name(layer)
    return dataclasses.replace(base, name=name, batch=int(batch), seqlen=1, chunk=1, h0_recipe="normal",
                               dt_zero_frac=0.0)


def run_decode(args, shape):
    """ssd_step throughput: each step reads and writes the float32 state once (HBM-bound)."""
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    from selective_state_space_gb300 import api
    from selective_state_space_gb300.build import build
    build()
    inp = workloads.make_inputs(shape)
    d = {k: (None if v is None else v.to(dev)) for k, v in inp.tensors().items()}
    x, dt, Bm, Cm = d["x"][:, 0], d["dt"][:, 0], d["B"][:, 0], d["C"][:, 0]
    h = d["h0"].clone()
    y = torch.empty_like(x)
    stream = torch.cuda.current_stream(dev)

    def step():
        api.ssd_step(x, dt, d["A"], Bm, Cm, d["D"], h, y=y, stream=stream)

    e = esize(shape.dtype)
    state = shape.batch * shape.nheads * shape.headdim * shape.dstate * 4
    alg = (2 * state + 2 * shape.batch * shape.nheads * shape.headdim * e + shape.batch * shape.nheads * e
           + 2 * shape.batch * shape.ngroups * shape.dstate * e + 2 * shape.nheads * 4)
    flush = alg < 2 * L2_BYTES
    scrub = torch.empty(512 * 2**20, dtype=torch.uint8, device=dev) if flush else None
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(0) as clk:
        # warm-up inside the sampled window, right before the timed steps (the sampler's start-up
        # leaves the GPU idle for a moment)
        for _ in range(max(3, args.warmup)):
            step()
        torch.cuda.synchronize()
        if not flush:
            start.record(stream)
            for _ in range(args.steps):
                step()
            end.record(stream)
            torch.cuda.synchronize()
            ms = start.elapsed_time(end)
        else:
            ms = 0.0
            for i in range(args.steps):
                scrub.fill_(i & 0xff)
                start.record(stream)
                step()
                end.record(stream)
                torch.cuda.synchronize()
                ms += start.elapsed_time(end)
    ms_per_step = ms / args.steps
    peaks, peak_kind = load_peaks()
    peak = float(peaks["hbm_gbs"])
    achieved = alg / (ms_per_step * 1e-3) / 1e9
    line = {
        "metric": DECODE_METRIC, "value": shape.batch / (ms_per_step * 1e-3), "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32 (state), " + shape.dtype + " (x, B, C)",
        "data": "synthetic",
        "config": {"workload": shape.name, "batch": shape.batch, "nheads": shape.nheads, "headdim": shape.headdim,
                   "dstate": shape.dstate, "ngroups": shape.ngroups, "input_dtype": shape.dtype,
                   "l2": ("flushed between steps: each step timed alone after writing a 512 MB buffer" if flush
                          else "no flush: the state read and written per step exceeds twice the 129 MB L2")},
        "roofline": {"kernel": "ssd_step", "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": f"{peak_kind} hbm_gbs", "alg_bytes_per_launch": alg,
                     "traffic": None},
        "gpu_launches": args.steps,
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)


BWD_METRIC = "ssd_bwd_tokens_per_s"
# float32 CUDA-core peak of one GB300: 152 SMs x 128 FP32 lanes x 2 flop (FMA) x 2070 MHz
FP32_ALU_TFLOPS = 152 * 128 * 2 * 2.070e9 / 1e12


def bwd_alg_flops(s: workloads.Shape) -> float:
    """Algorithmic flops of the chunked gradient pass, per (batch, chunk): per head
    10TSH (five contractions of 2TSH each: the forward chunk state, the entering-state
    gradient, Lam B, Lam^T x and h_in^T dy) + T(T+1)(2H + 2S) (dy.x and the contractions of
    v, dB and dC, lower triangles) + 6SH (both state passes and <Lam, h_in>), plus per
    group T(T+1) S (C B^T, lower triangle)."""
    T, S, H = s.chunk, s.dstate, s.headdim
    per_head = 10 * T * S * H + T * (T + 1) * (2 * H + 2 * S) + 6 * S * H
    return float(s.batch * s.nchunks * (s.nheads * per_head + s.ngroups * T * (T + 1) * S))


def bwd_cpu_baseline(inp, gin, budget_s: float):
    """The gradient oracle as it stands, on (batch, head) pairs at full sequence length, one pair per
    call with every core on the pairs of a window; tokens/s scaled to the whole workload."""
    import oracle
    s = inp.shape
    cores = oracle.default_threads()
    hpg = s.nheads // s.ngroups
    windows = list(_head_windows(s, cores))
    done, rounds, t0 = 0, 0, time.perf_counter()
    while True:
        b, lo, hi = windows[rounds % len(windows)]
        glo, ghi = lo // hpg, (hi - 1) // hpg + 1
        oracle.ssd_bwd_seq(inp.x[b:b + 1, :, lo:hi], inp.dt[b:b + 1, :, lo:hi], inp.A[lo:hi],
                           inp.B[b:b + 1, :, glo:ghi], inp.C[b:b + 1, :, glo:ghi], inp.D[lo:hi],
                           gin.dy[b:b + 1, :, lo:hi], h0=None if inp.h0 is None else inp.h0[b:b + 1, lo:hi],
                           dh_final=None if gin.dh_final is None else gin.dh_final[b:b + 1, lo:hi], nthreads=cores)
        done += hi - lo
        rounds += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    el = time.perf_counter() - t0
    return {"value": done * s.seqlen / s.nheads / el, "unit": UNIT, "cores": cores, "model": cpu_model(), "kind": "oracle",
            "sample": f"{done} (batch, head) pairs (workload has {s.batch * s.nheads}) at full length L={s.seqlen}, "
                      f"reverse-mode float64 recurrence, {el:.1f} s; tokens/s scaled to the whole workload"}


def run_bwd_reference(args, shape):
    """The reference arm of the gradient pass: the oracle on the host cores, rank 0 only."""
    if int(os.environ.get("RANK", "0")) != 0:
        return
    import oracle
    oracle.build()
    inp = workloads.make_inputs(shape)
    gin = workloads.make_grad_inputs(shape)
    vals = [bwd_cpu_baseline(inp, gin, max(1.0, args.ref_step_s)) for _ in range(args.warmup + args.steps)]
    vals = vals[args.warmup:]
    tok = statistics.median(v["value"] for v in vals)
    print(json.dumps({"impl": "reference", "metric": BWD_METRIC, "value": tok, "unit": UNIT, "n_gpus": 1,
                      "steps": args.steps, "warmup": args.warmup, "ms_per_step": shape.tokens / tok * 1e3,
                      "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                      "data": "synthetic", "config": config_of(shape), "cpu_baseline": dict(vals[0], value=tok),
                      "e2e": {"value": tok, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
                      "gpu_launches": 0}), flush=True)


def run_bwd(args, shape):
    """ssd_bwd throughput on one layer: the whole gradient pass (forward recompute included)
    per step, inputs and upstream gradients resident on the device."""
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    from selective_state_space_gb300 import api
    from selective_state_space_gb300.build import build
    build()
    inp = workloads.make_inputs(shape)
    gin = workloads.make_grad_inputs(shape)
    d = {k: (None if v is None else v.to(dev)) for k, v in inp.tensors().items()}
    dy, dhf = gin.dy.to(dev), gin.dh_final.to(dev)
    desc = api.desc_for(d["x"], d["B"], shape.chunk)
    ws = torch.empty(max(api.bwd_workspace_size(desc), 256), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        return api.ssd_bwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], dy, shape.chunk, d["h0"], dhf,
                           workspace=ws, stream=stream)

    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(0) as clk:
        for _ in range(max(3, args.warmup)):
            step()
        torch.cuda.synchronize()
        start.record(stream)
        for _ in range(args.steps):
            step()
        end.record(stream)
        torch.cuda.synchronize()
    ms_per_step = start.elapsed_time(end) / args.steps
    e = esize(shape.dtype)
    io = 2 * step_io_bytes(shape) + shape.batch * shape.seqlen * shape.nheads * shape.headdim * e   # + dy
    flops = bwd_alg_flops(shape)
    peaks, peak_kind = load_peaks()
    line = {
        "metric": BWD_METRIC, "value": shape.tokens / (ms_per_step * 1e-3), "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32 (CUDA cores), " + shape.dtype + " (inputs, gradients)",
        "data": "synthetic", "config": dict(config_of(shape), l2="no flush: inputs, gradients and workspace per step "
                                            "exceed twice the 129 MB L2"),
        "roofline": {"kernel": "ssd_bwd (whole pass)", "bound": "alu", "achieved": flops / (ms_per_step * 1e-3) / 1e12,
                     "peak": FP32_ALU_TFLOPS, "unit": "TFLOP/s", "frac": flops / (ms_per_step * 1e-3) / 1e12 / FP32_ALU_TFLOPS,
                     "peak_source": "derived: 152 SMs x 128 FP32 lanes x 2 x 2070 MHz", "alg_flops_per_step": flops,
                     "traffic": None},
        "hbm_roofline": {"alg_bytes_per_step": io, "achieved_gbs": io / (ms_per_step * 1e-3) / 1e9,
                         "peak_gbs": float(peaks["hbm_gbs"]),
                         "frac": io / (ms_per_step * 1e-3) / 1e9 / float(peaks["hbm_gbs"])},
        "e2e": None,
        "gpu_launches": 10 * args.steps,
        "clocks": clk.summary(),
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = bwd_cpu_baseline(inp, gin, args.cpu_budget_s)
    print(json.dumps(line), flush=True)


S6_METRIC = "s6_fwd_tokens_per_s"
# exp2 rate of the special-function units: 152 SMs x 32 per clock (the doubled exponential rate of this
# Blackwell part; 16 per clock on earlier parts) x 2070 MHz
SFU_EX2_PER_S = 152 * 32 * 2.070e9


def s6_cpu_baseline(inp, budget_s: float):
    """The S6 oracle as it stands on sampled channels at full length, on every core: each oracle call
    scans one channel (ctypes releases the interpreter lock), and a thread pool runs one call per core."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    s = inp.shape
    cores = oracle.default_threads()
    cpg = s.dim // s.ngroups
    t = inp.tensors()

    def one(i):
        b, d = i % s.batch, (i * 7919) % s.dim
        g = d // cpg
        oracle.s6_fwd_seq(t["x"][b:b + 1, d:d + 1], t["delta"][b:b + 1, d:d + 1], t["A"][d:d + 1],
                          t["B"][b:b + 1, g:g + 1], t["C"][b:b + 1, g:g + 1],
                          None if t["D"] is None else t["D"][d:d + 1],
                          None if t["h0"] is None else t["h0"][b:b + 1, d:d + 1])

    done, t0 = 0, time.perf_counter()
    with ThreadPoolExecutor(max_workers=cores) as ex:
        while time.perf_counter() - t0 < budget_s:
            list(ex.map(one, range(done, done + cores)))
            done += cores
    el = time.perf_counter() - t0
    tok = done * s.seqlen / s.dim                             # channels -> whole-workload tokens (B L per B dim)
    return {"value": tok / el, "unit": "tokens/s", "cores": cores, "model": cpu_model(), "kind": "oracle",
            "sample": f"{done} channels (workload has {s.batch * s.dim}) at full length L={s.seqlen}, sequential "
                      f"float64 recurrence, {el:.1f} s; tokens/s scaled to the whole workload"}


def run_s6(args, shape):
    """ssd_s6_fwd throughput: inputs resident; one step = the scan of every channel of the batch."""
    if args.impl == "reference":
        if int(os.environ.get("RANK", "0")) != 0:
            return
        import oracle
        oracle.build()
        inp = workloads.make_s6_inputs(shape)
        vals = [s6_cpu_baseline(inp, max(1.0, args.ref_step_s)) for _ in range(args.warmup + args.steps)][args.warmup:]
        tok = statistics.median(v["value"] for v in vals)
        print(json.dumps({"impl": "reference", "metric": S6_METRIC, "value": tok, "unit": "tokens/s", "n_gpus": 1,
                          "steps": args.steps, "warmup": args.warmup, "ms_per_step": shape.tokens / tok * 1e3,
                          "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                          "data": "synthetic", "config": {"workload": shape.name},
                          "cpu_baseline": dict(vals[0], value=tok),
                          "e2e": {"value": tok, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
                          "gpu_launches": 0}), flush=True)
        return
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    from selective_state_space_gb300 import api
    from selective_state_space_gb300.build import build
    build()
    inp = workloads.make_s6_inputs(shape)
    d = {k: (None if v is None else v.to(dev)) for k, v in inp.tensors().items()}
    y = torch.empty_like(d["x"])
    stream = torch.cuda.current_stream(dev)
    e = esize(shape.dtype)
    nx = shape.batch * shape.dim * shape.seqlen
    nbc = shape.batch * shape.ngroups * shape.dstate * shape.seqlen
    state = shape.batch * shape.dim * shape.dstate * 4
    alg = 3 * nx * e + 2 * nbc * e + shape.dim * shape.dstate * 4 + (shape.dim * 4 if shape.skip else 0) \
        + (state if shape.h0 else 0) + state
    exps = nx * shape.dstate
    flush = alg < 2 * L2_BYTES
    scrub = torch.empty(512 * 2**20, dtype=torch.uint8, device=dev) if flush else None
    hf = torch.empty((shape.batch, shape.dim, shape.dstate), dtype=torch.float32, device=dev)

    def step():
        api.s6_fwd(d["x"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["h0"], y=y, stream=stream)

    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(0) as clk:
        for _ in range(max(3, args.warmup)):
            step()
        torch.cuda.synchronize()
        ms = 0.0
        if not flush:
            start.record(stream)
            for _ in range(args.steps):
                step()
            end.record(stream)
            torch.cuda.synchronize()
            ms = start.elapsed_time(end)
        else:
            for i in range(args.steps):
                scrub.fill_(i & 0xff)
                start.record(stream)
                step()
                end.record(stream)
                torch.cuda.synchronize()
                ms += start.elapsed_time(end)
    ms_per_step = ms / args.steps
    sec = ms_per_step * 1e-3
    peaks, peak_kind = load_peaks()
    hbm_peak = float(peaks["hbm_gbs"])
    t_hbm, t_sfu = alg / (hbm_peak * 1e9), exps / SFU_EX2_PER_S
    if t_hbm >= t_sfu:
        roof = {"bound": "hbm", "achieved": alg / sec / 1e9, "peak": hbm_peak, "unit": "GB/s",
                "frac": alg / sec / 1e9 / hbm_peak, "peak_source": f"{peak_kind} hbm_gbs"}
    else:
        roof = {"bound": "alu", "achieved": exps / sec / 1e12, "peak": SFU_EX2_PER_S / 1e12, "unit": "Tex2/s",
                "frac": exps / sec / SFU_EX2_PER_S,
                "peak_source": "derived: 152 SMs x 32 exp2 per clock x 2070 MHz (special-function units)"}
    roof.update({"kernel": "k_s6_scan", "alg_bytes_per_launch": alg, "exp2_per_launch": exps, "traffic": None,
                 "hbm_frac": alg / sec / 1e9 / hbm_peak, "sfu_frac": exps / sec / SFU_EX2_PER_S})
    line = {
        "metric": S6_METRIC, "value": shape.tokens / sec, "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32 (state and arithmetic), " + shape.dtype + " (x, delta, B, C, y)",
        "data": "synthetic",
        "config": {"workload": shape.name, "batch": shape.batch, "seqlen": shape.seqlen, "dim": shape.dim,
                   "dstate": shape.dstate, "ngroups": shape.ngroups, "input_dtype": shape.dtype,
                   "l2": ("flushed between steps: each step timed alone after writing a 512 MB buffer" if flush
                          else "no flush: compulsory I/O per step exceeds twice the 129 MB L2")},
        "roofline": roof, "e2e": None, "gpu_launches": args.steps, "clocks": clk.summary(),
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = s6_cpu_baseline(inp, args.cpu_budget_s)
    print(json.dumps(line), flush=True)


def time_fwd_device(shape, steps: int, warmup: int, dev) -> tuple:
    """ms per ssd_fwd step of `shape` with its inputs resident (back to back, or each step
    alone after an L2 flush when the workload fits in L2), and its plan."""
    from selective_state_space_gb300 import api
    inp = workloads.make_inputs(shape)
    d = {k: (None if v is None else v.to(dev)) for k, v in inp.tensors().items()}
    desc = api.desc_for(d["x"], d["B"], shape.chunk)
    plan = api.fwd_plan(desc)
    ws = api.alloc_workspace(desc, dev)
    y = torch.empty_like(d["x"])
    hf = torch.empty((shape.batch, shape.nheads, shape.headdim, shape.dstate), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        api.ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], shape.chunk, d["h0"], y=y, h_final=hf,
                    workspace=ws, stream=stream)

    for _ in range(max(3, warmup)):
        step()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if not needs_l2_flush(shape):
        start.record(stream)
        for _ in range(steps):
            step()
        end.record(stream)
        torch.cuda.synchronize()
        ms = start.elapsed_time(end)
    else:
        scrub = torch.empty(512 * 2**20, dtype=torch.uint8, device=dev)
        ms = 0.0
        for i in range(steps):
            scrub.fill_(i & 0xff)
            start.record(stream)
            step()
            end.record(stream)
            torch.cuda.synchronize()
            ms += start.elapsed_time(end)
    return ms / steps, plan


# The second workload the default line also reports, timed in the same run: the long-context
# prefill, whose super-chunk cut needs the chunk_state and state_passing passes in full.
SECOND_WORKLOAD = "long-prefill-64k"


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="mamba2-2.7b-layer")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget-s", type=float, default=12.0)
    ap.add_argument("--ref-step-s", type=float, default=2.0)
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--pass", dest="which", default="fwd", choices=["fwd", "bwd"],
                    help="bwd: time the gradient pass (ssd_bwd) of the workload instead of the forward pass")
    args = ap.parse_args()
    dshape = parse_decode(args.workload)
    if dshape is not None:
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the decode workloads time ssd_step only"}))
            return
        run_decode(args, dshape)
        return
    if args.workload.startswith("s6-"):
        run_s6(args, workloads.s6_by_name(args.workload))
        return
    shape = workloads.by_name(args.workload)
    if args.which == "bwd":
        if args.impl == "reference":
            run_bwd_reference(args, shape)
            return
        run_bwd(args, shape)
        return
    if args.impl == "reference":
        run_reference(args, shape)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)

    from selective_state_space_gb300 import api
    from selective_state_space_gb300.build import build
    build()
    inp = workloads.make_inputs(shape)
    d = {k: (None if v is None else v.to(dev)) for k, v in inp.tensors().items()}
    desc = api.desc_for(d["x"], d["B"], shape.chunk)
    tc = api.uses_tensor_cores(desc)
    plan = api.fwd_plan(desc)
    ws = api.alloc_workspace(desc, dev)
    y = torch.empty_like(d["x"])
    hf = torch.empty((shape.batch, shape.nheads, shape.headdim, shape.dstate), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(events=None):
        api.ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], shape.chunk, d["h0"], y=y, h_final=hf,
                    workspace=ws, stream=stream, events=events)

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(8)] for _ in range(args.steps)]
    for row in ev:          # torch creates the underlying CUDA event on first record
        for e in row:
            e.record(stream)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    flush = needs_l2_flush(shape)
    scrub = torch.empty(512 * 2**20, dtype=torch.uint8, device=dev) if flush else None
    with ClockSampler(local_rank) as clk:
        # warm-up inside the sampled window, right before the timed steps (the sampler's start-up
        # leaves the GPU idle for a moment)
        for _ in range(max(3, args.warmup)):
            step()
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        # the headline: K plain forward passes, nothing else on the stream (or, for a
        # workload that fits in L2, each pass timed alone after an L2 flush)
        if not flush:
            start.record(stream)
            for i in range(args.steps):
                step()
            end.record(stream)
            torch.cuda.synchronize()
            ms = start.elapsed_time(end)
        else:
            ms = 0.0
            for i in range(args.steps):
                scrub.fill_(i & 0xff)
                start.record(stream)
                step()
                end.record(stream)
                torch.cuda.synchronize()
                ms += start.elapsed_time(end)
        # the same K passes again with events around each stage (ssd_fwd_timed): the
        # per-kernel durations for the roofline; the events cost a few microseconds per
        # pass, so this pass does not feed the headline
        for i in range(args.steps):
            if flush:
                scrub.fill_(i & 0xff)
            step(ev[i])
        torch.cuda.synchronize()
    if dist:
        dist.barrier()
    ms = max_over_ranks(ms, dist, dev)
    ms_per_step = ms / args.steps
    stage_ms = {st: statistics.mean(ev[i][2 * j].elapsed_time(ev[i][2 * j + 1]) for i in range(args.steps))
                for j, st in enumerate(STAGES)}

    # end to end through the C ABI on host buffers (ssd_fwd_host): every step copies its pinned
    # host inputs in and y and h_final back out, the batch cut into slices whose copies overlap
    # the computation of the others
    host = {k: (None if v is None else v.pin_memory()) for k, v in inp.tensors().items()}
    y_host = torch.empty(y.shape, dtype=y.dtype, pin_memory=True)
    hf_host = torch.empty(hf.shape, dtype=hf.dtype, pin_memory=True)
    h2d = sum(v.numel() * v.element_size() for v in host.values() if v is not None)
    d2h = y_host.numel() * y_host.element_size() + hf_host.numel() * hf_host.element_size()
    host_buf = torch.empty(api.host_buffer_size(desc), dtype=torch.uint8, device=dev)

    def e2e_step():
        api.ssd_fwd_host(host["x"], host["dt"], host["A"], host["B"], host["C"], host["D"], shape.chunk, host["h0"],
                         y=y_host, h_final=hf_host, device_buffer=host_buf, stream=stream)

    e2e_step()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / args.e2e_steps
    e2e_ms = max_over_ranks(e2e_ms, dist, dev)

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return

    peaks, peak_kind = load_peaks()
    sb = stage_bytes(shape, plan)
    top = max(STAGES, key=lambda s_: stage_ms[s_] if sb[s_] else -1.0)
    kname = top
    # the dominant kernel's algorithmic bytes are the compulsory I/O of the step --
    # every input read once and every output written once, intermediates excluded (the scan reads
    # every input and writes every output of the step)
    alg_top = sb["step"]
    achieved = alg_top / (stage_ms[top] * 1e-3) / 1e9
    # a kernel timed inside a long step: burst copy bandwidth is the only HBM figure measured
    peak = float(peaks["hbm_gbs"])
    tokens_per_s = whole_job_rate(world, shape.tokens, ms_per_step)
    flops = alg_flops(shape)
    line = {
        "metric": METRIC, "value": tokens_per_s, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": ("tf32 (float32 inputs)" if shape.dtype == "f32" else "bf16") if tc
        else ("f32" if shape.dtype == "f32" else "f32 (bf16 inputs)"),
        "data": "synthetic", "config": dict(config_of(shape), parallelism=f"replicas{world}",
                                            tensor_cores=tc),
        "tflops": flops / (ms_per_step * 1e-3) / 1e12,
        "roofline": {"kernel": kname, "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": f"{peak_kind} hbm_gbs",
                     "alg_bytes_per_launch": alg_top, "traffic": traffic_record(kname, shape.name),
                     "plan_bytes_per_launch": sb[top],
                     "plan_frac": sb[top] / (stage_ms[top] * 1e-3) / 1e9 / peak},
        "step_roofline": {"alg_bytes": sb["step"], "alg_flops": flops,
                          "roofline_ms": max(sb["step"] / (peak * 1e9), flops / (float(peaks["bf16_tflops"]) * 1e12)) * 1e3,
                          "frac": max(sb["step"] / (peak * 1e9), flops / (float(peaks["bf16_tflops"]) * 1e12)) * 1e3 / ms_per_step},
        "plan": plan,
        "stages_ms": {s_: (stage_ms[s_] if sb[s_] else None) for s_ in STAGES},
        "stages_plan_gbs": {s_: (sb[s_] / (stage_ms[s_] * 1e-3) / 1e9 if sb[s_] else None) for s_ in STAGES},
        "e2e": {"value": whole_job_rate(world, shape.tokens, e2e_ms), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "call": "ssd_fwd_host (pinned host buffers; the batch in slices whose copies overlap the computation)"},
        "gpu_launches": plan["kernel_launches"] * args.steps,
        "clocks": clk.summary(),
    }
    if shape.name == "mamba2-2.7b-layer":
        # the second workload, timed the same way in the same process, on this rank alone
        s2 = workloads.by_name(SECOND_WORKLOAD)
        with ClockSampler(local_rank) as clk2:
            ms2, plan2 = time_fwd_device(s2, args.steps, args.warmup, dev)
        sb2 = stage_bytes(s2, plan2)
        roof2 = max(sb2["step"] / (peak * 1e9), alg_flops(s2) / (float(peaks["bf16_tflops"]) * 1e12)) * 1e3
        line["second_workload"] = {
            "workload": s2.name, "config": config_of(s2), "ms_per_step": ms2, "steps": args.steps,
            "warmup": max(3, args.warmup), "value": s2.tokens / (ms2 * 1e-3), "unit": UNIT,
            "step_roofline": {"alg_bytes": sb2["step"], "roofline_ms": roof2, "frac": roof2 / ms2},
            "plan": plan2, "clocks": clk2.summary(),
        }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(inp, args.cpu_budget_s)
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
