"""Benchmark of the GB300 fused attention forward.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-all]

One step = one fused attention forward (every step of the path runs in the
CUDA library) over one batch of the workload's synthetic inputs.  The headline
workload is the dense fp16 attention B=4, H=16, L=1024, D=64 (with lse).
Rank 0 prints one JSON line.  Under torchrun (N > 1) every rank runs an
independent replica on its own GPU (the forward needs no exchange between
GPUs), ranks meet at a barrier around the timed region and the slowest rank's
time is reported; ``value`` is the work of all ranks over that time.

``--impl reference`` times the CPU fp64 oracle instead (the slow program the
library is checked against) on the host cores, one head of the workload per
step; under torchrun only rank 0 runs it.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from attn_inputs import HEADLINE, MASK_NAMES, WORKLOADS, make_workload_inputs  # noqa: E402

L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
METRIC = "attention fwd TFLOP/s (unmasked FLOPs) and % of roofline per mask kind, 1×GB300"
KERNEL_SOURCES = ["attn_fwd_kernel.cuh", "ptx.cuh", "attn_api.cu"]


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(WORKLOADS))
    ap.add_argument("--no-all", action="store_true",
                    help="skip the per-mask-kind measurements of the other workloads")
    ap.add_argument("--soak-s", type=float, default=2.0,
                    help="seconds of untimed launches before the timed region (clock sampling)")
    ap.add_argument("--bwd-only", action="store_true",
                    help="time only the backward (attn_bwd) on --workload and print one line "
                         "(for profiler runs)")
    ap.add_argument("--fp8v-only", action="store_true",
                    help="time only the FP8 P.V variant (attn_fwd_fp8v) on --workload and print one "
                         "line (for profiler runs)")
    ap.add_argument("--threads", type=int, default=None,
                    help="host threads of the CPU oracle (--impl reference and the CPU baseline; "
                         "default: every core)")
    ap.add_argument("--shape", default=None,
                    help="an ad hoc problem B,H,L,D,MASK,DTYPE[,BS] (MASK dense|causal|block_diag, "
                         "DTYPE fp16|bf16) in place of --workload, same input recipe (seed 42, N(0,1)); "
                         "for profiler runs on reduced sizes")
    ap.add_argument("--lean", action="store_true",
                    help="only the device-timed line: no soak, e2e, CPU baseline or other "
                         "workloads (for profiler runs)")
    return ap.parse_args()


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "attention_forward_15_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary of this kernel and
    workload, if it was taken on the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("kernel_sources_sha256_16") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (every 200 ms) of SM clock and throttle reasons."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines: list[str] = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------- our arm

def rotation_sets(w, dev, nbytes_set):
    """Enough copies of the inputs/outputs that one pass over them exceeds
    twice the L2, so consecutive steps read their inputs from HBM."""
    return max(2, math.ceil(2 * L2_BYTES / nbytes_set))


def make_device_inputs(w, dev):
    """The workload's inputs from the seeded CPU recipe (the same values the
    parity tests check), copied to the device."""
    return tuple(t.to(dev) for t in make_workload_inputs(w))


def time_workload(af, w, dev, steps, warmup, soak_s=0.0, sampler=None, dist=None, fp8v=False):
    """Device time per step (ms) of the forward on workload w (``fp8v``: the
    FP8 P.V variant, V given as e5m2 V^T).

    Steps rotate over enough input/output sets that each step reads its
    inputs from HBM, and are replayed from CUDA graphs (the launch loop is
    captured once: per-call host work such as tensor-map encoding is not in
    the timed region, only the kernels).  Returns (ms_per_step, info)."""
    q, k, v = make_device_inputs(w, dev)
    if fp8v:
        v = v.float().to(torch.float8_e5m2).transpose(-1, -2).contiguous()
    per_set = 3 * q.numel() * q.element_size() + v.numel() * v.element_size() + w.B * w.H * w.L * 4
    nsets = rotation_sets(w, dev, per_set)
    sets = []
    for s in range(nsets):
        qs, ks, vs = (q, k, v) if s == 0 else (q.clone(), k.clone(), v.clone())
        sets.append((qs, ks, vs, torch.empty_like(q),
                     torch.empty((w.B, w.H, w.L), dtype=torch.float32, device=dev)))

    def step(i):
        qs, ks, vs, o, lse = sets[i % nsets]
        if fp8v:
            af.fwd_fp8v(qs, ks, vs, w.mask, w.block_size, w.sm_scale, out=o, lse_out=lse)
        else:
            af.fwd(qs, ks, vs, w.mask, w.block_size, w.sm_scale, out=o, lse_out=lse)

    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        for i in range(max(warmup, 1)):
            step(i)
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize(dev)

    chunk = min(steps, max(nsets, 1000 // nsets * nsets))
    graphs = []
    def capture(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(n):
                step(i)
        return g
    full = capture(chunk)
    rem = steps % chunk
    tail = capture(rem) if rem else None
    torch.cuda.synchronize(dev)
    replays = steps // chunk

    def run_timed_region():
        for _ in range(replays):
            full.replay()
        if tail is not None:
            tail.replay()

    if soak_s > 0:
        if sampler:
            sampler.start()
        t_end = time.perf_counter() + soak_s
        while time.perf_counter() < t_end:
            full.replay()
            torch.cuda.synchronize(dev)
    stream = torch.cuda.current_stream(dev)
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    run_timed_region()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    if dist:
        dist.barrier()
    ms = e0.elapsed_time(e1) / steps
    # Spread of the step time, outside the timed region: 30 replays of a graph
    # of nsets steps (one pass over the rotating sets), each timed alone.
    small = capture(nsets)
    samples = []
    for _ in range(30):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        small.replay()
        b.record(stream)
        torch.cuda.synchronize(dev)
        samples.append(a.elapsed_time(b) / nsets)
    samples.sort()
    dist_ms = {"p10": round(samples[3], 5), "median": round(statistics.median(samples), 5),
               "p90": round(samples[26], 5), "replays": 30, "steps_per_replay": nsets}
    st, det = af.last_device_status(dev.index)
    if st != 0:
        raise RuntimeError(f"device status {st} (detail {det:#x}) after the timed region")
    del graphs
    return ms, {"rotating_sets": nsets, "set_bytes": per_set, "graph_launches": chunk,
                "step_ms_spread": dist_ms}


def time_bwd(af, w, dev, steps, warmup):
    """Device time per step (ms) of the backward on workload w: o and lse from
    one forward per input set, dout drawn like the inputs; sets rotate past L2
    and the steps replay from a CUDA graph (three kernels per step)."""
    q, k, v = make_device_inputs(w, dev)
    per_set = 8 * q.numel() * q.element_size()
    nsets = rotation_sets(w, dev, per_set)
    lib = af.load_library()
    sets = []
    for s in range(nsets):
        qs, ks, vs = (q, k, v) if s == 0 else (q.clone(), k.clone(), v.clone())
        g = torch.randn(q.shape, device=dev).to(q.dtype)
        o, lse = af.fwd(qs, ks, vs, w.mask, w.block_size, w.sm_scale)
        ws = torch.empty(max(16, lib.attn_bwd_workspace_size(w.B, w.H, w.L)), dtype=torch.uint8, device=dev)
        sets.append((qs, ks, vs, o, lse, g, torch.empty_like(q), torch.empty_like(q), torch.empty_like(q), ws))

    def step(i):
        qs, ks, vs, o, lse, g, dq, dk, dv, ws = sets[i % nsets]
        af.bwd(qs, ks, vs, o, lse, g, w.mask, w.block_size, w.sm_scale, dq=dq, dk=dk, dv=dv, workspace=ws)

    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        for i in range(max(warmup, 1)):
            step(i)
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(steps):
            step(i)
    torch.cuda.synchronize(dev)
    stream = torch.cuda.current_stream(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    g.replay()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    st, det = af.last_device_status(dev.index)
    if st != 0:
        raise RuntimeError(f"device status {st} (detail {det:#x}) after the backward")
    return e0.elapsed_time(e1) / steps


def time_e2e(af, w, dev, steps, warmup):
    """End to end through the public host API: each step copies q, k, v from
    pinned host memory, runs the forward and copies o and lse back."""
    q, k, v = (t.pin_memory() for t in make_workload_inputs(w))
    staging: dict = {}
    for _ in range(max(warmup, 1)):
        af.fwd_host(q, k, v, w.mask, w.block_size, w.sm_scale, device=dev.index, staging=staging)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(steps):
        af.fwd_host(q, k, v, w.mask, w.block_size, w.sm_scale, device=dev.index, staging=staging)
    dt = (time.perf_counter() - t0) / steps
    h2d = 3 * q.numel() * q.element_size()
    d2h = staging["o_h"].numel() * staging["o_h"].element_size() + staging["lse_h"].numel() * 4
    return dt, h2d, d2h


# ----------------------------------------------------------------- oracle (CPU)

def oracle_sample(w, n_heads: int, reps: int = 1, threads: int | None = None):
    """Time the CPU fp64 oracle on the first n_heads (b, h) heads of workload
    w (all rows of each), reps times over, on `threads` host threads (default
    all); returns (seconds, flops of the sample, threads)."""
    import oracle
    q, k, v = make_workload_inputs(w)
    BH = w.B * w.H
    n_heads = max(1, min(n_heads, BH))
    qf, kf, vf = (t.reshape(BH, 1, w.L, w.D)[:n_heads].contiguous() for t in (q, k, v))
    threads = threads or os.cpu_count() or 1
    oracle.load()
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle.attention(qf, kf, vf, w.mask, w.block_size, w.sm_scale, nthreads=threads)
    dt = time.perf_counter() - t0
    import attention_forward_15_gb300 as af
    flops, _ = af.work(1, n_heads, w.L, w.D, w.mask, w.block_size, w.dtype)
    return dt, flops * reps, threads


def cpu_baseline(w, target_s: float = 10.0):
    """Oracle throughput on the host cores on a bounded sample of workload w
    (calibrated on one head, then enough heads for about target_s seconds; a
    workload whose every head takes less than that is run whole, repeated)."""
    dt1, f1, threads = oracle_sample(w, 1)
    n = max(1, min(w.B * w.H, int(target_s / max(dt1, 1e-3))))
    reps = 1
    if n > 1:
        dt, f, threads = oracle_sample(w, n)
    else:
        dt, f = dt1, f1
    if n == w.B * w.H and dt < 0.5 * target_s:
        reps = max(1, min(64, int(target_s / max(dt, 1e-3))))
        if reps > 1:
            dt, f, threads = oracle_sample(w, n, reps)
    what = f"all {w.L} rows of {n} of the {w.B * w.H} (b,h) heads"
    if reps > 1:
        what += f", the whole workload {reps} times"
    # the same oracle on one thread, one head
    dt_1t, f_1t, _ = oracle_sample(w, 1, threads=1)
    return {"value": f / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{what}, fp64, {dt:.2f} s wall",
            "single_thread": {"value": f_1t / dt_1t / 1e12, "unit": "TFLOP/s", "cores": 1,
                              "sample": f"all {w.L} rows of 1 (b,h) head, fp64, {dt_1t:.2f} s wall"}}


# ----------------------------------------------------------------- ranks

def reduce_max(x: float, dist, dev) -> float:
    """Max of x over all ranks (x itself without a process group)."""
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_step: float, world: int, ms_per_step: float) -> float:
    """Whole-job throughput: every rank runs the same per-rank work, timed by
    the slowest rank."""
    return flops_per_step * world / (ms_per_step * 1e-3) / 1e12


# ----------------------------------------------------------------- main

def roofline_for(w, flops, nbytes, ms, peaks, peaks_kind, traffic):
    t = ms * 1e-3
    tc = peaks["bf16_tflops"]            # fp16 and bf16 have the same dense tensor rate
    bw = peaks["hbm_gbs"]
    t_tensor = flops / (tc * 1e12)
    t_hbm = nbytes / (bw * 1e9)
    if t_tensor >= t_hbm:
        achieved = flops / t / 1e12
        return {"bound": "tensor", "achieved": round(achieved, 2), "peak": tc, "unit": "TFLOP/s",
                "frac": round(achieved / tc, 4), "traffic": traffic,
                "peak_source": f"{peaks_kind} bf16_tflops (burst; fp16 rate equal)"}
    achieved = nbytes / t / 1e9
    return {"bound": "hbm", "achieved": round(achieved, 1), "peak": bw, "unit": "GB/s",
            "frac": round(achieved / bw, 4), "traffic": traffic,
            "peak_source": f"{peaks_kind} hbm_gbs"}


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    w = WORKLOADS[args.workload] if args.shape is None else shape_workload(args.shape)

    if args.impl == "reference":
        if rank != 0:
            return
        run_reference(args, w, world)
        return

    import attention_forward_15_gb300 as af
    from attention_forward_15_gb300 import _build_ext
    if not os.path.exists(_build_ext.lib_path()):
        _build_ext.build()
    af.load_library()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the CUDA library has no CPU path)")
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as tdist
        tdist.init_process_group("nccl", device_id=dev)
        dist = tdist

    peaks, peaks_kind = load_peaks()
    if args.bwd_only:
        fb, _ = af.bwd_work(w.B, w.H, w.L, w.D, w.mask, w.block_size, w.dtype)
        msb = reduce_max(time_bwd(af, w, dev, args.steps, args.warmup), dist, dev)
        if rank == 0:
            print(json.dumps({"metric": "attention bwd TFLOP/s (2.5 x forward flops)", "workload": w.name,
                              "value": round(fb * world / (msb * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
                              "ms_per_step": round(msb, 5), "steps": args.steps, "warmup": args.warmup}),
                  flush=True)
        if dist:
            dist.destroy_process_group()
        return
    if args.fp8v_only:
        f8, _ = af.work(w.B, w.H, w.L, w.D, w.mask, w.block_size, w.dtype)
        ms8, _ = time_workload(af, w, dev, args.steps, args.warmup, fp8v=True)
        ms8 = reduce_max(ms8, dist, dev)
        if rank == 0:
            print(json.dumps({"metric": "attention fwd TFLOP/s, FP8 P.V variant", "workload": w.name,
                              "value": round(f8 * world / (ms8 * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
                              "ms_per_step": round(ms8, 5), "steps": args.steps, "warmup": args.warmup}),
                  flush=True)
        if dist:
            dist.destroy_process_group()
        return
    flops, nbytes = af.work(w.B, w.H, w.L, w.D, w.mask, w.block_size, w.dtype)
    if args.lean:
        args.soak_s, args.no_all = 0.0, True
    sampler = ClockSampler(dev.index) if rank == 0 and not args.lean else None
    ms, info = time_workload(af, w, dev, args.steps, args.warmup, soak_s=args.soak_s,
                             sampler=sampler, dist=dist)
    clocks = sampler.stop() if sampler else None
    ms = reduce_max(ms, dist, dev)

    if dist:
        dist.barrier()
    e2e_s, h2d, d2h = (None, 0, 0) if args.lean else \
        time_e2e(af, w, dev, max(10, min(args.steps, 200)), 3)
    if e2e_s is not None:
        e2e_s = reduce_max(e2e_s, dist, dev)

    per_mask = {}
    if not args.no_all:
        for name, ow in WORKLOADS.items():
            if name == w.name:
                continue
            f2, b2 = af.work(ow.B, ow.H, ow.L, ow.D, ow.mask, ow.block_size, ow.dtype)
            steps2 = max(5, min(args.steps, int(2e12 / f2) + 5, 200))
            ms2, _ = time_workload(af, ow, dev, steps2, 3)
            rl = roofline_for(ow, f2, b2, ms2, peaks, peaks_kind, ncu_traffic(name))
            # end to end through the host-buffer call, as for the main line
            e2e2, _, _ = time_e2e(af, ow, dev, 10, 2)
            per_mask[name] = {"mask": MASK_NAMES[ow.mask], "ms": round(ms2, 4),
                              "tflops": round(f2 / (ms2 * 1e-3) / 1e12, 2),
                              "roofline_bound": rl["bound"], "roofline_frac": rl["frac"],
                              "achieved": rl["achieved"], "unit": rl["unit"],
                              "e2e_ms": round(e2e2 * 1e3, 4),
                              "e2e_tflops": round(f2 / e2e2 / 1e12, 2)}
    # The FP8 P.V variant (V as e5m2, P rounded to e5m2) on three workloads.
    fp8_pv = {}
    if not args.no_all:
        for name in (w.name, "causal_b2h32l4096d128_bf16", "dense_b1h16l16384d256_bf16"):
            ow = WORKLOADS[name]
            f2, b2 = af.work(ow.B, ow.H, ow.L, ow.D, ow.mask, ow.block_size, ow.dtype)
            steps2 = max(5, min(args.steps, int(2e12 / f2) + 5, 200))
            ms2, _ = time_workload(af, ow, dev, steps2, 3, fp8v=True)
            fp8_pv[name] = {"mask": MASK_NAMES[ow.mask], "ms": round(ms2, 4),
                            "tflops": round(f2 / (ms2 * 1e-3) / 1e12, 2),
                            "frac_of_bf16_peak": round(f2 / (ms2 * 1e-3) / 1e12 / peaks["bf16_tflops"], 4)}
    # The backward (attn_bwd: dQ, dK, dV) at D = 64, 128 and 256.
    bwd_lines = {}
    if not args.no_all:
        for name in (w.name, "causal_b2h32l4096d128_bf16", "dense_b1h16l16384d256_bf16"):
            ow = WORKLOADS[name]
            fb, _ = af.bwd_work(ow.B, ow.H, ow.L, ow.D, ow.mask, ow.block_size, ow.dtype)
            msb = time_bwd(af, ow, dev, 40 if ow.L >= 4096 else 100, 3)
            bwd_lines[name] = {"mask": MASK_NAMES[ow.mask], "ms": round(msb, 4),
                               "tflops": round(fb / (msb * 1e-3) / 1e12, 2),
                               "frac_of_bf16_peak": round(fb / (msb * 1e-3) / 1e12 / peaks["bf16_tflops"], 4),
                               "flops": "2.5 x the forward's (S, dP, dV, dK, dQ)"}
    if dist:
        dist.barrier()
    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return

    value = job_tflops(flops, world, ms)
    cfg = w.describe()
    cfg.update({"parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                "l2": f"{info['rotating_sets']} rotating input/output sets of "
                      f"{info['set_bytes'] / 2**20:.1f} MiB (> 2x the 129 MB L2)",
                "launch": f"CUDA graph replay of {info['graph_launches']} launches",
                "flops_per_step": flops, "bytes_per_step": nbytes,
                "step_ms_spread": info["step_ms_spread"],
                "clocks_note": f"sampled over a {args.soak_s:.1f} s soak of the same graph "
                               "immediately before the timed region"})
    out = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16" if w.dtype == torch.float16 else "bf16", "data": "synthetic",
        "config": cfg,
        "roofline": roofline_for(w, flops, nbytes, ms, peaks, peaks_kind, ncu_traffic(w.name)),
        "e2e": None if e2e_s is None else {
            "value": round(job_tflops(flops, world, e2e_s * 1e3), 3), "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(e2e_s * 1e3, 4)},
        "gpu_launches": args.steps,
        "clocks": clocks,
        "per_workload": per_mask or None,
        "fp8_pv_variant": fp8_pv or None,
        "backward": bwd_lines or None,
    }
    out["cpu_baseline"] = None if args.lean else cpu_baseline(w)
    print(json.dumps(out), flush=True)
    if dist:
        dist.destroy_process_group()


def shape_workload(spec: str):
    """A workload from "B,H,L,D,MASK,DTYPE[,BS]" (sm_scale 1/sqrt(D), seed 42, N(0, 1))."""
    from attn_inputs import Workload
    f = spec.split(",")
    if len(f) not in (6, 7):
        raise SystemExit("--shape wants B,H,L,D,MASK,DTYPE[,BS]")
    masks = {v: k for k, v in MASK_NAMES.items()}
    dtypes = {"fp16": torch.float16, "bf16": torch.bfloat16}
    if f[4] not in masks or f[5] not in dtypes:
        raise SystemExit(f"--shape: MASK one of {sorted(masks)}, DTYPE one of {sorted(dtypes)}")
    B, H, L, D = (int(x) for x in f[:4])
    mask = masks[f[4]]
    dt = dtypes[f[5]]
    bs = int(f[6]) if len(f) == 7 else 0
    if (mask == masks["block_diag"]) != (bs > 0) or (bs > 0 and L % bs):
        raise SystemExit("--shape: a block size (dividing L) for block_diag, and only for it")
    return Workload(f"{f[4]}_b{B}h{H}l{L}d{D}_{f[5]}" + (f"_bs{bs}" if bs else ""), B, H, L, D, mask, dt,
                    1.0 / math.sqrt(D), bs)


def attended_pairs(w) -> float:
    """Attended (i, j) pairs of one head: L^2 dense, L(L+1)/2 causal, L*bs
    block-diagonal."""
    if w.mask == 0:
        return float(w.L) * w.L
    if w.mask == 1:
        return w.L * (w.L + 1) / 2.0
    return float(w.L) * w.block_size


def run_reference(args, w, world):
    """The oracle as the reference arm: each step computes one (b,h) head of
    the workload in fp64 on the host cores."""
    import oracle
    q, k, v = make_workload_inputs(w)
    BH = w.B * w.H
    threads = args.threads or os.cpu_count() or 1
    oracle.load()
    heads = [t.reshape(BH, 1, w.L, w.D) for t in (q, k, v)]

    def step(i):
        h = i % BH
        oracle.attention(heads[0][h:h + 1], heads[1][h:h + 1], heads[2][h:h + 1], w.mask,
                         w.block_size, w.sm_scale, nthreads=threads)
    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(i)
    dt = (time.perf_counter() - t0) / args.steps
    f_head = 4.0 * w.D * attended_pairs(w)
    value = f_head / dt / 1e12
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": w.describe(),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"one (b,h) head of {BH} per step, all {w.L} rows, fp64"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


if __name__ == "__main__":
    main()
