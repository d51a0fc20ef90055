#!/usr/bin/env python3
"""Throughput of the fused adaLN row kernels on one GB300 (or N replicas).

Metric: fused norm+modulate achieved HBM GB/s and % of the GB300 roofline;
rows/s.  A step is one pass of the FLUX.1-shaped LayerNorm + modulate site
over one batch: x [1, 4608, 3072] and its CFG pair x [2, 4608, 3072] with
per-batch scale/shift rows (two launches of ln_modulate).  Algorithmic bytes
are the minimum traffic: read x, scale, shift once, write out once.

Inputs are seeded synthetic tensors (workloads.py), resident in HBM, rotated
over enough buffer sets that every timed step reads from DRAM, not L2.  The
timed region is bracketed by a barrier and a device synchronise; kernels are
timed with CUDA events on the stream they run on.  Besides the headline the
JSON line carries: the roofline of the dominant kernel, the oracle timed on
the host cores (cpu_baseline), an end-to-end number through the C ABI from
pinned host buffers (e2e), sampled SM clocks, and a per-entry-point table on
the other model-site shapes.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl rmsmod|reference]

For N > 1 launch one process per GPU (torchrun); every rank runs its own
replica of the step (weak scaling, no data-path collective).
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused norm+modulate achieved HBM GB/s and % of GB300 roofline; rows/s"
WORKLOAD = "flux_ln_modulate_1x4608x3072+cfg_2x4608x3072"
NOMINAL_HBM_GBS = 8000.0
# ~20 ms of GPU sleep before a timed burst, so launches queue up ahead
PRIME_CYCLES = 40_000_000
FALLBACK_HBM_GBS = 6800.0


# --------------------------------------------------------------------------
# small utilities
# --------------------------------------------------------------------------

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            p = json.load(fh)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def timed_over_ranks(pg, device, run):
    """The timed region of one replica per rank: a barrier on both sides of
    `run()`, which returns this rank's device-timed milliseconds (with a
    device synchronise on both sides of its events), then the maximum over
    the ranks -- the job ends with its slowest replica."""
    if pg is not None:
        pg.barrier()
    ms = run()
    if pg is not None:
        pg.barrier()
        import torch

        t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
        pg.all_reduce(t, op=pg.ReduceOp.MAX)
        ms = float(t.item())
    return ms


def job_throughput(world, units_per_replica, steps, total_ms):
    """Whole-job throughput: the units every rank processed over the
    max-over-ranks time (weak scaling: each replica runs the full step)."""
    return world * units_per_replica * steps / (total_ms * 1e-3)


def emit(rank, line):
    """One JSON line, from rank 0 only."""
    if rank == 0:
        print(json.dumps(line), flush=True)


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling in the background."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.tmp = None
        self.marks = []

    def start(self):
        self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu=timestamp,{self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.tmp, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def mark(self, label):
        self.marks.append((label, time.time()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        rows = []
        try:
            with open(self.tmp.name) as fh:
                for line in fh:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) >= 9:
                        rows.append(parts)
            os.unlink(self.tmp.name)
        except Exception:
            pass
        return rows

    @staticmethod
    def summarise(rows):
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        smax = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        reasons = set()
        for r in rows:
            for name, v in zip(names[1:], r[5:9]):
                if v.strip().lower() in ("active", "0x1", "yes"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(rows)}


# --------------------------------------------------------------------------
# the reference arm: the CPU oracle, as it stands
# --------------------------------------------------------------------------

def run_reference(args, rank, world):
    if rank != 0:
        return 0
    import numpy as np

    import oracle
    import workloads as W

    oracle.build()
    B1 = W.WORKLOADS["ln_modulate_flux_1x4608x3072"].make()
    B2 = W.WORKLOADS["ln_modulate_flux_cfg_2x4608x3072"].make()
    # bounded sample per step: 8 rows of the B=1 tensor and 8 rows of each
    # CFG batch (16 rows), the same mix as the GPU step
    r1, r2 = 8, 8
    x1 = np.ascontiguousarray(B1["x"][:, :r1])
    x2 = np.ascontiguousarray(B2["x"][:, :r2])
    D = B1["D"]
    rows = r1 + 2 * r2
    step_bytes = rows * D * 4 + 2 * D * 2 + 2 * 2 * D * 2

    def step():
        oracle.ln_modulate(x1, B1["scale"], B1["shift"])
        oracle.ln_modulate(x2, B2["scale"], B2["shift"])

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    value = step_bytes * args.steps / dt / 1e9
    sample = (f"per step {rows} rows of D=3072 ({r1} of x[1,4608,3072], {r2} per CFG batch of "
              f"x[2,4608,3072]), single-threaded C oracle")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "rows_per_step": rows},
        "rows_per_s": rows * args.steps / dt,
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# --------------------------------------------------------------------------
# the CUDA arm
# --------------------------------------------------------------------------

# sources each kernel is built from (a change to any of them makes a stored
# DRAM-traffic figure stale)
KERNEL_SOURCES = {
    "row_kernel": ("row_kernels.cu", "device_common.cuh", "launch.h"),
    "row_kernel_ws": ("row_kernels.cu", "device_common.cuh", "launch.h"),
    "row_kernel_coop": ("row_kernels.cu", "device_common.cuh", "launch.h"),
    "qk_kernel": ("qk_kernel.cu", "device_common.cuh", "launch.h"),
    "wan_kernel": ("wan_kernel.cu", "device_common.cuh", "launch.h"),
    "bwd_ws_kernel": ("backward.cu", "device_common.cuh", "launch.h"),
    "tokens_top_kernel": ("backward.cu", "device_common.cuh", "launch.h"),
    "ew_kernel": ("elementwise.cu", "device_common.cuh", "launch.h"),
}


# the dominant kernel of each per-entry-point table row (for its traffic record)
ROW_KERNEL = {
    "ln_modulate_flux_1x4608x3072": "row_kernel_ws",
    "ln_modulate_flux_2x4608x3072": "row_kernel_ws",
    "rmsnorm_modulate_1x4216x4096": "row_kernel_ws",
    "gated_rmsnorm_modulate_1x4216x4096": "row_kernel_ws",
    "ln_modulate_folded_flux_2x4608x3072": "row_kernel_ws",
    "qk_layernorm_1x4352x32x128": "qk_kernel",
    "qk_layernorm_qkv_strided_1x4352x32x128": "qk_kernel",
    "rmsnorm_silu_cl_wan_c96": "wan_kernel",
    "rmsnorm_silu_cl_wan_c192": "wan_kernel",
    "rmsnorm_silu_cl_wan_c384": "wan_kernel",
    "modulate_scale_shift_bf16_1x4608x3072": "ew_kernel",
    "modulate_scale_shift_f16_1x4608x3072": "ew_kernel",
    "residual_gate_add_1x4216x4096": "ew_kernel",
    "conv_bias_epilogue_wan_c96": "ew_kernel",
    "conv_bias_epilogue_residual_wan_c96": "ew_kernel",
    "ln_modulate_backward_flux_1x4608x3072": "bwd_ws_kernel",
}


def source_digest(kernel: str) -> str:
    import hashlib

    src = os.path.join(ROOT, "rmsnorm_modulate_gb300", "csrc")
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(src, f), "rb") as fh:
            h.update(f.encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_record(kernel: str, workload: str):
    """DRAM bytes (read + write) per launch from the committed ncu summary
    table, if it was taken on the kernel's current source (each row records
    the digest of the sources the kernel is built from)."""
    path = os.path.join(ROOT, "profiles", "traffic.md")
    digest = source_digest(kernel)
    try:
        with open(path) as fh:
            for line in fh:
                cells = [c.strip() for c in line.strip().strip("|").split("|")]
                if len(cells) >= 4 and cells[0] == kernel and cells[1] == workload:
                    if cells[2] == digest:
                        return int(float(cells[3]))
    except OSError:
        pass
    return None


def cpu_baseline(seconds: float):
    import numpy as np

    import oracle
    import workloads as W

    oracle.build()
    B1 = W.WORKLOADS["ln_modulate_flux_1x4608x3072"].make()
    x = np.ascontiguousarray(B1["x"][:, :64])
    D = B1["D"]
    per = 64 * D * 4 + 2 * D * 2
    n = 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        oracle.ln_modulate(x, B1["scale"], B1["shift"])
        n += 1
    dt = time.perf_counter() - t0
    line = {"value": per * n / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{n} calls x 64 rows of x[1,4608,3072] (D=3072) through the single-"
                      f"threaded C oracle, {dt:.1f} s"}
    # the same oracle, row-parallel: one host thread per core, each calling
    # the (unchanged, single-threaded) C oracle on its own 64-row block of
    # x[1,4608,3072] (ctypes releases the interpreter lock during the call)
    from concurrent.futures import ThreadPoolExecutor

    cores = min(len(os.sched_getaffinity(0)), 4608 // 64)
    blocks = [np.ascontiguousarray(B1["x"][:, 64 * i:64 * (i + 1)]) for i in range(cores)]

    def work(xb):
        k = 0
        t_end = time.perf_counter() + seconds / 2
        while time.perf_counter() < t_end:
            oracle.ln_modulate(xb, B1["scale"], B1["shift"])
            k += 1
        return k

    t0 = time.perf_counter()
    with ThreadPoolExecutor(max_workers=cores) as ex:
        calls = sum(ex.map(work, blocks))
    dt = time.perf_counter() - t0
    line["row_parallel"] = {
        "value": per * calls / dt / 1e9, "unit": "GB/s", "cores": cores,
        "sample": f"{calls} calls x 64 rows on {cores} threads (one 64-row block each), "
                  f"{dt:.1f} s"}
    return line


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="rmsmod", choices=["rmsmod", "reference"])
    ap.add_argument("--no-kernels", action="store_true", help="skip the per-entry-point table")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--only", default=None,
                    help="time only the per-entry-point table rows whose name contains this "
                         "text (a small, fixed-shape run for profilers); prints one JSON line")
    ap.add_argument("--iters", type=int, default=200, help="launches per table row")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    rank, world, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if args.only is not None:
        return run_only(args, local)

    import numpy as np
    import torch

    import workloads as W
    from rmsnorm_modulate_gb300 import _build

    if rank == 0:
        _build.build()
    torch.cuda.set_device(local)
    pg = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        pg = dist
        if rank != 0:
            _build.build()  # no-op once rank 0 has built
        dist.barrier()
    import rmsnorm_modulate_gb300 as rm

    lib = rm.library()
    dev = torch.device("cuda", local)
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 126 * 2 ** 20))
    peak, peak_kind = peaks()

    # ---- inputs (identical bits to the test-suite's) --------------------
    def to_dev(bits):
        a = np.ascontiguousarray(bits)
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)

    w1 = W.WORKLOADS["ln_modulate_flux_1x4608x3072"].make()
    w2 = W.WORKLOADS["ln_modulate_flux_cfg_2x4608x3072"].make()
    D = w1["D"]
    rows1, rows2 = w1["B"] * w1["S"], w2["B"] * w2["S"]
    sc1, sh1 = to_dev(w1["scale"]), to_dev(w1["shift"])
    sc2, sh2 = to_dev(w2["scale"]), to_dev(w2["shift"])
    x1_0, x2_0 = to_dev(w1["x"]), to_dev(w2["x"])
    set_bytes = (rows1 + rows2) * D * 2 * 2
    nsets = max(2, -(-4 * l2 // set_bytes) + 1)
    sets = []
    for i in range(nsets):
        x1 = x1_0 if i == 0 else x1_0.clone()
        x2 = x2_0 if i == 0 else x2_0.clone()
        sets.append((x1, x2, torch.empty_like(x1), torch.empty_like(x2)))
    step_bytes = rows1 * D * 4 + 2 * D * 2 + rows2 * D * 4 + 2 * 2 * D * 2
    step_rows = rows1 + rows2
    # the two launches per step as ready-made C-ABI argument tuples
    stream = torch.cuda.Stream(device=dev)
    sp = ctypes.c_void_p(stream.cuda_stream)
    P = ctypes.c_void_p
    calls = []
    for x1, x2, o1, o2 in sets:
        calls.append(((P(x1.data_ptr()), P(sc1.data_ptr()), P(sh1.data_ptr()), P(o1.data_ptr()),
                       1, rows1, D, 0, ctypes.c_float(1e-6), None, None, sp),
                      (P(x2.data_ptr()), P(sc2.data_ptr()), P(sh2.data_ptr()), P(o2.data_ptr()),
                       2, w2["S"], D, D, ctypes.c_float(1e-6), None, None, sp)))
    f = lib.ln_modulate

    def launch(i):
        a, b = calls[i % nsets]
        if f(*a) != 0 or f(*b) != 0:
            raise RuntimeError("ln_modulate launch failed")

    uuid = getattr(props, "uuid", None)
    gpu_id = f"GPU-{uuid}" if uuid is not None else str(local)
    sampler = ClockSampler(gpu_id)
    sampler.start()

    # ---- warm-up (plus a short untimed ramp so clocks settle) ------------
    torch.cuda.synchronize(dev)  # the input sets were copied on the default stream
    with torch.cuda.stream(stream):
        t_ramp = time.time()
        i = 0
        while i < args.warmup or time.time() - t_ramp < 0.3:
            launch(i)
            i += 1
            if i % 256 == 0:
                stream.synchronize()
        stream.synchronize()

    # ---- timed region -----------------------------------------------------
    # A short GPU sleep first lets the host queue launches ahead of the GPU,
    # so the K steps run back to back; CUDA events on the launch stream
    # bracket exactly the K steps (the sleep lies before the start event).
    def timed_steps():
        e_start = torch.cuda.Event(enable_timing=True)
        e_end = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        sampler.mark("timed_start")
        with torch.cuda.stream(stream):
            torch.cuda._sleep(PRIME_CYCLES)
            e_start.record(stream)
            for i in range(args.steps):
                a, b = calls[i % nsets]
                if f(*a) != 0 or f(*b) != 0:
                    raise RuntimeError("ln_modulate launch failed")
            e_end.record(stream)
        torch.cuda.synchronize(dev)
        sampler.mark("timed_end")
        return e_start.elapsed_time(e_end)

    total_ms = timed_over_ranks(pg, dev, timed_steps)
    ms_per_step = total_ms / args.steps
    value = job_throughput(world, step_bytes, args.steps, total_ms) / 1e9
    # the dominant (and only) kernel of the step is ln_modulate; its average
    # launch moves step_bytes / 2 in ms_per_step / 2
    achieved = step_bytes / (ms_per_step * 1e-3) / 1e9
    b1 = rows1 * D * 4 + 2 * D * 2
    b2 = rows2 * D * 4 + 2 * 2 * D * 2

    # per-launch split (outside the timed region): each shape back to back
    def back_to_back(which, n=200):
        with torch.cuda.stream(stream):
            torch.cuda._sleep(PRIME_CYCLES)
            s0 = torch.cuda.Event(enable_timing=True)
            s1 = torch.cuda.Event(enable_timing=True)
            s0.record(stream)
            for i in range(n):
                if f(*calls[i % nsets][which]) != 0:
                    raise RuntimeError("ln_modulate launch failed")
            s1.record(stream)
        torch.cuda.synchronize(dev)
        return s0.elapsed_time(s1) / n

    # the same bytes moved by a plain device-to-device copy (x -> out, the
    # same rotating buffers, timed the same way): the practical ceiling of a
    # launch this short
    def copy_back_to_back(which, n=200):
        with torch.cuda.stream(stream):
            torch.cuda._sleep(PRIME_CYCLES)
            s0 = torch.cuda.Event(enable_timing=True)
            s1 = torch.cuda.Event(enable_timing=True)
            s0.record(stream)
            for i in range(n):
                st = sets[i % nsets]
                st[2 + which].copy_(st[which])
            s1.record(stream)
        torch.cuda.synchronize(dev)
        return s0.elapsed_time(s1) / n

    t1, t2 = back_to_back(0), back_to_back(1)
    c1, c2 = copy_back_to_back(0), copy_back_to_back(1)
    per_launch = {
        "ln_modulate_1x4608x3072": {"us": 1e3 * t1, "gbs": b1 / (t1 * 1e-3) / 1e9,
                                    "copy_us": 1e3 * c1, "of_copy_speed": c1 / t1},
        "ln_modulate_2x4608x3072": {"us": 1e3 * t2, "gbs": b2 / (t2 * 1e-3) / 1e9,
                                    "copy_us": 1e3 * c2, "of_copy_speed": c2 / t2},
    }
    # DRAM bytes of the average launch (the step is one launch of each shape)
    t_b1 = traffic_record("row_kernel_ws", "ln_modulate_flux_1x4608x3072")
    t_b2 = traffic_record("row_kernel_ws", "ln_modulate_flux_2x4608x3072")
    traffic = (t_b1 + t_b2) / 2 if t_b1 is not None and t_b2 is not None else None

    # ---- end to end through the binding from pinned host buffers ---------
    # Every step copies its inputs host -> device, runs the two launches and
    # copies both outputs device -> host.  Steps are pipelined over two
    # buffer sets and three streams (the copy engines of both directions and
    # the SMs work on different steps at once); all of every step's copies lie
    # inside the timed region.
    e2e = None
    if not args.no_e2e:
        nset = 2
        hx1 = [torch.empty(x1_0.shape, dtype=torch.bfloat16).pin_memory() for _ in range(nset)]
        hx2 = [torch.empty(x2_0.shape, dtype=torch.bfloat16).pin_memory() for _ in range(nset)]
        for h_ in hx1:
            h_.copy_(x1_0.cpu())
        for h_ in hx2:
            h_.copy_(x2_0.cpu())
        ho1 = [torch.empty_like(hx1[0]).pin_memory() for _ in range(nset)]
        ho2 = [torch.empty_like(hx2[0]).pin_memory() for _ in range(nset)]
        hmod = [[t.cpu().pin_memory() for t in (sc1, sh1, sc2, sh2)] for _ in range(nset)]
        dx1 = [sets[k][0] for k in range(nset)]
        dx2 = [sets[k][1] for k in range(nset)]
        do1 = [sets[k][2] for k in range(nset)]
        do2 = [sets[k][3] for k in range(nset)]
        dmod = [[torch.empty_like(t) for t in (sc1, sh1, sc2, sh2)] for _ in range(nset)]
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event() for _ in range(nset)]
        ev_run = [torch.cuda.Event() for _ in range(nset)]
        ev_out = [torch.cuda.Event() for _ in range(nset)]
        e_steps = max(3, min(args.steps, 200))

        def e2e_step(i):
            k = i % nset
            with torch.cuda.stream(s_in):
                s_in.wait_event(ev_run[k])          # step i - 2 is done reading set k
                dx1[k].copy_(hx1[k], non_blocking=True)
                dx2[k].copy_(hx2[k], non_blocking=True)
                for d_, h_ in zip(dmod[k], hmod[k]):
                    d_.copy_(h_, non_blocking=True)
                ev_in[k].record(s_in)
            stream.wait_event(ev_in[k])
            stream.wait_event(ev_out[k])            # step i - 2's outputs have left set k
            sc1d, sh1d, sc2d, sh2d = dmod[k]
            rm.ln_modulate(dx1[k], sc1d, sh1d, out=do1[k], stream=stream)
            rm.ln_modulate(dx2[k], sc2d, sh2d, out=do2[k], stream=stream)
            ev_run[k].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_run[k])
                ho1[k].copy_(do1[k], non_blocking=True)
                ho2[k].copy_(do2[k], non_blocking=True)
                ev_out[k].record(s_out)

        for i in range(4):
            e2e_step(i)
        torch.cuda.synchronize(dev)

        def timed_e2e():
            s0 = torch.cuda.Event(enable_timing=True)
            s1 = torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize(dev)
            with torch.cuda.stream(s_in):
                torch.cuda._sleep(PRIME_CYCLES)
                s0.record(s_in)
            for i in range(e_steps):
                e2e_step(i)
            s_out.wait_event(ev_run[(e_steps - 1) % nset])
            with torch.cuda.stream(s_out):
                s1.record(s_out)
            torch.cuda.synchronize(dev)
            return s0.elapsed_time(s1)

        e_ms = timed_over_ranks(pg, dev, timed_e2e)
        h2d = (hx1[0].numel() + hx2[0].numel() + sum(t.numel() for t in hmod[0])) * 2
        d2h = (ho1[0].numel() + ho2[0].numel()) * 2
        e2e = {"value": job_throughput(world, step_bytes, e_steps, e_ms) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e_steps,
               "ms_per_step": e_ms / e_steps,
               "pipelining": "2 buffer sets, host->device / compute / device->host on 3 streams"}

    # ---- the other entry points on their model-site shapes ---------------
    kernels = None
    if not args.no_kernels:
        kernels = kernel_table(rm, lib, dev, stream, l2, peak)
    clocks = ClockSampler.summarise(sampler.stop())

    if rank != 0:
        if pg is not None:
            pg.destroy_process_group()
        return 0
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "rows_per_step": step_rows, "D": D,
                   "bytes_per_step": step_bytes,
                   "l2": f"{nsets} rotating input/output sets, {nsets * set_bytes / 2**20:.0f} "
                         f"MiB > 4x the {l2 / 2**20:.0f} MiB L2",
                   "parallelism": f"replicas x{world}"},
        "rows_per_s": job_throughput(world, step_rows, args.steps, total_ms),
        "pct_of_roofline": 100.0 * value / world / peak,
        "pct_of_nominal_8tbs": 100.0 * value / world / NOMINAL_HBM_GBS,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": "row_kernel_ws<LN, V=12> (ln_modulate, D=3072: statistics and "
                               "output warps around a 16-row TMA ring; 4 + 8 warps for the "
                               "16-row items of B=1, 8 + 4 for the 31-row items of B=2)",
                     "traffic_per": "average launch of the step (B=1 and B=2 shapes), steady "
                                    "state: mean of 8 back-to-back launches per shape, each "
                                    "carrying the previous launch's L2 write-back",
                     "peak_kind": f"{peak_kind} copy bandwidth (burst)",
                     "algorithmic_bytes_per_launch": {"B1": b1, "B2": b2}},
        "per_launch": per_launch,
        "gpu_launches": 2 * args.steps,
        "clocks": clocks,
        "e2e": e2e,
        "cpu_baseline": cpu_baseline(args.cpu_seconds) if world == 1 else None,
        "kernels": kernels,
    }
    emit(rank, line)
    if pg is not None:
        pg.destroy_process_group()
    return 0


def run_only(args, local):
    import torch

    from rmsnorm_modulate_gb300 import _build

    _build.build()
    import rmsnorm_modulate_gb300 as rm

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 126 * 2 ** 20))
    peak, _ = peaks()
    stream = torch.cuda.Stream(device=dev)
    rows = kernel_table(rm, rm.library(), dev, stream, l2, peak, iters=args.iters,
                        only=args.only)
    print(json.dumps({"only": args.only, "kernels": rows}))
    return 0


def kernel_table(rm, lib, dev, stream, l2, peak, iters=200, only=None):
    """Every fused entry point on its model-site shape: median launch time
    over rotating buffers, achieved GB/s against the algorithmic bytes.
    Inputs are drawn on the device (seeded, same distributions as
    workloads.py); these rows measure speed only."""
    import torch

    import workloads as W

    g = torch.Generator(device=dev)
    g.manual_seed(0)

    def normal(shape, std=1.0, mean=0.0, dtype=torch.bfloat16):
        t = torch.randn(*shape, generator=g, device=dev, dtype=torch.float32)
        return (t * std + mean).to(dtype)

    rows = {}

    def want(name):
        return only is None or only in name

    def timed(name, bytes_, nrows, calls):
        """Launches back to back after a GPU sleep (the host runs ahead), timed
        as a burst by two events; per launch = burst / launches."""
        nsets = len(calls)
        # the inputs were drawn on the default stream; the launches run on
        # `stream`: finish the draws first (an in-place row would otherwise
        # race its own inputs, and a row that read an unfinished buffer keeps
        # whatever it wrote)
        torch.cuda.synchronize(dev)
        with torch.cuda.stream(stream):
            for i in range(5):
                calls[i % nsets]()
            stream.synchronize()
            # the host cost of one call (binding checks, views): the GPU sleep
            # must outlast queueing all `iters` calls, or the burst would time
            # the host
            h0 = time.perf_counter()
            for i in range(5):
                calls[i % nsets]()
            host_s = (time.perf_counter() - h0) / 5
            stream.synchronize()
            torch.cuda._sleep(max(PRIME_CYCLES, int(3 * iters * host_s * 2.1e9)))
            s0 = torch.cuda.Event(enable_timing=True)
            s1 = torch.cuda.Event(enable_timing=True)
            s0.record(stream)
            q0 = time.perf_counter()
            for i in range(iters):
                calls[i % nsets]()
            queue_s = (time.perf_counter() - q0) / iters
            s1.record(stream)
        torch.cuda.synchronize(dev)
        per = s0.elapsed_time(s1) / iters
        gbs = bytes_ / (per * 1e-3) / 1e9
        rows[name] = {"us": per * 1e3, "gbs": gbs, "frac": gbs / peak,
                      "frac_nominal_8tbs": gbs / NOMINAL_HBM_GBS, "host_us": host_s * 1e6,
                      # host time per call while queueing the burst: well below
                      # "us" means the launches ran back to back on the GPU
                      "host_queue_us": queue_s * 1e6,
                      "rows_per_s": nrows / (per * 1e-3), "bytes": bytes_, "sets": nsets,
                      # every buffer the rotation touches fits in L2 (small shapes)
                      "l2_resident": nsets * bytes_ < l2}
        kern = ROW_KERNEL.get(name)
        if kern is not None:
            # steady-state DRAM bytes per launch from the committed ncu table
            # (only while the kernel's sources match the recorded digest)
            rows[name]["traffic"] = traffic_record(kern, name)
            rows[name]["traffic_kernel"] = kern

    def nsets_for(set_bytes):
        """Enough rotating sets that each launch's buffers were evicted from L2."""
        return 1 if set_bytes >= 4 * l2 else min(16, -(-4 * l2 // set_bytes) + 1)

    # LayerNorm + modulate: the small config (L2-resident at any rotation,
    # latency-bound) and the FLUX.1 site with B = 1 and the CFG pair
    name = "ln_modulate_1x256x1024"
    if want(name):
        x = normal((1, 256, 1024))
        sc, sh = normal((1, 1, 1024), 0.1), normal((1, 1, 1024), 0.1)
        outs = [torch.empty_like(x) for _ in range(8)]
        timed(name, 256 * 1024 * 4 + 4 * 1024, 256,
              [lambda o=o: rm.ln_modulate(x, sc, sh, out=o, stream=stream) for o in outs])
    # the same small launch as a CUDA graph of 1000 launches (no host in the
    # loop): what one launch costs the GPU when nothing else hides it
    name = "ln_modulate_1x256x1024_graph1000"
    if want(name):
        x = normal((1, 256, 1024))
        sc, sh = normal((1, 1, 1024), 0.1), normal((1, 1, 1024), 0.1)
        outs = [torch.empty_like(x) for _ in range(8)]
        cap = torch.cuda.Stream(device=dev)
        torch.cuda.synchronize(dev)  # inputs drawn on the default stream
        with torch.cuda.stream(cap):
            for o in outs:  # first calls (launch attributes) outside the capture
                rm.ln_modulate(x, sc, sh, out=o, stream=cap)
        cap.synchronize()
        graph = torch.cuda.CUDAGraph()
        try:
            with torch.cuda.graph(graph, stream=cap):
                for i in range(1000):
                    rm.ln_modulate(x, sc, sh, out=outs[i % 8], stream=cap)
        except Exception as exc:  # capture refused: report it, keep the table
            rows[name] = {"error": f"{type(exc).__name__}: {exc}"[:200]}
            graph = None
    if want(name) and graph is not None:
        with torch.cuda.stream(cap):
            graph.replay()
            cap.synchronize()
            torch.cuda._sleep(PRIME_CYCLES)
            s0 = torch.cuda.Event(enable_timing=True)
            s1 = torch.cuda.Event(enable_timing=True)
            s0.record(cap)
            graph.replay()
            s1.record(cap)
        torch.cuda.synchronize(dev)
        per = s0.elapsed_time(s1) / 1000
        bytes_ = 256 * 1024 * 4 + 4 * 1024
        rows[name] = {"us": per * 1e3, "gbs": bytes_ / (per * 1e-3) / 1e9,
                      "frac": bytes_ / (per * 1e-3) / 1e9 / peak, "launches": 1000,
                      "rows_per_s": 256 / (per * 1e-3), "bytes": bytes_, "sets": 8}
        del graph
    for B in (1, 2):
        name = f"ln_modulate_flux_{B}x4608x3072"
        if not want(name):
            continue
        S, D = 4608, 3072
        n = nsets_for(B * S * D * 4)
        xs = [normal((B, S, D)) for _ in range(n)]
        sc, sh = normal((B, 1, D), 0.1), normal((B, 1, D), 0.1)
        os_ = [torch.empty_like(xs[0]) for _ in range(n)]
        timed(name, B * S * D * 4 + 2 * B * D * 2, B * S,
              [lambda a=a, o=o: rm.ln_modulate(a, sc, sh, out=o, stream=stream)
               for a, o in zip(xs, os_)])
        del xs, os_

    # the FLUX.1 text stream (1, 512, 3072): a short launch, L2-resident
    name = "ln_modulate_flux_text_1x512x3072"
    if want(name):
        S, D = 512, 3072
        n = nsets_for(S * D * 4)
        xs = [normal((1, S, D)) for _ in range(n)]
        sc, sh = normal((1, 1, D), 0.1), normal((1, 1, D), 0.1)
        os_ = [torch.empty_like(xs[0]) for _ in range(n)]
        timed(name, S * D * 4 + 2 * D * 2, S,
              [lambda a=a, o=o: rm.ln_modulate(a, sc, sh, out=o, stream=stream)
               for a, o in zip(xs, os_)])
        del xs, os_

    # the standalone elementwise chains: FLUX.1's modulate at the image and
    # text stream shapes (bf16 and fp16), ERNIE-Image's residual gate, the
    # Wan VAE conv-bias epilogue with and without the residual h
    for S in (4608, 512):
        for dt, tag in ((torch.bfloat16, "bf16"), (torch.float16, "f16")):
            name = f"modulate_scale_shift_{tag}_1x{S}x3072"
            if not want(name):
                continue
            D = 3072
            n = nsets_for(S * D * 4)
            ys = [normal((1, S, D), dtype=dt) for _ in range(n)]
            sc, sh = normal((1, 1, D), 0.1, dtype=dt), normal((1, 1, D), 0.1, dtype=dt)
            os_ = [torch.empty_like(ys[0]) for _ in range(n)]
            timed(name, S * D * 4 + 2 * D * 2, S,
                  [lambda a=a, o=o: rm.modulate_scale_shift(a, sc, sh, out=o, stream=stream)
                   for a, o in zip(ys, os_)])
            del ys, os_
    name = "residual_gate_add_1x4216x4096"
    if want(name):
        S, D = 4216, 4096
        n = nsets_for(S * D * 6)
        rs_in = [normal((1, S, D)) for _ in range(n)]
        us = [normal((1, S, D)) for _ in range(n)]
        gate = normal((1, 1, D), 0.1)
        os_ = [torch.empty_like(rs_in[0]) for _ in range(n)]
        timed(name, S * D * 6 + D * 2, S,
              [lambda a=a, u=u, o=o: rm.residual_gate_add(a, gate, u, out=o, stream=stream)
               for a, u, o in zip(rs_in, us, os_)])
        del rs_in, us, os_
    for with_h in (False, True):
        C = 96
        name = f"conv_bias_epilogue{'_residual' if with_h else ''}_wan_c{C}"
        if not want(name):
            continue
        npx = W.WAN_PIXELS
        xw = normal((npx, C))
        hw = normal((npx, C)) if with_h else None
        bias = normal((C,), 0.1, dtype=torch.float32)
        ow = torch.empty_like(xw)
        timed(name, npx * C * (6 if with_h else 4) + C * 4, npx,
              [lambda: rm.conv_bias_epilogue(xw, bias, hw, out=ow, stream=stream)])
        del xw, hw, ow

    # the single-rounding tier on the CFG pair
    name = "ln_modulate_folded_flux_2x4608x3072"
    if want(name):
        B, S, D = 2, 4608, 3072
        n = nsets_for(B * S * D * 4)
        xs = [normal((B, S, D)) for _ in range(n)]
        sc, sh = normal((B, 1, D), 0.1), normal((B, 1, D), 0.1)
        os_ = [torch.empty_like(xs[0]) for _ in range(n)]
        timed(name, B * S * D * 4 + 2 * B * D * 2, B * S,
              [lambda a=a, o=o: rm.ln_modulate_folded(a, sc, sh, out=o, stream=stream)
               for a, o in zip(xs, os_)])
        del xs, os_

    # backward of LN + modulate (grad_x and the token sums), FLUX.1 B=1 site;
    # algorithmic bytes: read x and grad_out once, write grad_x once (+ the
    # fp32 modulation gradients and the per-row statistics)
    name = "ln_modulate_backward_flux_1x4608x3072"
    if want(name):
        B, S, D = 1, 4608, 3072
        n = nsets_for(B * S * D * 6)
        xs = [normal((B, S, D)) for _ in range(n)]
        gs = [normal((B, S, D), 0.5) for _ in range(n)]
        gxs = [torch.empty_like(xs[0]) for _ in range(n)]
        sc, sh = normal((B, 1, D), 0.1), normal((B, 1, D), 0.1)
        means = [torch.empty(B * S, dtype=torch.float32, device=dev) for _ in range(n)]
        rstds = [torch.empty_like(means[0]) for _ in range(n)]
        for a, m, r in zip(xs, means, rstds):
            rm.ln_modulate(a, sc, sh, mean_out=m, rstd_out=r, stream=stream)
        gsc = torch.empty(B, D, dtype=torch.float32, device=dev)
        gsh = torch.empty_like(gsc)
        ws = torch.empty(rm.backward_workspace_bytes(B, S, D), dtype=torch.uint8, device=dev)
        timed(name, B * S * D * 6 + B * S * 8 + 2 * B * D * 4 + B * D * 2, B * S,
              [lambda a=a, g=g, o=o, m=m, r=r: rm.ln_modulate_backward(
                  a, sc, g, m, r, grad_x=o, grad_scale=gsc, grad_shift=gsh, workspace=ws,
                  stream=stream)
               for a, g, o, m, r in zip(xs, gs, gxs, means, rstds)])
        del xs, gs, gxs

    # RMSNorm + modulate and the gated site, ERNIE-Image
    S, D = 4216, 4096
    w = normal((D,), 0.05, 1.0)
    sc, sh = normal((1, 1, D), 0.1), normal((1, 1, D), 0.1)
    name = "rmsnorm_modulate_1x4216x4096"
    if want(name):
        n = nsets_for(S * D * 4)
        xs = [normal((1, S, D)) for _ in range(n)]
        os_ = [torch.empty_like(xs[0]) for _ in range(n)]
        timed(name, S * D * 4 + 3 * D * 2, S,
              [lambda a=a, o=o: rm.rmsnorm_modulate(a, w, sc, sh, out=o, stream=stream)
               for a, o in zip(xs, os_)])
        del xs, os_
    name = "gated_rmsnorm_modulate_1x4216x4096"
    if want(name):
        n = nsets_for(S * D * 8)
        rs_in = [normal((1, S, D)) for _ in range(n)]
        us = [normal((1, S, D)) for _ in range(n)]
        gate = normal((1, 1, D), 0.1)
        rs = [torch.empty_like(rs_in[0]) for _ in range(n)]
        os_ = [torch.empty_like(rs_in[0]) for _ in range(n)]
        timed(name, S * D * 8 + 4 * D * 2, S,
              [lambda a=a, u=u, r=r, o=o: rm.gated_rmsnorm_modulate(a, u, gate, w, sc, sh,
                                                                    res_out=r, out=o,
                                                                    stream=stream)
               for a, u, r, o in zip(rs_in, us, rs, os_)])
        del rs_in, us, rs, os_

    # qk-LayerNorm, GLM-Image
    name = "qk_layernorm_1x4352x32x128"
    if want(name):
        R = 4352 * 32
        n = nsets_for(2 * R * 128 * 4)
        qs = [normal((R, 128), 2.0) for _ in range(n)]
        ks = [normal((R, 128), 2.0) for _ in range(n)]
        wq, bq = normal((128,), 0.05, 1.0), normal((128,), 0.02)
        wk, bk = normal((128,), 0.05, 1.0), normal((128,), 0.02)
        qo = [torch.empty_like(qs[0]) for _ in range(n)]
        ko = [torch.empty_like(qs[0]) for _ in range(n)]
        timed(name, 2 * R * 128 * 4 + 4 * 128 * 2, 2 * R,
              [lambda a=a, b=b, c=c, d=d: rm.qk_layernorm(a, b, wq, bq, wk, bk, q_out=c,
                                                          k_out=d, stream=stream)
               for a, b, c, d in zip(qs, ks, qo, ko)])
        del qs, ks, qo, ko

    # the same site on q / k slices of a fused QKV projection [S, 3, 32, 128],
    # normalised in place inside the buffer
    name = "qk_layernorm_qkv_strided_1x4352x32x128"
    if want(name):
        T, H, hd = 4352 * 1, 32, 128
        n = nsets_for(3 * T * H * hd * 2)
        qkvs = [normal((T, 3, H, hd), 2.0) for _ in range(n)]
        wq, bq = normal((hd,), 0.05, 1.0), normal((hd,), 0.02)
        wk, bk = normal((hd,), 0.05, 1.0), normal((hd,), 0.02)
        views = [(t[:, 0], t[:, 1]) for t in qkvs]
        timed(name, 2 * T * H * hd * 4 + 4 * hd * 2, 2 * T * H,
              [lambda q=q, k=k: rm.qk_layernorm(q, k, wq, bq, wk, bk, q_out=q, k_out=k,
                                                stream=stream)
               for q, k in views])
        del views
        del qkvs

    # channels-last RMSNorm + SiLU, Wan VAE
    for C in (96, 192, 384):
        name = f"rmsnorm_silu_cl_wan_c{C}"
        if not want(name):
            continue
        npx = W.WAN_PIXELS
        xw = normal((npx, C))
        bias = normal((C,), 0.1, dtype=torch.float32)
        gam = normal((C,), 0.05, 1.0)
        ow = torch.empty_like(xw)
        timed(name, npx * C * 4 + C * 4 + C * 2, npx,
              [lambda: rm.rmsnorm_silu_cl(xw, bias, gam, out=ow, stream=stream)])
        del xw, ow
    torch.cuda.synchronize(dev)
    return rows


if __name__ == "__main__":
    sys.exit(main())
