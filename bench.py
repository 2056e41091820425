#!/usr/bin/env python3
"""Throughput of the constraint-planned tcgen05 GEMM on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload gemm_4096|gemm_512|gemm_batched|gemm_ragged]

A step is one pass of the hot path over one batch of synthetic input: the
planned configuration (memoised after the first call) and one launch of the
persistent GEMM kernel through the C ABI.  Inputs are seeded (synth_inputs),
resident in HBM before the timed region; L2 (129 MB) is flushed between
timed steps by writing a 256 MB buffer, outside the per-step CUDA events.

One JSON line is printed by rank 0.  ``value`` is whole-job TFLOP/s (2*b*M*N*K
per step per rank over the max-over-ranks mean kernel time); ``e2e`` is the
same metric through the same call with pinned host buffers and the H2D/D2H
copies inside the timed region; ``roofline`` relates the kernel to the
measured bf16 tensor peak; ``cpu_baseline`` times the float64 oracle on the
host cores on a bounded row sample.  ``--impl reference`` times that oracle
alone (the deliberately slow CPU program the pages' method is checked
against).  With N > 1 ranks each GPU runs an independent replica (the GEMM
has no exchange step).
"""

from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth_inputs as S  # noqa: E402

L2_FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="gemm_4096",
                    choices=["gemm_4096", "gemm_512", "gemm_batched", "gemm_ragged"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="CPU time budget of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return FALLBACK_PEAKS, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "tile_size_decision_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh", ".h", ".cpp")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources (source hash recorded beside the figure)."""
    path = os.path.join(ROOT, "profiles", f"traffic_{workload}.txt")
    if not os.path.exists(path):
        return None
    fields = {}
    with open(path) as f:
        for line in f:
            if "=" in line and not line.startswith("#"):
                k, v = line.split("=", 1)
                fields[k.strip()] = v.strip()
    if fields.get("source_hash") != kernel_source_hash():
        return None
    try:
        return int(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# --------------------------------------------------------------------------- #
# CPU oracle timing (the baseline and the reference arm)
# --------------------------------------------------------------------------- #

def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


def oracle_sample(wl, budget_s: float, a=None, b=None):
    """Time the float64 oracle GEMM on row blocks of A until the budget is
    spent.  Returns (tflops, seconds, rows_done, description)."""
    from oracle import gemm as og

    if a is None:
        a, b = S.gemm_inputs(wl)
    a64_all = a if wl.b == 1 else a[0]
    b_item = b if wl.b == 1 else b[0]
    rows = max(1, min(wl.m, 256))
    done = 0
    t0 = time.perf_counter()
    while True:
        r0 = done % wl.m
        r1 = min(r0 + rows, wl.m)
        blk = S.widen(a64_all[r0:r1], wl.in_dtype)
        og.gemm(blk, S.widen(b_item, wl.in_dtype))
        done += r1 - r0
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    flops = 2.0 * done * wl.n * wl.k
    desc = (f"float64 oracle C=A*B on {done} rows of A (blocks of {rows}) x full B "
            f"({wl.k}x{wl.n}), one batch item, widening included")
    return flops / dt / 1e12, dt, done, desc


# --------------------------------------------------------------------------- #
# Clock sampling during the timed region
# --------------------------------------------------------------------------- #

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.TemporaryFile(mode="w+")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-i", str(self.idx), "-lms", "100"], stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.seek(0)
        rows = [r for r in csv.reader(io.StringIO(self.file.read())) if len(r) >= 9]
        if not rows:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[j] for r in rows for j in range(4)
                          if r[5 + j].strip().lower() == "active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# --------------------------------------------------------------------------- #
# Our arm
# --------------------------------------------------------------------------- #

def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import tile_size_decision_gb300 as tiles

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    tiles.load()
    wl = S.WORKLOADS[args.workload]
    a_np, b_np = S.gemm_inputs(wl)

    def host_tensor(x, dt):
        t = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16) if dt == S.BF16 \
            else torch.from_numpy(x)
        return t.pin_memory()

    tdt = {S.F16: torch.float16, S.BF16: torch.bfloat16, S.F32: torch.float32}
    a_h, b_h = host_tensor(a_np, wl.in_dtype), host_tensor(b_np, wl.in_dtype)
    a_d, b_d = a_h.to(dev), b_h.to(dev)
    c_d = torch.empty(wl.c_shape(), dtype=tdt[wl.out_dtype], device=dev)
    c_h = torch.empty(wl.c_shape(), dtype=tdt[wl.out_dtype]).pin_memory()
    ws = tiles.workspace(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        if wl.b > 1:
            tiles.gemm_batched(a_d, b_d, out=c_d, workspace=ws, stream=stream)
        else:
            tiles.gemm(a_d, b_d, out=c_d, workspace=ws, stream=stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    tiles.check(ws, stream)

    verdict = tiles.plan(wl.m, wl.n, wl.k, b=wl.b, in_dtype=wl.in_dtype, out_dtype=wl.out_dtype,
                         device=tiles.device_query(local_rank))[0][0]

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    wall = time.perf_counter() - t_wall
    clocks = sampler.stop()
    tiles.check(ws, stream)
    kernel_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms = float(np.mean(kernel_ms))

    # End to end through the same call with pinned host buffers.
    e_starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    e_ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush.zero_()
        e_starts[i].record(stream)
        a_d.copy_(a_h, non_blocking=True)
        b_d.copy_(b_h, non_blocking=True)
        step()
        c_h.copy_(c_d, non_blocking=True)
        e_ends[i].record(stream)
    torch.cuda.synchronize()
    tiles.check(ws, stream)
    e2e_ms = float(np.mean([s.elapsed_time(e) for s, e in zip(e_starts, e_ends)]))

    t = torch.tensor([ms, e2e_ms], dtype=torch.float64, device=dev)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    ms, e2e_ms = float(t[0]), float(t[1])

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tf, secs, rows, desc = oracle_sample(wl, args.cpu_seconds, a_np, b_np)
        cpu = {"value": tf, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
               "sample": desc, "seconds": round(secs, 2)}

    if rank == 0:
        peaks, src = load_peaks()
        flops = wl.flops
        achieved = flops / (ms * 1e-3) / 1e12
        value = world * achieved
        e2e = world * flops / (e2e_ms * 1e-3) / 1e12
        peak = peaks["bf16_tflops"]
        c = verdict.cfg
        in_b = 2
        out_b = S.DTYPE_BYTES[wl.out_dtype]
        line = {
            "metric": "GEMM TFLOP/s at 4096^3 fp16 and % of GB300 dense tensor peak (1 GPU)",
            "value": round(value, 2),
            "unit": "TFLOP/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(ms, 5),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "f16" if wl.in_dtype == S.F16 else "bf16",
            "data": "synthetic",
            "impl": "ours",
            "config": {
                "workload": wl.name, "b": wl.b, "m": wl.m, "n": wl.n, "k": wl.k,
                "in_dtype": wl.in_dtype, "out_dtype": wl.out_dtype, "accumulate": "f32",
                "distribution": wl.dist, "seed": wl.seed,
                "tile": {"bm": c.bm, "bn": c.bn, "bk": c.bk, "stages": c.stages,
                         "cta_group": c.cta_group, "grid_tiles": verdict.grid,
                         "waves": verdict.waves, "last_wave_fill": round(verdict.last_wave_fill, 4)},
                "c0_bytes": verdict.c0_bytes,
                "l2": "flushed between timed steps (256 MB write, outside the kernel events)",
                "parallelism": f"replicas x{world}",
            },
            "roofline": {
                "bound": "tensor", "achieved": round(achieved, 2), "peak": peak,
                "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                "peak_source": f"{src} bf16 burst (fp16 shares the bf16 tensor rate)",
                "traffic": recorded_traffic(wl.name),
                "frac_of_nominal_2250": round(achieved / 2250.0, 4),
            },
            "e2e": {"value": round(e2e, 2), "unit": "TFLOP/s",
                    "h2d_bytes_per_step": int(wl.b * (wl.m * wl.k + wl.k * wl.n) * in_b),
                    "d2h_bytes_per_step": int(wl.b * wl.m * wl.n * out_b),
                    "ms_per_step": round(e2e_ms, 4)},
            "gpu_launches": args.steps,
            "clocks": clocks,
            "wall_s_timed_region": round(wall, 4),
            "kernel_ms_min": round(min(kernel_ms), 5),
            "kernel_ms_median": round(float(np.median(kernel_ms)), 5),
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


# --------------------------------------------------------------------------- #
# Reference arm: the float64 oracle on the host cores
# --------------------------------------------------------------------------- #

def run_reference(args, rank, world):
    if rank != 0:
        return
    wl = S.WORKLOADS[args.workload]
    a, b = S.gemm_inputs(wl)
    per_step = max(2.0, min(10.0, 150.0 / max(args.steps + args.warmup, 1)))
    for _ in range(args.warmup):
        oracle_sample(wl, min(per_step, 2.0), a, b)
    times, flops = [], 0.0
    descs = []
    for _ in range(args.steps):
        tf, secs, rows, desc = oracle_sample(wl, per_step, a, b)
        times.append(secs)
        flops += tf * 1e12 * secs
        descs.append(rows)
    total = sum(times)
    value = flops / total / 1e12
    line = {
        "metric": "GEMM TFLOP/s at 4096^3 fp16 and % of GB300 dense tensor peak (1 GPU)",
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * total / max(args.steps, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": {"workload": wl.name, "b": wl.b, "m": wl.m, "n": wl.n, "k": wl.k,
                   "in_dtype": wl.in_dtype, "out_dtype": wl.out_dtype},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": blas_threads(),
                         "kind": "oracle",
                         "sample": f"float64 oracle on row blocks of A, {per_step:.1f} s per step, "
                                   f"{int(np.mean(descs))} rows per step on average"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    rank, world, local_rank = dist_env()
    if args.gpus != world and world > 1:
        print(f"warning: --gpus {args.gpus} but WORLD_SIZE {world}", file=sys.stderr)
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        if args.warmup < 3:
            print("warning: fewer than 3 warm-up steps", file=sys.stderr)
        run_ours(args, rank, world, local_rank)
    return 0


if __name__ == "__main__":
    sys.exit(main())
