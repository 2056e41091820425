#!/usr/bin/env python3
"""Throughput of the constraint-planned tcgen05 GEMM on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload gemm_4096|gemm_512|gemm_batched|gemm_ragged|conv_htiled]

A step is one pass of the hot path over one batch of synthetic input: the
planned configuration (memoised after the first call) and one launch of the
persistent GEMM kernel through the C ABI.  Inputs are seeded (synth_inputs),
resident in HBM before the timed region.  The K timed steps run back to back
between one pair of CUDA events, cycling through R copies of the operands:
between two uses of one copy the other R - 1 copies, at least twice the
129 MB L2, pass through it, so no step finds its inputs in L2 and none needs
a flush (inputs larger than L2).  Per-step figures with L2 flushed between
steps (a 256 MB write outside per-step events) are reported beside it.

One JSON line is printed by rank 0.  ``value`` is whole-job TFLOP/s (2*b*M*N*K
per step per rank over the max-over-ranks time per step); ``e2e`` is the
same metric through the same call with pinned host buffers and the H2D/D2H
copies inside the timed region; ``roofline`` relates the kernel to the
measured bf16 tensor peak; ``cpu_baseline`` times the float64 oracle on the
host cores on a bounded row sample.  ``--impl reference`` times that oracle
alone (the deliberately slow CPU program the pages' method is checked
against).  With N > 1 ranks each GPU runs an independent replica (the GEMM
has no exchange step).

The default single-GPU run of the 4096^3 headline adds, after the headline's
timed steps:
  timing     the step timed on its own at least 50 times with L2 flushed and
             50 times L2-warm (mean, median, minimum);
  sustained  about 2.5 s of back-to-back launches between one pair of
             events, with the SM clock sampled inside that window: TFLOP/s
             against the measured sustained bf16 peak, and the cycles per
             launch at the clock it ran at;
  workloads  the other four seeded workloads (gemm_512, gemm_batched,
             gemm_ragged, conv_htiled), each measured like the headline
             (at least 50 rotating steps, then 50 flushed and 50 warm ones
             on their own) with its roofline, its
             recorded DRAM traffic, its clock record and the oracle timed on
             a bounded sample of it.
"""

from __future__ import annotations

import argparse
import csv
import hashlib
import re
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
L2_BYTES = 129 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="gemm_4096",
                    choices=["gemm_4096", "gemm_512", "gemm_batched", "gemm_ragged",
                             "conv_htiled"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="CPU time budget of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--extra-cpu-seconds", type=float, default=3.0,
                    help="CPU time budget of the oracle sample of each further workload")
    ap.add_argument("--no-extras", action="store_true",
                    help="gemm_4096 only: skip the 50-iteration timings, the sustained leg and "
                         "the other four workloads")
    ap.add_argument("--sustained-seconds", type=float, default=2.5,
                    help="length of the sustained back-to-back leg")
    ap.add_argument("--workload-sustained-seconds", type=float, default=0.8,
                    help="length of each further workload's back-to-back leg (its clock record)")
    ap.add_argument("--e2e-chunks", type=int, default=4, metavar="P",
                    help="pieces of the end-to-end call (uploads, kernels, downloads overlap)")
    ap.add_argument("--autotune", type=int, default=4, metavar="K",
                    help="GEMM workloads: time the planner's top K configurations (with "
                         "their last-round schedules) before the timed steps and run the "
                         "fastest; 0 runs the planner's first choice")
    return ap.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def max_over_ranks(values, dist, world, device):
    """Elementwise maximum of per-rank timings: the slowest replica sets the
    job's time.  With one rank the values come back unchanged."""
    import torch

    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t]


def job_throughput(world, units_per_replica, seconds):
    """Whole-job throughput of independent replicas (weak scaling): the units
    every rank processed over the slowest rank's time."""
    return world * units_per_replica / seconds


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return FALLBACK_PEAKS, "fallback"


# Sources that decide a workload's kernels and launch shapes: a recorded
# DRAM figure stays valid while these files are unchanged.
SHARED_SOURCES = ("sm103_ptx.cuh", "tiles_internal.h", "planner.cpp", "gemm_sm103a.cuh")
WORKLOAD_SOURCES = {
    "gemm": ("gemm_sm103a.cu", "api.cu"),
    "conv": ("conv_sm103a.cuh", "conv_sm103a.cu", "conv_tma_sm103a.cu"),
}


def code_only(text: str) -> str:
    """C/C++/CUDA source without comments and with whitespace collapsed: an
    edit to a comment leaves a recorded figure valid, a code change does not.
    (String literals holding comment markers are not special-cased; the
    hashed sources have none that matter.)"""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash(workload: str, read=None) -> str:
    """Hash of the code (comments dropped) of the sources a workload's kernels
    and launch shapes come from; `read(name)` returns a source's text."""
    kind = "conv" if workload.startswith("conv") else "gemm"
    csrc = os.path.join(ROOT, "tile_size_decision_gb300", "csrc")
    if read is None:
        def read(name):
            with open(os.path.join(csrc, name), encoding="utf-8") as f:
                return f.read()
    h = hashlib.sha256()
    for name in sorted(SHARED_SOURCES + WORKLOAD_SOURCES[kind]):
        h.update(name.encode() + code_only(read(name)).encode())
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
    if fields.get("source_hash") != kernel_source_hash(workload):
        return None
    try:
        return int(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


L2_NOTE = ("inputs larger than L2: the timed GPU steps run back to back over R copies of the "
           "operands, and the R - 1 other copies touched between two uses of one copy hold at "
           "least twice the 129 MB L2 (no flush); the per-step figures under 'flushed' write a "
           "256 MB buffer between steps instead; the CPU oracle arm has no L2")


def rotation_sets(set_bytes: int) -> int:
    """Copies of a workload's operands (inputs and output) that the timed
    steps cycle through: enough that the other copies touched between two
    uses of one hold at least twice the L2."""
    return max(2, -(-2 * L2_BYTES // max(int(set_bytes), 1)) + 1)


def workload_config(wl, world=1):
    """The workload as both arms describe it in their line's config: shapes,
    dtypes, distribution, seed, the L2 treatment and the replicas."""
    if isinstance(wl, S.ConvWorkload):
        base = {"workload": wl.name, "n": wl.n, "c": wl.c, "h": wl.h, "w": wl.w,
                "c_out": wl.c_out, "kh": wl.kh, "kw": wl.kw, "stride": [wl.sh, wl.sw],
                "pad": [wl.ph, wl.pw], "dil": [wl.dh, wl.dw], "tile_oh": wl.tile_oh}
    else:
        base = {"workload": wl.name, "b": wl.b, "m": wl.m, "n": wl.n, "k": wl.k}
    return dict(base, in_dtype=wl.in_dtype, out_dtype=wl.out_dtype, accumulate="f32",
                distribution=wl.dist, seed=wl.seed, l2=L2_NOTE,
                parallelism=f"replicas x{world}")


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


def oracle_conv_sample(wl, budget_s: float, x=None, w=None):
    """Time the float64 oracle convolution image by image until the budget is
    spent.  Returns (tflops, seconds, images_done, description)."""
    from oracle import conv as oc

    if x is None:
        x, w = S.conv_inputs(wl)
    w64 = S.widen(w, wl.in_dtype)
    done = 0
    t0 = time.perf_counter()
    while True:
        i = done % wl.n
        oc.conv2d(S.widen(x[i:i + 1], wl.in_dtype), w64, (wl.sh, wl.sw), (wl.ph, wl.ph),
                  (wl.pw, wl.pw), (wl.dh, wl.dw))
        done += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    flops = wl.flops / wl.n * done
    desc = (f"float64 oracle direct convolution (kh*kw shifted matmuls) on {done} images "
            f"of {wl.n}, widening included")
    return flops / dt / 1e12, dt, done, desc


# --------------------------------------------------------------------------- #
# Clock sampling during the timed region
# --------------------------------------------------------------------------- #

class ClockSampler:
    """nvidia-smi samples of the SM clock, its maximum, the power and the
    throttle reasons, every 100 ms, each stamped with the host clock so that
    a summary can keep the samples of one time window."""

    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.file = None
        self.rows = []

    def start(self):
        try:
            self.file = tempfile.TemporaryFile(mode="w+")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-i", str(self.idx), "-lms", "100"], stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        """Stop sampling and keep the parsed rows."""
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.seek(0)
        self.rows = parse_clock_rows(self.file.read())

    def summary(self, t0=None, t1=None):
        """Median SM clock, its maximum and the throttle reasons of the
        samples taken in [t0, t1] (host time.time(); all samples when no
        window is given)."""
        return summarize_clocks(self.rows, t0, t1)


def parse_clock_rows(text: str):
    """Rows of the sampler's CSV as dicts: t (host seconds since the epoch),
    sm, max (MHz), power (W), reasons (the active throttle reasons)."""
    rows = []
    for r in csv.reader(io.StringIO(text)):
        if len(r) < 10:
            continue
        try:
            t = time.mktime(time.strptime(r[0].strip().split(".")[0], "%Y/%m/%d %H:%M:%S"))
            frac = r[0].strip().split(".")
            t += float("0." + frac[1]) if len(frac) > 1 and frac[1].isdigit() else 0.0
        except (ValueError, IndexError):
            t = None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        reasons = [ClockSampler.REASONS[j] for j in range(4)
                   if r[6 + j].strip().lower() == "active"]
        rows.append({"t": t, "sm": num(r[2]), "max": num(r[3]), "power": num(r[4]),
                     "reasons": reasons})
    return rows


def summarize_clocks(rows, t0=None, t1=None):
    if t0 is not None:
        rows = [r for r in rows if r["t"] is not None and t0 <= r["t"] <= t1]
    if not rows:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
    sm = [r["sm"] for r in rows if r["sm"] is not None]
    mx = [r["max"] for r in rows if r["max"] is not None]
    pw = [r["power"] for r in rows if r["power"] is not None]
    return {"sm_mhz": float(np.median(sm)) if sm else None,
            "sm_max_mhz": max(mx) if mx else None,
            "reasons": sorted({x for r in rows for x in r["reasons"]}),
            "samples": len(rows),
            "power_w_median": float(np.median(pw)) if pw else None}


# --------------------------------------------------------------------------- #
# Our arm
# --------------------------------------------------------------------------- #

class Job:
    """One workload prepared on a device: pinned host inputs, resident device
    inputs and output (copy 0 of the rotation, beside copies 1 .. R-1), the
    step (one call through the C ABI on copy i % R) and the figures the JSON
    line reports."""


def gemm_job(wl, dev, tiles, torch):
    a_np, b_np = S.gemm_inputs(wl)
    j = Job()
    j.host_in = [host_tensor(a_np, wl.in_dtype, torch), host_tensor(b_np, wl.in_dtype, torch)]
    j.dev_in = [t.to(dev) for t in j.host_in]
    j.out = torch.empty(wl.c_shape(), dtype=TORCH_DT(torch)[wl.out_dtype], device=dev)
    j.host_out = torch.empty(wl.c_shape(), dtype=j.out.dtype).pin_memory()
    a_d, b_d = j.dev_in

    verdict = tiles.plan(wl.m, wl.n, wl.k, b=wl.b, in_dtype=wl.in_dtype, out_dtype=wl.out_dtype,
                         device=tiles.device_query(dev.index or 0))[0][0]
    # A workspace with room for every last-round schedule the autotune
    # times: the planner's own choice, and a K split of its tile (partials).
    c = verdict.cfg
    ksplit = tiles.make_config(c.bm, c.bn, c.bk, c.stages, c.threads, c.instr, c.acc_bufs,
                               c.cta_group, tail="ksplit")
    j.ws = max(tiles.gemm_workspace(a_d, b_d, j.out), tiles.gemm_workspace(a_d, b_d, j.out, ksplit),
               key=lambda t: t.numel())
    j.set_bytes = sum(t.numel() * t.element_size() for t in (a_d, b_d, j.out))
    j.sets = [(a_d, b_d, j.out)] + [(a_d.clone(), b_d.clone(), torch.empty_like(j.out))
                                    for _ in range(rotation_sets(j.set_bytes) - 1)]

    def step(i, stream):
        a, b, out = j.sets[i % len(j.sets)]
        if wl.b > 1:
            tiles.gemm_batched(a, b, out=out, workspace=j.ws, stream=stream)
        else:
            tiles.gemm(a, b, out=out, workspace=j.ws, stream=stream)

    j.step = step

    def e2e_step(stream, chunks):
        # The host-buffer call: uploads, GEMMs and downloads in overlapping pieces.
        tiles.gemm_host(j.host_in[0], j.host_in[1], j.host_out, a_d, b_d, j.out, workspace=j.ws,
                        stream=stream, chunks=chunks)

    j.e2e_step = e2e_step
    j.launches = 1
    j.flops = wl.flops
    j.bound = "tensor"
    j.bytes = wl.b * (wl.m * wl.k + wl.k * wl.n) * 2 + wl.b * wl.m * wl.n * S.DTYPE_BYTES[wl.out_dtype]
    sch = tiles.gemm_schedule(a_d, b_d, j.out, workspace=j.ws)
    j.config = workload_config(wl)
    # How this library runs it (reported beside the config, under "plan").
    j.plan = {
        "tile": {"bm": c.bm, "bn": c.bn, "bk": c.bk, "stages": c.stages,
                 "cta_group": c.cta_group, "grid_tiles": verdict.grid, "waves": verdict.waves,
                 "last_wave_fill": round(verdict.last_wave_fill, 4),
                 "tail_k_parts": verdict.tail_split},
        "schedule": {"tiles": sch.tiles, "resident_groups": sch.resident_groups,
                     "full_units": sch.full_units, "units": sch.units, "groups": sch.groups,
                     "tail": ["whole", "n_halves", "k_split"][sch.tail_mode],
                     "k_parts": sch.ksplit, "workspace_bytes": sch.workspace_bytes},
        "c0_bytes": verdict.c0_bytes,
    }
    j.dtype = "f16" if wl.in_dtype == S.F16 else "bf16"
    j.oracle = lambda budget: oracle_sample(wl, budget, a_np, b_np)

    def autotune(top_k):
        # The measured shortlist (outside the timed steps): the winner becomes
        # the problem's tuned configuration, which the steps' calls use.
        best, rows = tiles.gemm_autotune(a_d, b_d, j.out, top_k=top_k, reps=10, workspace=j.ws,
                                         batched=wl.b > 1)
        tiles.check(j.ws)
        sch_t = tiles.gemm_schedule(a_d, b_d, j.out, workspace=j.ws)
        return {"top_k": top_k, "reps": 10,
                "winner": {"bm": best.bm, "bn": best.bn, "stages": best.stages,
                           "cta_group": best.cta_group,
                           "tail": ["whole", "n_halves", "k_split"][sch_t.tail_mode],
                           "k_parts": sch_t.ksplit},
                "planner_choice_kept": (best.bm, best.bn, best.stages, best.cta_group,
                                        sch_t.tail_mode) == (c.bm, c.bn, c.stages, c.cta_group,
                                                             sch.tail_mode),
                "shortlist_us": [
                    [f'{r["bm"]}x{r["bn"]}/{r["stages"]}/cg{r["cta_group"]}/{r["tail_mode"]}'
                     + ("/planner" if r["tail_asked"] == 0 else ""),
                     round(r["us"], 2)] for r in rows if r["status"] == 0]}

    j.autotune = autotune
    c_lib = [torch.empty_like(j.out) for _ in j.sets]

    def library_step(i):
        a, b, _ = j.sets[i % len(j.sets)]
        torch.matmul(a, b, out=c_lib[i % len(j.sets)])

    j.library_step = library_step if j.out.dtype == a_d.dtype else None
    return j


def conv_job(wl, dev, tiles, torch):
    x_np, w_np = S.conv_inputs(wl)
    j = Job()
    j.host_in = [host_tensor(x_np, wl.in_dtype, torch), host_tensor(w_np, wl.in_dtype, torch)]
    j.dev_in = [t.to(dev) for t in j.host_in]
    shape = (wl.n, wl.c_out, wl.oh, wl.ow)
    j.out = torch.empty(shape, dtype=TORCH_DT(torch)[wl.out_dtype], device=dev)
    j.host_out = torch.empty(shape, dtype=j.out.dtype).pin_memory()
    x_d, w_d = j.dev_in
    # A workspace sized for the TMA im2col producer (the default path).
    j.ws = tiles.conv_workspace(x_d, w_d, (wl.sh, wl.sw), (wl.ph, wl.pw), (wl.dh, wl.dw),
                                wl.tile_oh)
    j.set_bytes = sum(t.numel() * t.element_size() for t in (x_d, w_d, j.out))
    j.sets = [(x_d, w_d, j.out)] + [(x_d.clone(), w_d.clone(), torch.empty_like(j.out))
                                    for _ in range(rotation_sets(j.set_bytes) - 1)]

    def step(i, stream):
        x, w, out = j.sets[i % len(j.sets)]
        tiles.conv2d_htiled(x, w, (wl.sh, wl.sw), (wl.ph, wl.pw), (wl.dh, wl.dw), wl.tile_oh,
                            out=out, workspace=j.ws, stream=stream)

    j.step = step

    def e2e_step(stream, chunks):
        # The host-buffer call: uploads, convolutions and downloads in
        # overlapping runs of images.
        tiles.conv2d_host(j.host_in[0], j.host_in[1], j.host_out, x_d, w_d, j.out,
                          (wl.sh, wl.sw), (wl.ph, wl.pw), (wl.dh, wl.dw), wl.tile_oh,
                          workspace=j.ws, stream=stream, chunks=chunks)

    j.e2e_step = e2e_step
    # One convolution launch per 128 H-tiles (the NCHW input is read in
    # place), after a filter reorder launch unless the filter is 3x3 over 64
    # channels, which goes to tensor memory straight from its OIHW rows.
    j.reorder_launches = 0 if (wl.kh * wl.kw == 9 and wl.c == 64 and wl.c_out <= 128) else 1
    j.launches = j.reorder_launches + -(-(-(-wl.oh // wl.tile_oh)) // 128)
    j.flops = wl.flops
    j.bound = "hbm"
    j.bytes = (x_np.size + w_np.size) * 2 + int(np.prod(shape)) * S.DTYPE_BYTES[wl.out_dtype]
    n_ht = -(-wl.oh // wl.tile_oh)
    rows = [tiles.htile_rows(wl.h, wl.kh, wl.sh, wl.ph, wl.dh, o0, min(o0 + wl.tile_oh, wl.oh))
            for o0 in range(0, wl.oh, wl.tile_oh)]
    halo_bytes = sum(min(r.in_end, wl.h) - r.in_start for r in rows) * wl.n * wl.c * wl.w * 2
    j.config = workload_config(wl)
    # How this library runs it (reported beside the config, under "plan").
    j.plan = {
        "h_tiles": n_ht,
        "gemm_per_tile": {"m": wl.c_out, "n": wl.tile_oh * wl.ow, "k": wl.c * wl.kh * wl.kw},
        "input_bytes_with_halo": halo_bytes,
        "producer": ("tma: the NCHW input read in place; per (kernel row, 64 channels) a TMA box "
                     "of the input row, transposed by warps of the kernel into stride-phase "
                     "planes that serve every tap as the MMA B operand; filter in tensor memory "
                     "(built from its OIHW rows) as the A operand"),
        "workspace_bytes": int(j.ws.numel()),
    }
    j.dtype = "f16" if wl.in_dtype == S.F16 else "bf16"
    j.oracle = lambda budget: oracle_conv_sample(wl, budget, x_np, w_np)
    return j


def TORCH_DT(torch):
    return {S.F16: torch.float16, S.BF16: torch.bfloat16, S.F32: torch.float32}


def host_tensor(x, dt, torch):
    t = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16) if dt == S.BF16 \
        else torch.from_numpy(x)
    return t.pin_memory()


def timed_rotating(job, stream, steps, start=0):
    """Milliseconds per step of `steps` back-to-back steps over the job's
    operand copies (step i uses copy i % R, from i = start), between one pair
    of CUDA events on `stream`, and the host-clock window (time.time()) they
    ran in."""
    import torch

    s_ev = torch.cuda.Event(enable_timing=True)
    e_ev = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0 = time.time()
    s_ev.record(stream)
    for i in range(start, start + steps):
        job.step(i, stream)
    e_ev.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    return s_ev.elapsed_time(e_ev) / steps, (t0, t1)


def timed_steps(job, stream, flush, steps, warm=False):
    """Milliseconds of each of `steps` steps on operand copy 0, each
    bracketed by CUDA events on `stream`; before each step L2 is flushed (a
    256 MB write outside the events) unless `warm`.  Also returns the
    host-clock window (time.time()) that the steps ran in."""
    import torch

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    torch.cuda.synchronize()
    t0 = time.time()
    for i in range(steps):
        if not warm:
            flush.zero_()
        starts[i].record(stream)
        job.step(0, stream)
        ends[i].record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    return [s.elapsed_time(e) for s, e in zip(starts, ends)], (t0, t1)


def roofline(job, ms, peaks, src, workload):
    """The roofline object of one workload's kernel at `ms` per step."""
    achieved = job.flops / (ms * 1e-3) / 1e12
    if job.bound == "tensor":
        peak = peaks["bf16_tflops"]
        roof = {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak,
                "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                "peak_source": f"{src} bf16 burst (fp16 shares the bf16 tensor rate)",
                "frac_of_nominal_2250": round(achieved / 2250.0, 4)}
    else:
        gbs = job.bytes / (ms * 1e-3) / 1e9
        peak = peaks["hbm_gbs"]
        roof = {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                "frac": round(gbs / peak, 4), "peak_source": f"{src} HBM copy bandwidth",
                "algorithmic_bytes": job.bytes,
                "timed_over": f"the whole step ({job.launches} launch(es): "
                              + ("the filter reorder, then " if job.reorder_launches else "")
                              + "the convolution)"}
    roof["traffic"] = recorded_traffic(workload)
    return roof


def ms_stats(ms):
    return {"iterations": len(ms), "mean_ms": round(float(np.mean(ms)), 5),
            "median_ms": round(float(np.median(ms)), 5), "min_ms": round(float(np.min(ms)), 5)}


def sustained_leg(job, stream, seconds, gpu_index, peaks, src):
    """Back-to-back launches of the step over the rotating operand copies
    (no flush) between one pair of CUDA events for about `seconds`, with the
    clocks sampled inside that window: the throughput under the power cap
    and the clock-normalised time."""
    import torch

    probe, _ = timed_rotating(job, stream, 20)
    n = max(50, int(seconds * 1e3 / max(probe, 1e-3)))
    sampler = ClockSampler(gpu_index)
    sampler.start()
    time.sleep(0.3)
    s_ev = torch.cuda.Event(enable_timing=True)
    e_ev = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0 = time.time()
    s_ev.record(stream)
    for i in range(n):
        job.step(i, stream)
    e_ev.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    sampler.stop()
    total_ms = s_ev.elapsed_time(e_ev)
    us = 1e3 * total_ms / n
    tflops = job.flops * n / (total_ms * 1e-3) / 1e12
    clk = sampler.summary(t0, t1)
    out = {"launches": n, "seconds": round(total_ms / 1e3, 3), "us_per_launch": round(us, 3),
           "tflops": round(tflops, 2), "clocks": clk}
    if job.bound == "tensor":
        out.update({"frac_of_sustained": round(tflops / peaks["bf16_tflops_sustained"], 4),
                    "frac_of_burst": round(tflops / peaks["bf16_tflops"], 4),
                    "peak_source": f"{src} bf16 sustained (a seconds-long loop under the power cap)"})
    else:
        gbs = job.bytes * n / (total_ms * 1e-3) / 1e9
        out.update({"gbs": round(gbs, 1), "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 4),
                    "peak_source": f"{src} HBM copy bandwidth (back to back over the rotating "
                                   "operand copies)"})
    if clk["sm_mhz"]:
        # Time x clock: the cycles one launch takes at the clock it ran at.
        out["kcycles_per_launch"] = round(us * clk["sm_mhz"] / 1e3, 1)
        if clk["sm_max_mhz"]:
            out["tflops_at_max_clock"] = round(tflops * clk["sm_max_mhz"] / clk["sm_mhz"], 1)
    return out


def make_job(name, dev, tiles, torch):
    wl = S.WORKLOADS[name]
    return (conv_job if isinstance(wl, S.ConvWorkload) else gemm_job)(wl, dev, tiles, torch), wl


def workload_entry(name, args, dev, tiles, torch, stream, flush, peaks, src, gpu_index):
    """One non-headline workload measured like the headline: warm-up, then
    at least 50 back-to-back steps over its rotating operand copies (its
    value and roofline), 50 flushed and 50 L2-warm steps on their own, and
    the oracle timed on a bounded sample of it."""
    job, wl = make_job(name, dev, tiles, torch)
    entry = {"config": job.config, "plan": job.plan}
    if getattr(job, "autotune", None) and args.autotune > 0:
        entry["plan"]["autotune"] = job.autotune(args.autotune)
    sampler = ClockSampler(gpu_index)
    sampler.start()
    time.sleep(0.3)
    for i in range(args.warmup):
        job.step(i, stream)
    tiles.check(job.ws, stream)
    n = max(args.steps, 50)
    mean, (t0, t1) = timed_rotating(job, stream, n, start=args.warmup)
    ms, _ = timed_steps(job, stream, flush, n)
    warm, _ = timed_steps(job, stream, flush, n, warm=True)
    sampler.stop()
    tiles.check(job.ws, stream)
    # A short back-to-back leg under load: its clock samples are the
    # workload's clock record (the flushed steps last milliseconds).
    busy = sustained_leg(job, stream, args.workload_sustained_seconds, gpu_index, peaks, src)
    tiles.check(job.ws, stream)
    entry.update({
        "value": round(job.flops / (mean * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
        "ms_per_step": round(mean, 5), "steps": n, "operand_copies": len(job.sets),
        "flushed": dict(ms_stats(ms), tflops_median=round(
            job.flops / (float(np.median(ms)) * 1e-3) / 1e12, 2)),
        "l2_warm": dict(ms_stats(warm), tflops_median=round(
            job.flops / (float(np.median(warm)) * 1e-3) / 1e12, 2)),
        "roofline": roofline(job, mean, peaks, src, name),
        "gpu_launches": n * job.launches,
        "clocks": busy["clocks"],
        "clocks_timed_steps": dict(sampler.summary(t0, t1), whole_leg=sampler.summary()),
        "sustained": {key: val for key, val in busy.items() if key != "clocks"},
    })
    if not args.no_cpu_baseline:
        tf, secs, _, desc = job.oracle(args.extra_cpu_seconds)
        entry["cpu_baseline"] = {"value": tf, "unit": "TFLOP/s", "cores": blas_threads(),
                                 "kind": "oracle", "sample": desc, "seconds": round(secs, 2)}
    return entry


EXTRA_WORKLOADS = ("gemm_512", "gemm_batched", "gemm_ragged", "conv_htiled")


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import tile_size_decision_gb300 as tiles

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    tiles.load()
    job, wl = make_job(args.workload, dev, tiles, torch)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    peaks, src = load_peaks()

    if getattr(job, "autotune", None) and args.autotune > 0:
        job.plan["autotune"] = job.autotune(args.autotune)
    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    # The warm-up steps run right before the timed ones, after the sampler's
    # start-up pause, so that the timed steps start from a busy GPU; the
    # rotation continues from them.
    for i in range(args.warmup):
        job.step(i, stream)
    tiles.check(job.ws, stream)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    ms, (t0, t1) = timed_rotating(job, stream, args.steps, start=args.warmup)
    if world > 1:
        dist.barrier()
    wall = time.perf_counter() - t_wall
    sampler.stop()
    tiles.check(job.ws, stream)
    # The headline's clock record: every sample from the warm-up to the end
    # of the timed steps (the timed region itself lasts milliseconds; the
    # sustained leg below samples a seconds-long window under load).
    clocks = dict(sampler.summary(), samples_in_timed_window=sampler.summary(t0, t1)["samples"])

    # End to end through the library's host-buffer call (pinned host buffers):
    # every step uploads the inputs and downloads the result.
    e_starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    e_ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    job.e2e_step(stream, args.e2e_chunks)          # untimed: creates the copy streams
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush.zero_()
        e_starts[i].record(stream)
        job.e2e_step(stream, args.e2e_chunks)
        e_ends[i].record(stream)
    torch.cuda.synchronize()
    tiles.check(job.ws, stream)
    e2e_ms = float(np.mean([s.elapsed_time(e) for s, e in zip(e_starts, e_ends)]))

    ms, e2e_ms = max_over_ranks([ms, e2e_ms], dist, world, dev)

    # Context only (not on this library's path): cuBLAS through torch.matmul
    # on the same operand copies, timed the same way.
    context = None
    if getattr(job, "library_step", None) is not None:
        for i in range(args.warmup):
            job.library_step(i)
        torch.cuda.synchronize()
        s_ev = torch.cuda.Event(enable_timing=True)
        e_ev = torch.cuda.Event(enable_timing=True)
        s_ev.record(stream)
        for i in range(args.warmup, args.warmup + args.steps):
            job.library_step(i)
        e_ev.record(stream)
        torch.cuda.synchronize()
        lib_mean = s_ev.elapsed_time(e_ev) / args.steps
        context = {"cublas_torch_matmul": {
            "ms_per_step": round(lib_mean, 5),
            "tflops": round(job.flops / (lib_mean * 1e-3) / 1e12, 2),
            "note": "torch.matmul on the same device operand copies, timed the same way; "
                    "context, not a baseline"}}

    # What the line reports of the headline job (the job is released before
    # the other workloads run).
    head = {"dtype": job.dtype, "config": job.config, "plan": job.plan,
            "roofline": roofline(job, ms, peaks, src,
                                                                            args.workload),
            "h2d": int(sum(t.numel() * t.element_size() for t in job.host_in)),
            "d2h": int(job.host_out.numel() * job.host_out.element_size()),
            "launches": job.launches, "copies": len(job.sets)}

    # The same step timed at least 50 times, L2 flushed and L2 warm, and a
    # sustained, clock-sampled leg of back-to-back launches.
    extras = world == 1 and args.workload == "gemm_4096" and not args.no_extras
    timing = sustained = None
    if extras:
        n = max(args.steps, 50)
        fl, _ = timed_steps(job, stream, flush, n)
        wm, _ = timed_steps(job, stream, flush, n, warm=True)
        tiles.check(job.ws, stream)
        timing = {"flushed": dict(ms_stats(fl), tflops_median=round(
                      job.flops / (float(np.median(fl)) * 1e-3) / 1e12, 2)),
                  "l2_warm": dict(ms_stats(wm), tflops_median=round(
                      job.flops / (float(np.median(wm)) * 1e-3) / 1e12, 2))}
        sustained = sustained_leg(job, stream, args.sustained_seconds, local_rank, peaks, src)
        tiles.check(job.ws, stream)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tf, secs, _, desc = job.oracle(args.cpu_seconds)
        cpu = {"value": tf, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
               "sample": desc, "seconds": round(secs, 2)}

    workloads = None
    if extras:
        del job
        torch.cuda.empty_cache()
        workloads = {}
        for name in EXTRA_WORKLOADS:
            workloads[name] = workload_entry(name, args, dev, tiles, torch, stream, flush, peaks,
                                             src, local_rank)
            torch.cuda.empty_cache()

    if rank == 0:
        value = job_throughput(world, wl.flops, ms * 1e-3) / 1e12
        e2e = job_throughput(world, wl.flops, e2e_ms * 1e-3) / 1e12
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
            "dtype": head["dtype"],
            "data": "synthetic",
            "impl": "ours",
            "config": dict(head["config"], parallelism=f"replicas x{world}"),
            "plan": head["plan"],
            "roofline": head["roofline"],
            "e2e": {"value": round(e2e, 2), "unit": "TFLOP/s",
                    "call": "tiles_gemm_host" if args.workload.startswith("gemm") else "tiles_conv2d_host",
                    "pieces": args.e2e_chunks,
                    "h2d_bytes_per_step": head["h2d"],
                    "d2h_bytes_per_step": head["d2h"],
                    "ms_per_step": round(e2e_ms, 4)},
            "gpu_launches": args.steps * head["launches"],
            "clocks": clocks,
            "wall_s_timed_region": round(wall, 4),
            "operand_copies": head["copies"],
            "cpu_baseline": cpu,
        }
        if timing is not None:
            line["timing"] = timing
        if sustained is not None:
            line["sustained"] = sustained
        if workloads is not None:
            line["workloads"] = workloads
        if context is not None:
            line["context"] = context
        if args.workload != "gemm_4096":
            line["metric"] = f"TFLOP/s of {args.workload} (a parity workload, not the headline)"
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
    if isinstance(wl, S.ConvWorkload):
        x, w = S.conv_inputs(wl)
        sample = lambda budget: oracle_conv_sample(wl, budget, x, w)  # noqa: E731
    else:
        a, b = S.gemm_inputs(wl)
        sample = lambda budget: oracle_sample(wl, budget, a, b)  # noqa: E731
    config = workload_config(wl, world)
    per_step = max(2.0, min(10.0, 150.0 / max(args.steps + args.warmup, 1)))
    for _ in range(args.warmup):
        sample(min(per_step, 2.0))
    times, flops, desc = [], 0.0, ""
    for _ in range(args.steps):
        tf, secs, _, desc = sample(per_step)
        times.append(secs)
        flops += tf * 1e12 * secs
    total = sum(times)
    value = flops / total / 1e12
    line = {
        "metric": "GEMM TFLOP/s at 4096^3 fp16 and % of GB300 dense tensor peak (1 GPU)",
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * total / max(args.steps, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference", "config": config,
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": blas_threads(),
                         "kind": "oracle",
                         "sample": f"{desc}; {per_step:.1f} s of CPU work per step"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    if args.workload != "gemm_4096":
        line["metric"] = f"TFLOP/s of {args.workload} (a parity workload, not the headline)"
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
