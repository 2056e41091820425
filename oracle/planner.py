"""Tile-size constraint procedure, page mode (oracle; test infrastructure only).

Source: the page "04-tile-size-decision" (its README's "目的" block and the
four checks it names, whose numbers the page's script tile_decision.py and
its printed outputs fix).  A GEMM tile (bm x bn, K step bk, a pipeline of
`stages`, a block of `threads`) is checked against

  C3  the MMA instruction shape: the tile edges and the thread count are
      whole multiples of the MMA family's shape, within the block limit;
  C1  on-chip capacity: `stages` copies of the A and B slices fit one
      block's shared memory;
  C2  register pressure: the accumulator tile, spread over the threads and
      rounded to the per-warp register granule, fits the per-thread limit;
then the resident blocks per SM follow from the scarcest of registers,
shared memory and threads, and

  C4  waves: the tiles run in waves of the resident blocks; a last wave
      under half full is a tail warning, fewer tiles than SMs an idle one;
  C0  DRAM traffic without caches: every tile streams its panels of A and B
      once, C is written once:
          C0 = in_bytes*b*M*N*K*(1/bn + 1/bm) + out_bytes*b*M*N

A sweep over the page's candidate grid keeps the feasible tiles and ranks
them by least traffic, then most resident blocks, then least shared memory.

The page's numbers carry some conventions that its printed outputs make
observable, and that are kept here:
  * C2 counts the accumulators alone (no other registers).
  * Blocks by shared memory divide the per-SM capacity, not the per-block one.
  * With no resident block the resident count is taken as 1, so waves = tiles.
  * The binding resource is the first scarcest in the order regs, smem,
    threads; the 32-block hardware cap never binds by name.
  * Traffic ranks by Python's round() (half to even) of the float64 C0, and
    ties keep the enumeration order (bm, bn, bk, stages, threads ascending).

Readings where the page is silent: C0 takes a batch b and separate input and
output widths (the README's formula has b; with b=1 and equal widths it is
the script's own expression), evaluated left to right in IEEE float64; the
tile counts use exact integer ceilings.
"""

from __future__ import annotations

import itertools
from dataclasses import dataclass, field

# Failure tags (the page prints them as message prefixes).
C1 = "C1"
C2 = "C2"
C3 = "C3"
OCC = "C1/C2"

# Warning tags.
W_TAIL = "C4-tail"
W_IDLE = "C4-idle"

# The page's instruction-shape table: the multiples of (M edge, N edge, K
# step, threads) for warp-level mma m16n8k16, warpgroup-level wgmma
# m64nNk16, and scalar code.
INSTR_MULTIPLES = {
    "mma": (16, 8, 16, 32),
    "wgmma": (64, 8, 16, 128),
    "simt": (1, 1, 1, 32),
}


@dataclass(frozen=True)
class DeviceModel:
    """The page's hardware parameters (H100/H200 defaults)."""

    smem_per_sm: int = 228 * 1024
    smem_per_block_max: int = 227 * 1024
    regs_per_sm: int = 65536
    max_threads_per_sm: int = 2048
    max_threads_per_block: int = 1024
    max_blocks_per_sm: int = 32
    regs_per_thread_max: int = 255
    reg_granularity_per_warp: int = 256
    warp_size: int = 32
    sm_count: int = 132


def cli_device(sm_count: int = 132, smem_kb: int = 228) -> DeviceModel:
    """The device the page's command line describes: its --smem-kb is per SM,
    and one block may use all of it but 1 KB."""
    return DeviceModel(sm_count=sm_count, smem_per_sm=smem_kb * 1024,
                       smem_per_block_max=smem_kb * 1024 - 1024)


@dataclass(frozen=True)
class TileConfig:
    bm: int
    bn: int
    bk: int
    stages: int = 3
    threads: int = 128
    instr: str = "wgmma"


@dataclass
class Verdict:
    cfg: TileConfig
    smem_per_stage: int = 0
    smem_total: int = 0
    accum_per_thread: int = 0
    regs_per_thread: int = 0
    regs_per_block: int = 0
    blocks_by_regs: int = 0
    blocks_by_smem: int = 0
    blocks_by_threads: int = 0
    blocks_per_sm: int = 0
    grid: int = 0
    waves: int = 0
    last_wave_fill: float = 0.0
    c0_bytes: float = 0.0
    failures: list = field(default_factory=list)   # tags, in the order found
    warnings: list = field(default_factory=list)
    binding: str = ""

    @property
    def feasible(self) -> bool:
        return not self.failures


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def shape_violations(cfg: TileConfig, dev: DeviceModel) -> int:
    """C3: how many of the shape conditions the configuration breaks (each
    tile edge and the thread count a multiple of the MMA family's shape; no
    more threads than a block may have)."""
    multiples = INSTR_MULTIPLES[cfg.instr]
    values = (cfg.bm, cfg.bn, cfg.bk, cfg.threads)
    broken = sum(1 for value, mult in zip(values, multiples) if value % mult)
    return broken + (cfg.threads > dev.max_threads_per_block)


def accumulator_registers(cfg: TileConfig, dev: DeviceModel, accum_bytes: int):
    """C2: (accumulators per thread, 32-bit registers per thread once a
    warp's share is rounded up to whole allocation granules)."""
    per_thread = ceil_div(cfg.bm * cfg.bn, cfg.threads)
    lane_words = per_thread * accum_bytes // 4
    warp_regs = ceil_div(lane_words * dev.warp_size, dev.reg_granularity_per_warp) \
        * dev.reg_granularity_per_warp
    return per_thread, warp_regs // dev.warp_size


def residency(regs_per_block: int, smem_per_block: int, threads: int, dev: DeviceModel):
    """Blocks one SM holds by each resource, the resident count (the scarcest,
    capped by the block limit) and the binding resource ("" when none fits)."""
    fits = {
        "regs": dev.regs_per_sm // max(regs_per_block, 1),
        "smem": dev.smem_per_sm // max(smem_per_block, 1),
        "threads": dev.max_threads_per_sm // max(threads, 1),
    }
    scarcest = min(fits.values())
    resident = max(min(scarcest, dev.max_blocks_per_sm), 0)
    binding = next(name for name, n in fits.items() if n == scarcest) if resident else ""
    return fits, resident, binding


def evaluate(cfg: TileConfig, dev: DeviceModel, elem_bytes: int = 2,
             accum_bytes: int = 4) -> Verdict:
    """C3, C1 and C2 for one configuration, then its residency."""
    v = Verdict(cfg=cfg)
    v.failures += [C3] * shape_violations(cfg, dev)
    # C1: a stage holds the A slice (bm x bk) and the B slice (bk x bn).
    v.smem_per_stage = (cfg.bm + cfg.bn) * cfg.bk * elem_bytes
    v.smem_total = v.smem_per_stage * cfg.stages
    if v.smem_total > dev.smem_per_block_max:
        v.failures.append(C1)
    v.accum_per_thread, v.regs_per_thread = accumulator_registers(cfg, dev, accum_bytes)
    if v.regs_per_thread > dev.regs_per_thread_max:
        v.failures.append(C2)
    v.regs_per_block = v.regs_per_thread * cfg.threads
    fits, v.blocks_per_sm, v.binding = residency(v.regs_per_block, v.smem_total, cfg.threads, dev)
    v.blocks_by_regs, v.blocks_by_smem, v.blocks_by_threads = \
        fits["regs"], fits["smem"], fits["threads"]
    if v.blocks_per_sm == 0:
        v.failures.append(OCC)
    return v


def finish_parallelism(v: Verdict, m: int, n: int, dev: DeviceModel, b: int = 1) -> Verdict:
    """C4: the output tiles (times the batch b) in waves of the resident
    blocks; the fill of the last wave is 1.0 when the waves come out even."""
    v.grid = b * ceil_div(m, v.cfg.bm) * ceil_div(n, v.cfg.bn)
    resident = max(v.blocks_per_sm * dev.sm_count, 1)
    v.waves = ceil_div(v.grid, resident)
    leftover = v.grid % resident
    v.last_wave_fill = leftover / resident if leftover else 1.0
    if v.waves > 1 and v.last_wave_fill < 0.5:
        v.warnings.append(W_TAIL)
    if v.grid < dev.sm_count:
        v.warnings.append(W_IDLE)
    return v


def c0_bytes(m: int, n: int, k: int, bm: int, bn: int, in_bytes: int = 2,
             out_bytes: int | None = None, b: int = 1) -> float:
    """C0: cache-less DRAM traffic of the tiled GEMM: A is streamed N/bn
    times and B M/bm times (no ceilings), C written once."""
    if out_bytes is None:
        out_bytes = in_bytes
    return in_bytes * b * m * n * k * (1 / bn + 1 / bm) + out_bytes * b * m * n


# The page's candidate grid.
SWEEP_BM = (16, 32, 64, 128, 256)
SWEEP_BN = (16, 32, 64, 128, 256)
SWEEP_BK = (16, 32, 64, 128)
SWEEP_STAGES = (2, 3, 4)
SWEEP_THREADS = (128, 256, 512)


def candidates(k: int, instr: str):
    """Configurations of the page's grid in its enumeration order: K steps
    beyond K and thread counts off the family's multiple are left out."""
    tmult = INSTR_MULTIPLES[instr][3]
    for bm, bn, bk, stages, threads in itertools.product(SWEEP_BM, SWEEP_BN, SWEEP_BK,
                                                         SWEEP_STAGES, SWEEP_THREADS):
        if bk <= k and threads % tmult == 0:
            yield TileConfig(bm, bn, bk, stages, threads, instr)


@dataclass
class SweepResult:
    ranked: list            # feasible verdicts, best first
    n_tied_best: int        # how many share the minimum rounded C0
    best_fill: float        # the largest last-wave fill among them


def rank_key(v: Verdict):
    """Least traffic, then most resident blocks, then least shared memory."""
    return (round(v.c0_bytes), -v.blocks_per_sm, v.smem_total)


def sweep(m: int, n: int, k: int, dev: DeviceModel, instr: str = "wgmma", b: int = 1,
          in_bytes: int = 2, out_bytes: int | None = None) -> SweepResult:
    """The feasible configurations of the page's grid, ranked (a stable sort,
    so ties keep the enumeration order)."""
    kept = []
    for cfg in candidates(k, instr):
        v = evaluate(cfg, dev, elem_bytes=in_bytes)
        if v.feasible:
            finish_parallelism(v, m, n, dev, b)
            v.c0_bytes = c0_bytes(m, n, k, cfg.bm, cfg.bn, in_bytes, out_bytes, b)
            kept.append(v)
    kept.sort(key=rank_key)
    if not kept:
        return SweepResult(kept, 0, 0.0)
    best = round(kept[0].c0_bytes)
    tied = sum(round(v.c0_bytes) == best for v in kept)
    return SweepResult(kept, tied, max(v.last_wave_fill for v in kept))
