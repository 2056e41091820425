"""GB300 mode of the tile planner (oracle; test infrastructure only).

This library's extension of the page's constraints (README of
"04-tile-size-decision": C3 instruction shape, C1 capacity, C2 registers,
C4 waves and last-wave fill, C0 traffic) to its sm_103a kernels, written
independently of the C++ planner so that the two can be compared bit for
bit.  No page fixes these rules; the README's known-limitations section says
what fixes them instead: C1 and C2 are bounds that the real kernel has to
confirm.  So the kernel-dependent numbers are inputs here, never literals:

  * the compiled tiles (bm, bn, cta_group) come from the library's variant
    list; the pipeline depth of each is derived, not listed: the deepest
    stage count (at most MAX_STAGES) that passes C1;
  * the kernels' register figure, the co-resident CTA pairs, the operand
    fill rate, the K-split hand-off rate and latency and the CTA pairs'
    launch cost are fields of the device record, which callers fill from the
    runtime (GPU tests) or from the library's preset (host tests).

What pins them: GPU tests compare C1's total with the dynamic shared memory
the runtime reports for each compiled kernel, the register figure with its
register count, the resident groups with the runtime's occupancy (blocks per
SM, co-resident clusters), and the ranking with measured launch times; host
tests compare the time estimate with a brute-force simulation of the
persistent schedule.  The pieces shared with the page (C0, the fill
formula, the binding order) are pinned through the page-mode tests.

Rules
  C3   tcgen05.mma kind::f16: 128 rows per CTA (bm = 128 * cta_group,
       cta_group 1 or 2), bn a multiple of 16 in [16, 256], bk a multiple of
       16; the kernels' layout adds bk * in_bytes == 128 (one swizzle atom),
       (bn / cta_group) a multiple of 64, 192 threads, 1-2 accumulators,
       1-MAX_STAGES stages.  One violation per failed condition.
  C1   stages * ((bm + bn) / cg) * bk * in_bytes + the epilogue's staging
       (four 32-row x 128-byte boxes) + the barrier block + 1 KB of
       alignment slack <= smem_per_block_max.  The page's C1 counts the A/B
       tiles alone and names what it leaves out.
  C2   TMEM: acc_bufs * bn fp32 columns, allocated as a power of two >= 32,
       <= tmem_cols.
  residency  least of regs (kernel_regs_per_thread * threads), smem,
       threads, TMEM blocks per SM; ties go to regs, smem, threads, tmem.
  C4   tiles = b * ceil(M/bm) * ceil(N/bn); resident groups = blocks per
       SM times the SMs (one CTA per tile) or the co-resident CTA pairs
       (cta_pairs, else sm_count // 2); waves; fill as on the page.
  C0   the page's expression with b, in_bytes, out_bytes.
  time est_clocks = whole rounds * K blocks * unit + the last round's cost,
       unit = max(mma, fill) with mma = (bm/cg)*bn*bk*2 // mma_flops_per_clk
       and fill = ceil(stage bytes / fill_bytes_per_clk).  The last round
       (when tiles % resident > 0) takes the cheapest of: whole tiles;
       N-halves (whole B atoms, and the rest fills at most half the groups)
       at the half-width tile's unit; K parts s = 2 .. min(resident // rest,
       MAX_TAIL_PARTS, K blocks) at ceil(K blocks / s) * unit + (s - 1) *
       reduce, reduce = 2 * ceil((bm/cg)*bn*4 / partial_bytes_per_clk) +
       handoff_clocks (a part's fp32 partial goes out and comes back).
       Ties keep that order and the fewer parts.  tail_split reports s, -1
       for N-halves, 0 for whole tiles.  A CTA-pair kernel adds
       pair_launch_clocks, its extra fixed cost per launch.
  rank (est_clocks, round(C0), -blocks per SM, smem_total), stable over the
       variant order.
"""

from __future__ import annotations

from dataclasses import dataclass, field

from . import planner as page

THREADS = 192                  # warp-specialised block: producer, MMA, 4 epilogue warps
EPILOGUE_BYTES = 4 * 32 * 128  # one 32-row x 128-byte staging box per epilogue warp
BARRIER_BYTES = 256            # mbarriers, the TMEM address slot, the abort flag
ALIGN_SLACK = 1024             # operand tiles start on a 1024-byte swizzle atom
MAX_STAGES = 8
MAX_TAIL_PARTS = 8


@dataclass(frozen=True)
class GB300Device:
    """Hardware and kernel facts.  The kernel-dependent fields have no
    defaults: a caller supplies them from an observation or a preset."""

    kernel_regs_per_thread: int
    fill_bytes_per_clk: int
    partial_bytes_per_clk: int
    handoff_clocks: int
    pair_launch_clocks: int
    cta_pairs: int = 0          # co-resident 2-CTA clusters; 0 = sm_count // 2
    smem_per_sm: int = 228 * 1024
    smem_per_block_max: int = 227 * 1024
    regs_per_sm: int = 65536
    max_threads_per_sm: int = 2048
    max_blocks_per_sm: int = 32
    sm_count: int = 148
    tmem_cols: int = 512
    mma_flops_per_clk: int = 8192


@dataclass(frozen=True)
class GB300Config:
    bm: int
    bn: int
    bk: int
    stages: int
    threads: int = THREADS
    acc_bufs: int = 2
    cta_group: int = 1


@dataclass
class GB300Verdict:
    cfg: GB300Config
    c3_violations: int = 0
    failures: list = field(default_factory=list)
    smem_per_stage: int = 0
    smem_total: int = 0
    tmem_cols_alloc: int = 0
    regs_per_thread: int = 0
    regs_per_block: int = 0
    blocks_by_regs: int = 0
    blocks_by_smem: int = 0
    blocks_by_threads: int = 0
    blocks_by_tmem: int = 0
    blocks_per_sm: int = 0
    binding: str = ""
    grid: int = 0
    waves: int = 0
    last_wave_fill: float = 0.0
    warnings: list = field(default_factory=list)
    c0_bytes: float = 0.0
    est_clocks: int = 0
    tail_split: int = 0


def _tmem_alloc(cols: int) -> int:
    p = 32
    while p < cols:
        p *= 2
    return p


def stage_bytes(bm: int, bn: int, bk: int, cg: int, in_bytes: int = 2) -> int:
    """One pipeline stage of one CTA: its bm/cg rows of A and bn/cg columns
    of B, bk deep."""
    return (bm // cg + bn // cg) * bk * in_bytes


def c1_total(bm: int, bn: int, bk: int, cg: int, stages: int, in_bytes: int = 2) -> int:
    return stage_bytes(bm, bn, bk, cg, in_bytes) * stages + EPILOGUE_BYTES + BARRIER_BYTES \
        + ALIGN_SLACK


def evaluate(cfg: GB300Config, dev: GB300Device, in_bytes: int = 2) -> GB300Verdict:
    v = GB300Verdict(cfg=cfg)
    cg = cfg.cta_group if cfg.cta_group in (1, 2) else 1
    conditions = (
        cfg.cta_group in (1, 2),
        cfg.bm == 128 * cg,
        cfg.bn % 16 == 0 and 16 <= cfg.bn <= 256,
        cfg.bk % 16 == 0 and cfg.bk * in_bytes == 128,
        (cfg.bn // cg) % 64 == 0,
        cfg.threads == THREADS,
        1 <= cfg.acc_bufs <= 2,
        1 <= cfg.stages <= MAX_STAGES,
    )
    v.c3_violations = sum(not ok for ok in conditions)
    if v.c3_violations:
        v.failures.append(page.C3)
    v.smem_per_stage = stage_bytes(cfg.bm, cfg.bn, cfg.bk, cg, in_bytes)
    v.smem_total = c1_total(cfg.bm, cfg.bn, cfg.bk, cg, cfg.stages, in_bytes)
    if v.smem_total > dev.smem_per_block_max:
        v.failures.append(page.C1)
    v.tmem_cols_alloc = _tmem_alloc(max(cfg.acc_bufs * cfg.bn, 1))
    if v.tmem_cols_alloc > dev.tmem_cols:
        v.failures.append(page.C2)
    v.regs_per_thread = dev.kernel_regs_per_thread
    v.regs_per_block = dev.kernel_regs_per_thread * cfg.threads
    supply_demand = (
        ("regs", dev.regs_per_sm, v.regs_per_block),
        ("smem", dev.smem_per_sm, v.smem_total),
        ("threads", dev.max_threads_per_sm, cfg.threads),
        ("tmem", dev.tmem_cols, v.tmem_cols_alloc),
    )
    fits = {name: supply // max(demand, 1) for name, supply, demand in supply_demand}
    v.blocks_by_regs, v.blocks_by_smem = fits["regs"], fits["smem"]
    v.blocks_by_threads, v.blocks_by_tmem = fits["threads"], fits["tmem"]
    scarcest = min(fits.values())
    v.blocks_per_sm = max(min(scarcest, dev.max_blocks_per_sm), 0)
    if v.blocks_per_sm == 0:
        v.failures.append(page.OCC)
    else:
        v.binding = next(name for name, _, _ in supply_demand if fits[name] == scarcest)
    return v


def deepest_stages(bm: int, bn: int, cg: int, dev: GB300Device, in_bytes: int = 2) -> int:
    """The pipeline depth of a compiled tile: the most stages (up to
    MAX_STAGES) that still pass C1; 0 when not even one does."""
    bk = 128 // in_bytes
    best = 0
    for st in range(1, MAX_STAGES + 1):
        if c1_total(bm, bn, bk, cg, st, in_bytes) <= dev.smem_per_block_max:
            best = st
    return best


def resident_groups(v: GB300Verdict, dev: GB300Device) -> int:
    cg = max(v.cfg.cta_group, 1)
    slots = dev.cta_pairs if (cg == 2 and dev.cta_pairs > 0) else dev.sm_count // cg
    return max(v.blocks_per_sm * slots, 1)


def finish_parallelism(v: GB300Verdict, dev: GB300Device, b: int, m: int, n: int) -> None:
    cfg = v.cfg
    v.grid = b * page.ceil_div(m, cfg.bm) * page.ceil_div(n, cfg.bn)
    resident = resident_groups(v, dev)
    v.waves = page.ceil_div(v.grid, resident)
    rem = v.grid % resident
    v.last_wave_fill = rem / resident if rem else 1.0
    v.warnings = []
    if v.waves > 1 and v.last_wave_fill < 0.5:
        v.warnings.append(page.W_TAIL)
    if v.grid < dev.sm_count:
        v.warnings.append(page.W_IDLE)


def unit_clocks(dev: GB300Device, bm: int, bn: int, bk: int, cg: int) -> int:
    """Clocks of one K block of one tile: the MMA's or the operand fill's,
    whichever is longer."""
    mma = (bm // cg) * bn * bk * 2 // dev.mma_flops_per_clk
    fill = page.ceil_div(stage_bytes(bm, bn, bk, cg), dev.fill_bytes_per_clk)
    return max(mma, fill)


def reduce_clocks(dev: GB300Device, bm: int, bn: int, cg: int) -> int:
    """Clocks one extra K part adds to the last part: its fp32 partial tile
    per CTA written and read back, plus the hand-off's fixed latency."""
    return 2 * page.ceil_div((bm // cg) * bn * 4, max(dev.partial_bytes_per_clk, 1)) \
        + dev.handoff_clocks


def nhalf_applies(cfg: GB300Config, grid: int, resident: int) -> bool:
    """A last round filling at most half the groups, with N-halves that are
    whole 64-column B atoms per CTA."""
    cg = max(cfg.cta_group, 1)
    half = cfg.bn // 2
    if half % cg or (half // cg) % 64:
        return False
    rest = grid % resident
    return 0 < rest and 2 * rest <= resident


def tail_choice(v: GB300Verdict, dev: GB300Device, kblocks: int, resident: int):
    """(mode, parts, clocks) of the last round: whole tiles, N-halves or K
    parts, whichever the model makes cheapest (ties keep that order and the
    fewer parts)."""
    cfg = v.cfg
    cg = max(cfg.cta_group, 1)
    unit = unit_clocks(dev, cfg.bm, cfg.bn, cfg.bk, cg)
    best = ("whole", 0, kblocks * unit)
    rest = v.grid % resident
    if rest == 0:
        return best
    if nhalf_applies(cfg, v.grid, resident):
        t = kblocks * unit_clocks(dev, cfg.bm, cfg.bn // 2, cfg.bk, cg)
        if t < best[2]:
            best = ("nhalf", 0, t)
    reduce = reduce_clocks(dev, cfg.bm, cfg.bn, cg)
    for s in range(2, min(resident // rest, MAX_TAIL_PARTS, kblocks) + 1):
        t = page.ceil_div(kblocks, s) * unit + (s - 1) * reduce
        if t < best[2]:
            best = ("ksplit", s, t)
    return best


def est_clocks(v: GB300Verdict, dev: GB300Device, k: int) -> int:
    cfg = v.cfg
    cg = max(cfg.cta_group, 1)
    kblocks = page.ceil_div(k, cfg.bk)
    unit = unit_clocks(dev, cfg.bm, cfg.bn, cfg.bk, cg)
    resident = resident_groups(v, dev)
    mode, parts, clocks = tail_choice(v, dev, kblocks, resident)
    v.tail_split = parts if mode == "ksplit" else (-1 if mode == "nhalf" else 0)
    rest = v.grid % resident
    launch = dev.pair_launch_clocks if cfg.cta_group == 2 else 0
    return (v.grid // resident) * kblocks * unit + (clocks if rest else 0) + launch


def compiled_configs(tiles, dev: GB300Device, in_bytes: int = 2) -> list:
    """Configurations of the compiled tiles (bm, bn, cta_group), each at
    its deepest stage count."""
    bk = 128 // in_bytes
    return [GB300Config(bm, bn, bk, deepest_stages(bm, bn, cg, dev, in_bytes), cta_group=cg)
            for bm, bn, cg in tiles]


def plan(b: int, m: int, n: int, k: int, dev: GB300Device, tiles, in_bytes: int = 2,
         out_bytes: int = 2) -> list:
    """Feasible verdicts of the compiled tiles, best first."""
    kept = []
    for cfg in compiled_configs(tiles, dev, in_bytes):
        v = evaluate(cfg, dev, in_bytes)
        if v.failures:
            continue
        finish_parallelism(v, dev, b, m, n)
        v.c0_bytes = page.c0_bytes(m, n, k, cfg.bm, cfg.bn, in_bytes, out_bytes, b)
        v.est_clocks = est_clocks(v, dev, k)
        kept.append(v)
    kept.sort(key=lambda v: (v.est_clocks, round(v.c0_bytes), -v.blocks_per_sm, v.smem_total))
    return kept
