"""GB300 mode of the tile planner (oracle; test infrastructure only).

Parity unpinned: no page fixes these rules.  They extend the page's
constraint order (tile_decision.py: C3 -> C1 -> C2 -> occupancy -> C4 -> C0)
to the sm_103a kernels of this library, and this module restates them
independently of the C++ planner so the two can be compared bit for bit.
The parts that reduce to the page (C0, the fill formula, the binding order)
are pinned through the page-mode tests.

Rules
  C3   tcgen05.mma kind::f16: 128 rows per CTA (bm = 128 * cta_group,
       cta_group 1 or 2), bn a multiple of 16 in [16, 256], bk a multiple of
       16; the kernels' layout adds bk * in_bytes == 128 (one swizzle atom),
       (bn / cta_group) a multiple of 64, 192 threads, 1-2 accumulators,
       1-8 stages.  One violation count per failed condition.
  C1   stages * ((bm/cg)*bk + bk*(bn/cg)) * in_bytes + 16384 (the
       epilogue's staging: four 32-row x 128-byte boxes, from which TMA
       stores write C) + 256 (barriers) + 1024 (alignment slack)
       <= smem_per_block_max.  The page's C1 counts the A/B tiles alone and
       names the epilogue, barriers and padding it leaves out.
  C2   TMEM: acc_bufs * bn fp32 columns, allocated as a power of two >= 32,
       <= tmem_cols.
  occupancy  least of regs (kernel_regs_per_thread * threads), smem,
       threads, TMEM; binding order regs, smem, threads, tmem.
  C4   grid = b * ceil(M/bm) * ceil(N/bn); resident = max(bps * slots, 1)
       with slots = sm_count for one CTA per tile and the co-resident CTA
       pairs (cta_pairs, else sm_count // 2) for pairs; waves; fill as on the
       page.
  C0   the page's expression with b, in_bytes, out_bytes.
  time est_clocks = (grid // resident) * ceil(K/bk) * unit + the last
       round's cost, unit = max(mma, fill), mma = (bm/cg)*bn*bk*2 //
       mma_flops_per_clk, fill = ceil(smem_per_stage / fill_bytes_per_clk).
       The last round (when grid % resident > 0) takes the cheapest of:
       whole tiles ceil(K/bk) * unit; N-halves (if whole B atoms and the rest
       fills at most half the groups) ceil(K/bk) * unit of the half-width
       tile; K parts s in 2..min(resident // rest, 8, K blocks):
       ceil(K/bk / s) * unit + (s-1) * reduce with reduce =
       2 * ceil((bm/cg)*bn*4 / PARTIAL_BYTES_PER_CLK) + 2048: a K part's
       fp32 partial goes out and comes back at 32 bytes per clock per SM,
       the rate measured for it on GB300 (not the operand fill rate).
       tail_split reports s, -1 for N-halves, 0 for whole tiles.
  rank (est_clocks, round(C0), -bps, smem_total), stable over the variant
       order.
"""

from __future__ import annotations

from dataclasses import dataclass, field

from . import planner as page

# Compiled variants (bm, bn, cta_group, stages), in enumeration order.
VARIANTS = ((128, 64, 1, 8), (128, 128, 1, 6), (128, 192, 1, 5), (128, 256, 1, 4),
            (256, 128, 2, 8), (256, 256, 2, 6))

THREADS = 192
EPILOGUE_BYTES = 4 * 32 * 128
BARRIER_BYTES = 256
ALIGN_SLACK = 1024
MAX_STAGES = 8


@dataclass(frozen=True)
class GB300Device:
    smem_per_sm: int = 228 * 1024
    smem_per_block_max: int = 227 * 1024
    regs_per_sm: int = 65536
    max_threads_per_sm: int = 2048
    max_blocks_per_sm: int = 32
    sm_count: int = 148
    tmem_cols: int = 512
    mma_flops_per_clk: int = 8192
    fill_bytes_per_clk: int = 64
    kernel_regs_per_thread: int = 168
    cta_pairs: int = 0          # co-resident 2-CTA clusters; 0 = sm_count // 2


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


def evaluate(cfg: GB300Config, dev: GB300Device, in_bytes: int = 2) -> GB300Verdict:
    v = GB300Verdict(cfg=cfg)
    cg = cfg.cta_group
    bad = [cg not in (1, 2)]
    cgs = cg if cg in (1, 2) else 1
    bad += [
        cfg.bm != 128 * cgs,
        cfg.bn % 16 != 0 or cfg.bn < 16 or cfg.bn > 256,
        cfg.bk % 16 != 0 or cfg.bk * in_bytes != 128,
        (cfg.bn // cgs) % 64 != 0,
        cfg.threads != THREADS,
        not 1 <= cfg.acc_bufs <= 2,
        not 1 <= cfg.stages <= MAX_STAGES,
    ]
    v.c3_violations = sum(bad)
    if v.c3_violations:
        v.failures.append(page.C3)
    v.smem_per_stage = ((cfg.bm // cgs) * cfg.bk + cfg.bk * (cfg.bn // cgs)) * in_bytes
    v.smem_total = v.smem_per_stage * cfg.stages + EPILOGUE_BYTES + BARRIER_BYTES + ALIGN_SLACK
    if v.smem_total > dev.smem_per_block_max:
        v.failures.append(page.C1)
    v.tmem_cols_alloc = _tmem_alloc(max(cfg.acc_bufs * cfg.bn, 1))
    if v.tmem_cols_alloc > dev.tmem_cols:
        v.failures.append(page.C2)
    v.regs_per_thread = dev.kernel_regs_per_thread
    v.regs_per_block = dev.kernel_regs_per_thread * cfg.threads
    v.blocks_by_regs = dev.regs_per_sm // max(v.regs_per_block, 1)
    v.blocks_by_smem = dev.smem_per_sm // max(v.smem_total, 1)
    v.blocks_by_threads = dev.max_threads_per_sm // max(cfg.threads, 1)
    v.blocks_by_tmem = dev.tmem_cols // max(v.tmem_cols_alloc, 1)
    counts = (("regs", v.blocks_by_regs), ("smem", v.blocks_by_smem),
              ("threads", v.blocks_by_threads), ("tmem", v.blocks_by_tmem))
    least = min(c for _, c in counts)
    v.blocks_per_sm = max(min(least, dev.max_blocks_per_sm), 0)
    if v.blocks_per_sm == 0:
        v.failures.append(page.OCC)
    else:
        v.binding = next(name for name, c in counts if c == least)
    return v


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


MAX_TAIL_PARTS = 8


HANDOFF_CLOCKS = 2048
PARTIAL_BYTES_PER_CLK = 32


def _stage_bytes(bm: int, bn: int, bk: int, cg: int, in_bytes: int = 2) -> int:
    return ((bm // cg) * bk + bk * (bn // cg)) * in_bytes


def _unit(dev: GB300Device, bm: int, bn: int, bk: int, cg: int) -> int:
    mma = (bm // cg) * bn * bk * 2 // dev.mma_flops_per_clk
    fill = page.ceil_div(_stage_bytes(bm, bn, bk, cg), dev.fill_bytes_per_clk)
    return max(mma, fill)


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
    unit = _unit(dev, cfg.bm, cfg.bn, cfg.bk, cg)
    best = ("whole", 0, kblocks * unit)
    rest = v.grid % resident
    if rest == 0:
        return best
    if nhalf_applies(cfg, v.grid, resident):
        t = kblocks * _unit(dev, cfg.bm, cfg.bn // 2, cfg.bk, cg)
        if t < best[2]:
            best = ("nhalf", 0, t)
    reduce = 2 * page.ceil_div((cfg.bm // cg) * cfg.bn * 4, PARTIAL_BYTES_PER_CLK) + HANDOFF_CLOCKS
    for s in range(2, min(resident // rest, MAX_TAIL_PARTS, kblocks) + 1):
        t = page.ceil_div(kblocks, s) * unit + (s - 1) * reduce
        if t < best[2]:
            best = ("ksplit", s, t)
    return best


def est_clocks(v: GB300Verdict, dev: GB300Device, k: int) -> int:
    cfg = v.cfg
    cg = max(cfg.cta_group, 1)
    kblocks = page.ceil_div(k, cfg.bk)
    unit = _unit(dev, cfg.bm, cfg.bn, cfg.bk, cg)
    resident = resident_groups(v, dev)
    mode, parts, clocks = tail_choice(v, dev, kblocks, resident)
    v.tail_split = parts if mode == "ksplit" else (-1 if mode == "nhalf" else 0)
    rest = v.grid % resident
    return (v.grid // resident) * kblocks * unit + (clocks if rest else 0)


def plan(b: int, m: int, n: int, k: int, dev: GB300Device, in_bytes: int = 2,
         out_bytes: int = 2) -> list:
    kept = []
    for bm, bn, cg, stages in VARIANTS:
        cfg = GB300Config(bm, bn, 128 // in_bytes, stages, cta_group=cg)
        v = evaluate(cfg, dev, in_bytes)
        if v.failures:
            continue
        finish_parallelism(v, dev, b, m, n)
        v.c0_bytes = page.c0_bytes(m, n, k, bm, bn, in_bytes, out_bytes, b)
        v.est_clocks = est_clocks(v, dev, k)
        kept.append(v)
    kept.sort(key=lambda v: (v.est_clocks, round(v.c0_bytes), -v.blocks_per_sm, v.smem_total))
    return kept
