"""Tile-size constraint procedure, page mode (oracle; test infrastructure only).

Restates, step by step, the checks of the page
"04-tile-size-decision/tile_decision.py" (sections: ``Device``, ``Config``,
``Verdict`` records; ``INSTR_SHAPES``; ``evaluate``; ``finish_parallelism``;
``dram_traffic``; ``sweep``; ``main``) and the README on the same site
("目的" block: C0 = b*M*N*K*(1/block_N + 1/block_M) + b*M*N).

Order of the checks, as on the page:
  C3 instruction shape -> C1 on-chip capacity -> C2 register pressure ->
  occupancy and the binding resource -> C4 waves and last-wave fill -> C0 DRAM
  traffic -> sweep, filter, sort.

Page quirks kept on purpose (each is observable in the page's printed output):
  * C2 counts accumulators only and rounds to 256 registers per warp.
  * blocks_by_smem divides by shared memory per SM (not per block).
  * With 0 blocks per SM the resident count is clamped to 1, so waves = grid.
  * The binding label is the first minimum in the order regs, smem, threads.
  * The sort key is (round(C0), -blocks_per_sm, smem_total), stable over the
    enumeration order bm, bn, bk, stages, threads.

Readings where the pages are silent:
  * C0 with a batch b and separate input/output widths:
        in_bytes*b*M*N*K*(1/bn + 1/bm) + out_bytes*b*M*N
    evaluated left to right in IEEE float64; with b=1 and in=out=elem this is
    the page's own expression.
  * ceil(M/bm) is the exact integer ceiling; the page's float ceiling equals
    it for every block size below 2**22.
"""

from __future__ import annotations

from dataclasses import dataclass, field

# Failure tags (the page writes them as message prefixes).
C1 = "C1"
C2 = "C2"
C3 = "C3"
OCC = "C1/C2"

# Warning tags.
W_TAIL = "C4-tail"
W_IDLE = "C4-idle"

# (M multiple, N multiple, K multiple, thread multiple) per MMA family, from
# the page's instruction-shape table (mma m16n8k16 warp-level, wgmma m64nNk16
# warpgroup-level, scalar).
INSTR_MULTIPLES = {
    "mma": (16, 8, 16, 32),
    "wgmma": (64, 8, 16, 128),
    "simt": (1, 1, 1, 32),
}


@dataclass(frozen=True)
class DeviceModel:
    """Hardware parameters of the page's ``Device`` record (H100/H200 defaults)."""

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
    """The device the page's command line builds: per-block shared memory is
    the per-SM figure minus 1 KB."""
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


def check_instruction_shape(v: Verdict, dev: DeviceModel) -> None:
    """C3: every tile edge and the thread count are multiples of the MMA shape;
    the block may not exceed the per-block thread limit."""
    cfg = v.cfg
    mm, nm, km, tm = INSTR_MULTIPLES[cfg.instr]
    for value, mult in ((cfg.bm, mm), (cfg.bn, nm), (cfg.bk, km), (cfg.threads, tm)):
        if value % mult:
            v.failures.append(C3)
    if cfg.threads > dev.max_threads_per_block:
        v.failures.append(C3)


def check_capacity(v: Verdict, dev: DeviceModel, elem_bytes: int) -> None:
    """C1: one stage holds a bm x bk slice of A and a bk x bn slice of B; the
    pipeline keeps `stages` of them; the total must fit one block's smem."""
    cfg = v.cfg
    v.smem_per_stage = (cfg.bm * cfg.bk + cfg.bk * cfg.bn) * elem_bytes
    v.smem_total = v.smem_per_stage * cfg.stages
    if v.smem_total > dev.smem_per_block_max:
        v.failures.append(C1)


def check_registers(v: Verdict, dev: DeviceModel, accum_bytes: int) -> None:
    """C2: the bm x bn accumulator spread over the block's threads, counted in
    32-bit registers and rounded up to the per-warp allocation granule."""
    cfg = v.cfg
    v.accum_per_thread = ceil_div(cfg.bm * cfg.bn, cfg.threads)
    words = v.accum_per_thread * accum_bytes // 4
    per_warp = ceil_div(words * dev.warp_size, dev.reg_granularity_per_warp) \
        * dev.reg_granularity_per_warp
    v.regs_per_thread = per_warp // dev.warp_size
    if v.regs_per_thread > dev.regs_per_thread_max:
        v.failures.append(C2)
    v.regs_per_block = v.regs_per_thread * cfg.threads


def occupancy(v: Verdict, dev: DeviceModel) -> None:
    """Resident blocks per SM: the least of what registers, shared memory and
    threads allow, capped by the hardware block limit.  The binding resource
    is the first of regs, smem, threads that reaches that least value."""
    cfg = v.cfg
    v.blocks_by_regs = dev.regs_per_sm // max(v.regs_per_block, 1)
    v.blocks_by_smem = dev.smem_per_sm // max(v.smem_total, 1)
    v.blocks_by_threads = dev.max_threads_per_sm // max(cfg.threads, 1)
    least = min(v.blocks_by_regs, v.blocks_by_smem, v.blocks_by_threads)
    v.blocks_per_sm = max(min(least, dev.max_blocks_per_sm), 0)
    if v.blocks_per_sm == 0:
        v.failures.append(OCC)
        return
    for name, count in (("regs", v.blocks_by_regs), ("smem", v.blocks_by_smem),
                        ("threads", v.blocks_by_threads)):
        if count == least:
            v.binding = name
            break


def evaluate(cfg: TileConfig, dev: DeviceModel, elem_bytes: int = 2,
             accum_bytes: int = 4) -> Verdict:
    """C3, C1, C2 and occupancy for one configuration, in the page's order."""
    v = Verdict(cfg=cfg)
    check_instruction_shape(v, dev)
    check_capacity(v, dev, elem_bytes)
    check_registers(v, dev, accum_bytes)
    occupancy(v, dev)
    return v


def finish_parallelism(v: Verdict, m: int, n: int, dev: DeviceModel, b: int = 1) -> Verdict:
    """C4: output tiles, waves over the resident blocks, last-wave fill.

    ``b`` multiplies the tile count (a batch of independent GEMMs); b=1 is the
    page.  Fill is 1.0 when the tiles divide the resident count exactly.
    """
    cfg = v.cfg
    v.grid = b * ceil_div(m, cfg.bm) * ceil_div(n, cfg.bn)
    resident = max(v.blocks_per_sm * dev.sm_count, 1)
    v.waves = ceil_div(v.grid, resident)
    rem = v.grid % resident
    v.last_wave_fill = rem / resident if rem else 1.0
    if v.waves > 1 and v.last_wave_fill < 0.5:
        v.warnings.append(W_TAIL)
    if v.grid < dev.sm_count:
        v.warnings.append(W_IDLE)
    return v


def c0_bytes(m: int, n: int, k: int, bm: int, bn: int, in_bytes: int = 2,
             out_bytes: int | None = None, b: int = 1) -> float:
    """C0: cache-less DRAM traffic of the tiled GEMM.

    Every output tile streams a bm x K panel of A and a K x bn panel of B, so
    A is read ceil-free N/bn times and B M/bm times; C is written once.
    """
    if out_bytes is None:
        out_bytes = in_bytes
    return in_bytes * b * m * n * k * (1 / bn + 1 / bm) + out_bytes * b * m * n


SWEEP_BM = (16, 32, 64, 128, 256)
SWEEP_BN = (16, 32, 64, 128, 256)
SWEEP_BK = (16, 32, 64, 128)
SWEEP_STAGES = (2, 3, 4)
SWEEP_THREADS = (128, 256, 512)


@dataclass
class SweepResult:
    ranked: list            # feasible verdicts, best first
    n_tied_best: int        # how many share the minimum rounded C0
    best_fill: float        # the largest last-wave fill among them


def sweep(m: int, n: int, k: int, dev: DeviceModel, instr: str = "wgmma", b: int = 1,
          in_bytes: int = 2, out_bytes: int | None = None) -> SweepResult:
    """Enumerate the page's candidate grid, keep the feasible ones, rank them.

    Ranking: least rounded C0 first, then more resident blocks, then less
    shared memory; ties keep the enumeration order (bm, bn, bk, stages,
    threads, each ascending).  Python's round() rounds half to even.
    b, in_bytes and out_bytes extend C0 and C4 as the README's C0 does; the
    defaults are the page's sweep.
    """
    tmult = INSTR_MULTIPLES[instr][3]
    kept = []
    for bm in SWEEP_BM:
        for bn in SWEEP_BN:
            for bk in SWEEP_BK:
                if bk > k:
                    continue
                for stages in SWEEP_STAGES:
                    for threads in SWEEP_THREADS:
                        if threads % tmult:
                            continue
                        v = evaluate(TileConfig(bm, bn, bk, stages, threads, instr), dev,
                                     elem_bytes=in_bytes)
                        if not v.feasible:
                            continue
                        finish_parallelism(v, m, n, dev, b)
                        v.c0_bytes = c0_bytes(m, n, k, bm, bn, in_bytes, out_bytes, b)
                        kept.append(v)
    kept.sort(key=lambda v: (round(v.c0_bytes), -v.blocks_per_sm, v.smem_total))
    if kept:
        best = round(kept[0].c0_bytes)
        tied = sum(1 for v in kept if round(v.c0_bytes) == best)
        fill = max(v.last_wave_fill for v in kept)
    else:
        tied, fill = 0, 0.0
    return SweepResult(kept, tied, fill)
