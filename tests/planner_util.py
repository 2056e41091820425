"""Helpers shared by the planner tests: the oracle's GB300 device record
filled from the library's device record (preset or queried), and the
library's compiled tiles."""

from oracle import planner_gb300 as OG


def oracle_device(dev) -> OG.GB300Device:
    """The oracle's device record with every field taken from the library's
    record `dev` (a tiles_device from a preset or a runtime query)."""
    return OG.GB300Device(
        kernel_regs_per_thread=dev.kernel_regs_per_thread,
        fill_bytes_per_clk=dev.fill_bytes_per_clk,
        partial_bytes_per_clk=dev.partial_bytes_per_clk,
        handoff_clocks=dev.handoff_clocks,
        pair_launch_clocks=dev.pair_launch_clocks,
        cta_pairs=dev.cta_pairs,
        smem_per_sm=dev.smem_per_sm,
        smem_per_block_max=dev.smem_per_block_max,
        regs_per_sm=dev.regs_per_sm,
        max_threads_per_sm=dev.max_threads_per_sm,
        max_blocks_per_sm=dev.max_blocks_per_sm,
        sm_count=dev.sm_count,
        tmem_cols=dev.tmem_cols,
        mma_flops_per_clk=dev.mma_flops_per_clk,
    )


def compiled_tiles(T) -> list:
    """(bm, bn, cta_group) of every compiled GEMM variant, in the library's
    order."""
    return [(c.bm, c.bn, c.cta_group) for c in T.gemm_variants()]
