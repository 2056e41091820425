"""Command-line tile planner over the C ABI.

Takes the flags of the page's script (tile_decision.py, "main": --m --n --k
--instr --sm-count --smem-kb --block-m --block-n --block-k --stages --threads
--topk --diagnose) with the same meanings, so that a command written for the
page's script asks this library the same question.  Without --diagnose it
ranks every feasible configuration (the page's sweep); with --diagnose it
checks the one configuration the block flags give.

Additions for GB300: --mode gb300 ranks the configurations the sm_103a
kernels implement (tcgen05 shapes, TMEM, CTA pairs, the time model with the
last-round schedule), --device N takes the hardware model from a GPU,
--b/--in-dtype/--out-dtype set the batch and data types, --acc-bufs and
--cta-group complete a GB300 configuration, and --json prints one JSON
object instead of the table.

    python -m tile_size_decision_gb300.cli --topk 10
    python -m tile_size_decision_gb300.cli --diagnose --block-m 128 --block-n 256 --block-k 64
    python -m tile_size_decision_gb300.cli --mode gb300 --m 5000 --n 3000 --k 4096
"""
from __future__ import annotations

import argparse
import json
import sys

from . import _abi
import tile_size_decision_gb300 as T

BINDINGS = {0: "", 1: "regs", 2: "smem", 3: "threads", 4: "tmem"}
FAILURES = ((0x1, "C3"), (0x2, "C1"), (0x4, "C2"), (0x8, "OCC"))
WARNINGS = ((0x1, "tail"), (0x2, "idle"))
INSTRS = sorted(_abi.INSTR_CODES)

# The page's defaults apply in page mode; GB300 mode has its own.
PAGE_DEFAULTS = dict(m=4096, n=4096, k=4096, instr="wgmma", sm_count=132, smem_kb=228,
                     block_m=128, block_n=128, block_k=32, stages=3, threads=256, topk=15)
GB300_DEFAULTS = dict(m=4096, n=4096, k=4096, instr="tcgen05", block_m=256, block_n=256,
                      block_k=64, threads=192, topk=15)


def compiled_stages(bm: int, bn: int, cta_group: int) -> int:
    """The pipeline depth of the compiled kernel with this tile (GB300 mode's
    default --stages); 2 for a tile no kernel was compiled for."""
    for c in T.gemm_variants():
        if (c.bm, c.bn, c.cta_group) == (bm, bn, cta_group):
            return c.stages
    return 2


def parse(argv=None):
    p = argparse.ArgumentParser(
        prog="python -m tile_size_decision_gb300.cli",
        description="Check GEMM tile configurations against C0-C4 and rank them.")
    p.add_argument("--m", type=int)
    p.add_argument("--n", type=int)
    p.add_argument("--k", type=int)
    p.add_argument("--instr", choices=INSTRS)
    p.add_argument("--sm-count", type=int, help="SMs (page mode default 132)")
    p.add_argument("--smem-kb", type=int, help="shared memory per SM, KB (page mode default 228)")
    p.add_argument("--block-m", type=int)
    p.add_argument("--block-n", type=int)
    p.add_argument("--block-k", type=int)
    p.add_argument("--stages", type=int)
    p.add_argument("--threads", type=int)
    p.add_argument("--topk", type=int, help="rows of the ranking to print")
    p.add_argument("--diagnose", action="store_true",
                   help="check the configuration the block flags give")
    # GB300 additions
    p.add_argument("--mode", choices=["pages", "gb300"], default="pages")
    p.add_argument("--device", type=int, default=-1,
                   help="take the hardware model from CUDA device N (default: a preset)")
    p.add_argument("--b", type=int, default=1, help="batch of equally shaped GEMMs")
    p.add_argument("--in-dtype", choices=["f16", "bf16"], default="f16")
    p.add_argument("--out-dtype", choices=["f16", "bf16", "f32"], default=None)
    p.add_argument("--acc-bufs", type=int, default=2, help="GB300: TMEM accumulators")
    p.add_argument("--cta-group", type=int, default=None, help="GB300: 1 or 2 SMs per MMA")
    p.add_argument("--json", action="store_true")
    a = p.parse_args(argv)
    defaults = PAGE_DEFAULTS if a.mode == "pages" else GB300_DEFAULTS
    for key, val in defaults.items():
        if getattr(a, key, None) is None:
            setattr(a, key, val)
    if a.cta_group is None:
        a.cta_group = 0 if a.mode == "pages" else (2 if a.block_m == 256 else 1)
    if a.stages is None:
        a.stages = compiled_stages(a.block_m, a.block_n, a.cta_group)
    return a


def device_for(a) -> _abi.Device:
    if a.device >= 0:
        dev = T.device_query(a.device)
    else:
        dev = T.device_preset("h100_pages" if a.mode == "pages" else "gb300")
    # The page's --sm-count/--smem-kb: per-block shared memory is the per-SM
    # figure less the 1 KB the hardware reserves per block.
    if a.sm_count is not None:
        dev.sm_count = a.sm_count
    if a.smem_kb is not None:
        dev.smem_per_sm = a.smem_kb * 1024
        dev.smem_per_block_max = a.smem_kb * 1024 - 1024
    return dev


def bits(value, table):
    return [name for bit, name in table if value & bit]


def verdict_dict(v: _abi.Verdict) -> dict:
    c = v.cfg
    return {
        "bm": c.bm, "bn": c.bn, "bk": c.bk, "stages": c.stages, "threads": c.threads,
        "instr": c.instr, "acc_bufs": c.acc_bufs, "cta_group": c.cta_group,
        "smem_per_stage": v.smem_per_stage, "smem_total": v.smem_total,
        "accum_per_thread": v.accum_per_thread, "regs_per_thread": v.regs_per_thread,
        "regs_per_block": v.regs_per_block,
        "blocks_by": {"regs": v.blocks_by_regs, "smem": v.blocks_by_smem,
                      "threads": v.blocks_by_threads, "tmem": v.blocks_by_tmem},
        "blocks_per_sm": v.blocks_per_sm, "tmem_cols": v.tmem_cols_alloc,
        "binding": BINDINGS.get(v.binding, str(v.binding)),
        "failures": bits(v.failures, FAILURES), "c3_violations": v.c3_violations,
        "warnings": bits(v.warnings, WARNINGS),
        "grid": v.grid, "waves": v.waves, "last_wave_fill": v.last_wave_fill,
        "c0_bytes": v.c0_bytes, "est_clocks": v.est_clocks, "tail_split": v.tail_split,
    }


def run(a) -> dict:
    dev = device_for(a)
    out = {
        "mode": a.mode,
        "device": {"sm_count": dev.sm_count, "smem_per_sm": dev.smem_per_sm,
                   "smem_per_block_max": dev.smem_per_block_max, "regs_per_sm": dev.regs_per_sm,
                   "tmem_cols": dev.tmem_cols},
        "target": {"b": a.b, "m": a.m, "n": a.n, "k": a.k, "in_dtype": a.in_dtype,
                   "out_dtype": a.out_dtype or a.in_dtype, "instr": a.instr},
    }
    if a.diagnose:
        acc = 0 if a.mode == "pages" else a.acc_bufs
        cfg = T.make_config(a.block_m, a.block_n, a.block_k, a.stages, a.threads, a.instr, acc,
                            a.cta_group)
        in_bytes = 2
        v = T.evaluate(dev, cfg, in_bytes, 4)
        T.finish_parallelism(dev, v, a.m, a.n, b=a.b)
        out["diagnosis"] = verdict_dict(v)
        # C0 of the requested tile (the sweep ranks by it; a single check
        # reports it too).
        out_bytes = {"f16": 2, "bf16": 2, "f32": 4}[a.out_dtype or a.in_dtype]
        out["diagnosis"]["c0_bytes"] = T.c0_bytes(a.m, a.n, a.k, a.block_m, a.block_n, in_bytes,
                                                  out_bytes, b=a.b)
        return out
    ranked, feasible = T.plan(a.m, a.n, a.k, b=a.b, in_dtype=a.in_dtype, out_dtype=a.out_dtype,
                              mode=a.mode, instr=a.instr, device=dev)
    out["feasible"] = feasible
    out["ranked"] = [verdict_dict(v) for v in ranked[:max(a.topk, 0)]]
    if ranked:
        best = ranked[0].c0_bytes
        out["tied_at_best_c0"] = sum(1 for v in ranked if round(v.c0_bytes) == round(best))
    return out


def print_table(res: dict, file=None) -> None:
    file = file or sys.stdout
    d, t = res["device"], res["target"]
    print(f"hardware: {d['sm_count']} SMs, {d['smem_per_sm'] // 1024} KB shared memory per SM "
          f"({d['smem_per_block_max'] // 1024} KB per block), {d['regs_per_sm']} registers per SM"
          + (f", {d['tmem_cols']} TMEM columns" if res["mode"] == "gb300" else ""), file=file)
    print(f"problem:  {t['b']} x {t['m']}x{t['n']}x{t['k']}  {t['in_dtype']} -> {t['out_dtype']}, "
          f"fp32 accumulate, {t['instr']}, {res['mode']} rules", file=file)
    if "diagnosis" in res:
        v = res["diagnosis"]
        status = "passes" if not v["failures"] else "fails " + ", ".join(v["failures"])
        print(f"\n{v['bm']}x{v['bn']}x{v['bk']}, {v['stages']} stages, {v['threads']} threads: "
              f"{status}", file=file)
        rows = [
            ("C1 shared memory", f"{v['smem_per_stage']} B/stage, {v['smem_total']} B in all, "
                                 f"limit {d['smem_per_block_max']} B"),
            ("C2 accumulators", f"{v['accum_per_thread']} per thread -> {v['regs_per_thread']} "
                                f"registers/thread, {v['regs_per_block']}/block"
                                + (f", {v['tmem_cols']} TMEM columns" if v["tmem_cols"] else "")),
            ("occupancy", f"regs {v['blocks_by']['regs']}, smem {v['blocks_by']['smem']}, "
                          f"threads {v['blocks_by']['threads']}"
                          + (f", tmem {v['blocks_by']['tmem']}" if res["mode"] == "gb300" else "")
                          + f" -> {v['blocks_per_sm']} blocks/SM, bound by {v['binding'] or '-'}"),
            ("C4 waves", f"{v['grid']} tiles, {v['waves']} waves, last wave "
                         f"{100 * v['last_wave_fill']:.0f}% full"
                         + (f" ({', '.join(v['warnings'])})" if v["warnings"] else "")),
            ("C0 traffic", f"{v['c0_bytes'] / 1e6:.1f} MB"),
        ]
        for name, text in rows:
            print(f"  {name:18s} {text}", file=file)
        return
    print(f"\n{res['feasible']} feasible configurations; "
          f"{res.get('tied_at_best_c0', 0)} share the least C0\n", file=file)
    hdr = (f"{'#':>3} {'bm':>4} {'bn':>4} {'bk':>3} {'st':>2} {'thr':>4} {'cg':>2} "
           f"{'C0 MB':>9} {'smem KB':>8} {'regs':>4} {'blk/SM':>6} {'waves':>5} {'last%':>5} "
           f"{'bound':>7}")
    if res["mode"] == "gb300":
        hdr += f" {'est clk':>9} {'tail':>5}"
    print(hdr, file=file)
    for i, v in enumerate(res["ranked"], 1):
        row = (f"{i:>3} {v['bm']:>4} {v['bn']:>4} {v['bk']:>3} {v['stages']:>2} {v['threads']:>4} "
               f"{v['cta_group']:>2} {v['c0_bytes'] / 1e6:>9.1f} {v['smem_total'] / 1024:>8.1f} "
               f"{v['regs_per_thread']:>4} {v['blocks_per_sm']:>6} {v['waves']:>5} "
               f"{100 * v['last_wave_fill']:>5.0f} {v['binding'] or '-':>7}")
        if res["mode"] == "gb300":
            tail = {0: "whole", -1: "halves"}.get(v["tail_split"], f"K/{v['tail_split']}")
            row += f" {v['est_clocks']:>9} {tail:>5}"
        print(row, file=file)


def main(argv=None) -> int:
    a = parse(argv)
    res = run(a)
    if a.json:
        print(json.dumps(res))
    else:
        print_table(res)
    return 0


if __name__ == "__main__":
    sys.exit(main())
