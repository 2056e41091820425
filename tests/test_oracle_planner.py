"""Pins for the oracle planner (page mode).

Three kinds of pin:
  * values the pages print (tests/golden/planner_pages.json, each cited);
  * closed forms from the tiling tutorial (capacity, registers, intensity);
  * opt-in: a differential run of the page's own script over a grid of
    shapes, devices and instruction families.  The page text is third-party
    content from the open web, so the run happens only when the variable
    TILES_PAGES_DIR names a directory holding the page text, and then in an
    isolated interpreter (python -I -S: no site packages, no user paths, no
    environment) in a scratch directory, with a time limit.  Nothing of the
    script is stored here.
"""

import json
import os
import re
import subprocess
import sys

import pytest

from oracle import planner as P
from oracle import gemm as G

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "planner_pages.json")
# Directory of the source pages' text, for the opt-in differential run.
PAGES_ENV = "TILES_PAGES_DIR"


@pytest.fixture(scope="module")
def golden():
    with open(GOLDEN) as f:
        return json.load(f)


def row_fields(v: P.Verdict):
    """A ranked verdict rendered with the precision the page prints."""
    c = v.cfg
    return (c.bm, c.bn, c.bk, c.stages, c.threads, f"{v.c0_bytes / 1e6:.1f}",
            f"{v.smem_total / 1024:.1f}", v.regs_per_thread, v.blocks_per_sm, v.waves,
            f"{v.last_wave_fill * 100:.0f}", v.binding)


def test_sweep_default_matches_printed(golden):
    g = golden["sweep_default"]
    a = g["args"]
    dev = P.cli_device(a["sm_count"], a["smem_kb"])
    res = P.sweep(a["m"], a["n"], a["k"], dev, a["instr"])
    assert len(res.ranked) == g["feasible"]
    for v, want in zip(res.ranked, g["top_rows"]):
        assert row_fields(v) == (want["bm"], want["bn"], want["bk"], want["stages"],
                                 want["threads"], want["traffic_mb"], want["smem_kb"],
                                 want["regs_per_thread"], want["blocks_per_sm"], want["waves"],
                                 want["tail_pct"], want["binding"])
    assert res.n_tied_best == g["tied_at_min"]
    assert f"{res.best_fill * 100:.0f}" == g["best_fill_pct"]
    # 1107.3 MB is the 256x256 tile's C0 at 4096^3 exactly: 2*4096^3*(2/256) + 2*4096^2.
    assert res.ranked[0].c0_bytes == 1107296256.0


def test_diagnose_over_budget(golden):
    g = golden["diagnose_over_budget"]
    c = g["cfg"]
    dev = P.cli_device()
    v = P.evaluate(P.TileConfig(c["bm"], c["bn"], c["bk"], c["stages"], c["threads"], c["instr"]), dev)
    assert f"{v.smem_per_stage / 1024:.1f}" == g["smem_per_stage_kb"]
    assert f"{v.smem_total / 1024:.1f}" == g["smem_total_kb"]
    assert v.smem_total == g["c1_total_bytes"]
    assert dev.smem_per_block_max == g["c1_limit_bytes"]
    assert v.accum_per_thread == g["accum_per_thread"]
    assert v.regs_per_thread == g["regs_per_thread"]
    assert v.regs_per_block == g["regs_per_block"]
    assert (v.blocks_by_regs, v.blocks_by_smem, v.blocks_by_threads, v.blocks_per_sm) == (
        g["blocks_by_regs"], g["blocks_by_smem"], g["blocks_by_threads"], g["blocks_per_sm"])
    assert v.failures == g["failures"]
    assert v.binding == ""
    # Zero resident blocks: the resident count is clamped to 1, so every tile is a wave.
    P.finish_parallelism(v, 4096, 4096, dev)
    assert v.grid == 256 and v.waves == 256


def test_tutorial_capacity(golden):
    g = golden["tutorial_capacity"]
    a100 = P.DeviceModel(smem_per_sm=g["a100_smem_kb"] * 1024,
                         smem_per_block_max=g["a100_smem_kb"] * 1024)
    s = g["small"]
    v = P.evaluate(P.TileConfig(s["bm"], s["bn"], s["bk"], s["stages"], 128, "mma"), a100,
                   elem_bytes=s["elem_bytes"])
    assert v.smem_total == s["smem_bytes"]
    assert v.blocks_by_smem == g["blocks_for_small"]
    assert P.C1 not in v.failures
    big = g["large"]
    v = P.evaluate(P.TileConfig(big["bm"], big["bn"], big["bk"], big["stages"], 128, "mma"),
                   a100, elem_bytes=big["elem_bytes"])
    assert v.smem_total == big["smem_bytes"]
    assert P.C1 in v.failures


def test_tutorial_registers(golden):
    g = golden["tutorial_registers"]
    v = P.evaluate(P.TileConfig(g["bm"], g["bn"], 32, 2, g["threads"], "mma"), P.DeviceModel())
    # The page's C2 counts the accumulators (16) and rounds to the warp granule:
    # 16 registers x 32 lanes = 512 = 2 granules -> 16 per thread.
    assert v.accum_per_thread == g["accumulators"]
    assert v.regs_per_thread == 16
    # The tutorial's alternative estimate adds a fixed overhead.
    assert g["bm"] * g["bn"] // g["threads"] + g["overhead"] == g["estimate"]


def test_tutorial_intensity(golden):
    g = golden["tutorial_intensity"]
    naive = G.arithmetic_intensity_naive(g["k"], g["elem_bytes"])
    tiled = G.arithmetic_intensity_tiled(g["tile"], g["tile"], g["k"], g["elem_bytes"])
    assert naive == g["naive_flop_per_byte"]
    assert tiled == g["tiled_flop_per_byte"]
    assert tiled / naive == g["ratio"]


def test_c0_batch_term_and_widths():
    # C0 is linear in b, and with b=1 and equal widths it is the page's
    # expression; the output term scales with the output width alone.
    one = P.c0_bytes(4096, 4096, 4096, 128, 256)
    assert P.c0_bytes(4096, 4096, 4096, 128, 256, b=16) == 16 * one
    base = P.c0_bytes(5000, 3000, 4096, 128, 256, in_bytes=2, out_bytes=2)
    wide = P.c0_bytes(5000, 3000, 4096, 128, 256, in_bytes=2, out_bytes=4)
    assert wide - base == 2 * 5000 * 3000
    # Closed form at a square tile: reads 2*elem*M*N*K/bm + writes elem*M*N.
    assert P.c0_bytes(1024, 1024, 1024, 64, 64) == 2 * 2 * 1024 ** 3 / 64 + 2 * 1024 ** 2


def test_c4_fill_and_warnings():
    dev = P.cli_device(sm_count=148)
    v = P.evaluate(P.TileConfig(128, 256, 64, 3, 256), dev)
    P.finish_parallelism(v, 4096, 4096, dev)
    # 512 tiles over 148 resident blocks: 4 waves, last wave 68 of 148.
    assert (v.grid, v.waves) == (512, 4)
    assert v.last_wave_fill == 68 / 148
    assert P.W_TAIL in v.warnings
    # Exact division gives a full last wave.
    v = P.finish_parallelism(P.evaluate(v.cfg, dev), 128 * 148, 256, dev)
    assert v.last_wave_fill == 1.0 and v.waves == 1 and not v.warnings
    # Fewer tiles than SMs: the idle warning.
    v = P.finish_parallelism(P.evaluate(v.cfg, dev), 128, 256 * 7, dev)
    assert v.warnings == [P.W_IDLE]


def test_binding_order_prefers_regs_on_ties():
    dev = P.DeviceModel()
    # 256 threads with 128x128 (64 regs) and smem 64 KB: regs -> 4, smem -> 3.
    v = P.evaluate(P.TileConfig(128, 128, 64, 2, 256), dev)
    assert (v.blocks_by_regs, v.blocks_by_smem, v.blocks_by_threads) == (4, 3, 8)
    assert v.binding == "smem"
    # A tie between regs and smem: 128 threads hold 128 accumulators each
    # (16384 regs/block -> 4 blocks) and 3 stages of 16 KB leave room for 4.
    v = P.evaluate(P.TileConfig(128, 128, 32, 3, 128), dev)
    assert (v.blocks_by_regs, v.blocks_by_smem, v.blocks_by_threads) == (4, 4, 16)
    assert v.binding == "regs"
    # Threads bind: 1024-thread blocks, 2 per SM.
    v = P.evaluate(P.TileConfig(64, 64, 64, 4, 1024), dev)
    assert (v.blocks_by_regs, v.blocks_by_smem, v.blocks_by_threads) == (8, 3, 2)
    assert v.binding == "threads"


# --------------------------------------------------------------------------- #
# Differential run of the page's own script
# --------------------------------------------------------------------------- #

def _pages_lines():
    """Lines of the page text that prints the planner script."""
    pages = os.environ.get(PAGES_ENV, "")
    if not pages:
        pytest.skip(f"opt-in: set {PAGES_ENV} to the directory of the source pages' text")
    if not os.path.isdir(pages):
        pytest.skip(f"{PAGES_ENV}={pages!r} is not a directory")
    for name in sorted(os.listdir(pages)):
        if not name.endswith(".md"):
            continue
        with open(os.path.join(pages, name), encoding="utf-8") as f:
            lines = f.read().split("\n")
        if any(l.startswith("#!/usr/bin/env python3") for l in lines):
            return lines
    pytest.skip("no mounted page prints the planner script")


def _script_path(tmp_path_factory):
    lines = _pages_lines()
    start = next(i for i, l in enumerate(lines) if l.startswith("#!/usr/bin/env python3"))
    end = next(i for i in range(start, len(lines)) if "raise SystemExit(main())" in lines[i])
    d = tmp_path_factory.mktemp("page_script")
    p = d / "planner_page.py"
    p.write_text("\n".join(lines[start:end + 1]) + "\n", encoding="utf-8")
    return str(p)


@pytest.fixture(scope="module")
def page_script(tmp_path_factory):
    return _script_path(tmp_path_factory)


def run_script(path, *args):
    # Isolated interpreter, empty environment, the script's own scratch
    # directory as the working directory, bounded time.
    out = subprocess.run([sys.executable, "-I", "-S", path, *map(str, args)],
                         capture_output=True, text=True, timeout=120, env={},
                         cwd=os.path.dirname(path))
    assert out.returncode == 0, out.stderr
    return out.stdout


ROW = re.compile(r"^\s*(\d+)\s+(\d+)\s+(\d+)\s+(\d+)\s+(\d+)\s+([\d.]+)\s+([\d.]+)\s+(\d+)\s+(\d+)"
                 r"\s+(\d+)\s+(\d+)%\s+(\w+)\s*$")


def parse_sweep(text):
    feasible = int(re.search(r"feasible configurations found: (\d+)", text).group(1))
    rows = []
    for line in text.splitlines():
        m = ROW.match(line)
        if m:
            g = m.groups()
            rows.append((int(g[0]), int(g[1]), int(g[2]), int(g[3]), int(g[4]), g[5], g[6],
                         int(g[7]), int(g[8]), int(g[9]), g[10], g[11]))
    tied = int(re.search(r"tied at the minimum traffic: (\d+)", text).group(1))
    fill = re.search(r"best last-wave fill among feasible configurations: (\d+)%", text).group(1)
    return feasible, rows, tied, fill


SWEEP_CASES = [
    # (m, n, k, instr, sm_count, smem_kb)
    (4096, 4096, 4096, "wgmma", 132, 228),
    (4096, 4096, 4096, "mma", 132, 228),
    (4096, 4096, 4096, "wgmma", 108, 164),
    (5000, 3000, 4096, "wgmma", 148, 228),
    (2048, 2048, 1024, "mma", 148, 228),
    (512, 512, 512, "simt", 148, 228),
    (100, 37, 24, "wgmma", 132, 100),
    (128, 12544, 576, "wgmma", 148, 228),
]


@pytest.mark.parametrize("case", SWEEP_CASES, ids=lambda c: "x".join(map(str, c)))
def test_sweep_matches_page_script(page_script, case):
    m, n, k, instr, sms, kb = case
    text = run_script(page_script, "--m", m, "--n", n, "--k", k, "--instr", instr,
                      "--sm-count", sms, "--smem-kb", kb, "--topk", 100000)
    feasible, rows, tied, fill = parse_sweep(text)
    res = P.sweep(m, n, k, P.cli_device(sms, kb), instr)
    assert len(res.ranked) == feasible
    assert [row_fields(v) for v in res.ranked] == rows
    assert res.n_tied_best == tied
    assert f"{res.best_fill * 100:.0f}" == fill


DIAG_NUMS = [
    (r"C1 shared/stage\s+([\d.]+) KB -> total\s+([\d.]+) KB", ("smem_per_stage_kb", "smem_total_kb")),
    (r"C2 accumulators\s+(\d+)/thread ->\s+(\d+) regs/thread \(warp-rounded\),\s+(\d+) regs/block",
     ("accum", "regs", "regs_block")),
    (r"occupancy: regs -> (\d+) blk/SM, smem -> (\d+), threads -> (\d+)\s+=> (\d+) blk/SM",
     ("by_regs", "by_smem", "by_threads", "bps")),
    (r"binding=(\w*)", ("binding",)),
    (r"C4 grid\s+(\d+) tiles over\s+(\d+)-warp blocks -> (\d+) wave\(s\), last wave\s+([\d.]+)% full",
     ("grid", "warps", "waves", "fill")),
]


def parse_diag(text):
    out = {}
    for pat, names in DIAG_NUMS:
        m = re.search(pat, text)
        assert m, pat
        out.update(zip(names, m.groups()))
    out["fail"] = [l.split("FAIL", 1)[1].split()[0] for l in text.splitlines() if "FAIL" in l]
    out["warn"] = [l.split("warn", 1)[1].split()[0] for l in text.splitlines()
                   if l.strip().startswith("warn")]
    return out


def oracle_diag(v: P.Verdict):
    warn_tags = {P.W_TAIL: "C4", P.W_IDLE: "C4"}
    return {
        "smem_per_stage_kb": f"{v.smem_per_stage / 1024:.1f}",
        "smem_total_kb": f"{v.smem_total / 1024:.1f}",
        "accum": str(v.accum_per_thread), "regs": str(v.regs_per_thread),
        "regs_block": str(v.regs_per_block),
        "by_regs": str(v.blocks_by_regs), "by_smem": str(v.blocks_by_smem),
        "by_threads": str(v.blocks_by_threads), "bps": str(v.blocks_per_sm),
        "binding": v.binding,
        "grid": str(v.grid), "warps": str(v.blocks_per_sm * v.cfg.threads // 32),
        "waves": str(v.waves), "fill": f"{v.last_wave_fill * 100:.1f}",
        "fail": list(v.failures), "warn": [warn_tags[w] for w in v.warnings],
    }


DIAG_CASES = [
    # (bm, bn, bk, stages, threads, instr, m, n, sms, kb)
    (128, 256, 64, 3, 256, "wgmma", 4096, 4096, 132, 228),
    (256, 256, 64, 4, 256, "wgmma", 4096, 4096, 132, 228),
    (256, 256, 64, 3, 256, "wgmma", 4096, 4096, 132, 228),
    (128, 128, 32, 2, 256, "mma", 4096, 4096, 108, 164),
    (100, 24, 20, 2, 96, "wgmma", 5000, 3000, 148, 228),
    (64, 8, 16, 4, 2048, "mma", 513, 77, 148, 228),
    (16, 16, 16, 2, 32, "simt", 128, 128, 148, 228),
    (256, 128, 128, 2, 512, "wgmma", 5000, 3000, 148, 228),
    (128, 192, 64, 4, 384, "wgmma", 4096, 4096, 148, 228),
]


@pytest.mark.parametrize("case", DIAG_CASES, ids=lambda c: "_".join(map(str, c)))
def test_diagnose_matches_page_script(page_script, case):
    bm, bn, bk, st, thr, instr, m, n, sms, kb = case
    text = run_script(page_script, "--diagnose", "--block-m", bm, "--block-n", bn,
                      "--block-k", bk, "--stages", st, "--threads", thr, "--instr", instr,
                      "--m", m, "--n", n, "--sm-count", sms, "--smem-kb", kb)
    dev = P.cli_device(sms, kb)
    v = P.evaluate(P.TileConfig(bm, bn, bk, st, thr, instr), dev)
    P.finish_parallelism(v, m, n, dev)
    assert oracle_diag(v) == parse_diag(text)
