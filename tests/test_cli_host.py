"""The command-line planner (the page's flags over the C ABI): its answers
against the values the page prints and against the oracle's sweep."""
import io
import json
from contextlib import redirect_stdout

import pytest

import tile_size_decision_gb300 as T
from tile_size_decision_gb300 import cli
from oracle import planner as P

import os
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "planner_pages.json")


@pytest.fixture(scope="module")
def golden():
    T.load()
    with open(GOLDEN) as f:
        return json.load(f)


def run_json(*argv):
    buf = io.StringIO()
    with redirect_stdout(buf):
        assert cli.main(list(argv) + ["--json"]) == 0
    return json.loads(buf.getvalue())


def test_default_sweep_is_the_printed_one(golden):
    g = golden["sweep_default"]
    a = g["args"]
    res = run_json("--m", str(a["m"]), "--n", str(a["n"]), "--k", str(a["k"]), "--instr", a["instr"],
                   "--sm-count", str(a["sm_count"]), "--smem-kb", str(a["smem_kb"]),
                   "--topk", str(len(g["top_rows"])))
    # The page's defaults are the same question with no flags at all.
    assert run_json("--topk", str(len(g["top_rows"]))) == res
    assert res["feasible"] == g["feasible"]
    assert res["tied_at_best_c0"] == g["tied_at_min"]
    for v, want in zip(res["ranked"], g["top_rows"]):
        got = (v["bm"], v["bn"], v["bk"], v["stages"], v["threads"], f"{v['c0_bytes'] / 1e6:.1f}",
               f"{v['smem_total'] / 1024:.1f}", v["regs_per_thread"], v["blocks_per_sm"],
               v["waves"], f"{v['last_wave_fill'] * 100:.0f}", v["binding"])
        assert got == (want["bm"], want["bn"], want["bk"], want["stages"], want["threads"],
                       want["traffic_mb"], want["smem_kb"], want["regs_per_thread"],
                       want["blocks_per_sm"], want["waves"], want["tail_pct"], want["binding"])
    assert f"{res['ranked'][0]['last_wave_fill'] * 100:.0f}" == g["best_fill_pct"]


def test_diagnose_over_budget_is_the_printed_one(golden):
    g = golden["diagnose_over_budget"]
    c = g["cfg"]
    res = run_json("--diagnose", "--block-m", str(c["bm"]), "--block-n", str(c["bn"]),
                   "--block-k", str(c["bk"]), "--stages", str(c["stages"]),
                   "--threads", str(c["threads"]), "--instr", c["instr"])
    v = res["diagnosis"]
    assert v["smem_total"] == g["c1_total_bytes"]
    assert res["device"]["smem_per_block_max"] == g["c1_limit_bytes"]
    assert f"{v['smem_per_stage'] / 1024:.1f}" == g["smem_per_stage_kb"]
    assert (v["accum_per_thread"], v["regs_per_thread"], v["regs_per_block"]) == (
        g["accum_per_thread"], g["regs_per_thread"], g["regs_per_block"])
    assert (v["blocks_by"]["regs"], v["blocks_by"]["smem"], v["blocks_by"]["threads"],
            v["blocks_per_sm"]) == (g["blocks_by_regs"], g["blocks_by_smem"],
                                    g["blocks_by_threads"], g["blocks_per_sm"])
    # The page names the no-block-fits failure "C1/C2"; the ABI's bit is OCC.
    named = {"C1": "C1", "C2": "C2", "C1/C2": "OCC"}
    assert sorted(v["failures"]) == sorted(named[f] for f in g["failures"])
    assert v["binding"] == ""
    assert v["grid"] == 256 and v["waves"] == 256


@pytest.mark.parametrize("m,n,k,instr,sm,smem", [
    (1000, 3000, 512, "mma", 108, 164),
    (4096, 1024, 8192, "wgmma", 132, 228),
    (333, 4097, 96, "simt", 80, 96),
])
def test_sweep_matches_the_oracle(m, n, k, instr, sm, smem):
    res = run_json("--m", str(m), "--n", str(n), "--k", str(k), "--instr", instr,
                   "--sm-count", str(sm), "--smem-kb", str(smem), "--topk", "100000")
    dev = P.cli_device(sm, smem)
    ref = P.sweep(m, n, k, dev, instr)
    assert res["feasible"] == len(ref.ranked)
    for v, r in zip(res["ranked"], ref.ranked):
        assert (v["bm"], v["bn"], v["bk"], v["stages"], v["threads"]) == (
            r.cfg.bm, r.cfg.bn, r.cfg.bk, r.cfg.stages, r.cfg.threads)
        assert v["c0_bytes"] == r.c0_bytes and v["waves"] == r.waves
        assert v["last_wave_fill"] == r.last_wave_fill and v["binding"] == r.binding


def test_gb300_mode_ranks_the_pair_tile_first():
    res = run_json("--mode", "gb300", "--sm-count", "148")
    best = res["ranked"][0]
    assert (best["bm"], best["bn"], best["stages"], best["cta_group"]) == (256, 256, 6, 2)
    assert best["grid"] == 256 and best["waves"] == 4 and best["tail_split"] == -1
    assert res["device"]["tmem_cols"] == 512


def test_text_output_mentions_every_row():
    buf = io.StringIO()
    with redirect_stdout(buf):
        cli.main(["--topk", "5"])
    lines = buf.getvalue().splitlines()
    assert lines[0].startswith("hardware: 132 SMs")
    rows = [ln.split() for ln in lines if ln.split() and ln.split()[0].isdigit()]
    assert sum(1 for r in rows if len(r) > 10) == 5


def test_gb300_diagnose_defaults_are_the_compiled_bench_kernel():
    # With no flags but the mode, --diagnose checks the 256x256 CTA-pair
    # tile at the depth it was compiled with, which passes every constraint.
    T.load()
    res = run_json("--mode", "gb300", "--diagnose")
    v = res["diagnosis"]
    assert (v["bm"], v["bn"], v["cta_group"]) == (256, 256, 2)
    compiled = {(c.bm, c.bn, c.cta_group): c.stages for c in T.gemm_variants()}
    assert v["stages"] == compiled[(256, 256, 2)]
    assert v["failures"] == [] and v["blocks_per_sm"] == 1
    # One stage deeper no longer fits (C1), and the shared memory is reported.
    deeper = run_json("--mode", "gb300", "--diagnose", "--stages", str(v["stages"] + 1))
    assert "C1" in deeper["diagnosis"]["failures"]
