"""Host-side checks of the C ABI (no GPU needed).

  * libtiles.so loads and exports every function include/tiles.h declares;
  * the C++ planner matches the oracle bit for bit: page mode against the
    page restatement (ranked lists, every field, floats by their bits) and
    GB300 mode against the GB300 restatement;
  * tiles_htile_rows and tiles_c0_bytes against the oracle;
  * argument validation returns the documented status before any CUDA call.
"""

import ctypes as C
import os
import random
import re

import pytest

import tile_size_decision_gb300 as T
from tile_size_decision_gb300 import _abi
from oracle import conv as OC
from oracle import planner as OP
from oracle import planner_gb300 as OG
from tests.planner_util import compiled_tiles, oracle_device

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tiles.h")


@pytest.fixture(scope="module")
def lib():
    from tile_size_decision_gb300 import build
    build.build()
    return T.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tiles_\w+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 16
    for name in names:
        assert hasattr(lib, name), name
        assert name in _abi.SIGNATURES, f"binding lacks {name}"
    assert set(_abi.SIGNATURES) == set(names)


def test_status_strings(lib):
    assert lib.tiles_status_string(0) == b"TILES_OK"
    assert lib.tiles_status_string(-6) == b"TILES_ERR_TIMEOUT"
    assert lib.tiles_workspace_bytes() >= 4


# --------------------------------------------------------------------------- #
# Planner parity, page mode
# --------------------------------------------------------------------------- #

def page_device(sm_count, smem_kb):
    d = T.device_preset("h100_pages")
    d.sm_count = sm_count
    d.smem_per_sm = smem_kb * 1024
    d.smem_per_block_max = smem_kb * 1024 - 1024
    return d


BIND = {"": 0, "regs": 1, "smem": 2, "threads": 3, "tmem": 4}
FAILBIT = {OP.C3: _abi.FAIL_C3, OP.C1: _abi.FAIL_C1, OP.C2: _abi.FAIL_C2, OP.OCC: _abi.FAIL_OCC}
WARNBIT = {OP.W_TAIL: _abi.WARN_TAIL, OP.W_IDLE: _abi.WARN_IDLE}


def fhex(x):
    return float(x).hex()


def page_fields_native(v):
    c = v.cfg
    return (c.bm, c.bn, c.bk, c.stages, c.threads, v.smem_per_stage, v.smem_total,
            v.accum_per_thread, v.regs_per_thread, v.regs_per_block, v.blocks_by_regs,
            v.blocks_by_smem, v.blocks_by_threads, v.blocks_per_sm, v.binding, v.failures,
            v.c3_violations, v.grid, v.waves, fhex(v.last_wave_fill), v.warnings,
            fhex(v.c0_bytes))


def page_fields_oracle(v):
    c = v.cfg
    fails = 0
    for f in v.failures:
        fails |= FAILBIT[f]
    warns = 0
    for w in v.warnings:
        warns |= WARNBIT[w]
    return (c.bm, c.bn, c.bk, c.stages, c.threads, v.smem_per_stage, v.smem_total,
            v.accum_per_thread, v.regs_per_thread, v.regs_per_block, v.blocks_by_regs,
            v.blocks_by_smem, v.blocks_by_threads, v.blocks_per_sm, BIND[v.binding], fails,
            v.failures.count(OP.C3), v.grid, v.waves, fhex(v.last_wave_fill), warns,
            fhex(v.c0_bytes))


PAGE_PLANS = [
    # (b, m, n, k, instr, sm, smem_kb, in_dtype, out_dtype)
    (1, 4096, 4096, 4096, "wgmma", 132, 228, "f16", "f16"),
    (1, 4096, 4096, 4096, "mma", 108, 164, "f16", "f16"),
    (16, 2048, 2048, 1024, "wgmma", 148, 228, "bf16", "bf16"),
    (1, 5000, 3000, 4096, "simt", 148, 228, "bf16", "f32"),
    (3, 77, 1000, 24, "mma", 100, 96, "f16", "f32"),
]


@pytest.mark.parametrize("case", PAGE_PLANS, ids=lambda c: "_".join(map(str, c)))
def test_page_plan_matches_oracle(lib, case):
    b, m, n, k, instr, sm, kb, di, do = case
    dev = page_device(sm, kb)
    native, nf = T.plan(m, n, k, b=b, in_dtype=di, out_dtype=do, mode="pages", instr=instr,
                        device=dev)
    ib = 2
    ob = 4 if do == "f32" else 2
    ref = OP.sweep(m, n, k, OP.cli_device(sm, kb), instr, b=b, in_bytes=ib, out_bytes=ob)
    assert nf == len(ref.ranked)
    assert [page_fields_native(v) for v in native] == [page_fields_oracle(v) for v in ref.ranked]


def test_page_evaluate_random_configs(lib):
    rng = random.Random(1234)
    for _ in range(2000):
        instr = rng.choice(["mma", "wgmma", "simt"])
        cfg = OP.TileConfig(rng.choice([8, 16, 24, 32, 64, 100, 128, 192, 256, 512]),
                            rng.choice([8, 16, 24, 32, 64, 100, 128, 192, 256, 512]),
                            rng.choice([8, 16, 32, 48, 64, 128]), rng.randint(1, 6),
                            rng.choice([32, 64, 96, 128, 256, 384, 512, 1024, 2048]), instr)
        sm, kb = rng.choice([(132, 228), (148, 228), (108, 164), (80, 100)])
        eb = rng.choice([1, 2, 4])
        ab = rng.choice([2, 4])
        m, n, b = rng.randint(1, 20000), rng.randint(1, 20000), rng.randint(1, 8)
        dev = OP.cli_device(sm, kb)
        ref = OP.evaluate(cfg, dev, elem_bytes=eb, accum_bytes=ab)
        OP.finish_parallelism(ref, m, n, dev, b)
        nd = page_device(sm, kb)
        v = T.evaluate(nd, T.make_config(cfg.bm, cfg.bn, cfg.bk, cfg.stages, cfg.threads, instr),
                       eb, ab)
        T.finish_parallelism(nd, v, m, n, b)
        ref.c0_bytes = 0.0
        assert page_fields_native(v) == page_fields_oracle(ref), cfg


def test_c0_bytes_bitwise(lib):
    rng = random.Random(7)
    for _ in range(3000):
        b, m, n, k = rng.randint(1, 64), rng.randint(1, 1 << 16), rng.randint(1, 1 << 16), \
            rng.randint(1, 1 << 16)
        bm, bn = rng.choice([16, 64, 128, 192, 256]), rng.choice([16, 48, 64, 128, 256])
        ib, ob = rng.choice([1, 2, 4]), rng.choice([2, 4])
        assert fhex(T.c0_bytes(m, n, k, bm, bn, ib, ob, b)) == \
            fhex(OP.c0_bytes(m, n, k, bm, bn, ib, ob, b))


def test_htile_rows_match_oracle(lib):
    for H in (1, 5, 9, 17, 224):
        for kh in (1, 3, 5):
            for sh in (1, 2, 3):
                for pt in range(kh):
                    for d in (1, 2):
                        OH = OC.out_size(H, kh, sh, pt, pt, d)
                        for tile in (1, 2, 16):
                            for o0, o1 in OC.htile_ranges(max(OH, 0), tile):
                                r = OC.htile_rows(H, kh, sh, pt, d, o0, o1)
                                t = T.htile_rows(H, kh, sh, pt, d, o0, o1)
                                assert (t.in_start, t.in_end, t.in_span, t.pt, t.pb, t.halo) == (
                                    r.in_start, r.in_end, r.in_span, r.pt, r.pb, r.halo)


def test_conv_out_hw_matches_oracle(lib):
    d = _abi.ConvDesc()
    oh, ow = C.c_int32(0), C.c_int32(0)
    for h, k, s, p, dil in [(224, 3, 2, 1, 1), (9, 3, 2, 1, 1), (5, 5, 1, 2, 2), (7, 1, 3, 0, 1),
                            (1, 1, 1, 0, 1), (17, 5, 4, 3, 2)]:
        d.n, d.c, d.h, d.w, d.c_out, d.kh, d.kw = 1, 1, h, h + 3, 1, k, k
        d.sh, d.sw, d.ph, d.pw, d.dh, d.dw = s, s, p, p, dil, dil
        assert lib.tiles_conv_out_hw(C.byref(d), C.byref(oh), C.byref(ow)) == _abi.OK
        assert (oh.value, ow.value) == (OC.out_size(h, k, s, p, p, dil),
                                        OC.out_size(h + 3, k, s, p, p, dil))
        assert T.conv_out_hw(h, h + 3, k, k, (s, s), (p, p), (dil, dil)) == (oh.value, ow.value)
    d.h, d.kh, d.ph, d.dh = 2, 5, 0, 1          # no window fits
    assert lib.tiles_conv_out_hw(C.byref(d), C.byref(oh), C.byref(ow)) == _abi.ERR_INVALID_ARG
    d.h, d.sh = 9, 0
    assert lib.tiles_conv_out_hw(C.byref(d), C.byref(oh), C.byref(ow)) == _abi.ERR_INVALID_ARG


# --------------------------------------------------------------------------- #
# Planner parity, GB300 mode
# --------------------------------------------------------------------------- #

def gb300_fields_native(v):
    c = v.cfg
    return (c.bm, c.bn, c.bk, c.stages, c.threads, c.acc_bufs, c.cta_group, v.smem_per_stage,
            v.smem_total, v.tmem_cols_alloc, v.regs_per_thread, v.regs_per_block,
            v.blocks_by_regs, v.blocks_by_smem, v.blocks_by_threads, v.blocks_by_tmem,
            v.blocks_per_sm, v.binding, v.failures, v.c3_violations, v.grid, v.waves,
            fhex(v.last_wave_fill), v.warnings, fhex(v.c0_bytes), v.est_clocks, v.tail_split)


def gb300_fields_oracle(v):
    c = v.cfg
    fails = 0
    for f in v.failures:
        fails |= FAILBIT[f]
    warns = 0
    for w in v.warnings:
        warns |= WARNBIT[w]
    return (c.bm, c.bn, c.bk, c.stages, c.threads, c.acc_bufs, c.cta_group, v.smem_per_stage,
            v.smem_total, v.tmem_cols_alloc, v.regs_per_thread, v.regs_per_block,
            v.blocks_by_regs, v.blocks_by_smem, v.blocks_by_threads, v.blocks_by_tmem,
            v.blocks_per_sm, BIND[v.binding], fails, v.c3_violations, v.grid, v.waves,
            fhex(v.last_wave_fill), warns, fhex(v.c0_bytes), v.est_clocks, v.tail_split)


GB300_PLANS = [
    (1, 512, 512, 512, "f16", "f32", 148),
    (1, 4096, 4096, 4096, "f16", "f16", 148),
    (16, 2048, 2048, 1024, "bf16", "bf16", 148),
    (1, 5000, 3000, 4096, "bf16", "f32", 148),
    (8, 128, 1792, 576, "f16", "f16", 148),
    (1, 4096, 4096, 4096, "f16", "f16", 152),
    (1, 1, 1, 1, "bf16", "bf16", 160),
]


@pytest.mark.parametrize("pairs", [0, 72, 74, 76])
def test_gb300_plan_with_measured_pairs(lib, pairs):
    dev = T.device_preset("gb300")
    dev.sm_count = 152
    dev.cta_pairs = pairs
    native, nf = T.plan(4096, 4096, 4096, in_dtype="f16", device=dev)
    ref = OG.plan(1, 4096, 4096, 4096, oracle_device(dev), compiled_tiles(T), 2, 2)
    assert [gb300_fields_native(v) for v in native] == [gb300_fields_oracle(v) for v in ref]


@pytest.mark.parametrize("case", GB300_PLANS, ids=lambda c: "_".join(map(str, c)))
def test_gb300_plan_matches_oracle(lib, case):
    b, m, n, k, di, do, sm = case
    dev = T.device_preset("gb300")
    dev.sm_count = sm
    native, nf = T.plan(m, n, k, b=b, in_dtype=di, out_dtype=do, mode="gb300", device=dev)
    ref = OG.plan(b, m, n, k, oracle_device(dev), compiled_tiles(T), 2, 4 if do == "f32" else 2)
    assert nf == len(ref) == len(T.gemm_variants())
    assert [gb300_fields_native(v) for v in native] == [gb300_fields_oracle(v) for v in ref]


@pytest.mark.parametrize("field,values", [
    ("kernel_regs_per_thread", (96, 168, 176, 256)),
    ("fill_bytes_per_clk", (16, 48, 64, 128)),
    ("partial_bytes_per_clk", (0, 8, 32, 256)),
    ("handoff_clocks", (0, 512, 2048, 20000)),
    ("pair_launch_clocks", (0, 4500, 40000, 200000)),
])
def test_gb300_plan_follows_every_model_input(lib, field, values):
    # The kernel-dependent numbers are inputs of both planners: varying any
    # one of them (on shapes whose last round admits every schedule) keeps
    # the two in step, and each changes some ranking or estimate.
    shapes = [(1, 4096, 4096, 4096), (16, 2048, 2048, 1024), (1, 5000, 3000, 4096),
              (1, 3000, 2000, 1536), (1, 512, 512, 512)]
    seen = set()
    for val in values:
        dev = T.device_preset("gb300")
        dev.sm_count = 152
        setattr(dev, field, val)
        out = []
        for b, m, n, k in shapes:
            native, _ = T.plan(m, n, k, b=b, in_dtype="bf16", device=dev)
            ref = OG.plan(b, m, n, k, oracle_device(dev), compiled_tiles(T), 2, 2)
            got = [gb300_fields_native(v) for v in native]
            assert got == [gb300_fields_oracle(v) for v in ref], (field, val, m, n, k)
            out.append(tuple(got))
        seen.add(tuple(out))
    assert len(seen) > 1, f"{field} changes nothing"


def test_gb300_evaluate_random_configs(lib):
    rng = random.Random(99)
    dev = T.device_preset("gb300")
    odev = oracle_device(dev)
    for _ in range(1500):
        cfg = OG.GB300Config(rng.choice([64, 128, 256, 384]), rng.choice([16, 48, 64, 128, 192,
                                                                           256, 320, 512]),
                             rng.choice([16, 32, 64, 128]), rng.randint(1, 10),
                             rng.choice([128, 192, 256]), rng.randint(0, 3), rng.randint(0, 3))
        ib = rng.choice([1, 2, 4])
        ref = OG.evaluate(cfg, odev, ib)
        m, n, b = rng.randint(1, 9000), rng.randint(1, 9000), rng.randint(1, 4)
        if ref.cfg.cta_group < 1:
            continue
        OG.finish_parallelism(ref, odev, b, m, n)
        v = T.evaluate(dev, T.make_config(cfg.bm, cfg.bn, cfg.bk, cfg.stages, cfg.threads,
                                          "tcgen05", cfg.acc_bufs, cfg.cta_group), ib, 4)
        T.finish_parallelism(dev, v, m, n, b)
        assert gb300_fields_native(v)[:-3] == gb300_fields_oracle(ref)[:-3], cfg


# Dynamic shared memory the 256x256 CTA-pair GEMM kernel asked for at launch,
# as ncu reported it (launch__shared_mem_per_block_dynamic, 214.272 KB) in
# the 4096^3 capture.
MEASURED_SMEM_256x256_PAIR = 214272


def test_compiled_variants_are_the_deepest_pipelines_that_fit(lib):
    # The library's compiled variants, as configurations: every stage count
    # is the one the oracle derives from C1 (the deepest that fits 227 KB,
    # or the 8-stage barrier array), and C1's total for the bench kernel
    # equals what its launch requested as ncu observed it.
    dev = T.device_preset("gb300")
    odev = oracle_device(dev)
    variants = T.gemm_variants()
    assert len(variants) == lib.tiles_gemm_variant_count() >= 1
    for c in variants:
        assert (c.bk, c.threads, c.acc_bufs, c.instr, c.tail) == (64, 192, 2, _abi.INSTR_TCGEN05, 0)
        assert c.stages == OG.deepest_stages(c.bm, c.bn, c.cta_group, odev), (c.bm, c.bn)
        ref = OG.evaluate(OG.GB300Config(c.bm, c.bn, 64, c.stages, cta_group=c.cta_group), odev)
        v = T.evaluate(dev, c, 2, 4)
        assert v.smem_total == ref.smem_total and not ref.failures and not v.failures
        if (c.bm, c.bn, c.cta_group) == (256, 256, 2):
            assert v.smem_total == MEASURED_SMEM_256x256_PAIR
        if c.stages < OG.MAX_STAGES:
            deeper = OG.evaluate(OG.GB300Config(c.bm, c.bn, 64, c.stages + 1, cta_group=c.cta_group),
                                 odev)
            assert "C1" in deeper.failures
    out = _abi.Config()
    assert lib.tiles_gemm_variant(len(variants), C.byref(out)) == _abi.ERR_INVALID_ARG
    assert lib.tiles_gemm_variant(-1, C.byref(out)) == _abi.ERR_INVALID_ARG


def simulated_makespan(v, dev, k):
    """Clocks of the persistent schedule worked out unit by unit: units are
    the whole tiles, then the last round's tiles in their schedule (whole,
    two N-halves each, or s K parts each covering K blocks [p*kb//s,
    (p+1)*kb//s)); CTA group g runs units g, g + G, ... in turn (G = the
    smaller of the units and the resident groups); a unit costs its K
    blocks times the clocks of one K block at its width, and the last K part
    of a split tile, once its own K blocks are done, waits for its leading
    parts to be done and then adds one partial read-back per leading part.
    A CTA-pair launch adds its fixed cost (pair_launch_clocks)."""
    cfg = v.cfg
    cg = cfg.cta_group
    kb = -(-k // cfg.bk)
    resident = OG.resident_groups(v, dev)
    rest = v.grid % resident
    mode, parts, _ = OG.tail_choice(v, dev, kb, resident)
    full_unit = OG.unit_clocks(dev, cfg.bm, cfg.bn, cfg.bk, cg)
    units = [(kb * full_unit, None, 0)] * (v.grid - rest)       # (cost, tile, part)
    for t in range(rest):
        if mode == "nhalf":
            half = OG.unit_clocks(dev, cfg.bm, cfg.bn // 2, cfg.bk, cg)
            units += [(kb * half, None, 0)] * 2
        elif mode == "ksplit":
            for p in range(parts):
                blocks = (p + 1) * kb // parts - p * kb // parts
                units.append((blocks * full_unit, t, p))
        else:
            units.append((kb * full_unit, None, 0))
    groups = min(len(units), resident)
    clock = [0] * groups
    done = {}
    reduce = OG.reduce_clocks(dev, cfg.bm, cfg.bn, cg)
    for u, (cost, tile, part) in enumerate(units):
        g = u % groups
        finish = clock[g] + cost
        if tile is not None and part == parts - 1:
            finish = max([finish] + [done[(tile, p)] for p in range(parts - 1)])
            finish += (parts - 1) * reduce
        clock[g] = finish
        if tile is not None:
            done[(tile, part)] = clock[g]
    return max(clock) + (dev.pair_launch_clocks if cg == 2 else 0)


@pytest.mark.parametrize("sm,pairs", [(148, 0), (152, 76), (152, 74), (160, 0)])
def test_gb300_estimate_is_the_simulated_schedule(lib, sm, pairs):
    # The time estimate's round arithmetic against a unit-by-unit simulation
    # of the persistent schedule, over shapes whose last rounds take every
    # schedule (whole tiles, N-halves, 2-8 K parts) on every compiled tile.
    dev = T.device_preset("gb300")
    dev.sm_count, dev.cta_pairs = sm, pairs
    odev = oracle_device(dev)
    rng = random.Random(sm * 1000 + pairs)
    shapes = [(1, 4096, 4096, 4096), (16, 2048, 2048, 1024), (1, 5000, 3000, 4096),
              (1, 512, 512, 512), (1, 3000, 2000, 1536), (1, 256, 256, 16384)]
    shapes += [(rng.randint(1, 4), rng.randint(1, 6000), rng.randint(1, 6000),
                rng.randint(1, 9000)) for _ in range(60)]
    modes = set()
    for b, m, n, k in shapes:
        for cfg in OG.compiled_configs(compiled_tiles(T), odev):
            v = OG.evaluate(cfg, odev)
            OG.finish_parallelism(v, odev, b, m, n)
            est = OG.est_clocks(v, odev, k)
            assert est == simulated_makespan(v, odev, k), (b, m, n, k, cfg)
            modes.add(min(v.tail_split, 2))
    assert modes == {-1, 0, 2}, modes


def test_gb300_choice_at_the_bench_shape(lib):
    dev = T.device_preset("gb300")
    best = T.plan(4096, 4096, 4096, in_dtype="f16", device=dev)[0][0]
    # The CTA-pair 256x256 tile: same wave-quantised MMA time as 128x256 but
    # a third less operand traffic per SM, and the least C0.
    assert (best.cfg.bm, best.cfg.bn, best.cfg.stages, best.cfg.cta_group) == (256, 256, 6, 2)
    assert best.grid == 256 and best.waves == 4
    # 256 tiles on 74 pairs: 3 whole rounds and 34 tiles left, which fill
    # at most half the pairs, so they run as 68 N-half tiles: 64 K blocks
    # of the half-width unit (384 clocks, fill-bound) = 24,576 clocks,
    # against 32 * 512 + 2 * 4096 + 2048 = 26,624 for two K parts.
    assert best.tail_split == -1


# --------------------------------------------------------------------------- #
# Argument validation (returns before any CUDA call)
# --------------------------------------------------------------------------- #

def _desc(**kw):
    d = _abi.GemmDesc()
    d.m, d.n, d.k, d.batch = 64, 64, 64, 1
    d.a, d.b, d.c = 0x10000, 0x20000, 0x30000
    d.lda = d.ldb = d.ldc = 64
    d.a_dtype = d.b_dtype = _abi.F16
    d.c_dtype = _abi.F32
    for k, v in kw.items():
        setattr(d, k, v)
    return d


@pytest.mark.parametrize("kw,status", [
    (dict(a=None), _abi.ERR_INVALID_ARG),
    (dict(m=0), _abi.ERR_INVALID_ARG),
    (dict(batch=2), _abi.ERR_INVALID_ARG),
    (dict(a_dtype=_abi.F32, b_dtype=_abi.F32), _abi.ERR_UNSUPPORTED_DTYPE),
    (dict(b_dtype=_abi.BF16), _abi.ERR_UNSUPPORTED_DTYPE),
    (dict(c_dtype=7), _abi.ERR_UNSUPPORTED_DTYPE),
    (dict(lda=60, k=60, ldb=64), _abi.ERR_MISALIGNED),
    (dict(a=0x10002), _abi.ERR_MISALIGNED),
    (dict(lda=32), _abi.ERR_INVALID_ARG),
    (dict(m=1 << 31), _abi.ERR_TOO_LARGE),
])
def test_gemm_validation(lib, kw, status):
    d = _desc(**kw)
    assert lib.tiles_gemm(C.byref(d), None, None, 0, None) == status
    assert lib.tiles_last_error() != b""


def test_host_calls_check_arguments_before_any_cuda_call(lib):
    # Host-buffer calls reject missing buffers and piece counts outside
    # 1..16 before touching a device.
    d = _desc()
    h = C.c_void_p(0x40000)
    assert lib.tiles_gemm_host(C.byref(d), None, None, h, h, 4, None, 0, None) == _abi.ERR_INVALID_ARG
    assert lib.tiles_gemm_host(None, None, h, h, h, 4, None, 0, None) == _abi.ERR_INVALID_ARG
    for chunks in (0, 17):
        assert lib.tiles_gemm_host(C.byref(d), None, h, h, h, chunks, None, 0, None) == \
            _abi.ERR_INVALID_ARG
        assert b"chunks" in lib.tiles_last_error()
    cd = _abi.ConvDesc()
    cd.n, cd.c, cd.h, cd.w, cd.c_out, cd.kh, cd.kw = 1, 8, 9, 9, 4, 3, 3
    cd.sh = cd.sw = cd.dh = cd.dw = 1
    cd.x, cd.wt, cd.y = 0x10000, 0x20000, 0x30000
    assert lib.tiles_conv2d_host(C.byref(cd), 4, None, h, None, h, 2, None, 0, None) == \
        _abi.ERR_INVALID_ARG
    assert lib.tiles_conv2d_host(C.byref(cd), 4, None, h, h, h, 0, None, 0, None) == \
        _abi.ERR_INVALID_ARG
    cd.kh = 0
    assert lib.tiles_conv2d_host(C.byref(cd), 4, None, h, h, h, 2, None, 0, None) == \
        _abi.ERR_INVALID_ARG


def test_plan_validation(lib):
    dev = T.device_preset("gb300")
    p = _abi.Problem()
    p.b, p.m, p.n, p.k = 1, 0, 4, 4
    nf = C.c_int(-1)
    assert lib.tiles_plan(C.byref(dev), C.byref(p), None, 0, C.byref(nf)) == _abi.ERR_INVALID_ARG
    assert nf.value == 0
    p.m = 4
    p.in_dtype = 9
    assert lib.tiles_plan(C.byref(dev), C.byref(p), None, 0, C.byref(nf)) != _abi.OK
    t = _abi.HTile()
    assert lib.tiles_htile_rows(9, 3, 2, 1, 1, 2, 2, C.byref(t)) == _abi.ERR_INVALID_ARG


def test_binding_exports_every_listed_name():
    for name in T.__all__:
        assert hasattr(T, name), name


def test_drop_stage_hook_validates_before_arming(lib):
    # The planted-fault hook takes a limit in (0, 1e10] ns; a negative stage
    # disarms whatever is armed.  No GPU is touched by arming.
    assert lib.tiles_selftest_drop_stage(0, 0) == _abi.ERR_INVALID_ARG
    assert lib.tiles_selftest_drop_stage(3, 10_000_000_001) == _abi.ERR_INVALID_ARG
    assert lib.tiles_selftest_drop_stage(3, 50_000_000) == _abi.OK
    assert lib.tiles_selftest_drop_stage(-1, 0) == _abi.OK


def test_kernel_calls_refuse_a_missing_workspace_before_any_launch(lib):
    # Descriptor checks come first; then the workspace check, still before
    # any device work (a GEMM needs the device for its plan, so only the
    # order of the checks is visible here: a bad descriptor is reported as
    # such even with no workspace).
    d = _desc(a=None)
    assert lib.tiles_gemm(C.byref(d), None, None, 0, None) == _abi.ERR_INVALID_ARG
    assert b"null matrix pointer" in lib.tiles_last_error()
    cd = _abi.ConvDesc()
    cd.n, cd.c, cd.h, cd.w, cd.c_out, cd.kh, cd.kw = 1, 8, 9, 9, 4, 3, 3
    cd.sh = cd.sw = cd.dh = cd.dw = 1
    cd.x, cd.wt, cd.y = 0x10000, 0x20000, 0x30000
    assert lib.tiles_conv2d_htiled(C.byref(cd), 4, None, None, 0, None) == _abi.ERR_INVALID_ARG
    assert b"workspace" in lib.tiles_last_error()
