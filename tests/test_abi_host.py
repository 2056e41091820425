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
    odev = OG.GB300Device(sm_count=152, fill_bytes_per_clk=dev.fill_bytes_per_clk,
                          kernel_regs_per_thread=dev.kernel_regs_per_thread, cta_pairs=pairs)
    ref = OG.plan(1, 4096, 4096, 4096, odev, 2, 2)
    assert [gb300_fields_native(v) for v in native] == [gb300_fields_oracle(v) for v in ref]


@pytest.mark.parametrize("case", GB300_PLANS, ids=lambda c: "_".join(map(str, c)))
def test_gb300_plan_matches_oracle(lib, case):
    b, m, n, k, di, do, sm = case
    dev = T.device_preset("gb300")
    dev.sm_count = sm
    native, nf = T.plan(m, n, k, b=b, in_dtype=di, out_dtype=do, mode="gb300", device=dev)
    odev = OG.GB300Device(sm_count=sm, fill_bytes_per_clk=dev.fill_bytes_per_clk,
                          kernel_regs_per_thread=dev.kernel_regs_per_thread,
                          cta_pairs=dev.cta_pairs)
    ref = OG.plan(b, m, n, k, odev, 2, 4 if do == "f32" else 2)
    assert nf == len(ref) == len(OG.VARIANTS)
    assert [gb300_fields_native(v) for v in native] == [gb300_fields_oracle(v) for v in ref]


def test_gb300_evaluate_random_configs(lib):
    rng = random.Random(99)
    dev = T.device_preset("gb300")
    odev = OG.GB300Device(fill_bytes_per_clk=dev.fill_bytes_per_clk,
                          kernel_regs_per_thread=dev.kernel_regs_per_thread)
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


def test_gb300_c1_is_the_kernels_shared_memory(lib):
    # C1's total for the bench kernel equals what its launch requested, and
    # every compiled stage count is the deepest one that fits 227 KB (or
    # the 8-stage barrier array): one stage more fails C1.
    dev = T.device_preset("gb300")
    odev = OG.GB300Device(fill_bytes_per_clk=dev.fill_bytes_per_clk,
                          kernel_regs_per_thread=dev.kernel_regs_per_thread)
    for bm, bn, cg, st in OG.VARIANTS:
        cfg = OG.GB300Config(bm, bn, 64, st, cta_group=cg)
        ref = OG.evaluate(cfg, odev, 2)
        v = T.evaluate(dev, T.make_config(bm, bn, 64, st, 192, "tcgen05", 2, cg), 2, 4)
        assert v.smem_total == ref.smem_total and not ref.failures, (bm, bn, cg)
        if (bm, bn, cg) == (256, 256, 2):
            assert v.smem_total == MEASURED_SMEM_256x256_PAIR
        if st < OG.MAX_STAGES:
            deeper = OG.evaluate(OG.GB300Config(bm, bn, 64, st + 1, cta_group=cg), odev, 2)
            assert "C1" in deeper.failures, (bm, bn, cg, st)


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
