"""The GB300 planner against what the hardware reports and measures.

The README of the tile-size-decision page lists, among its known
limitations, that C1 and C2 are bounds that the real kernel has to confirm
and that the script measures nothing.  These tests make that confirmation:

  * C1: the planner's (and the oracle's) shared-memory total of each compiled
    kernel is exactly the dynamic shared memory the kernel requests, as the
    CUDA runtime reports it, with nothing static beside it;
  * C2 / registers: the register figure the planner uses covers the count
    the runtime reports for every compiled kernel, which spills nothing;
  * residency and C4: the oracle's blocks per SM equal the runtime's
    occupancy calculator, and its resident CTA groups equal the blocks per
    SM times the SMs (one CTA per tile) or the co-resident clusters (CTA
    pairs);
  * the oracle's GB300 plan, fed the device record the runtime query fills,
    is the native plan bit for bit;
  * ranking: on the four GEMM workloads the planner's first choice (with its
    own last-round schedule) runs within 3% of the fastest candidate of the
    measured shortlist (timed again, alternating with the fastest, when the
    shortlist's one-after-another timings put it outside), and the time estimate orders the shortlist's
    configurations as they measure wherever it separates them by more than
    20% (the model's error band, from measured shortlists of 16 shapes).
"""

import pytest

import synth_inputs as S
from oracle import planner_gb300 as OG

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import tile_size_decision_gb300 as T  # noqa: E402
from tests.planner_util import compiled_tiles, oracle_device  # noqa: E402


@pytest.fixture(scope="module")
def dev():
    T.load()
    torch.cuda.set_device(0)
    return T.device_query(0)


def test_runtime_confirms_c1_registers_and_residency(dev):
    preset = T.device_preset("gb300")
    odev = oracle_device(dev)
    variants = T.gemm_variants()
    regs_seen = 0
    for i, c in enumerate(variants):
        info = T.gemm_variant_info(i)
        assert (info.cfg.bm, info.cfg.bn, info.cfg.stages, info.cfg.cta_group) == \
            (c.bm, c.bn, c.stages, c.cta_group)
        ref = OG.evaluate(OG.GB300Config(c.bm, c.bn, c.bk, c.stages, cta_group=c.cta_group), odev)
        native = T.evaluate(dev, c, 2, 4)
        assert not ref.failures and not native.failures
        # C1 is what the launch asks for and is opted in to.
        assert info.dynamic_smem_bytes == ref.smem_total == native.smem_total, (c.bm, c.bn)
        assert info.max_dynamic_smem_bytes == info.dynamic_smem_bytes
        assert info.static_smem_bytes == 0
        # Registers: the planner's figure covers the kernel's; no spills.
        assert info.local_bytes_per_thread == 0, (c.bm, c.bn)
        assert 0 < info.regs_per_thread <= dev.kernel_regs_per_thread
        assert info.regs_per_thread <= preset.kernel_regs_per_thread
        regs_seen = max(regs_seen, info.regs_per_thread)
        # Residency: the occupancy calculator's blocks per SM and groups.
        assert ref.blocks_per_sm == native.blocks_per_sm == info.blocks_per_sm, (c.bm, c.bn)
        assert OG.resident_groups(ref, odev) == info.resident_groups, (c.bm, c.bn)
        if c.cta_group == 1:
            assert info.resident_groups == info.blocks_per_sm * dev.sm_count
        else:
            assert info.resident_groups == dev.cta_pairs <= dev.sm_count // 2
    # The queried register figure is the largest count, warp-granule rounded.
    granule = dev.reg_granularity_per_warp // dev.warp_size
    assert dev.kernel_regs_per_thread == -(-regs_seen // granule) * granule


@pytest.mark.parametrize("name", ["gemm_512", "gemm_4096", "gemm_batched", "gemm_ragged"])
def test_oracle_plan_on_the_queried_device(dev, name):
    wl = S.WORKLOADS[name]
    native, nf = T.plan(wl.m, wl.n, wl.k, b=wl.b, in_dtype=wl.in_dtype, out_dtype=wl.out_dtype,
                        device=dev)
    ref = OG.plan(wl.b, wl.m, wl.n, wl.k, oracle_device(dev), compiled_tiles(T), 2,
                  S.DTYPE_BYTES[wl.out_dtype])
    assert nf == len(ref)
    got = [(v.cfg.bm, v.cfg.bn, v.cfg.stages, v.cfg.cta_group, v.smem_total, v.blocks_per_sm,
            v.grid, v.waves, float(v.last_wave_fill).hex(), float(v.c0_bytes).hex(),
            v.est_clocks, v.tail_split) for v in native]
    want = [(v.cfg.bm, v.cfg.bn, v.cfg.stages, v.cfg.cta_group, v.smem_total, v.blocks_per_sm,
             v.grid, v.waves, float(v.last_wave_fill).hex(), float(v.c0_bytes).hex(),
             v.est_clocks, v.tail_split) for v in ref]
    assert got == want


def operands(wl):
    """Device operands of a workload's shape (values do not matter here)."""
    dt = {S.F16: torch.float16, S.BF16: torch.bfloat16}[wl.in_dtype]
    out_dt = {S.F16: torch.float16, S.BF16: torch.bfloat16, S.F32: torch.float32}[wl.out_dtype]
    g = torch.Generator(device="cuda")
    g.manual_seed(wl.seed)
    a = torch.randn(wl.a_shape(), device="cuda", generator=g).to(dt)
    b = torch.randn(wl.b_shape(), device="cuda", generator=g).to(dt)
    c = torch.empty(wl.c_shape(), device="cuda", dtype=out_dt)
    return a, b, c


def alternate_times(a, b, c, ws, batched, cfg_x, cfg_y, rounds=7, launches=20):
    """Median microseconds per launch of two configurations, each timed as
    `launches` back-to-back launches between one pair of events, the two
    alternating for `rounds` rounds."""
    def run(cfg):
        if batched:
            T.gemm_batched(a, b, out=c, cfg=cfg, workspace=ws)
        else:
            T.gemm(a, b, out=c, cfg=cfg, workspace=ws)

    times = ([], [])
    for cfg in (cfg_x, cfg_y):
        run(cfg)
    torch.cuda.synchronize()
    for _ in range(rounds):
        for i, cfg in enumerate((cfg_x, cfg_y)):
            s = torch.cuda.Event(enable_timing=True)
            e = torch.cuda.Event(enable_timing=True)
            s.record()
            for _ in range(launches):
                run(cfg)
            e.record()
            torch.cuda.synchronize()
            times[i].append(1000.0 * s.elapsed_time(e) / launches)
    T.check(ws)
    med = lambda v: sorted(v)[len(v) // 2]
    return med(times[0]), med(times[1])


@pytest.mark.parametrize("name", ["gemm_4096", "gemm_batched", "gemm_ragged", "gemm_512"])
def test_planner_choice_against_the_measured_shortlist(dev, name):
    wl = S.WORKLOADS[name]
    a, b, c = operands(wl)
    T.tuned_clear()
    ranked, _ = T.plan(wl.m, wl.n, wl.k, b=wl.b, in_dtype=wl.in_dtype, out_dtype=wl.out_dtype,
                       device=dev)
    top = ranked[:4]
    first = top[0].cfg
    # Room for every schedule the shortlist times, K splits included.
    ws = max((T.gemm_workspace(a, b, c, T.make_config(v.cfg.bm, v.cfg.bn, v.cfg.bk, v.cfg.stages,
                                                      v.cfg.threads, v.cfg.instr, v.cfg.acc_bufs,
                                                      v.cfg.cta_group, tail="ksplit"))
              for v in top), key=lambda t: t.numel())
    try:
        _, rows = T.gemm_autotune(a, b, c, top_k=len(top), reps=25, workspace=ws,
                                  batched=wl.b > 1)
        T.check(ws)
    finally:
        T.tuned_clear()
    ran = [r for r in rows if r["status"] == 0]
    fastest = min(r["us"] for r in ran)

    def own(cfg):
        # A configuration with its planner-chosen last round (tail "auto").
        return next(r for r in ran if (r["bm"], r["bn"], r["stages"], r["cta_group"]) ==
                    (cfg.bm, cfg.bn, cfg.stages, cfg.cta_group) and r["tail_asked"] == 0)

    table = [(v.cfg.bm, v.cfg.bn, v.cfg.cta_group, v.est_clocks, own(v.cfg)["us"]) for v in top]
    # 3%, or 0.3 us on launches of a few microseconds (their jitter).  The
    # shortlist times its candidates one after another, so a clock that
    # drifts between them can misorder two close ones: a first choice
    # outside the band is timed again against the fastest, alternately.
    us_first = own(first)["us"]
    if us_first > max(1.03 * fastest, fastest + 0.3):
        best = min(ran, key=lambda r: r["us"])
        cfg_best = T.make_config(best["bm"], best["bn"], first.bk, best["stages"], first.threads,
                                 first.instr, first.acc_bufs, best["cta_group"],
                                 tail=best["tail_asked"])
        us_first, fastest = alternate_times(a, b, c, ws, wl.b > 1, first, cfg_best)
    assert us_first <= max(1.03 * fastest, fastest + 0.3), (table, fastest, us_first)
    for i, (_, _, _, est_i, us_i) in enumerate(table):
        for _, _, _, est_j, us_j in table[i + 1:]:
            if est_i < 0.8 * est_j:
                assert us_i < us_j, table
            if est_j < 0.8 * est_i:
                assert us_j < us_i, table
