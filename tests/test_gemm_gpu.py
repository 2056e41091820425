"""GPU parity of the tcgen05 GEMM against the float64 oracle.

Every case runs through the C ABI (tiles_gemm / tiles_gemm_batched via the
binding) and compares element by element with oracle.gemm under
|C - C_ref| <= 1e-3 * sum|A||B| + ulp_out(C_ref), or exactly where the inputs
make the fp32 result exact.
"""

import numpy as np
import pytest

import synth_inputs as S
from oracle import gemm as OG
from oracle import tolerance as OT

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import tile_size_decision_gb300 as T  # noqa: E402
from tests.gpu_util import TORCH_DT, to_cuda, to_f64, empty_out  # noqa: E402

# Compiled variants: (bn, cta_group) -> stages.
VARIANTS = {(64, 1): 8, (128, 1): 6, (192, 1): 5, (256, 1): 4, (128, 2): 8, (256, 2): 6}
VARIANT_IDS = [f"bn{bn}_cg{cg}" for bn, cg in VARIANTS]


def variant(v):
    bn, cg = v
    return T.make_config(128 * cg, bn, 64, VARIANTS[v], 192, "tcgen05", 2, cg)


@pytest.fixture(scope="module")
def ws():
    T.load()
    return T.workspace()


def run_gemm(a_np, b_np, in_dt, out_dt, cfg=None, ws=None, pitch_a=None, pitch_b=None,
             pitch_c=None):
    a = to_cuda(a_np, in_dt, pitch_a)
    b = to_cuda(b_np, in_dt, pitch_b)
    c = empty_out((a_np.shape[0], b_np.shape[1]), out_dt, pitch_c)
    T.gemm(a, b, out=c, cfg=cfg, workspace=ws)
    T.check(ws)
    return c


def assert_close(got, a64, b64, out_dt):
    ref = OG.gemm(a64, b64)
    bound = OG.gemm_bound(a64, b64)
    ok, worst, idx = OT.check(got, ref, bound, out_dt)
    assert ok, f"worst ratio {worst} at {idx}: got {got[idx]} want {ref[idx]}"


@pytest.mark.parametrize("v", list(VARIANTS), ids=VARIANT_IDS)
def test_identity_exact(ws, v):
    # C = I x B must return B exactly: catches swizzle, descriptor and
    # row/column placement mistakes in every variant.
    bn, cg = v
    m = k = 128 * cg
    n = 2 * bn
    a = S.quantise(np.eye(m, k), S.F16)
    b = S.random_matrix(1, (k, n), S.F16)
    c = run_gemm(a, b, S.F16, S.F32, variant(v), ws)
    assert np.array_equal(to_f64(c), S.widen(b, S.F16))


@pytest.mark.parametrize("v", list(VARIANTS), ids=VARIANT_IDS)
def test_permutation_exact(ws, v):
    bn, cg = v
    rng = np.random.default_rng(3)
    m = k = 512
    n = bn + 64
    perm = rng.permutation(m)
    a = S.quantise(np.eye(m)[perm], S.BF16)
    b = S.random_matrix(2, (k, n), S.BF16)
    c = run_gemm(a, b, S.BF16, S.F32, variant(v), ws)
    assert np.array_equal(to_f64(c), S.widen(b, S.BF16)[perm])


@pytest.mark.parametrize("v", list(VARIANTS), ids=VARIANT_IDS)
@pytest.mark.parametrize("dt", [S.F16, S.BF16])
def test_integer_inputs_exact(ws, v, dt):
    # Entries in [-2, 2] and K = 320: every partial sum is an integer below
    # 2^24, so the fp32 accumulation is exact whatever its order.
    bn, cg = v
    m, n, k = 200 * cg + 57, 3 * bn - 16, 320
    a = S.integer_matrix(5, (m, k), dt)
    b = S.integer_matrix(6, (k, n), dt)
    c = run_gemm(a, b, dt, S.F32, variant(v), ws)
    assert np.array_equal(to_f64(c), OG.gemm(S.widen(a, dt), S.widen(b, dt)))


SHAPES = [
    (1, 1, 1), (1, 8, 8), (7, 24, 16), (16, 16, 17), (128, 64, 64), (129, 136, 80),
    (130, 136, 80), (255, 257, 63), (256, 256, 128), (300, 200, 100), (64, 520, 1000),
    (1000, 8, 8), (517, 611, 129),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("out_dt", [S.F32, S.F16, S.BF16])
def test_small_shapes_planned(ws, shape, out_dt):
    m, n, k = shape
    in_dt = S.BF16 if out_dt == S.BF16 else S.F16
    a = S.random_matrix(10 + m, (m, k), in_dt)
    b = S.random_matrix(20 + n, (k, n), in_dt)
    pa, pb = -(-k // 8) * 8, -(-n // 8) * 8
    pc = -(-n // 8) * 8 if out_dt != S.F32 else -(-n // 4) * 4
    c = run_gemm(a, b, in_dt, out_dt, None, ws, pa, pb, pc)
    assert_close(to_f64(c), S.widen(a, in_dt), S.widen(b, in_dt), out_dt)


@pytest.mark.parametrize("v", list(VARIANTS), ids=VARIANT_IDS)
def test_ragged_every_variant_with_canaries(ws, v):
    # Output written into the interior of a larger buffer: rows past M and
    # columns past N (the canary band) must stay untouched.
    bn, cg = v
    m, n, k = 333 * cg, 2 * bn + 40, 200
    a = S.random_matrix(31, (m, k), S.F16, "normal")
    b = S.random_matrix(32, (k, n), S.F16, "normal")
    big = torch.full((m + 3, n + 24), 12345.0, dtype=torch.float32, device="cuda")
    c = big[:m, :n]
    T.gemm(to_cuda(a, S.F16, -(-k // 8) * 8), to_cuda(b, S.F16, -(-n // 8) * 8), out=c,
           cfg=variant(v), workspace=ws)
    T.check(ws)
    host = to_f64(big)
    assert np.all(host[m:, :] == 12345.0) and np.all(host[:, n:] == 12345.0)
    assert_close(host[:m, :n], S.widen(a, S.F16), S.widen(b, S.F16), S.F32)


@pytest.mark.parametrize("v", list(VARIANTS), ids=VARIANT_IDS)
@pytest.mark.parametrize("out_dt", [S.F16, S.BF16])
def test_ragged_16bit_output_stays_inside_m_and_n(ws, v, out_dt):
    # 16-bit C leaves through 64-column TMA store boxes of 32 rows; the
    # tensor map over C clips them at M and N, so the canary band past N
    # (inside the row pitch) and the rows past M stay untouched.
    bn, cg = v
    m, n, k = 333 * cg, 2 * bn + 40, 200
    in_dt = S.BF16 if out_dt == S.BF16 else S.F16
    a = S.random_matrix(33, (m, k), in_dt, "normal")
    b = S.random_matrix(34, (k, n), in_dt, "normal")
    canary = 1536.0                      # exact in fp16 and bf16
    big = torch.full((m + 3, n + 24), canary, dtype=TORCH_DT[out_dt], device="cuda")
    c = big[:m, :n]
    T.gemm(to_cuda(a, in_dt, -(-k // 8) * 8), to_cuda(b, in_dt, -(-n // 8) * 8), out=c,
           cfg=variant(v), workspace=ws)
    T.check(ws)
    host = to_f64(big)
    assert np.all(host[m:, :] == canary) and np.all(host[:, n:] == canary)
    assert_close(host[:m, :n], S.widen(a, in_dt), S.widen(b, in_dt), out_dt)


@pytest.mark.parametrize("v", [(128, 1), (256, 2), (192, 1)], ids=["bn128_cg1", "bn256_cg2",
                                                                   "bn192_cg1"])
@pytest.mark.parametrize("out_dt", [S.F32, S.F16, S.BF16])
def test_batched_output_gaps_stay_untouched(ws, v, out_dt):
    # C's items sit in a larger buffer: each item's rows past M and columns
    # past N, and the rows between items, belong to nobody.  The 3-D tensor
    # map over C (item pitch = the buffer's) must keep every store inside
    # its own item's M x N.
    bn, cg = v
    bsz, m, n, k = 3, 130 * cg + 7, bn + 72, 128
    in_dt = S.BF16 if out_dt == S.BF16 else S.F16
    a = S.random_matrix(43, (bsz, m, k), in_dt, "normal")
    b = S.random_matrix(44, (bsz, k, n), in_dt, "normal")
    canary = 1536.0
    big = torch.full((bsz, m + 9, n + 40), canary, dtype=TORCH_DT[out_dt], device="cuda")
    c = big[:, :m, :n]
    T.gemm_batched(to_cuda(a, in_dt), to_cuda(b, in_dt), out=c, cfg=variant(v), workspace=ws)
    T.check(ws)
    host = to_f64(big)
    assert np.all(host[:, m:, :] == canary) and np.all(host[:, :, n:] == canary)
    assert_close(host[:, :m, :n], S.widen(a, in_dt), S.widen(b, in_dt), out_dt)


@pytest.mark.parametrize("v", [None] + list(VARIANTS), ids=["planned"] + VARIANT_IDS)
def test_batched_small(ws, v):
    bsz, m, n, k = 5, 300, 200, 96
    a = S.random_matrix(41, (bsz, m, k), S.BF16, "normal")
    b = S.random_matrix(42, (bsz, k, n), S.BF16, "normal")
    c = empty_out((bsz, m, n), S.BF16)
    T.gemm_batched(to_cuda(a, S.BF16), to_cuda(b, S.BF16), out=c,
                   cfg=variant(v) if v else None, workspace=ws)
    T.check(ws)
    assert_close(to_f64(c), S.widen(a, S.BF16), S.widen(b, S.BF16), S.BF16)


@pytest.mark.parametrize("v", [(128, 1), (256, 2)], ids=["bn128_cg1", "bn256_cg2"])
def test_batched_rows_do_not_leak_between_items(ws, v):
    # M not a multiple of the tile: a tile's rows past M must read zeros, not
    # the next batch item's rows.  Item t of A is all (t+1), B all ones.
    bsz, m, n, k = 3, 70, 256, 64
    a = np.stack([np.full((m, k), t + 1.0) for t in range(bsz)])
    a = S.quantise(a, S.F16)
    b = S.quantise(np.ones((bsz, k, n)), S.F16)
    c = empty_out((bsz, m, n), S.F32)
    T.gemm_batched(to_cuda(a, S.F16), to_cuda(b, S.F16), out=c, cfg=variant(v), workspace=ws)
    T.check(ws)
    got = to_f64(c)
    for t in range(bsz):
        assert np.all(got[t] == (t + 1) * k)


def full_workload(name, small_ws=None):
    # The launch configuration bench.py times: the planned tile and a
    # workspace sized for the K-split last round (unless small_ws is given).
    wl = S.WORKLOADS[name]
    a, b = S.gemm_inputs(wl)
    ta, tb = to_cuda(a, wl.in_dtype), to_cuda(b, wl.in_dtype)
    c = empty_out(wl.c_shape(), wl.out_dtype)
    ws = small_ws if small_ws is not None else T.gemm_workspace(ta, tb, c)
    if wl.b > 1:
        T.gemm_batched(ta, tb, out=c, workspace=ws)
    else:
        T.gemm(ta, tb, out=c, workspace=ws)
    T.check(ws)
    return wl, a, b, to_f64(c)


@pytest.mark.parametrize("name", ["gemm_512", "gemm_4096", "gemm_batched", "gemm_ragged"])
def test_workload_full_parity(ws, name):
    wl, a, b, got = full_workload(name)
    assert_close(got, S.widen(a, wl.in_dtype), S.widen(b, wl.in_dtype), wl.out_dtype)


@pytest.mark.parametrize("name", ["gemm_4096", "gemm_ragged"])
def test_workload_parity_without_workspace_room(ws, name):
    # With only the 256-byte workspace the last round falls back to N-halves
    # (or whole tiles); the result must be the same within tolerance.
    wl, a, b, got = full_workload(name, small_ws=ws)
    assert_close(got, S.widen(a, wl.in_dtype), S.widen(b, wl.in_dtype), wl.out_dtype)


def test_repeat_is_deterministic(ws):
    wl = S.WORKLOADS["gemm_ragged"]
    a, b = S.gemm_inputs(wl)
    ta, tb = to_cuda(a, wl.in_dtype), to_cuda(b, wl.in_dtype)
    c1 = T.gemm(ta, tb, out_dtype="f32", workspace=ws)
    c2 = T.gemm(ta, tb, out_dtype="f32", workspace=ws)
    T.check(ws)
    assert torch.equal(c1, c2)


def test_bounded_wait_reports_timeout_and_context_survives(ws):
    T.selftest_wait_timeout(ws, 50_000_000)       # 50 ms
    with pytest.raises(T.TilesError) as e:
        T.check(ws)
    assert e.value.status == -6
    # The error word was cleared and the context still runs kernels.
    T.check(ws)
    a = S.integer_matrix(1, (128, 64), S.F16)
    b = S.integer_matrix(2, (64, 64), S.F16)
    c = run_gemm(a, b, S.F16, S.F32, None, ws)
    assert np.array_equal(to_f64(c), OG.gemm(S.widen(a, S.F16), S.widen(b, S.F16)))


def test_rejects_unaligned_pitch(ws):
    a = torch.zeros((64, 60), dtype=torch.float16, device="cuda")
    b = torch.zeros((60, 64), dtype=torch.float16, device="cuda")
    with pytest.raises(T.TilesError) as e:
        T.gemm(a, b, out_dtype="f32", workspace=ws)
    assert e.value.status == -3


def _groups(cg):
    return torch.cuda.get_device_properties(0).multi_processor_count // cg


@pytest.mark.parametrize("v", [(256, 2), (256, 1), (128, 1)], ids=["bn256_cg2", "bn256_cg1",
                                                                   "bn128_cg1"])
@pytest.mark.parametrize("rest", ["one", "half_round", "all_halves"])
@pytest.mark.parametrize("tail", ["auto_small_ws", "nhalf", "ksplit"])
def test_tail_rounds_split(ws, v, rest, tail):
    # Tile counts around the resident group count, so the last round is
    # split: into N-halves, along K (the workspace holds the partial tiles),
    # or as the planner picks with only the 256-byte workspace; one extra
    # tile, half a round extra, or a problem smaller than one round; N and M
    # are ragged.
    bn, cg = v
    g = _groups(cg)
    tiles = {"one": g + 1, "half_round": g + g // 2, "all_halves": 5}[rest]
    m, n, k = 128 * cg * tiles - 37, bn - 40, 1000
    a_np = S.random_matrix(51, (m, k), S.F16, "normal")
    b_np = S.random_matrix(52, (k, n), S.F16, "normal")
    a = to_cuda(a_np, S.F16, -(-k // 8) * 8)
    b = to_cuda(b_np, S.F16, -(-n // 8) * 8)
    c = empty_out((m, n), S.F32, -(-n // 4) * 4)
    bn_, cg_ = v
    cfg = T.make_config(128 * cg_, bn_, 64, VARIANTS[v], 192, "tcgen05", 2, cg_,
                        tail="auto" if tail == "auto_small_ws" else tail)
    w = ws if tail == "auto_small_ws" else T.gemm_workspace(a, b, c, cfg)
    sch = T.gemm_schedule(a, b, c, cfg, w)
    if tail == "ksplit":
        assert sch.tail_mode == 2 and sch.ksplit >= 2
        assert sch.units == sch.full_units + (sch.tiles - sch.full_units) * sch.ksplit
    if tail == "nhalf":
        assert sch.tail_mode == 1 and sch.units == sch.full_units + 2 * (sch.tiles - sch.full_units)
    for _ in range(3):          # reuse of the workspace across launches
        c.fill_(float("nan"))
        T.gemm(a, b, out=c, cfg=cfg, workspace=w)
        T.check(w)
        assert_close(to_f64(c), S.widen(a_np, S.F16), S.widen(b_np, S.F16), S.F32)


@pytest.mark.parametrize("v", [(256, 2), (256, 1), (128, 1)], ids=["bn256_cg2", "bn256_cg1",
                                                                   "bn128_cg1"])
@pytest.mark.parametrize("out_dt", [S.F16, S.BF16])
def test_ksplit_tail_16bit_output(ws, v, out_dt):
    # The last K part adds the partials and casts: a 16-bit C leaves in
    # 64-column boxes, two TMEM chunks each.  N and M are ragged, and the
    # canary band past N inside the row pitch stays untouched.
    bn, cg = v
    g = _groups(cg)
    m, n, k = 128 * cg * (g + 1) - 37, bn - 40, 1000
    in_dt = S.BF16 if out_dt == S.BF16 else S.F16
    a_np = S.random_matrix(53, (m, k), in_dt, "normal")
    b_np = S.random_matrix(54, (k, n), in_dt, "normal")
    a = to_cuda(a_np, in_dt, -(-k // 8) * 8)
    b = to_cuda(b_np, in_dt, -(-n // 8) * 8)
    canary = 1536.0
    big = torch.full((m, n + 16), canary, dtype=TORCH_DT[out_dt], device="cuda")
    c = big[:, :n]
    cfg = T.make_config(128 * cg, bn, 64, VARIANTS[v], 192, "tcgen05", 2, cg, tail="ksplit")
    w = T.gemm_workspace(a, b, c, cfg)
    sch = T.gemm_schedule(a, b, c, cfg, w)
    assert sch.tail_mode == 2 and sch.ksplit >= 2
    T.gemm(a, b, out=c, cfg=cfg, workspace=w)
    T.check(w)
    host = to_f64(big)
    assert np.all(host[:, n:] == canary)
    assert_close(host[:, :n], S.widen(a_np, in_dt), S.widen(b_np, in_dt), out_dt)


def test_ksplit_tail_is_deterministic(ws):
    wl = S.WORKLOADS["gemm_ragged"]
    a, b = S.gemm_inputs(wl)
    ta, tb = to_cuda(a, wl.in_dtype), to_cuda(b, wl.in_dtype)
    c1 = empty_out(wl.c_shape(), wl.out_dtype)
    # The planner's tile with its last round forced to K parts (the planner
    # itself prefers N-halves here).
    f = T.plan(wl.m, wl.n, wl.k, in_dtype=wl.in_dtype, out_dtype=wl.out_dtype,
               device=T.device_query(0))[0][0].cfg
    cfg = T.make_config(f.bm, f.bn, f.bk, f.stages, f.threads, f.instr, f.acc_bufs, f.cta_group,
                        tail="ksplit")
    w = T.gemm_workspace(ta, tb, c1, cfg)
    assert T.gemm_schedule(ta, tb, c1, cfg=cfg, workspace=w).tail_mode == 2
    T.gemm(ta, tb, out=c1, cfg=cfg, workspace=w)
    c2 = T.gemm(ta, tb, out_dtype="f32", cfg=cfg, workspace=w)
    T.check(w)
    assert torch.equal(c1, c2)


def test_schedule_of_the_bench_shape():
    # The 4096^3 fp16 GEMM plans the CTA-pair 256x256 tile; its 256 tiles run
    # in rounds of the co-resident pairs the device reports, and a last round
    # filling at most half of them runs as N-half tiles.
    a = torch.zeros((4096, 4096), dtype=torch.float16, device="cuda")
    c = torch.empty((4096, 4096), dtype=torch.float16, device="cuda")
    sch = T.gemm_schedule(a, a, c)
    dev = T.device_query(0)
    assert (sch.cfg.bm, sch.cfg.bn, sch.cfg.cta_group) == (256, 256, 2)
    assert sch.tiles == 256
    assert sch.resident_groups == dev.cta_pairs > 0
    rem = sch.tiles % sch.resident_groups
    if 0 < rem and 2 * rem <= sch.resident_groups:
        assert sch.full_units == sch.tiles - rem and sch.units == sch.full_units + 2 * rem
    else:
        assert sch.full_units == sch.units == sch.tiles
    assert sch.groups == min(sch.units, sch.resident_groups)


@pytest.mark.parametrize("tail", ["whole", "nhalf", "ksplit"])
def test_forced_tail_schedules(tail):
    # 256x256 pair tiles with one tile more than a round: each forced last-
    # round schedule runs as asked and gives the same result within tolerance.
    g = _groups(2)
    m, n, k = 256 * (g + 3) - 11, 256, 640
    a_np = S.random_matrix(61, (m, k), S.BF16, "normal")
    b_np = S.random_matrix(62, (k, n), S.BF16, "normal")
    a, b = to_cuda(a_np, S.BF16), to_cuda(b_np, S.BF16)
    c = empty_out((m, n), S.BF16)
    cfg = T.make_config(256, 256, 64, 6, 192, "tcgen05", 2, 2, tail=tail)
    w = T.gemm_workspace(a, b, c, cfg)
    sch = T.gemm_schedule(a, b, c, cfg, w)
    assert sch.tail_mode == {"whole": 0, "nhalf": 1, "ksplit": 2}[tail]
    T.gemm(a, b, out=c, cfg=cfg, workspace=w)
    T.check(w)
    assert_close(to_f64(c), S.widen(a_np, S.BF16), S.widen(b_np, S.BF16), S.BF16)


# --------------------------------------------------------------------------- #
# Extreme aspect ratios: long K, tall-skinny, very wide, many tiny items
# --------------------------------------------------------------------------- #

@pytest.mark.parametrize("m,n,k,in_dt,out_dt", [
    (128, 256, 32768, S.BF16, S.F32),     # 512 K blocks per tile
    (40000, 16, 64, S.F16, S.F16),        # 157 M blocks, one narrow N block
    (16, 50000, 128, S.F16, S.F32),       # one M block, 196+ N blocks
    (257, 4097, 72, S.BF16, S.BF16),      # ragged in every dimension
])
def test_extreme_aspect_ratios(ws, m, n, k, in_dt, out_dt):
    a = S.random_matrix(90 + m % 7, (m, k), in_dt, "normal")
    b = S.random_matrix(91 + n % 7, (k, n), in_dt, "normal")
    pa, pb = -(-k // 8) * 8, -(-n // 8) * 8
    pc = -(-n // 8) * 8 if out_dt != S.F32 else -(-n // 4) * 4
    big = T.gemm_workspace(to_cuda(a, in_dt, pa), to_cuda(b, in_dt, pb), empty_out((m, n), out_dt, pc))
    c = run_gemm(a, b, in_dt, out_dt, None, big, pa, pb, pc)
    assert_close(to_f64(c), S.widen(a, in_dt), S.widen(b, in_dt), out_dt)


@pytest.mark.parametrize("v", [(256, 2), (128, 1)], ids=["bn256_cg2", "bn128_cg1"])
def test_grouped_tile_order_covers_every_tile(ws, v):
    # A tall GEMM whose A panels (20 M blocks x K) exceed the scheduler's L2
    # share, so the tiles go in groups of 8 M blocks: two full groups, a last
    # group of 4 blocks ending in a ragged one, and a ragged N.  Every output
    # is written (NaN canary) and rows sampled in every group match the
    # oracle.
    bn, cg = v
    bm = 128 * cg
    m, n = bm * 19 + 37, 2 * bn + 40
    k = 4608 if cg == 2 else 9216
    assert -(-m // bm) * bm * k * 2 > (43 << 20)
    a = S.random_matrix(97, (m, k), S.F16, "normal")
    b = S.random_matrix(98, (k, n), S.F16, "normal")
    c = empty_out((m, n), S.F32)
    T.gemm(to_cuda(a, S.F16), to_cuda(b, S.F16), out=c, cfg=variant(v), workspace=ws)
    T.check(ws)
    got = to_f64(c)
    assert not np.isnan(got).any()
    rows = np.r_[0:8, 8 * bm - 4:8 * bm + 4, 16 * bm - 4:16 * bm + 4, m - 40:m]
    a64, b64 = S.widen(a[rows], S.F16), S.widen(b, S.F16)
    assert_close(got[rows], a64, b64, S.F32)


def test_many_tiny_batch_items(ws):
    batch, m, n, k = 1000, 16, 24, 32
    a = S.random_matrix(95, (batch, m, k), S.F16)
    b = S.random_matrix(96, (batch, k, n), S.F16)
    c = empty_out((batch, m, n), S.F32)
    T.gemm_batched(to_cuda(a, S.F16), to_cuda(b, S.F16), out=c, workspace=ws)
    T.check(ws)
    # Every item against the oracle (a batched float64 matmul).
    assert_close(to_f64(c), S.widen(a, S.F16), S.widen(b, S.F16), S.F32)
