"""Measured shortlist (tutorial, "自动调优"): the planner's top-k
configurations timed on the GPU, the fastest recorded and used by later
calls without a configuration; outputs stay within the oracle's bound."""
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
from tests.gpu_util import to_cuda, to_f64, empty_out  # noqa: E402


@pytest.fixture(autouse=True)
def clean_table():
    T.load()
    T.tuned_clear()
    yield
    T.tuned_clear()


def inputs(m, n, k, dt, seed):
    a = S.random_matrix(seed, (m, k), dt, "normal")
    b = S.random_matrix(seed + 1, (k, n), dt, "normal")
    return a, b


def key(dev, m, n, k, dt, out_dt, batch=1):
    return (dev.sm_count, batch, m, n, k, dt, out_dt)


def test_autotune_picks_a_shortlisted_config_and_later_calls_use_it():
    # 3000 x 2000 x 1536: a partial last round, so the tail schedules differ.
    m, n, k, dt, out_dt = 3000, 2000, 1536, S.BF16, S.F32
    a_np, b_np = inputs(m, n, k, dt, 40)
    a, b = to_cuda(a_np, dt), to_cuda(b_np, dt)
    c = empty_out((m, n), out_dt)
    dev = T.device_query(0)
    ws = T.gemm_workspace(a, b, c)
    top_k = 3
    ranked = T.plan(m, n, k, in_dtype=dt, out_dtype=out_dt, device=dev)[0][:top_k]
    shortlist = {(v.cfg.bm, v.cfg.bn, v.cfg.stages, v.cfg.cta_group) for v in ranked}
    best, rows = T.gemm_autotune(a, b, c, top_k=top_k, reps=3, workspace=ws)
    T.check(ws)
    ran = [r for r in rows if r["status"] == 0]
    assert ran and all(r["us"] > 0 for r in ran)
    assert {(r["bm"], r["bn"], r["stages"], r["cta_group"]) for r in rows} <= shortlist
    assert (best.bm, best.bn, best.stages, best.cta_group) in shortlist
    fastest = min(ran, key=lambda r: r["us"])   # the first of equal times, as the library keeps
    assert (fastest["bm"], fastest["bn"], fastest["tail_asked"]) == (best.bm, best.bn, best.tail)
    # The table now answers for this problem, and a call without cfg uses it.
    tuned = T.tuned_lookup(*key(dev, m, n, k, dt, out_dt))
    assert tuned is not None and (tuned.bm, tuned.bn, tuned.tail) == (best.bm, best.bn, best.tail)
    sch = T.gemm_schedule(a, b, c, workspace=ws)
    assert (sch.cfg.bm, sch.cfg.bn, sch.cfg.stages, sch.cfg.cta_group) == \
        (best.bm, best.bn, best.stages, best.cta_group)
    out = empty_out((m, n), out_dt)
    T.gemm(a, b, out=out, workspace=ws)
    T.check(ws)
    a64, b64 = S.widen(a_np, dt), S.widen(b_np, dt)
    ok, worst, idx = OT.check(to_f64(out), OG.gemm(a64, b64), OG.gemm_bound(a64, b64), out_dt)
    assert ok, f"worst ratio {worst} at {idx}"
    # Clearing the table restores the planner's first choice.
    T.tuned_clear()
    sch2 = T.gemm_schedule(a, b, c, workspace=ws)
    first = ranked[0].cfg
    assert (sch2.cfg.bm, sch2.cfg.bn, sch2.cfg.stages) == (first.bm, first.bn, first.stages)


def test_autotune_batched_and_saved_table_reloads(tmp_path):
    batch, m, n, k, dt = 4, 512, 768, 1024, S.F16
    a_np = S.random_matrix(50, (batch, m, k), dt)
    b_np = S.random_matrix(51, (batch, k, n), dt)
    a, b = to_cuda(a_np, dt), to_cuda(b_np, dt)
    c = empty_out((batch, m, n), dt)
    ws = T.workspace()
    best, rows = T.gemm_autotune(a, b, c, top_k=2, reps=2, workspace=ws)
    T.check(ws)
    dev = T.device_query(0)
    path = tmp_path / "tuned.txt"
    T.tuned_save(str(path))
    T.tuned_clear()
    assert T.tuned_lookup(*key(dev, m, n, k, dt, dt, batch)) is None
    T.tuned_load(str(path))
    again = T.tuned_lookup(*key(dev, m, n, k, dt, dt, batch))
    assert again is not None and (again.bm, again.bn, again.tail) == (best.bm, best.bn, best.tail)
    out = empty_out((batch, m, n), dt)
    T.gemm_batched(a, b, out=out, workspace=ws)
    T.check(ws)
    for i in range(batch):
        a64, b64 = S.widen(a_np[i], dt), S.widen(b_np[i], dt)
        ok, worst, idx = OT.check(to_f64(out[i]), OG.gemm(a64, b64), OG.gemm_bound(a64, b64), dt)
        assert ok, f"item {i}: worst ratio {worst} at {idx}"


def test_tuned_ksplit_without_workspace_room_falls_back():
    # A tuned K-split last round must not make a later call with the small
    # workspace fail: the schedule yields to one that fits.
    m, n, k, dt = 3000, 2000, 1536, S.BF16
    a_np, b_np = inputs(m, n, k, dt, 60)
    a, b = to_cuda(a_np, dt), to_cuda(b_np, dt)
    c = empty_out((m, n), dt)
    # Room for the partial tiles of a K-split last round of the planner's tile.
    f = T.plan(m, n, k, in_dtype=dt, out_dtype=dt, device=T.device_query(0))[0][0].cfg
    ks = T.make_config(f.bm, f.bn, f.bk, f.stages, f.threads, f.instr, f.acc_bufs, f.cta_group,
                       tail="ksplit")
    big = T.gemm_workspace(a, b, c, ks)
    best, rows = T.gemm_autotune(a, b, c, top_k=1, reps=2, workspace=big)
    small = T.workspace()
    out = empty_out((m, n), dt)
    T.gemm(a, b, out=out, workspace=small)
    T.check(small)
    a64, b64 = S.widen(a_np, dt), S.widen(b_np, dt)
    ok, worst, idx = OT.check(to_f64(out), OG.gemm(a64, b64), OG.gemm_bound(a64, b64), dt)
    assert ok, f"worst ratio {worst} at {idx}"


def test_autotune_argument_checks():
    a = torch.zeros((256, 256), dtype=torch.float16, device="cuda")
    b = torch.zeros((256, 256), dtype=torch.float16, device="cuda")
    c = torch.zeros((256, 256), dtype=torch.float16, device="cuda")
    ws = T.workspace()
    for top_k, reps in ((0, 3), (17, 3), (2, 0), (2, 101)):
        with pytest.raises(T.TilesError) as e:
            T.gemm_autotune(a, b, c, top_k=top_k, reps=reps, workspace=ws)
        assert e.value.status == -1
