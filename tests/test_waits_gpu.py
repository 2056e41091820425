"""The production kernels' own bounded waits, made to run out.

A planted fault (tiles_selftest_drop_stage) makes the first CTA group of
the next GEMM or TMA-convolution launch skip the loads and the arrival of one
pipeline stage, with a 50 ms limit on every wait of that launch.  The stage's
consumer then waits on a barrier that never completes; the kernel must record
the expiry, let its other roles stop (for a CTA pair, in both CTAs, through
the pair's closing cluster barrier), wait for its own copies and MMAs, free
its tensor memory and return.  Each test checks TILES_ERR_TIMEOUT from
tiles_check, that the error word is cleared by the read, and that the next
launch in the same context is correct against the float64 oracle.  No GPU
fault is injected: the waits end by their own limit.
"""

import numpy as np
import pytest

import synth_inputs as S
from oracle import conv as OC
from oracle import gemm as OG
from oracle import tolerance as OT

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import tile_size_decision_gb300 as T  # noqa: E402
from tile_size_decision_gb300 import _abi  # noqa: E402
from tests.gpu_util import to_cuda, to_f64, empty_out  # noqa: E402

LIMIT_NS = 50_000_000


@pytest.fixture(scope="module")
def ws():
    T.load()
    return T.workspace()


def expect_timeout(ws):
    with pytest.raises(T.TilesError) as e:
        T.check(ws)
    assert e.value.status == _abi.ERR_TIMEOUT
    T.check(ws)           # the read cleared the word


def gemm_variant(bn, cg):
    stages = {(c.bn, c.cta_group): c.stages for c in T.gemm_variants()}[(bn, cg)]
    return T.make_config(128 * cg, bn, 64, stages, 192, "tcgen05", 2, cg)


@pytest.mark.parametrize("bn,cg", [(128, 1), (256, 1), (128, 2), (256, 2)],
                         ids=["bn128_cg1", "bn256_cg1", "bn128_cg2", "bn256_cg2"])
@pytest.mark.parametrize("stage", [0, 5, 11])
def test_gemm_wait_expires_and_the_context_recovers(ws, bn, cg, stage):
    # 16 K blocks per tile, so every planted stage is one of the first
    # group's (its first unit) whatever the schedule.
    m, n, k = 640 * cg, 3 * bn, 1024
    a_np = S.random_matrix(300 + stage, (m, k), S.F16, "normal")
    b_np = S.random_matrix(301 + stage, (k, n), S.F16, "normal")
    a, b = to_cuda(a_np, S.F16), to_cuda(b_np, S.F16)
    cfg = gemm_variant(bn, cg)
    T.selftest_drop_stage(stage, LIMIT_NS)
    c = empty_out((m, n), S.F32)
    T.gemm(a, b, out=c, cfg=cfg, workspace=ws)
    expect_timeout(ws)
    # The other groups ran: tiles outside the first group's are written.
    got = to_f64(c)
    a64, b64 = S.widen(a_np, S.F16), S.widen(b_np, S.F16)
    ref, bound = OG.gemm(a64, b64), OG.gemm_bound(a64, b64)
    assert np.isfinite(got).sum() >= got.size // 2
    # The same GEMM again, no fault armed: correct, no timeout.
    c2 = empty_out((m, n), S.F32)
    T.gemm(a, b, out=c2, cfg=cfg, workspace=ws)
    T.check(ws)
    ok, worst, idx = OT.check(to_f64(c2), ref, bound, S.F32)
    assert ok, f"worst ratio {worst} at {idx}"


def test_disarmed_fault_plants_nothing(ws):
    T.selftest_drop_stage(0, LIMIT_NS)
    T.selftest_drop_stage(-1, 0)
    a_np = S.random_matrix(310, (256, 64), S.F16)
    b_np = S.random_matrix(311, (64, 256), S.F16)
    c = T.gemm(to_cuda(a_np, S.F16), to_cuda(b_np, S.F16), out_dtype="f32", workspace=ws)
    T.check(ws)
    a64, b64 = S.widen(a_np, S.F16), S.widen(b_np, S.F16)
    ok, _, _ = OT.check(to_f64(c), OG.gemm(a64, b64), OG.gemm_bound(a64, b64), S.F32)
    assert ok
    with pytest.raises(T.TilesError):
        T.selftest_drop_stage(0, 0)


@pytest.mark.parametrize("form,layout", [("rows_direct", "nchw"), ("rows", "nhwc"),
                                         ("tmem", "nhwc")])
@pytest.mark.parametrize("stage", [0, 3])
def test_conv_wait_expires_and_the_context_recovers(form, layout, stage):
    # 320 output rows over at most 152 CTAs: the first CTA runs at least two
    # rows, so every planted stage is one of its loads in every form.
    x_np = S.random_matrix(320 + stage, (8, 64, 80, 24), S.F16)
    w_np = S.random_matrix(321 + stage, (32, 64, 3, 3), S.F16)
    st, pad, dil, tile_oh = (2, 2), (1, 1), (1, 1), 4
    x = to_cuda(x_np, S.F16)
    if layout == "nhwc":
        x = x.permute(0, 2, 3, 1).contiguous()
    w = to_cuda(w_np, S.F16)
    cws = T.conv_workspace(x, w, st, pad, dil, tile_oh, layout=layout)
    cfg = T.make_config(128, 256, 64, 4, 192, "tcgen05", 0, 1, conv_weights=form)
    T.selftest_drop_stage(stage, LIMIT_NS)
    T.conv2d_htiled(x, w, st, pad, dil, tile_oh, out_dtype="f32", cfg=cfg, workspace=cws,
                    layout=layout)
    expect_timeout(cws)
    y = T.conv2d_htiled(x, w, st, pad, dil, tile_oh, out_dtype="f32", cfg=cfg, workspace=cws,
                        layout=layout)
    T.check(cws)
    x64, w64 = S.widen(x_np, S.F16), S.widen(w_np, S.F16)
    ref = OC.conv2d(x64, w64, st, (1, 1), (1, 1))
    bound = OC.conv2d(np.abs(x64), np.abs(w64), st, (1, 1), (1, 1))
    ok, worst, idx = OT.check(to_f64(y), ref, bound, S.F32)
    assert ok, f"worst ratio {worst} at {idx}"


def test_missing_workspace_is_rejected(ws):
    # Without a workspace an expired wait would go unreported, so the
    # kernel calls refuse to launch.
    a = to_cuda(S.random_matrix(330, (128, 64), S.F16), S.F16)
    b = to_cuda(S.random_matrix(331, (64, 128), S.F16), S.F16)
    with pytest.raises(T.TilesError) as e:
        T.gemm(a, b, out_dtype="f32")
    assert e.value.status == _abi.ERR_INVALID_ARG
    x = to_cuda(S.random_matrix(332, (1, 8, 9, 9), S.F16), S.F16)
    w = to_cuda(S.random_matrix(333, (4, 8, 3, 3), S.F16), S.F16)
    with pytest.raises(T.TilesError) as e:
        T.conv2d_htiled(x, w, (1, 1), (1, 1), (1, 1), 4, out_dtype="f32")
    assert e.value.status == _abi.ERR_INVALID_ARG
