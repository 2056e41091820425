"""GPU parity of the H-tiled implicit-GEMM convolution against the oracle.

The kernel consumes the H-tile rows (in_start, pt', real rows) that the
library's htile_rows computes on the host, i.e. the tiling tutorial's
"H/W 维切分的通用公式".  Cases: brute force on tiny shapes, integer inputs
(exact in fp32), tile heights from 1 row to more than OH (results must be
bit-identical: the K order per output never changes), more than one launch
of H-tiles, c_out above and below one 128-row block, canary guards around
the output, and the full convolution workload.
"""

import numpy as np
import pytest

import synth_inputs as S
from oracle import conv as OC
from oracle import tolerance as OT

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import tile_size_decision_gb300 as T  # noqa: E402
from tests.gpu_util import to_cuda, to_f64, TORCH_DT  # noqa: E402


@pytest.fixture(scope="module")
def ws():
    T.load()
    return T.workspace()


def tmem_fits(c, co, kh, kw):
    # The weights-in-tensor-memory form: one 128-channel output block and
    # kh*kw*ceil(c/64) K blocks of 32 columns next to two 16-column
    # accumulators in 512 columns.
    return co <= 128 and kh * kw * ((c + 63) // 64) * 32 + 32 <= 512


def run_conv(x_np, w_np, in_dt, out_dt, stride, pad, dil, tile_oh, ws, guard=0, producer="gather",
             layout="nchw"):
    # producer "gather": the small workspace (threads gather the operand);
    # "tma": a workspace sized for the TMA producer, weights where they fit
    # best; "tma_smem" / "tma_tmem" force the weights into shared or tensor
    # memory, "tma_tmem1" / "tma_tmem2" also fix one or two accumulators.
    x = to_cuda(x_np, in_dt)
    if layout == "nhwc":
        x = x.permute(0, 2, 3, 1).contiguous()
    w = to_cuda(w_np, in_dt)
    n, c, h, wd = x_np.shape
    co, _, kh, kw = w_np.shape
    oh = OC.out_size(h, kh, stride[0], pad[0], pad[0], dil[0])
    ow = OC.out_size(wd, kw, stride[1], pad[1], pad[1], dil[1])
    total = n * co * oh * ow
    flat = torch.full((total + 2 * guard,), 2048.0, dtype=TORCH_DT[out_dt], device="cuda")
    y = flat[guard:guard + total].view(n, co, oh, ow)
    if producer.startswith("tma"):
        ws = T.conv_workspace(x, w, stride, pad, dil, tile_oh, layout=layout)
        place = producer[4:] or "auto"
        acc = int(place[4:]) if place.startswith(("tmem", "rows")) and len(place) > 4 else 0
        cfg = T.make_config(128, 256, 64, 4, 192, "tcgen05", acc, 1,
                            conv_weights=place[:4] if place != "auto" else "auto")
    else:
        cfg = None
    T.conv2d_htiled(x, w, stride, pad, dil, tile_oh, out=y, workspace=ws, cfg=cfg, layout=layout)
    T.check(ws)
    host = to_f64(flat)
    if guard:
        assert np.all(host[:guard] == 2048.0) and np.all(host[guard + total:] == 2048.0)
    return host[guard:guard + total].reshape(n, co, oh, ow)


def check_against_oracle(got, x64, w64, stride, pad, dil, out_dt):
    ref = OC.conv2d(x64, w64, stride, (pad[0], pad[0]), (pad[1], pad[1]), dil)
    bound = OC.conv2d(np.abs(x64), np.abs(w64), stride, (pad[0], pad[0]), (pad[1], pad[1]), dil)
    ok, worst, idx = OT.check(got, ref, bound, out_dt)
    assert ok, f"worst ratio {worst} at {idx}: got {got[idx]} want {ref[idx]}"


TINY = [
    # (n, c, h, w, co, kh, kw, stride, pad, dil, tile_oh)
    (1, 8, 9, 9, 4, 3, 3, (2, 2), (1, 1), (1, 1), 2),     # the tutorial's H=9 example rows
    (2, 8, 7, 10, 16, 3, 3, (1, 1), (1, 1), (1, 1), 3),
    (1, 16, 12, 12, 8, 1, 1, (1, 1), (0, 0), (1, 1), 5),
    (1, 8, 11, 13, 5, 5, 3, (2, 1), (2, 1), (1, 2), 1),
    (3, 24, 16, 16, 130, 3, 3, (2, 2), (1, 1), (2, 2), 4),
    (1, 8, 20, 6, 8, 2, 2, (3, 3), (0, 1), (1, 1), 7),
]


@pytest.mark.parametrize("case", TINY, ids=lambda c: "_".join(str(v) for v in c[:7]))
def test_tiny_against_loops(ws, case):
    n, c, h, wd, co, kh, kw, st, pad, dil, tile = case
    x = S.random_matrix(1, (n, c, h, wd), S.F16)
    w = S.random_matrix(2, (co, c, kh, kw), S.F16)
    got = run_conv(x, w, S.F16, S.F32, st, pad, dil, tile, ws, guard=64)
    x64, w64 = S.widen(x, S.F16), S.widen(w, S.F16)
    ref = OC.conv2d_loops(x64, w64, st, pad, dil) if n * co * c * h * wd < 200000 else None
    if ref is not None:
        bound = OC.conv2d_loops(np.abs(x64), np.abs(w64), st, pad, dil)
        ok, worst, idx = OT.check(got, ref, bound, S.F32)
        assert ok, f"worst ratio {worst} at {idx}"
    check_against_oracle(got, x64, w64, st, pad, dil, S.F32)


@pytest.mark.parametrize("dt", [S.F16, S.BF16])
def test_integer_inputs_exact(ws, dt):
    x = S.integer_matrix(3, (2, 16, 30, 28), dt)
    w = S.integer_matrix(4, (40, 16, 3, 3), dt)
    got = run_conv(x, w, dt, S.F32, (2, 2), (1, 1), (1, 1), 4, ws)
    ref = OC.conv2d(S.widen(x, dt), S.widen(w, dt), (2, 2), (1, 1), (1, 1))
    assert np.array_equal(got, ref)


def test_tile_height_does_not_change_bits(ws):
    x = S.random_matrix(5, (2, 16, 37, 33), S.BF16, "normal")
    w = S.random_matrix(6, (64, 16, 3, 3), S.BF16, "normal")
    outs = [run_conv(x, w, S.BF16, S.F32, (2, 1), (1, 1), (1, 1), t, ws) for t in (1, 2, 3, 7, 19, 40)]
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])
    check_against_oracle(outs[0], S.widen(x, S.BF16), S.widen(w, S.BF16), (2, 1), (1, 1), (1, 1),
                         S.F32)


def test_more_h_tiles_than_one_launch(ws):
    # 300 output rows at tile height 1: three launches of at most 128 H-tiles.
    x = S.random_matrix(7, (1, 8, 300, 20), S.F16)
    w = S.random_matrix(8, (12, 8, 3, 3), S.F16)
    got = run_conv(x, w, S.F16, S.F16, (1, 1), (1, 1), (1, 1), 1, ws, guard=32)
    check_against_oracle(got, S.widen(x, S.F16), S.widen(w, S.F16), (1, 1), (1, 1), (1, 1), S.F16)


def test_many_output_channels_bf16_out(ws):
    x = S.random_matrix(9, (2, 32, 20, 20), S.BF16, "normal")
    w = S.random_matrix(10, (300, 32, 3, 3), S.BF16, "normal")
    got = run_conv(x, w, S.BF16, S.BF16, (1, 1), (1, 1), (1, 1), 6, ws, guard=16)
    check_against_oracle(got, S.widen(x, S.BF16), S.widen(w, S.BF16), (1, 1), (1, 1), (1, 1),
                         S.BF16)


def test_conv_workload_full(ws):
    wl = S.WORKLOADS["conv_htiled"]
    x, w = S.conv_inputs(wl)
    got = run_conv(x, w, wl.in_dtype, wl.out_dtype, (wl.sh, wl.sw), (wl.ph, wl.pw),
                   (wl.dh, wl.dw), wl.tile_oh, ws)
    assert got.shape == (wl.n, wl.c_out, wl.oh, wl.ow)
    check_against_oracle(got, S.widen(x, wl.in_dtype), S.widen(w, wl.in_dtype), (wl.sh, wl.sw),
                         (wl.ph, wl.pw), (wl.dh, wl.dw), wl.out_dtype)


def test_rejects_unaligned_weights(ws):
    x = torch.zeros((1, 3, 8, 8), dtype=torch.float16, device="cuda")
    w = torch.zeros((4, 3, 3, 3), dtype=torch.float16, device="cuda")   # K = 27
    with pytest.raises(T.TilesError) as e:
        T.conv2d_htiled(x, w, (1, 1), (1, 1), (1, 1), 4, workspace=ws)
    assert e.value.status == -3


# --------------------------------------------------------------------------- #
# The TMA im2col producer
# --------------------------------------------------------------------------- #

PLACES = ["smem", "tmem1", "tmem2", "rows"]


@pytest.mark.parametrize("case", TINY, ids=lambda c: "_".join(str(v) for v in c[:7]))
@pytest.mark.parametrize("layout", ["nchw", "nhwc"])
@pytest.mark.parametrize("place", PLACES)
def test_tma_tiny_against_loops(ws, case, layout, place):
    n, c, h, wd, co, kh, kw, st, pad, dil, tile = case
    if place.startswith(("tmem", "rows")) and not tmem_fits(c, co, kh, kw):
        pytest.skip("filter does not fit tensor memory")
    x = S.random_matrix(1, (n, c, h, wd), S.F16)
    w = S.random_matrix(2, (co, c, kh, kw), S.F16)
    got = run_conv(x, w, S.F16, S.F32, st, pad, dil, tile, ws, guard=64, producer="tma_" + place,
                   layout=layout)
    x64, w64 = S.widen(x, S.F16), S.widen(w, S.F16)
    if n * co * c * h * wd < 200000:
        ref = OC.conv2d_loops(x64, w64, st, pad, dil)
        bound = OC.conv2d_loops(np.abs(x64), np.abs(w64), st, pad, dil)
        ok, worst, idx = OT.check(got, ref, bound, S.F32)
        assert ok, f"worst ratio {worst} at {idx}"
    check_against_oracle(got, x64, w64, st, pad, dil, S.F32)


@pytest.mark.parametrize("dt", [S.F16, S.BF16])
@pytest.mark.parametrize("place", PLACES)
def test_tma_integer_inputs_exact(ws, dt, place):
    # 72 channels are 18 K blocks, more than tensor memory holds next to
    # the accumulators; the TMEM form takes 48 (one zero-padded block).
    c = 72 if place == "smem" else 48   # the tensor-memory forms hold 48 channels' filter
    x = S.integer_matrix(3, (2, c, 30, 28), dt)
    w = S.integer_matrix(4, (40, c, 3, 3), dt)
    got = run_conv(x, w, dt, S.F32, (2, 2), (1, 1), (1, 1), 4, ws, producer="tma_" + place)
    ref = OC.conv2d(S.widen(x, dt), S.widen(w, dt), (2, 2), (1, 1), (1, 1))
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("place", PLACES)
def test_tma_tile_height_does_not_change_bits(ws, place):
    x = S.random_matrix(5, (2, 16, 37, 34), S.BF16, "normal")
    w = S.random_matrix(6, (64, 16, 3, 3), S.BF16, "normal")
    outs = [run_conv(x, w, S.BF16, S.F32, (2, 1), (1, 1), (1, 1), t, ws, producer="tma_" + place)
            for t in (1, 2, 3, 7, 19, 40)]
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])
    check_against_oracle(outs[0], S.widen(x, S.BF16), S.widen(w, S.BF16), (2, 1), (1, 1), (1, 1),
                         S.F32)


@pytest.mark.parametrize("place", PLACES)
def test_tma_wide_rows_and_many_h_tiles(ws, place):
    # W wider than one TMA box (several column blocks) and 300 output rows at
    # tile height 1 (three launches of H-tiles).
    x = S.random_matrix(7, (1, 8, 300, 600), S.F16)
    w = S.random_matrix(8, (12, 8, 3, 3), S.F16)
    got = run_conv(x, w, S.F16, S.F16, (1, 2), (1, 1), (1, 1), 1, ws, guard=32,
                   producer="tma_" + place)
    check_against_oracle(got, S.widen(x, S.F16), S.widen(w, S.F16), (1, 2), (1, 1), (1, 1), S.F16)


def test_tma_channels_not_multiple_of_64(ws):
    x = S.random_matrix(9, (2, 40, 20, 22), S.BF16, "normal")
    w = S.random_matrix(10, (300, 40, 3, 3), S.BF16, "normal")
    got = run_conv(x, w, S.BF16, S.BF16, (1, 1), (1, 1), (1, 1), 6, ws, guard=16, producer="tma")
    check_against_oracle(got, S.widen(x, S.BF16), S.widen(w, S.BF16), (1, 1), (1, 1), (1, 1),
                         S.BF16)


@pytest.mark.parametrize("layout", ["nchw", "nhwc"])
@pytest.mark.parametrize("place", PLACES)
def test_tma_conv_workload_full(ws, layout, place):
    wl = S.WORKLOADS["conv_htiled"]
    x, w = S.conv_inputs(wl)
    got = run_conv(x, w, wl.in_dtype, wl.out_dtype, (wl.sh, wl.sw), (wl.ph, wl.pw),
                   (wl.dh, wl.dw), wl.tile_oh, ws, producer="tma_" + place, layout=layout)
    check_against_oracle(got, S.widen(x, wl.in_dtype), S.widen(w, wl.in_dtype), (wl.sh, wl.sw),
                         (wl.ph, wl.pw), (wl.dh, wl.dw), wl.out_dtype)


def test_default_producer_with_workspace_is_tma(ws):
    # cfg=None with a workspace of conv_workspace size takes the TMA producer,
    # whose K order (r, s, ci) differs from the gather's (ci, r, s): both
    # stay within tolerance of the oracle.
    wl = S.WORKLOADS["conv_htiled"]
    x_np, w_np = S.conv_inputs(wl)
    x, w = to_cuda(x_np, wl.in_dtype), to_cuda(w_np, wl.in_dtype)
    big = T.conv_workspace(x, w, (2, 2), (1, 1), (1, 1), 16)
    assert big.numel() > 8 * 64 * 224 * 224 * 2
    y1 = T.conv2d_htiled(x, w, (2, 2), (1, 1), (1, 1), 16, workspace=big)
    y2 = T.conv2d_htiled(x, w, (2, 2), (1, 1), (1, 1), 16, workspace=big,
                         cfg=T.make_config(128, 256, 64, 4, 192, "tcgen05", 2, 1))
    T.check(big)
    assert torch.equal(y1, y2)


@pytest.mark.parametrize("out_dt", [S.F16, S.BF16, S.F32])
@pytest.mark.parametrize("place", ["tmem", "tmem1", "tmem2", "rows", "rows1", "rows2"])
def test_tmem_weights_ragged_channels_and_columns(ws, out_dt, place):
    # c_out below 128 (zero rows of the tensor-memory filter), a channel
    # count that is not a multiple of 64, odd output widths (scalar tails)
    # and stride 1 and 3.
    for seed, (n, c, h, wd, co, st) in enumerate([(2, 24, 19, 27, 72, 1), (1, 56, 23, 41, 100, 3)]):
        x = S.random_matrix(20 + seed, (n, c, h, wd), S.BF16, "normal")
        w = S.random_matrix(30 + seed, (co, c, 3, 3), S.BF16, "normal")
        got = run_conv(x, w, S.BF16, out_dt, (st, st), (1, 1), (1, 1), 5, ws, guard=16,
                       producer="tma_" + place)
        check_against_oracle(got, S.widen(x, S.BF16), S.widen(w, S.BF16), (st, st), (1, 1),
                             (1, 1), out_dt)


def test_tmem_weights_refused_when_they_do_not_fit(ws):
    x = torch.zeros((1, 64, 8, 8), dtype=torch.float16, device="cuda")
    w = torch.zeros((200, 64, 3, 3), dtype=torch.float16, device="cuda")   # c_out > 128
    big = T.conv_workspace(x, w, (1, 1), (1, 1), (1, 1), 4)
    with pytest.raises(T.TilesError) as e:
        T.conv2d_htiled(x, w, (1, 1), (1, 1), (1, 1), 4, workspace=big,
                        cfg=T.make_config(128, 256, 64, 4, 192, "tcgen05", 2, 1, conv_weights="tmem"))
    assert e.value.status == -4


def test_nhwc_without_workspace_is_refused(ws):
    x = torch.zeros((1, 8, 8, 16), dtype=torch.float16, device="cuda")
    w = torch.zeros((4, 16, 3, 3), dtype=torch.float16, device="cuda")
    with pytest.raises(T.TilesError) as e:
        T.conv2d_htiled(x, w, (1, 1), (1, 1), (1, 1), 4, workspace=ws, layout="nhwc")
    assert e.value.status == -4


# --------------------------------------------------------------------------- #
# Tiling over the batch and the width (tiles_conv2d_tiled)
# --------------------------------------------------------------------------- #

def run_tiled(x_np, w_np, in_dt, out_dt, stride, pad, dil, tile_oh, tile_ow, tile_n, place,
              layout="nchw", guard=16):
    x = to_cuda(x_np, in_dt)
    if layout == "nhwc":
        x = x.permute(0, 2, 3, 1).contiguous()
    w = to_cuda(w_np, in_dt)
    n, c, h, wd = x_np.shape
    co, _, kh, kw = w_np.shape
    oh = OC.out_size(h, kh, stride[0], pad[0], pad[0], dil[0])
    ow = OC.out_size(wd, kw, stride[1], pad[1], pad[1], dil[1])
    total = n * co * oh * ow
    flat = torch.full((total + 2 * guard,), 2048.0, dtype=TORCH_DT[out_dt], device="cuda")
    y = flat[guard:guard + total].view(n, co, oh, ow)
    if place == "gather":
        ws, cfg = T.workspace(), None
    else:
        ws = T.conv_workspace(x, w, stride, pad, dil, tile_oh, layout=layout)
        acc = int(place[4:]) if place.startswith(("tmem", "rows")) and len(place) > 4 else 0
        cfg = T.make_config(128, 256, 64, 4, 192, "tcgen05", acc, 1, conv_weights=place[:4])
    T.conv2d_tiled(x, w, stride, pad, dil, tile_oh, tile_ow, tile_n, out=y, workspace=ws, cfg=cfg,
                   layout=layout)
    T.check(ws)
    host = to_f64(flat)
    assert np.all(host[:guard] == 2048.0) and np.all(host[guard + total:] == 2048.0)
    return host[guard:guard + total].reshape(n, co, oh, ow)


@pytest.mark.parametrize("place", ["smem", "tmem1", "tmem2"])
@pytest.mark.parametrize("layout", ["nchw", "nhwc"])
def test_w_and_batch_tiles_do_not_change_bits(place, layout):
    # The width's slices follow the rows' formulas; batch tiles need no halo.
    # For one producer every tiling gives the same bits, and the oracle's
    # tiled convolution (exactly the untiled one) bounds them.
    x = S.random_matrix(70, (3, 16, 21, 45), S.BF16, "normal")
    w = S.random_matrix(71, (40, 16, 3, 3), S.BF16, "normal")
    st, pad, dil = (2, 1), (1, 1), (1, 1)
    base = run_tiled(x, w, S.BF16, S.F32, st, pad, dil, 4, 0, 0, place, layout)
    for tile_ow, tile_n in ((1, 0), (5, 2), (8, 1), (17, 3), (40, 0), (45, 2)):
        got = run_tiled(x, w, S.BF16, S.F32, st, pad, dil, 4, tile_ow, tile_n, place, layout)
        assert np.array_equal(got, base), (tile_ow, tile_n)
    x64, w64 = S.widen(x, S.BF16), S.widen(w, S.BF16)
    ref = OC.conv2d_tiled(x64, w64, st, pad, dil, tile_oh=4, tile_ow=5, tile_n=2)
    bound = OC.conv2d(np.abs(x64), np.abs(w64), st, (pad[0], pad[0]), (pad[1], pad[1]), dil)
    ok, worst, idx = OT.check(base, ref, bound, S.F32)
    assert ok, f"worst ratio {worst} at {idx}"


def test_many_w_tiles_take_several_launches():
    # 150 output columns at tile_ow 1: three launches of at most 64 W-tiles,
    # 16-bit output with scalar stores at every tile edge.
    x = S.random_matrix(72, (1, 8, 6, 150), S.F16)
    w = S.random_matrix(73, (12, 8, 3, 3), S.F16)
    got = run_tiled(x, w, S.F16, S.F16, (1, 1), (1, 1), (1, 1), 2, 1, 0, "tmem")
    check_against_oracle(got, S.widen(x, S.F16), S.widen(w, S.F16), (1, 1), (1, 1), (1, 1), S.F16)


def test_gather_batch_tiles_and_w_tiles_refused():
    x = S.random_matrix(74, (5, 8, 12, 12), S.F16)
    w = S.random_matrix(75, (16, 8, 3, 3), S.F16)
    got = run_tiled(x, w, S.F16, S.F32, (1, 1), (1, 1), (1, 1), 3, 0, 2, "gather")
    check_against_oracle(got, S.widen(x, S.F16), S.widen(w, S.F16), (1, 1), (1, 1), (1, 1), S.F32)
    xt, wt_ = to_cuda(x, S.F16), to_cuda(w, S.F16)
    with pytest.raises(T.TilesError) as e:
        T.conv2d_tiled(xt, wt_, (1, 1), (1, 1), (1, 1), 3, 4, 0, workspace=T.workspace())
    assert e.value.status == -4


def test_conv_workload_tiled_over_w_and_batch():
    wl = S.WORKLOADS["conv_htiled"]
    x, w = S.conv_inputs(wl)
    got = run_tiled(x, w, wl.in_dtype, wl.out_dtype, (wl.sh, wl.sw), (wl.ph, wl.pw),
                    (wl.dh, wl.dw), wl.tile_oh, 56, 2, "tmem")
    check_against_oracle(got, S.widen(x, wl.in_dtype), S.widen(w, wl.in_dtype), (wl.sh, wl.sw),
                         (wl.ph, wl.pw), (wl.dh, wl.dw), wl.out_dtype)


@pytest.mark.parametrize("st,dil,kw", [((1, 1), (1, 1), 3), ((2, 2), (1, 1), 3), ((1, 3), (1, 2), 5),
                                       ((2, 2), (1, 3), 3), ((1, 1), (1, 1), 5), ((3, 2), (1, 1), 4)])
def test_rows_form_strides_and_dilations(st, dil, kw):
    # Tap s reads stride phase (s*dw) % sw from pixel (s*dw) // sw on: one,
    # two or more phase planes per input row, shifted descriptors for the rest.
    x = S.random_matrix(80, (2, 16, 15, 61), S.BF16, "normal")
    w = S.random_matrix(81, (24, 16, 3, kw), S.BF16, "normal")
    pad = (1, kw // 2)
    got = run_tiled(x, w, S.BF16, S.F32, st, pad, dil, 4, 0, 0, "rows")
    smem = run_tiled(x, w, S.BF16, S.F32, st, pad, dil, 4, 0, 0, "smem")
    assert np.array_equal(got, smem)
    check_against_oracle(got, S.widen(x, S.BF16), S.widen(w, S.BF16), st, pad, dil, S.F32)


@pytest.mark.parametrize("place", ["smem", "tmem", "rows", "gather"])
def test_single_output_channel_and_1x1(place):
    # c_out = 1 (127 zero rows in the tensor-memory filter) with a 3x3 window,
    # and a 1x1 stride-2 convolution (one tap, one phase plane).
    x = S.random_matrix(100, (2, 24, 17, 19), S.F16)
    w = S.random_matrix(101, (1, 24, 3, 3), S.F16)
    got = run_tiled(x, w, S.F16, S.F32, (1, 1), (1, 1), (1, 1), 5, 0, 0, place)
    check_against_oracle(got, S.widen(x, S.F16), S.widen(w, S.F16), (1, 1), (1, 1), (1, 1), S.F32)
    w1 = S.random_matrix(102, (32, 24, 1, 1), S.F16)
    got = run_tiled(x, w1, S.F16, S.F16, (2, 2), (0, 0), (1, 1), 3, 0, 0, place)
    check_against_oracle(got, S.widen(x, S.F16), S.widen(w1, S.F16), (2, 2), (0, 0), (1, 1), S.F16)


# --------------------------------------------------------------------------- #
# The rows form over an NCHW input read in place (transposer warps)
# --------------------------------------------------------------------------- #

def run_place(x_np, w_np, in_dt, out_dt, stride, pad, dil, tile_oh, conv_weights, acc=0,
              tile_ow=0, tile_n=0, layout="nchw", guard=16):
    """One TMA convolution with the filter placement forced; tile_ow and
    tile_n 0 take whole rows and the whole batch."""
    x = to_cuda(x_np, in_dt)
    if layout == "nhwc":
        x = x.permute(0, 2, 3, 1).contiguous()
    w = to_cuda(w_np, in_dt)
    n, c, h, wd = x_np.shape
    co, _, kh, kw = w_np.shape
    oh = OC.out_size(h, kh, stride[0], pad[0], pad[0], dil[0])
    ow = OC.out_size(wd, kw, stride[1], pad[1], pad[1], dil[1])
    total = n * co * oh * ow
    flat = torch.full((total + 2 * guard,), 2048.0, dtype=TORCH_DT[out_dt], device="cuda")
    y = flat[guard:guard + total].view(n, co, oh, ow)
    ws = T.conv_workspace(x, w, stride, pad, dil, tile_oh, layout=layout)
    cfg = T.make_config(128, 256, 64, 4, 192, "tcgen05", acc, 1, conv_weights=conv_weights)
    T.conv2d_tiled(x, w, stride, pad, dil, tile_oh, tile_ow, tile_n, out=y, workspace=ws, cfg=cfg,
                   layout=layout)
    T.check(ws)
    host = to_f64(flat)
    assert np.all(host[:guard] == 2048.0) and np.all(host[guard + total:] == 2048.0)
    return host[guard:guard + total].reshape(n, co, oh, ow)


# (n, c, h, w, c_out, kh, kw, stride, pad, dil, tile_oh): W a multiple of 8.
DIRECT_CASES = [
    (1, 8, 9, 16, 4, 3, 3, (2, 2), (1, 1), (1, 1), 2),       # the tutorial's H=9 rows, one channel group
    (2, 16, 12, 24, 24, 3, 3, (1, 1), (1, 1), (1, 1), 5),
    (1, 24, 15, 40, 72, 3, 3, (2, 2), (1, 1), (1, 1), 3),     # 24 channels: 3 of 8 groups live
    (2, 64, 14, 32, 128, 3, 3, (2, 2), (1, 1), (1, 1), 7),
    (1, 56, 11, 48, 100, 3, 3, (3, 3), (1, 1), (1, 1), 4),    # three phases, one shift
    (1, 32, 13, 56, 40, 3, 5, (1, 2), (1, 2), (1, 1), 6),
    (2, 16, 17, 64, 24, 3, 3, (2, 2), (2, 3), (1, 3), 5),     # dilation 3 at stride 2
    (1, 16, 10, 40, 16, 3, 2, (1, 3), (1, 0), (2, 1), 3),     # taps 0, 1 at stride 3: phase 2 unread
    (1, 72, 9, 32, 48, 1, 3, (1, 1), (0, 1), (1, 1), 4),      # two channel blocks
    (1, 8, 7, 8, 8, 3, 3, (1, 1), (2, 2), (1, 1), 9),         # more padding than one group
    (1, 16, 6, 16, 32, 1, 1, (2, 2), (0, 0), (1, 1), 2),      # 1x1 at stride 2: one phase plane
]


@pytest.mark.parametrize("case", DIRECT_CASES, ids=lambda c: "_".join(str(v) for v in c[:8]))
@pytest.mark.parametrize("out_dt", [S.F32, S.BF16])
def test_direct_rows_match_rows_form_bits(case, out_dt):
    # The transposer warps build the same planes the TMA loads from the NHWC
    # copy, and the MMAs run in the same order: identical bits.
    n, c, h, wd, co, kh, kw, st, pad, dil, tile = case
    x = S.random_matrix(110, (n, c, h, wd), S.BF16, "normal")
    w = S.random_matrix(111, (co, c, kh, kw), S.BF16, "normal")
    got = run_place(x, w, S.BF16, out_dt, st, pad, dil, tile, "rows_direct")
    rows = run_place(x, w, S.BF16, out_dt, st, pad, dil, tile, "rows")
    assert np.array_equal(got, rows)
    x64, w64 = S.widen(x, S.BF16), S.widen(w, S.BF16)
    if n * co * c * h * wd < 400000:
        ref = OC.conv2d_loops(x64, w64, st, pad, dil)
        bound = OC.conv2d_loops(np.abs(x64), np.abs(w64), st, pad, dil)
        ok, worst, idx = OT.check(got, ref, bound, out_dt)
        assert ok, f"worst ratio {worst} at {idx}"
    check_against_oracle(got, x64, w64, st, pad, dil, out_dt)


@pytest.mark.parametrize("acc", [1, 2])
def test_direct_rows_integer_inputs_exact(acc):
    x = S.integer_matrix(112, (2, 48, 30, 32), S.F16)
    w = S.integer_matrix(113, (40, 48, 3, 3), S.F16)
    got = run_place(x, w, S.F16, S.F32, (2, 2), (1, 1), (1, 1), 4, "rows_direct", acc=acc)
    ref = OC.conv2d(S.widen(x, S.F16), S.widen(w, S.F16), (2, 2), (1, 1), (1, 1))
    assert np.array_equal(got, ref)


def test_direct_rows_w_and_batch_tiles_do_not_change_bits():
    # Each W-tile's span starts at its own column (col0 mod 8 varies); batch
    # tiles start at their own image.
    x = S.random_matrix(114, (3, 16, 21, 48), S.BF16, "normal")
    w = S.random_matrix(115, (40, 16, 3, 3), S.BF16, "normal")
    st, pad, dil = (2, 1), (1, 1), (1, 1)
    base = run_place(x, w, S.BF16, S.F32, st, pad, dil, 4, "rows_direct")
    for tile_ow, tile_n in ((1, 0), (5, 2), (8, 1), (17, 3), (40, 0)):
        got = run_place(x, w, S.BF16, S.F32, st, pad, dil, 4, "rows_direct", tile_ow=tile_ow,
                        tile_n=tile_n)
        assert np.array_equal(got, base), (tile_ow, tile_n)
    check_against_oracle(base, S.widen(x, S.BF16), S.widen(w, S.BF16), st, pad, dil, S.F32)


@pytest.mark.parametrize("st", [(1, 1), (1, 2)])
def test_direct_rows_wide_spans(st):
    # Widths past one span (several column blocks per row); at stride 1 a
    # stage spans up to 249 columns, the transposers' 32 groups of 8.
    x = S.random_matrix(116, (1, 8, 5, 1000), S.F16)
    w = S.random_matrix(117, (12, 8, 3, 3), S.F16)
    got = run_place(x, w, S.F16, S.F16, st, (1, 1), (1, 1), 2, "rows_direct", guard=32)
    rows = run_place(x, w, S.F16, S.F16, st, (1, 1), (1, 1), 2, "rows", guard=32)
    assert np.array_equal(got, rows)
    check_against_oracle(got, S.widen(x, S.F16), S.widen(w, S.F16), st, (1, 1), (1, 1), S.F16)


def test_direct_rows_workload_and_auto():
    # The convolution workload: the direct form is what AUTO takes for it.
    wl = S.WORKLOADS["conv_htiled"]
    x_np, w_np = S.conv_inputs(wl)
    args = ((wl.sh, wl.sw), (wl.ph, wl.pw), (wl.dh, wl.dw), wl.tile_oh)
    got = run_place(x_np, w_np, wl.in_dtype, wl.out_dtype, *args, "rows_direct")
    auto = run_place(x_np, w_np, wl.in_dtype, wl.out_dtype, *args, "auto")
    assert np.array_equal(got, auto)
    check_against_oracle(got, S.widen(x_np, wl.in_dtype), S.widen(w_np, wl.in_dtype), *args[:3],
                         wl.out_dtype)


def test_direct_rows_refused_where_it_does_not_apply():
    w = torch.zeros((16, 16, 3, 3), dtype=torch.float16, device="cuda")
    cfg = T.make_config(128, 256, 64, 4, 192, "tcgen05", 0, 1, conv_weights="rows_direct")
    for shape, layout in (((1, 16, 8, 20), "nchw"),       # W not a multiple of 8
                          ((1, 8, 16, 16), "nhwc")):      # not an NCHW input
        x = torch.zeros(shape, dtype=torch.float16, device="cuda")
        ws = T.conv_workspace(x, w, (1, 1), (1, 1), (1, 1), 4, layout=layout)
        with pytest.raises(T.TilesError) as e:
            T.conv2d_htiled(x, w, (1, 1), (1, 1), (1, 1), 4, workspace=ws, cfg=cfg, layout=layout)
        assert e.value.status == -4


@pytest.mark.parametrize("case", [
    # (n, c, h, w, co, stride, dtype, layout): 3x3 filters over 64 input
    # channels (9 K blocks, which fit tensor memory), taken there straight
    # from their OIHW rows; c_out below 128 leaves TMEM rows zero-filled.
    (2, 64, 20, 24, 96, (1, 1), S.BF16, "nchw"),
    (1, 64, 17, 16, 128, (2, 2), S.F16, "nchw"),
    (2, 64, 12, 16, 40, (1, 1), S.F16, "nhwc"),
    (1, 64, 9, 8, 128, (2, 2), S.BF16, "nhwc"),
])
def test_raw_oihw_filter_in_tensor_memory(case):
    n, c, h, wd, co, st, dt, layout = case
    x_np = S.random_matrix(91, (n, c, h, wd), dt)
    w_np = S.random_matrix(92, (co, c, 3, 3), dt)
    x = to_cuda(x_np, dt)
    if layout == "nhwc":
        x = x.permute(0, 2, 3, 1).contiguous()
    w = to_cuda(w_np, dt)
    oh, ow = T.conv_out_hw(h, wd, 3, 3, st, (1, 1), (1, 1))
    y = torch.full((n, co, oh, ow), float("nan"), dtype=torch.float32, device="cuda")
    wsp = T.conv_workspace(x, w, st, (1, 1), (1, 1), 4, layout=layout)
    T.conv2d_htiled(x, w, st, (1, 1), (1, 1), 4, out=y, workspace=wsp, layout=layout)
    T.check(wsp)
    # The filter went to tensor memory from the caller's rows: nothing wrote
    # the workspace's reordered-filter area (it follows the 256-byte header).
    assert int(wsp[256:256 + co * 9 * c * 2].count_nonzero()) == 0
    check_against_oracle(to_f64(y), S.widen(x_np, dt), S.widen(w_np, dt), st, (1, 1), (1, 1),
                         S.F32)
