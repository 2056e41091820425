"""Pins for the H-tile row formulas and the float64 convolution oracle.

  * the tutorial's worked example (tests/golden/htile_example.json);
  * brute force: the seven-fold loop against the shifted-matmul evaluation;
  * a 1x1 stride-1 convolution reduces to a GEMM;
  * closed form on all-ones inputs (interior, edge and corner counts);
  * over a grid of H, kh, sh, pt, d and tile heights, the H-tiled convolution
    built from slices with (pt', pb') equals the untiled one exactly on
    integer inputs, every tile yields o1 - o0 rows, and adjacent interior
    tiles share exactly `halo` input rows.
"""

import itertools
import json
import os

import numpy as np
import pytest

import synth_inputs as S
from oracle import conv as C
from oracle import gemm as G

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "htile_example.json")


def test_worked_example():
    with open(GOLDEN) as f:
        g = json.load(f)
    p = g["params"]
    assert C.out_size(p["H"], p["kh"], p["sh"], p["pt"], p["pb_for_OH"], p["d"]) == p["OH"]
    assert C.out_size(p["H"], p["kh"], p["sh"], p["pt"], p["pt"], p["d"]) == p["OH"] + 1
    assert C.htile_ranges(p["OH"], p["tile_oh"]) == [(t["o0"], t["o1"]) for t in g["tiles"]]
    for t in g["tiles"]:
        r = C.htile_rows(p["H"], p["kh"], p["sh"], p["pt"], p["d"], t["o0"], t["o1"])
        assert (r.in_start, r.in_end, r.in_span, r.pt, r.pb) == (
            t["in_start"], t["in_end"], t["in_span"], t["pt"], t["pb"])
        assert r.halo == g["halo"]
    a = C.htile_rows(p["H"], p["kh"], p["sh"], p["pt"], p["d"], 0, 2)
    b = C.htile_rows(p["H"], p["kh"], p["sh"], p["pt"], p["d"], 2, 4)
    shared = set(range(a.in_start, a.in_end)) & set(range(b.in_start, b.in_end))
    assert shared == {g["shared_row"]}


CASES = [
    # (n, c, h, w, co, kh, kw, stride, pad, dil)
    (1, 1, 5, 5, 1, 3, 3, (1, 1), (1, 1), (1, 1)),
    (2, 3, 7, 6, 4, 3, 2, (2, 1), (1, 0), (1, 1)),
    (1, 2, 9, 9, 3, 3, 3, (2, 2), (1, 1), (2, 1)),
    (1, 2, 6, 8, 2, 1, 1, (1, 1), (0, 0), (1, 1)),
    (2, 1, 10, 4, 2, 5, 3, (3, 2), (2, 1), (1, 2)),
]


@pytest.mark.parametrize("case", CASES)
def test_brute_force_tiny(case):
    n, c, h, w, co, kh, kw, st, pad, dil = case
    x = S.widen(S.random_matrix(1, (n, c, h, w), S.F16), S.F16)
    wt = S.widen(S.random_matrix(2, (co, c, kh, kw), S.F16), S.F16)
    ref = C.conv2d(x, wt, st, (pad[0], pad[0]), (pad[1], pad[1]), dil)
    loops = C.conv2d_loops(x, wt, st, pad, dil)
    assert ref.shape == loops.shape
    np.testing.assert_allclose(ref, loops, rtol=0, atol=1e-12)
    pts = [(0, 0, 0, 0), (n - 1, co - 1, ref.shape[2] - 1, ref.shape[3] - 1),
           (0, co // 2, ref.shape[2] // 2, 0)]
    got = C.conv2d_points(x, wt, pts, st, pad, dil)
    np.testing.assert_allclose(got, [ref[p] for p in pts], rtol=0, atol=1e-12)
    bnd = C.conv2d_points(x, wt, pts, st, pad, dil, absolute=True)
    full_bnd = C.conv2d(np.abs(x), np.abs(wt), st, (pad[0], pad[0]), (pad[1], pad[1]), dil)
    np.testing.assert_allclose(bnd, [full_bnd[p] for p in pts], rtol=0, atol=1e-12)


def test_pointwise_conv_is_gemm():
    x = S.widen(S.random_matrix(3, (2, 5, 4, 6), S.BF16), S.BF16)
    wt = S.widen(S.random_matrix(4, (7, 5, 1, 1), S.BF16), S.BF16)
    y = C.conv2d(x, wt)
    for b in range(2):
        g = G.gemm(wt[:, :, 0, 0], x[b].reshape(5, 24)).reshape(7, 4, 6)
        np.testing.assert_allclose(y[b], g, rtol=0, atol=1e-12)


def test_all_ones_closed_form():
    c = 3
    y = C.conv2d(np.ones((1, c, 6, 5)), np.ones((1, c, 3, 3)), (1, 1), (1, 1), (1, 1))
    assert y.shape == (1, 1, 6, 5)
    assert y[0, 0, 2, 2] == 9 * c                   # interior: full window
    assert y[0, 0, 0, 0] == 4 * c                   # corner: 2x2 of the window
    assert y[0, 0, 0, 2] == 6 * c                   # top edge: 2x3
    assert y[0, 0, 3, 4] == 6 * c                   # right edge: 3x2
    # stride 2, pad 1 on 224 -> 112, the size used by the convolution workload
    assert C.out_size(224, 3, 2, 1, 1, 1) == 112


def _rows_used(H, kh, sh, pt, d, o0, o1):
    rows = set()
    for o in range(o0, o1):
        for r in range(kh):
            ih = o * sh - pt + r * d
            if 0 <= ih < H:
                rows.add(ih)
    return rows


def test_htiled_equals_untiled_exhaustive():
    rng = np.random.default_rng(11)
    checked = 0
    for H, kh, sh, d in itertools.product((1, 2, 5, 9, 16, 23, 40), (1, 2, 3, 5), (1, 2, 3),
                                          (1, 2)):
        for pt in range(kh):
            OH = C.out_size(H, kh, sh, pt, pt, d)
            if OH <= 0:
                continue
            x = rng.integers(-3, 4, size=(1, 2, H, 3)).astype(np.float64)
            w = rng.integers(-2, 3, size=(2, 2, kh, 2)).astype(np.float64)
            full = C.conv2d(x, w, (sh, 1), (pt, pt), (0, 0), (d, 1))
            for tile in (1, 2, 3, 5):
                tiled = C.conv2d_htiled(x, w, (sh, 1), (pt, 0), (d, 1), tile)
                assert np.array_equal(tiled, full), (H, kh, sh, pt, d, tile)
                for o0, o1 in C.htile_ranges(OH, tile):
                    t = C.htile_rows(H, kh, sh, pt, d, o0, o1)
                    used = _rows_used(H, kh, sh, pt, d, o0, o1)
                    # the slice covers every real row the tile's windows touch
                    assert used <= set(range(t.in_start, min(t.in_end, H)))
                    if o1 < OH and o0 * sh - pt >= 0:
                        nxt = C.htile_rows(H, kh, sh, pt, d, o1, min(o1 + tile, OH))
                        assert t.in_end - nxt.in_start == t.halo
                checked += 1
    assert checked > 500


def test_htile_rows_zero_and_negative_halo():
    # stride >= window: tiles do not overlap and the signed halo is <= 0
    t = C.htile_rows(H=10, kh=2, sh=3, pt=0, d=1, o0=0, o1=2)
    assert t.halo == -1
    # bottom pad: the last tile reaches past H
    t = C.htile_rows(H=9, kh=3, sh=2, pt=1, d=1, o0=4, o1=5)
    assert (t.in_start, t.in_end, t.pt, t.pb) == (7, 10, 0, 1)


def test_tiled_over_batch_h_and_w_equals_untiled():
    # The slicing formulas applied to both spatial dimensions, and batch
    # tiles without halo, rebuild the untiled convolution exactly (integer
    # inputs: every sum is exact in float64).
    rng = np.random.default_rng(12)
    checked = 0
    for (H, W), (kh, kw), (sh, sw), (ph, pw), (dh, dw) in itertools.product(
            ((9, 7), (16, 13), (5, 23)), ((3, 3), (2, 5), (1, 3)), ((1, 1), (2, 2), (3, 1)),
            ((0, 0), (1, 1), (1, 2)), ((1, 1), (2, 1))):
        if ph >= kh or pw >= kw:
            continue
        OH = C.out_size(H, kh, sh, ph, ph, dh)
        OW = C.out_size(W, kw, sw, pw, pw, dw)
        if OH <= 0 or OW <= 0:
            continue
        x = rng.integers(-3, 4, size=(3, 2, H, W)).astype(np.float64)
        w = rng.integers(-2, 3, size=(2, 2, kh, kw)).astype(np.float64)
        full = C.conv2d(x, w, (sh, sw), (ph, ph), (pw, pw), (dh, dw))
        for tile_oh, tile_ow, tile_n in ((1, 1, 1), (2, 3, 2), (OH, 2, 3), (3, OW, 1), (4, 5, 2)):
            tiled = C.conv2d_tiled(x, w, (sh, sw), (ph, pw), (dh, dw), tile_oh, tile_ow, tile_n)
            assert np.array_equal(tiled, full), (H, W, kh, kw, sh, sw, ph, pw, dh, dw,
                                                  tile_oh, tile_ow, tile_n)
            checked += 1
    assert checked > 200


def test_tiled_with_full_width_is_the_h_tiling():
    rng = np.random.default_rng(13)
    x = rng.standard_normal((2, 3, 11, 10))
    w = rng.standard_normal((4, 3, 3, 3))
    a = C.conv2d_tiled(x, w, (2, 1), (1, 1), (1, 1), tile_oh=2)
    b = C.conv2d_htiled(x, w, (2, 1), (1, 1), (1, 1), tile_oh=2)
    assert np.array_equal(a, b)


def test_w_tile_halo_columns():
    # Adjacent W-tiles share (kw-1)*d + 1 - sw input columns, as rows do.
    W, kw, sw, pw, d = 20, 3, 1, 1, 1
    OW = C.out_size(W, kw, sw, pw, pw, d)
    tiles = C.htile_ranges(OW, 6)
    for (q0, q1), (r0, r1) in zip(tiles, tiles[1:]):
        a = C.htile_rows(W, kw, sw, pw, d, q0, q1)
        b = C.htile_rows(W, kw, sw, pw, d, r0, r1)
        assert a.in_end - b.in_start == a.halo == 2
