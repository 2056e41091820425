"""H-tiling row formulas and a float64 direct convolution (test only).

Row formulas, from the tiling tutorial's section "H/W 维切分的通用公式", for an
output tile covering rows [o0, o1) of a convolution with input height H,
kernel height kh, stride sh, top padding pt and dilation d:

    in_start = max(0, o0*sh - pt)              first input row the tile reads
    in_end   = (o1 - 1)*sh - pt + (kh - 1)*d + 1   one past the last row
    in_span  = in_end - in_start               rows of the slice
    pt'      = max(0, pt - o0*sh)              top pad left for the sub-op
    pb'      = max(0, in_end - H)              bottom pad the sub-op needs
    halo     = (kh - 1)*d + 1 - sh             rows shared by adjacent tiles

Readings where the tutorial is silent:
  * in_span counts the pb' virtual rows when in_end > H; the real slice is
    [in_start, min(in_end, H)).
  * halo is reported signed; it is <= 0 when sh >= (kh-1)*d + 1.
  * Tiles are [t*tile_oh, min((t+1)*tile_oh, OH)); OH uses symmetric padding.

The convolution is the definition
    y[n, co, oh, ow] = sum_{ci, r, s} w[co, ci, r, s]
                       * x[n, ci, oh*sh - pt + r*dh, ow*sw - pw + s*dw]
with zeros outside the image, evaluated in float64 as kh*kw shifted matmuls.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class HTileRows:
    in_start: int
    in_end: int
    in_span: int
    pt: int
    pb: int
    halo: int


def htile_rows(H: int, kh: int, sh: int, pt: int, d: int, o0: int, o1: int) -> HTileRows:
    in_start = max(0, o0 * sh - pt)
    in_end = (o1 - 1) * sh - pt + (kh - 1) * d + 1
    return HTileRows(
        in_start=in_start,
        in_end=in_end,
        in_span=in_end - in_start,
        pt=max(0, pt - o0 * sh),
        pb=max(0, in_end - H),
        halo=(kh - 1) * d + 1 - sh,
    )


def out_size(size: int, k: int, stride: int, pad_lo: int, pad_hi: int, dil: int) -> int:
    return (size + pad_lo + pad_hi - (k - 1) * dil - 1) // stride + 1


def htile_ranges(OH: int, tile_oh: int):
    return [(o0, min(o0 + tile_oh, OH)) for o0 in range(0, OH, tile_oh)]


def conv2d(x64: np.ndarray, w64: np.ndarray, stride=(1, 1), pad_h=(0, 0), pad_w=(0, 0),
           dil=(1, 1)) -> np.ndarray:
    """Direct convolution, NCHW input, OIHW weights, float64.

    pad_h = (top, bottom) and pad_w = (left, right) may be asymmetric so that
    the H-tiled sub-operators (pt', pb') can be evaluated with it.
    """
    x64 = np.asarray(x64, dtype=np.float64)
    w64 = np.asarray(w64, dtype=np.float64)
    n, c, h, w = x64.shape
    co, c2, kh, kw = w64.shape
    if c != c2:
        raise ValueError("channel mismatch")
    sh, sw = stride
    dh, dw = dil
    oh = out_size(h, kh, sh, pad_h[0], pad_h[1], dh)
    ow = out_size(w, kw, sw, pad_w[0], pad_w[1], dw)
    y = np.zeros((n, co, max(oh, 0), max(ow, 0)), dtype=np.float64)
    if oh <= 0 or ow <= 0:
        return y
    xp = np.zeros((n, c, h + pad_h[0] + pad_h[1], w + pad_w[0] + pad_w[1]), dtype=np.float64)
    xp[:, :, pad_h[0]:pad_h[0] + h, pad_w[0]:pad_w[0] + w] = x64
    for r in range(kh):
        for s in range(kw):
            r0 = r * dh
            s0 = s * dw
            patch = xp[:, :, r0:r0 + sh * (oh - 1) + 1:sh, s0:s0 + sw * (ow - 1) + 1:sw]
            # [co, c] x [n, c, oh*ow] -> [n, co, oh*ow]
            y += np.matmul(w64[:, :, r, s], patch.reshape(n, c, oh * ow)).reshape(n, co, oh, ow)
    return y


def conv2d_loops(x64: np.ndarray, w64: np.ndarray, stride=(1, 1), pad=(0, 0), dil=(1, 1)):
    """The defining seven-fold loop with symmetric padding, for tiny shapes."""
    x64 = np.asarray(x64, dtype=np.float64)
    w64 = np.asarray(w64, dtype=np.float64)
    n, c, h, w = x64.shape
    co, _, kh, kw = w64.shape
    oh = out_size(h, kh, stride[0], pad[0], pad[0], dil[0])
    ow = out_size(w, kw, stride[1], pad[1], pad[1], dil[1])
    y = np.zeros((n, co, oh, ow), dtype=np.float64)
    for b in range(n):
        for o in range(co):
            for i in range(oh):
                for j in range(ow):
                    acc = 0.0
                    for ci in range(c):
                        for r in range(kh):
                            ih = i * stride[0] - pad[0] + r * dil[0]
                            if ih < 0 or ih >= h:
                                continue
                            for s in range(kw):
                                iw = j * stride[1] - pad[1] + s * dil[1]
                                if iw < 0 or iw >= w:
                                    continue
                                acc += w64[o, ci, r, s] * x64[b, ci, ih, iw]
                    y[b, o, i, j] = acc
    return y


def conv2d_htiled(x64: np.ndarray, w64: np.ndarray, stride=(1, 1), pad=(0, 0), dil=(1, 1),
                  tile_oh: int = 1) -> np.ndarray:
    """The convolution assembled tile by tile over H.

    Each tile convolves only its input slice [in_start, min(in_end, H)) with
    top pad pt' and bottom pad pb' from ``htile_rows`` (W keeps the original
    symmetric padding) and writes its o1 - o0 rows into the output.
    """
    x64 = np.asarray(x64, dtype=np.float64)
    n, c, h, w = x64.shape
    co, _, kh, kw = np.asarray(w64).shape
    oh = out_size(h, kh, stride[0], pad[0], pad[0], dil[0])
    ow = out_size(w, kw, stride[1], pad[1], pad[1], dil[1])
    y = np.zeros((n, co, oh, ow), dtype=np.float64)
    for o0, o1 in htile_ranges(oh, tile_oh):
        t = htile_rows(h, kh, stride[0], pad[0], dil[0], o0, o1)
        sl = x64[:, :, t.in_start:min(t.in_end, h), :]
        sub = conv2d(sl, w64, stride, (t.pt, t.pb), (pad[1], pad[1]), dil)
        if sub.shape[2] != o1 - o0:
            raise AssertionError(f"tile [{o0},{o1}) produced {sub.shape[2]} rows")
        y[:, :, o0:o1, :] = sub
    return y


def conv2d_tiled(x64: np.ndarray, w64: np.ndarray, stride=(1, 1), pad=(0, 0), dil=(1, 1),
                 tile_oh: int = 1, tile_ow: int | None = None, tile_n: int | None = None
                 ) -> np.ndarray:
    """The convolution assembled from independent sub-convolutions over
    batch tiles, H-tiles and W-tiles.

    The tutorial's slicing formulas ("H/W 维切分的通用公式") apply to each
    spatial dimension alike: an output tile [q0, q1) of the width reads the
    input columns [in_start, min(in_end, W)) with left pad pl' and right pad
    pr' from the same formulas (``htile_rows`` with the width's sizes).  A
    batch tile of images needs no halo at all (the tutorial's reason to tile
    the batch first, "为什么教学工程先切 batch 维"): each image is its own
    sub-problem.  Every tile convolves only its own slice.
    """
    x64 = np.asarray(x64, dtype=np.float64)
    n, c, h, w = x64.shape
    co, _, kh, kw = np.asarray(w64).shape
    oh = out_size(h, kh, stride[0], pad[0], pad[0], dil[0])
    ow = out_size(w, kw, stride[1], pad[1], pad[1], dil[1])
    tile_ow = ow if tile_ow is None else tile_ow
    tile_n = n if tile_n is None else tile_n
    y = np.zeros((n, co, oh, ow), dtype=np.float64)
    for n0 in range(0, n, tile_n):
        n1 = min(n0 + tile_n, n)
        for o0, o1 in htile_ranges(oh, tile_oh):
            th = htile_rows(h, kh, stride[0], pad[0], dil[0], o0, o1)
            for q0, q1 in htile_ranges(ow, tile_ow):
                tw = htile_rows(w, kw, stride[1], pad[1], dil[1], q0, q1)
                sl = x64[n0:n1, :, th.in_start:min(th.in_end, h), tw.in_start:min(tw.in_end, w)]
                sub = conv2d(sl, w64, stride, (th.pt, th.pb), (tw.pt, tw.pb), dil)
                if sub.shape[2:] != (o1 - o0, q1 - q0):
                    raise AssertionError(f"tile [{o0},{o1})x[{q0},{q1}) produced {sub.shape[2:]}")
                y[n0:n1, :, o0:o1, q0:q1] = sub
    return y


def conv2d_points(x64: np.ndarray, w64: np.ndarray, pts, stride=(1, 1), pad=(0, 0),
                  dil=(1, 1), absolute: bool = False) -> np.ndarray:
    """y (or its bound with |x|, |w|) at sampled points (n, co, oh, ow) only."""
    x64 = np.asarray(x64, dtype=np.float64)
    w64 = np.asarray(w64, dtype=np.float64)
    if absolute:
        x64 = np.abs(x64)
        w64 = np.abs(w64)
    _, c, h, w = x64.shape
    _, _, kh, kw = w64.shape
    out = np.empty(len(pts), dtype=np.float64)
    for t, (b, o, i, j) in enumerate(pts):
        acc = 0.0
        for r in range(kh):
            ih = i * stride[0] - pad[0] + r * dil[0]
            if ih < 0 or ih >= h:
                continue
            for s in range(kw):
                iw = j * stride[1] - pad[1] + s * dil[1]
                if iw < 0 or iw >= w:
                    continue
                acc += float(np.dot(w64[o, :, r, s], x64[b, :, ih, iw]))
        out[t] = acc
    return out
