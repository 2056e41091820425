"""Pass criterion for GPU results against the float64 oracle (test only).

    |C_gpu - C_ref| <= 1e-3 * S + ulp_out(|C_ref|)

S is sum_k |A_ik * B_kj| (or the convolution's analogue) and ulp_out is the
spacing of the output dtype at |C_ref|, so the last term covers the final
round-to-nearest cast to fp16/bf16/fp32.
"""

from __future__ import annotations

import numpy as np

# (mantissa bits, minimum normal exponent) of each output dtype.
_FORMATS = {
    "f16": (10, -14),
    "bf16": (7, -126),
    "f32": (23, -126),
}


def ulp(x: np.ndarray, dtype: str) -> np.ndarray:
    """Spacing of ``dtype`` at |x| (subnormal spacing below the normal range)."""
    mant, emin = _FORMATS[dtype]
    ax = np.abs(np.asarray(x, dtype=np.float64))
    _, e = np.frexp(ax)                 # ax = f * 2**e, f in [0.5, 1)
    exp = np.maximum(e - 1, emin)       # floor(log2 ax), clamped to normal range
    return np.ldexp(1.0, exp - mant)


def tolerance(ref: np.ndarray, bound: np.ndarray, out_dtype: str, rel: float = 1e-3) -> np.ndarray:
    return rel * np.asarray(bound, dtype=np.float64) + ulp(ref, out_dtype)


def check(got64: np.ndarray, ref: np.ndarray, bound: np.ndarray, out_dtype: str,
          rel: float = 1e-3):
    """Return (ok, worst_ratio, index) where ratio = |err| / tolerance."""
    got64 = np.asarray(got64, dtype=np.float64)
    err = np.abs(got64 - ref)
    tol = tolerance(ref, bound, out_dtype, rel)
    ratio = err / tol
    if ratio.size == 0:
        return True, 0.0, None
    bad = ~np.isfinite(got64)
    if bad.any():
        idx = np.unravel_index(int(np.argmax(bad)), bad.shape)
        return False, float("inf"), idx
    flat = int(np.argmax(ratio))
    worst = float(ratio.reshape(-1)[flat])
    return worst <= 1.0, worst, np.unravel_index(flat, ratio.shape)
