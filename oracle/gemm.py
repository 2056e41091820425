"""Float64 GEMM oracle (test infrastructure only).

The tiling tutorial states the problem as C = A x B with A of M x K, B of
K x N and C of M x N ("案例解释 / 前提"); each C[i, j] takes K multiplies and
K adds.  The tiled GPU method reaches exactly this sum, in another order, so
the oracle is the definition itself:

    C[b, i, j] = sum_k A[b, i, k] * B[b, k, j]

computed in float64 from the already-quantised inputs, with numpy's matmul as
the summation primitive.  ``gemm_loops`` is the same sum as three explicit
loops for tiny shapes; ``gemm_bound`` is S = |A| x |B|, the scale of the
tolerance.
"""

from __future__ import annotations

import numpy as np


def gemm(a64: np.ndarray, b64: np.ndarray) -> np.ndarray:
    """C = A x B in float64; leading batch axes broadcast as in matmul."""
    return np.matmul(np.asarray(a64, dtype=np.float64), np.asarray(b64, dtype=np.float64))


def gemm_bound(a64: np.ndarray, b64: np.ndarray) -> np.ndarray:
    """S[b, i, j] = sum_k |A[b, i, k]| * |B[b, k, j]|."""
    return np.matmul(np.abs(np.asarray(a64, dtype=np.float64)),
                     np.abs(np.asarray(b64, dtype=np.float64)))


def gemm_loops(a64: np.ndarray, b64: np.ndarray) -> np.ndarray:
    """The defining triple loop, for shapes of a few dozen per side."""
    a64 = np.asarray(a64, dtype=np.float64)
    b64 = np.asarray(b64, dtype=np.float64)
    m, k = a64.shape
    k2, n = b64.shape
    if k != k2:
        raise ValueError("inner dimensions differ")
    c = np.zeros((m, n), dtype=np.float64)
    for i in range(m):
        for j in range(n):
            acc = 0.0
            for kk in range(k):
                acc += a64[i, kk] * b64[kk, j]
            c[i, j] = acc
    return c


def gemm_rows(a64: np.ndarray, b64: np.ndarray, rows, cols) -> np.ndarray:
    """C at the sampled coordinates (rows[t], cols[t]) only: one dot product
    each, for checking outputs of problems too large to compute whole."""
    a64 = np.asarray(a64, dtype=np.float64)
    b64 = np.asarray(b64, dtype=np.float64)
    return np.einsum("tk,tk->t", a64[rows, :], b64[:, cols].T)


def gemm_rows_bound(a64: np.ndarray, b64: np.ndarray, rows, cols) -> np.ndarray:
    a64 = np.abs(np.asarray(a64, dtype=np.float64))
    b64 = np.abs(np.asarray(b64, dtype=np.float64))
    return np.einsum("tk,tk->t", a64[rows, :], b64[:, cols].T)


def arithmetic_intensity_naive(k: int, elem_bytes: int) -> float:
    """FLOP per byte when one thread computes one C[i, j] and reads its whole
    row of A and column of B from memory (tutorial, "Naive 方法")."""
    return (2 * k) / (2 * k * elem_bytes)


def arithmetic_intensity_tiled(bm: int, bn: int, k: int, elem_bytes: int) -> float:
    """FLOP per byte for one bm x bn output tile that reads a bm x K panel of A
    and a K x bn panel of B once (tutorial, "Tiled 方法分块复用数据")."""
    return (bm * bn * 2 * k) / ((bm + bn) * k * elem_bytes)
