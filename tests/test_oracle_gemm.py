"""Pins for the float64 GEMM oracle, the tolerance and the input generator.

The oracle is C = A x B (tiling tutorial, "案例解释 / 前提").  It is pinned by
brute force on tiny shapes (three explicit loops, a separate implementation
from the matmul primitive), by closed forms on structured inputs, and by the
identity; the tolerance's ulp is pinned against numpy's and torch's own
spacing; the bf16 rounding of the generator against torch's conversion.
"""

import numpy as np
import pytest

import synth_inputs as S
from oracle import gemm as G
from oracle import tolerance as T


@pytest.mark.parametrize("shape", [(1, 1, 1), (3, 5, 7), (17, 9, 33), (8, 16, 1), (1, 40, 2)])
def test_brute_force_tiny(shape):
    m, n, k = shape
    a = S.widen(S.random_matrix(10 + m, (m, k), S.F16), S.F16)
    b = S.widen(S.random_matrix(20 + n, (k, n), S.F16), S.F16)
    ref = G.gemm(a, b)
    loops = G.gemm_loops(a, b)
    assert ref.shape == (m, n)
    # fp16 inputs have 11-bit significands: every product is exact in float64
    # and a sum of a few dozen stays far from float64 rounding.
    np.testing.assert_allclose(ref, loops, rtol=0, atol=1e-12)


def test_closed_forms():
    m, n, k = 6, 5, 7
    i = np.arange(m, dtype=np.float64)[:, None]
    j = np.arange(n, dtype=np.float64)[None, :]
    # A[i,k] = i, B[k,j] = j  ->  C[i,j] = K*i*j
    a = np.repeat(i, k, axis=1)
    b = np.repeat(j, k, axis=0)
    assert np.array_equal(G.gemm(a, b), k * i * j)
    # A[i,k] = k, B[k,j] = 1  ->  C[i,j] = K(K-1)/2
    a = np.tile(np.arange(k, dtype=np.float64), (m, 1))
    assert np.array_equal(G.gemm(a, np.ones((k, n))), np.full((m, n), k * (k - 1) / 2))
    # A[i,k] = (-1)^k, B[k,j] = 1  ->  alternating sum: 1 if K odd else 0
    a = np.tile((-1.0) ** np.arange(k), (m, 1))
    assert np.array_equal(G.gemm(a, np.ones((k, n))), np.ones((m, n)))


def test_identity_and_permutation():
    rng = np.random.default_rng(5)
    b = S.widen(S.random_matrix(5, (64, 48), S.BF16), S.BF16)
    assert np.array_equal(G.gemm(np.eye(64), b), b)
    perm = rng.permutation(64)
    p = np.eye(64)[perm]            # row r of P selects row perm[r] of B
    assert np.array_equal(G.gemm(p, b), b[perm])
    # Non-square operands in the wrong order are refused, not silently mixed.
    with pytest.raises(ValueError):
        G.gemm(np.ones((3, 4)), np.ones((3, 4)))


def test_batched_is_per_slice():
    a = S.widen(S.random_matrix(1, (3, 4, 6), S.BF16, "normal"), S.BF16)
    b = S.widen(S.random_matrix(2, (3, 6, 5), S.BF16, "normal"), S.BF16)
    c = G.gemm(a, b)
    for t in range(3):
        np.testing.assert_allclose(c[t], G.gemm_loops(a[t], b[t]), rtol=0, atol=1e-12)


def test_bound_and_sampled_rows():
    a = S.widen(S.random_matrix(3, (20, 30), S.F16), S.F16)
    b = S.widen(S.random_matrix(4, (30, 10), S.F16), S.F16)
    c = G.gemm(a, b)
    s = G.gemm_bound(a, b)
    assert np.all(s >= np.abs(c) - 1e-12)
    assert np.array_equal(G.gemm_bound(np.abs(a), np.abs(b)), G.gemm(np.abs(a), np.abs(b)))
    rows = np.array([0, 19, 7, 7])
    cols = np.array([0, 9, 3, 4])
    np.testing.assert_allclose(G.gemm_rows(a, b, rows, cols), c[rows, cols], rtol=0, atol=1e-12)
    np.testing.assert_allclose(G.gemm_rows_bound(a, b, rows, cols), s[rows, cols], rtol=0,
                               atol=1e-12)


def test_ulp_matches_library_spacing():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.uniform(-70000, 70000, 500), rng.uniform(-1e-3, 1e-3, 500),
                        [1.0, 2.0, 65504.0, 6.103515625e-05, 3e-8]])
    h = x[np.abs(x) < 65504].astype(np.float16)
    assert np.array_equal(T.ulp(h.astype(np.float64), "f16"),
                          np.abs(np.spacing(h)).astype(np.float64))
    f = x.astype(np.float32)
    assert np.array_equal(T.ulp(f.astype(np.float64), "f32"),
                          np.abs(np.spacing(f)).astype(np.float64))
    torch = pytest.importorskip("torch")
    bb = torch.tensor(x, dtype=torch.float64).to(torch.bfloat16)
    up = torch.nextafter(bb.abs(), torch.full_like(bb, float("inf")))
    want = (up.double() - bb.abs().double()).numpy()
    assert np.array_equal(T.ulp(bb.double().numpy(), "bf16"), want)
    assert T.ulp(np.array([1.0]), "f16")[0] == 2.0 ** -10
    assert T.ulp(np.array([1.0]), "bf16")[0] == 2.0 ** -7


def test_tolerance_check_detects_error():
    ref = np.array([[1.0, 2.0], [3.0, 4.0]])
    bound = np.array([[10.0, 10.0], [10.0, 10.0]])
    ok, worst, _ = T.check(ref + 0.005, ref, bound, "f32")
    assert ok and worst < 1
    ok, worst, idx = T.check(ref + np.array([[0, 0], [0, 0.02]]), ref, bound, "f32")
    assert not ok and idx == (1, 1)
    ok, _, _ = T.check(np.array([[np.nan, 2.0], [3.0, 4.0]]), ref, bound, "f32")
    assert not ok


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.normal(0, 1, 20000), rng.normal(0, 1e-30, 1000),
                        rng.uniform(-3e38, 3e38, 1000)])
    bits = S.f64_to_bf16_bits(x)
    want = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16)
    assert np.array_equal(bits.view(np.int16), want.numpy())
    back = S.bf16_bits_to_f64(bits)
    assert np.array_equal(back, torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
                          .double().numpy())


def test_workload_recipes_are_seeded():
    wl = S.GemmWorkload("t", 1, 8, 6, 4, S.BF16, S.F32, "normal", 3, scale=0.5)
    a1, b1 = S.gemm_inputs(wl)
    a2, b2 = S.gemm_inputs(wl)
    assert np.array_equal(a1, a2) and np.array_equal(b1, b2)
    assert a1.dtype == np.uint16 and a1.shape == (8, 4) and b1.shape == (4, 6)
    conv = S.WORKLOADS["conv_htiled"]
    assert (conv.oh, conv.ow) == (112, 112)
    assert conv.flops == 2 * 8 * 128 * 112 * 112 * 64 * 9
    assert S.WORKLOADS["gemm_4096"].flops == 2 * 4096 ** 3
