"""tiles_gemm_noalloc: the GEMM for callers that cannot allocate device memory.

Such callers (code running inside an allocator or driver callback, under a
runtime that owns all device memory, or on a path that must not allocate)
cannot hand the library a workspace.  The entry point uses the library's
static device scratch instead.  These tests call it through the C ABI twice in
a row and compare each result with the float64 oracle under the parity
tolerance of the other GPU tests, and with the workspace-taking entry point
(tiles_gemm_batched, the same kernel and schedule) bit for bit.  The file is
named so that pytest collects it last.
"""

import ctypes as C

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
from tile_size_decision_gb300 import _abi  # noqa: E402
from tests.gpu_util import to_cuda, to_f64, empty_out  # noqa: E402


def desc_for(a, b, c, dt_in, dt_out):
    d = _abi.GemmDesc()
    d.batch, d.m, d.k = a.shape
    d.n = b.shape[2]
    d.a, d.b, d.c = a.data_ptr(), b.data_ptr(), c.data_ptr()
    d.lda, d.ldb, d.ldc = a.stride(1), b.stride(1), c.stride(1)
    d.stride_a, d.stride_b, d.stride_c = a.stride(0), b.stride(0), c.stride(0)
    d.a_dtype = d.b_dtype = _abi.DTYPE_CODES[dt_in]
    d.c_dtype = _abi.DTYPE_CODES[dt_out]
    return d


@pytest.mark.parametrize("case", [
    (3, 300, 520, 256, S.BF16, S.F32),
    (1, 1000, 1000, 512, S.F16, S.F16),
])
def test_noalloc_matches_workspace_gemm_on_two_calls(case):
    bsz, m, n, k, dt_in, dt_out = case
    lib = T.load()
    a_np = S.random_matrix(7, (bsz, m, k), dt_in, "normal")
    b_np = S.random_matrix(8, (bsz, k, n), dt_in, "normal")
    a, b = to_cuda(a_np, dt_in), to_cuda(b_np, dt_in)
    stream = torch.cuda.current_stream()
    handle = C.c_void_p(stream.cuda_stream)

    ws = T.workspace()
    same = empty_out((bsz, m, n), dt_out)
    d_ws = desc_for(a, b, same, dt_in, dt_out)
    assert lib.tiles_gemm_batched(C.byref(d_ws), None, ws.data_ptr(), ws.numel(), handle) == 0
    assert lib.tiles_check(ws.data_ptr(), handle) == 0
    same64 = to_f64(same)

    a64, b64 = S.widen(a_np, dt_in), S.widen(b_np, dt_in)
    ref, bound = OG.gemm(a64, b64), OG.gemm_bound(a64, b64)
    for call in range(2):
        out = empty_out((bsz, m, n), dt_out)
        d = desc_for(a, b, out, dt_in, dt_out)
        status = lib.tiles_gemm_noalloc(C.byref(d), None, handle, 1)
        assert status == 0, lib.tiles_last_error().decode()
        got = to_f64(out)
        ok, worst, idx = OT.check(got, ref, bound, dt_out)
        assert ok, f"call {call}: ratio {worst} at {idx}"
        assert np.array_equal(got, same64), f"call {call} differs from tiles_gemm_batched"


def test_noalloc_rejects_bad_arguments_before_launch():
    lib = T.load()
    d = _abi.GemmDesc()
    d.m = d.n = d.k = 64
    d.batch = 1
    d.a, d.b, d.c = 0x10000, 0x20000, 0x30002
    d.lda = d.ldb = d.ldc = 64
    d.a_dtype = d.b_dtype = _abi.F16
    d.c_dtype = _abi.F32
    assert lib.tiles_gemm_noalloc(C.byref(d), None, None, 1) == _abi.ERR_MISALIGNED
    # A K-split last round would need more scratch than the static array.
    d.c = 0x30000
    d.m = d.n = d.k = d.lda = d.ldb = d.ldc = 4096
    stages = {(c.bn, c.cta_group): c.stages for c in T.gemm_variants()}[(256, 2)]
    ks = T.make_config(256, 256, 64, stages, 192, "tcgen05", 2, 2, tail="ksplit")
    assert lib.tiles_gemm_noalloc(C.byref(d), C.byref(ks), None, 1) == _abi.ERR_TOO_LARGE


def test_noalloc_reports_a_timeout_once_then_clears_it():
    # A bounded wait that runs out in one no-alloc call (a planted fault:
    # the first CTA group skips one pipeline stage, 50 ms wait limit) is
    # recorded in the library's static scratch; the next call with wait != 0
    # reports it once and clears it, and the call after that is clean and
    # correct.
    lib = T.load()
    bsz, m, n, k = 2, 512, 384, 1024
    a_np = S.random_matrix(17, (bsz, m, k), S.F16, "normal")
    b_np = S.random_matrix(18, (bsz, k, n), S.F16, "normal")
    a, b = to_cuda(a_np, S.F16), to_cuda(b_np, S.F16)
    handle = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    out = empty_out((bsz, m, n), S.F32)
    d = desc_for(a, b, out, S.F16, S.F32)
    assert lib.tiles_selftest_drop_stage(3, 50_000_000) == 0
    assert lib.tiles_gemm_noalloc(C.byref(d), None, handle, 0) == 0
    assert lib.tiles_gemm_noalloc(C.byref(d), None, handle, 1) == _abi.ERR_TIMEOUT
    out2 = empty_out((bsz, m, n), S.F32)
    d2 = desc_for(a, b, out2, S.F16, S.F32)
    assert lib.tiles_gemm_noalloc(C.byref(d2), None, handle, 1) == 0
    a64, b64 = S.widen(a_np, S.F16), S.widen(b_np, S.F16)
    ok, worst, idx = OT.check(to_f64(out2), OG.gemm(a64, b64), OG.gemm_bound(a64, b64), S.F32)
    assert ok, f"ratio {worst} at {idx}"
