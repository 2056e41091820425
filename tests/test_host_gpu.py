"""End-to-end calls from host buffers (tiles_gemm_host, tiles_conv2d_host).

Each case starts from seeded host operands in page-locked memory, runs the
call, and checks the host result against the float64 oracle under the same
tolerance as the device calls.  The cases cover the ways the work is cut into
pieces: rows of one GEMM (ragged, and fewer rows than pieces), runs of batch
items (more pieces asked for than items), runs of images, and one piece; two
calls in a row reuse the library's copy streams and events.
"""

import threading

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
from tests.gpu_util import TORCH_DT  # noqa: E402


def pinned(arr: np.ndarray, dt: str):
    if dt == S.BF16:
        t = torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(arr))
    return t.pin_memory()


def host_f64(t) -> np.ndarray:
    return t.to(torch.float64).numpy()


@pytest.mark.parametrize("case", [
    # (batch, m, n, k, in, out, chunks)
    (1, 1000, 712, 320, S.F16, S.F32, 4),       # ragged rows: pieces of whole 256-row tiles
    (1, 200, 256, 512, S.BF16, S.BF16, 6),      # fewer rows than one tile: one piece
    (1, 2048, 1024, 1024, S.F16, S.F16, 1),     # a single piece
    (5, 300, 264, 200, S.BF16, S.F32, 2),       # runs of batch items
    (3, 128, 128, 64, S.F16, S.F16, 16),        # more pieces asked for than items
])
def test_gemm_host_matches_oracle(case):
    bsz, m, n, k, dt, odt, chunks = case
    a_np = S.random_matrix(71, (bsz, m, k), dt, "normal")
    b_np = S.random_matrix(72, (bsz, k, n), dt, "normal")
    a_h, b_h = pinned(a_np, dt), pinned(b_np, dt)
    c_h = torch.full((bsz, m, n), float("nan"), dtype=TORCH_DT[odt]).pin_memory()
    a_d = torch.empty_like(a_h, device="cuda")
    b_d = torch.empty_like(b_h, device="cuda")
    c_d = torch.empty((bsz, m, n), dtype=TORCH_DT[odt], device="cuda")
    ws = T.gemm_workspace(a_d, b_d, c_d)
    a64, b64 = S.widen(a_np, dt), S.widen(b_np, dt)
    ref, bound = OG.gemm(a64, b64), OG.gemm_bound(a64, b64)
    if bsz == 1:
        a_h, b_h, c_h, a_d, b_d, c_d = (t[0] for t in (a_h, b_h, c_h, a_d, b_d, c_d))
        ref, bound = ref[0], bound[0]
    for call in range(2):
        c_h.fill_(float("nan"))
        T.gemm_host(a_h, b_h, c_h, a_d, b_d, c_d, workspace=ws, chunks=chunks)
        torch.cuda.synchronize()
        T.check(ws)
        ok, worst, idx = OT.check(host_f64(c_h), ref, bound, odt)
        assert ok, f"call {call}: worst ratio {worst} at {idx}"


def test_gemm_host_equals_the_device_call_piece_by_piece():
    # One piece per 256-row tile block: each piece is the device GEMM of
    # those rows, so the host result equals the device call's, bit for bit.
    m, n, k = 1024, 512, 768
    a_np = S.random_matrix(73, (m, k), S.F16, "normal")
    b_np = S.random_matrix(74, (k, n), S.F16, "normal")
    a_h, b_h = pinned(a_np, S.F16), pinned(b_np, S.F16)
    c_h = torch.empty((m, n), dtype=torch.float32).pin_memory()
    a_d, b_d = a_h.cuda(), b_h.cuda()
    c_d = torch.empty((m, n), dtype=torch.float32, device="cuda")
    cfg = T.make_config(256, 256, 64, 6, 192, "tcgen05", 2, 2, tail="whole")
    ws = T.workspace()
    T.gemm_host(a_h, b_h, c_h, torch.empty_like(a_d), torch.empty_like(b_d), c_d, cfg=cfg,
                workspace=ws, chunks=4)
    torch.cuda.synchronize()
    dev = torch.empty((m, n), dtype=torch.float32, device="cuda")
    for r0 in range(0, m, 256):
        T.gemm(a_d[r0:r0 + 256], b_d, out=dev[r0:r0 + 256], cfg=cfg, workspace=ws)
    T.check(ws)
    assert torch.equal(c_h, dev.cpu())


@pytest.mark.parametrize("case", [
    # (n, c, h, w, co, stride, pad, layout, chunks)
    (4, 64, 56, 56, 128, (2, 2), (1, 1), "nchw", 3),
    (3, 16, 20, 24, 32, (1, 1), (1, 1), "nhwc", 8),
    (2, 8, 9, 16, 4, (2, 2), (1, 1), "nchw", 1),
])
def test_conv2d_host_matches_oracle(case):
    n, c, h, wd, co, st, pad, layout, chunks = case
    x_np = S.random_matrix(81, (n, c, h, wd), S.F16)
    w_np = S.random_matrix(82, (co, c, 3, 3), S.F16)
    x_in = x_np if layout == "nchw" else np.ascontiguousarray(x_np.transpose(0, 2, 3, 1))
    x_h, w_h = pinned(x_in, S.F16), pinned(w_np, S.F16)
    oh, ow = T.conv_out_hw(h, wd, 3, 3, st, pad, (1, 1))
    y_h = torch.full((n, co, oh, ow), float("nan"), dtype=torch.float16).pin_memory()
    x_d, w_d = torch.empty_like(x_h, device="cuda"), torch.empty_like(w_h, device="cuda")
    y_d = torch.empty((n, co, oh, ow), dtype=torch.float16, device="cuda")
    ws = T.conv_workspace(x_d, w_d, st, pad, (1, 1), 16, layout=layout)
    x64, w64 = S.widen(x_np, S.F16), S.widen(w_np, S.F16)
    ref = OC.conv2d(x64, w64, st, (pad[0], pad[0]), (pad[1], pad[1]), (1, 1))
    bound = OC.conv2d(np.abs(x64), np.abs(w64), st, (pad[0], pad[0]), (pad[1], pad[1]), (1, 1))
    for call in range(2):
        y_h.fill_(float("nan"))
        T.conv2d_host(x_h, w_h, y_h, x_d, w_d, y_d, st, pad, (1, 1), 16, workspace=ws,
                      layout=layout, chunks=chunks)
        torch.cuda.synchronize()
        T.check(ws)
        ok, worst, idx = OT.check(host_f64(y_h), ref, bound, S.F16)
        assert ok, f"call {call}: worst ratio {worst} at {idx}"


def test_host_calls_order_after_earlier_work_on_the_stream():
    # Work enqueued before the call (filling the device buffers with garbage)
    # precedes its uploads; work after it sees the downloaded result.
    m = n = k = 512
    a_np = S.random_matrix(75, (m, k), S.F16)
    b_np = S.random_matrix(76, (k, n), S.F16)
    a_h, b_h = pinned(a_np, S.F16), pinned(b_np, S.F16)
    c_h = torch.empty((m, n), dtype=torch.float32).pin_memory()
    a_d = torch.empty((m, k), dtype=torch.float16, device="cuda")
    b_d = torch.empty((k, n), dtype=torch.float16, device="cuda")
    c_d = torch.empty((m, n), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    ws = T.workspace()
    with torch.cuda.stream(s):
        for t in (a_d, b_d, c_d):
            t.fill_(7.0)
        T.gemm_host(a_h, b_h, c_h, a_d, b_d, c_d, workspace=ws, stream=s, chunks=3)
        after = c_d.clone()
    s.synchronize()
    a64, b64 = S.widen(a_np, S.F16), S.widen(b_np, S.F16)
    ok, worst, idx = OT.check(host_f64(c_h), OG.gemm(a64, b64), OG.gemm_bound(a64, b64), S.F32)
    assert ok, f"worst ratio {worst} at {idx}"
    assert torch.equal(after.cpu(), c_h)


def test_host_calls_from_threads_that_exit():
    # Each host thread has its own copy streams and events, released when
    # the thread exits.  Three threads call at once, each on its own stream
    # and buffers, and exit; then this thread calls.  Every result matches.
    m, n, k = 768, 512, 256
    a_np = S.random_matrix(77, (m, k), S.F16)
    b_np = S.random_matrix(78, (k, n), S.F16)
    a_h, b_h = pinned(a_np, S.F16), pinned(b_np, S.F16)
    a64, b64 = S.widen(a_np, S.F16), S.widen(b_np, S.F16)
    ref, bound = OG.gemm(a64, b64), OG.gemm_bound(a64, b64)
    outs, errors = [], []

    def call(idx):
        try:
            c_h = torch.full((m, n), float("nan"), dtype=torch.float32).pin_memory()
            a_d = torch.empty((m, k), dtype=torch.float16, device="cuda")
            b_d = torch.empty((k, n), dtype=torch.float16, device="cuda")
            c_d = torch.empty((m, n), dtype=torch.float32, device="cuda")
            s = torch.cuda.Stream()
            ws = T.workspace()                # each call has its own workspace
            T.gemm_host(a_h, b_h, c_h, a_d, b_d, c_d, workspace=ws, stream=s, chunks=2 + idx)
            s.synchronize()
            outs.append(c_h)
        except Exception as e:          # reported below, in the main thread
            errors.append(e)

    threads = [threading.Thread(target=call, args=(i,)) for i in range(3)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    call(3)
    assert not errors, errors
    assert len(outs) == 4
    for c_h in outs:
        ok, worst, idx = OT.check(host_f64(c_h), ref, bound, S.F32)
        assert ok, f"worst ratio {worst} at {idx}"
