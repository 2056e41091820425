"""tile_size_decision_gb300 — constraint-planned tiled GEMM and H-tiled
convolution for NVIDIA GB300 (sm_103a).

A thin Python binding over libtiles.so (C ABI in include/tiles.h).  The
binding only marshals arguments: planning (C0-C4), tensor-map encoding and
every kernel run in the native library.  PyTorch supplies device memory and
streams.  Names follow the C ABI without the ``tiles_`` prefix.
"""

from __future__ import annotations

import ctypes as C
import os

from . import _abi
from ._abi import TilesError, check as _check

__all__ = [
    "TilesError", "load", "version", "device_preset", "device_query", "evaluate",
    "finish_parallelism", "c0_bytes", "plan", "htile_rows", "workspace_bytes", "workspace",
    "gemm_variants", "gemm_variant_info",
    "gemm", "gemm_batched", "gemm_schedule", "gemm_workspace", "gemm_noalloc", "gemm_autotune",
    "gemm_host", "conv2d_host",
    "tuned_lookup", "tuned_save", "tuned_load", "tuned_clear", "conv2d_htiled", "conv2d_tiled",
    "conv_workspace",
    "conv_out_shape", "conv_out_hw", "check", "selftest_wait_timeout", "selftest_drop_stage",
    "make_config",
]


def load():
    return _abi.load()


def version() -> str:
    return load().tiles_version().decode()


def device_preset(name: str = "gb300") -> _abi.Device:
    d = _abi.Device()
    pid = {"h100_pages": _abi.DEV_H100_PAGES, "gb300": _abi.DEV_GB300}[name]
    _check(load().tiles_device_preset(pid, C.byref(d)), "tiles_device_preset")
    return d


def device_query(ordinal: int = 0) -> _abi.Device:
    d = _abi.Device()
    _check(load().tiles_device_query(ordinal, C.byref(d)), "tiles_device_query")
    return d


CONV_WEIGHTS = {"auto": _abi.CONV_W_AUTO, "smem": _abi.CONV_W_SMEM, "tmem": _abi.CONV_W_TMEM,
                "rows": _abi.CONV_W_TMEM_ROWS, "rows_direct": _abi.CONV_W_TMEM_ROWS_DIRECT}
TAILS = {"auto": _abi.TAIL_AUTO, "whole": _abi.TAIL_WHOLE, "nhalf": _abi.TAIL_NHALF,
         "ksplit": _abi.TAIL_KSPLIT}


def make_config(bm, bn, bk, stages=3, threads=128, instr="wgmma", acc_bufs=0,
                cta_group=0, tail="auto", conv_weights="auto") -> _abi.Config:
    c = _abi.Config()
    c.bm, c.bn, c.bk, c.stages, c.threads = bm, bn, bk, stages, threads
    c.instr = _abi.INSTR_CODES[instr] if isinstance(instr, str) else instr
    c.acc_bufs, c.cta_group = acc_bufs, cta_group
    c.tail = TAILS[tail] if isinstance(tail, str) else tail
    c.conv_weights = CONV_WEIGHTS[conv_weights] if isinstance(conv_weights, str) else conv_weights
    return c


def evaluate(dev: _abi.Device, cfg: _abi.Config, elem_bytes: int = 2,
             accum_bytes: int = 4) -> _abi.Verdict:
    v = _abi.Verdict()
    _check(load().tiles_evaluate(C.byref(dev), C.byref(cfg), elem_bytes, accum_bytes,
                                 C.byref(v)), "tiles_evaluate")
    return v


def finish_parallelism(dev: _abi.Device, v: _abi.Verdict, m: int, n: int,
                       b: int = 1) -> _abi.Verdict:
    _check(load().tiles_finish_parallelism(C.byref(dev), b, m, n, C.byref(v)),
           "tiles_finish_parallelism")
    return v


def c0_bytes(m, n, k, bm, bn, in_bytes=2, out_bytes=None, b=1) -> float:
    if out_bytes is None:
        out_bytes = in_bytes
    return load().tiles_c0_bytes(b, m, n, k, bm, bn, in_bytes, out_bytes)


def plan(m: int, n: int, k: int, b: int = 1, in_dtype: str = "f16", out_dtype: str | None = None,
         mode: str = "gb300", instr: str = "tcgen05", device: _abi.Device | None = None,
         capacity: int | None = None):
    """Ranked feasible verdicts (best first) and the count of feasible ones."""
    lib = load()
    if device is None:
        device = device_preset("gb300" if mode == "gb300" else "h100_pages")
    p = _abi.Problem()
    p.b, p.m, p.n, p.k = b, m, n, k
    p.in_dtype = _abi.DTYPE_CODES[in_dtype]
    p.out_dtype = _abi.DTYPE_CODES[out_dtype or in_dtype]
    p.instr = _abi.INSTR_CODES[instr]
    p.mode = {"pages": _abi.MODE_PAGES, "gb300": _abi.MODE_GB300}[mode]
    nf = C.c_int(0)
    _check(lib.tiles_plan(C.byref(device), C.byref(p), None, 0, C.byref(nf)), "tiles_plan")
    cap = nf.value if capacity is None else min(capacity, nf.value)
    out = (_abi.Verdict * max(cap, 1))()
    _check(lib.tiles_plan(C.byref(device), C.byref(p), out, cap, C.byref(nf)), "tiles_plan")
    return list(out[:cap]), nf.value


def gemm_variants() -> list:
    """The compiled GEMM kernel variants as configurations (no GPU needed)."""
    lib = load()
    out = []
    for i in range(lib.tiles_gemm_variant_count()):
        c = _abi.Config()
        _check(lib.tiles_gemm_variant(i, C.byref(c)), "tiles_gemm_variant")
        out.append(c)
    return out


def gemm_variant_info(index: int) -> _abi.VariantInfo:
    """What the CUDA runtime reports for compiled variant `index` on the
    current device: registers, shared memory, resident blocks and groups."""
    info = _abi.VariantInfo()
    _check(load().tiles_gemm_variant_info(index, C.byref(info)), "tiles_gemm_variant_info")
    return info


def htile_rows(H, kh, sh, pt, d, o0, o1) -> _abi.HTile:
    t = _abi.HTile()
    _check(load().tiles_htile_rows(H, kh, sh, pt, d, o0, o1, C.byref(t)), "tiles_htile_rows")
    return t


def workspace_bytes() -> int:
    return int(load().tiles_workspace_bytes())


# ---- kernels (need torch and a GPU) --------------------------------------------


_TORCH = None
_DTYPE_CODES = None
_RAW_STREAM = None


def _torch():
    global _TORCH
    if _TORCH is None:
        import torch
        _TORCH = torch
    return _TORCH


def _dtype_code(t) -> int:
    global _DTYPE_CODES
    if _DTYPE_CODES is None:
        torch = _torch()
        _DTYPE_CODES = {torch.float16: _abi.F16, torch.bfloat16: _abi.BF16,
                        torch.float32: _abi.F32}
    code = _DTYPE_CODES.get(t.dtype)
    if code is None:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return code


def _stream_handle(stream):
    """The CUDA stream handle of `stream`, or of the current device's current
    stream.  The latter is read through torch's raw-stream query where it
    exists (torch.cuda.current_stream() builds a Python object per call)."""
    global _RAW_STREAM
    if stream is not None:
        return C.c_void_p(stream.cuda_stream)
    if _RAW_STREAM is None:
        tc = _torch()._C
        if hasattr(tc, "_cuda_getCurrentRawStream") and hasattr(tc, "_cuda_getDevice"):
            get, dev = tc._cuda_getCurrentRawStream, tc._cuda_getDevice
            _RAW_STREAM = lambda: get(dev())
        else:
            cur = _torch().cuda.current_stream
            _RAW_STREAM = lambda: cur().cuda_stream
    return C.c_void_p(_RAW_STREAM())


def workspace(device=None):
    """A zeroed workspace tensor for the kernels' error word."""
    torch = _torch()
    return torch.zeros(workspace_bytes(), dtype=torch.uint8,
                       device=device if device is not None else "cuda")


def _cfg_ptr(cfg):
    return C.byref(cfg) if cfg is not None else None


def _check_operand(t, name):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.stride(-1) != 1:
        raise ValueError(f"{name} must have unit stride in its last dimension")


def _gemm_desc(a, b, out, batched: bool) -> _abi.GemmDesc:
    sa, sb, sc = a.stride(), b.stride(), out.stride()
    if not (a.is_cuda and b.is_cuda and out.is_cuda) or sa[-1] != 1 or sb[-1] != 1 or sc[-1] != 1:
        for t, nm in ((a, "a"), (b, "b"), (out, "out")):
            _check_operand(t, nm)
    ha, hb, hc = a.shape, b.shape, out.shape
    m, k, n = ha[-2], ha[-1], hb[-1]
    if hb[-2] != k or hc[-2] != m or hc[-1] != n:
        raise ValueError(f"shape mismatch: {tuple(ha)} x {tuple(hb)} -> {tuple(hc)}")
    d = _abi.GemmDesc()
    d.m, d.n, d.k = m, n, k
    d.batch = ha[0] if batched else 1
    d.a, d.b, d.c = a.data_ptr(), b.data_ptr(), out.data_ptr()
    d.lda, d.ldb, d.ldc = sa[-2], sb[-2], sc[-2]
    if batched:
        if hb[0] != d.batch or hc[0] != d.batch:
            raise ValueError("batch sizes differ")
        d.stride_a, d.stride_b, d.stride_c = sa[0], sb[0], sc[0]
    d.a_dtype, d.b_dtype, d.c_dtype = _dtype_code(a), _dtype_code(b), _dtype_code(out)
    return d


def _alloc_out(shape, like, out_dtype):
    torch = _torch()
    dt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16,
          None: like.dtype}[out_dtype] if not isinstance(out_dtype, torch.dtype) else out_dtype
    return torch.empty(shape, dtype=dt, device=like.device)


def gemm(a, b, out=None, out_dtype=None, cfg=None, workspace=None, stream=None):
    """out = a @ b for 2-D row-major CUDA tensors (fp16/bf16 in)."""
    if out is None:
        out = _alloc_out((a.shape[0], b.shape[1]), a, out_dtype)
    d = _gemm_desc(a, b, out, batched=False)
    ws = workspace.data_ptr() if workspace is not None else None
    wsb = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load().tiles_gemm(C.byref(d), _cfg_ptr(cfg), ws, wsb, _stream_handle(stream)),
           "tiles_gemm")
    return out


def gemm_autotune(a, b, out, top_k=4, reps=5, workspace=None, stream=None, batched=None):
    """Time the planner's top_k configurations for out = a @ b (each with
    every last-round schedule it admits) and record the fastest as the tuned
    configuration of the problem, which later calls with cfg=None use.
    Overwrites `out`.  Returns (best Config, list of per-candidate dicts)."""
    if batched is None:
        batched = a.dim() == 3
    d = _gemm_desc(a, b, out, batched=batched)
    ws = workspace.data_ptr() if workspace is not None else None
    wsb = workspace.numel() * workspace.element_size() if workspace is not None else 0
    cap = 3 * top_k
    res = (_abi.TuneResult * cap)()
    n = C.c_int(0)
    best = _abi.Config()
    _check(load().tiles_gemm_autotune(C.byref(d), top_k, reps, ws, wsb, _stream_handle(stream),
                                      res, cap, C.byref(n), C.byref(best)),
           "tiles_gemm_autotune")
    rows = []
    for r in res[:min(n.value, cap)]:
        rows.append({"bm": r.cfg.bm, "bn": r.cfg.bn, "stages": r.cfg.stages,
                     "cta_group": r.cfg.cta_group, "tail_asked": r.cfg.tail,
                     "tail_mode": ["none", "n_halves", "k_split"][r.tail_mode],
                     "ksplit": r.ksplit, "status": r.status, "us": r.us})
    return best, rows


def tuned_lookup(sm_count, b, m, n, k, in_dtype, out_dtype):
    """The tuned Config of a problem (dtypes as "f16"/"bf16"/"f32" or codes),
    or None."""
    in_dtype = _abi.DTYPE_CODES.get(in_dtype, in_dtype)
    out_dtype = _abi.DTYPE_CODES.get(out_dtype, out_dtype)
    cfg = _abi.Config()
    s = load().tiles_tuned_lookup(sm_count, b, m, n, k, in_dtype, out_dtype, C.byref(cfg))
    if s == _abi.ERR_INFEASIBLE:
        return None
    _check(s, "tiles_tuned_lookup")
    return cfg


def tuned_save(path):
    _check(load().tiles_tuned_save(os.fsencode(path)), "tiles_tuned_save")


def tuned_load(path):
    _check(load().tiles_tuned_load(os.fsencode(path)), "tiles_tuned_load")


def tuned_clear():
    _check(load().tiles_tuned_clear(), "tiles_tuned_clear")


def gemm_batched(a, b, out=None, out_dtype=None, cfg=None, workspace=None, stream=None):
    """out[t] = a[t] @ b[t] for 3-D CUDA tensors."""
    if out is None:
        out = _alloc_out((a.shape[0], a.shape[1], b.shape[2]), a, out_dtype)
    d = _gemm_desc(a, b, out, batched=True)
    ws = workspace.data_ptr() if workspace is not None else None
    wsb = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load().tiles_gemm_batched(C.byref(d), _cfg_ptr(cfg), ws, wsb, _stream_handle(stream)),
           "tiles_gemm_batched")
    return out


def _mirror(host, dev, nm):
    """A host tensor that mirrors a device tensor (same shape, dtype, strides)."""
    if host.is_cuda or tuple(host.shape) != tuple(dev.shape) or host.dtype != dev.dtype \
            or host.stride() != dev.stride():
        raise ValueError(f"{nm}: the host tensor must mirror its device tensor "
                         "(same shape, dtype and strides, in host memory)")


def gemm_host(a_host, b_host, out_host, a_dev, b_dev, out_dev, cfg=None, workspace=None,
              stream=None, chunks=4):
    """out_host = a_host @ b_host (2-D, or 3-D batched) through the device
    buffers a_dev, b_dev, out_dev: uploads, GEMMs and downloads in `chunks`
    overlapping pieces (tiles_gemm_host).  Host tensors should be pinned."""
    for h, dv, nm in ((a_host, a_dev, "a"), (b_host, b_dev, "b"), (out_host, out_dev, "out")):
        _mirror(h, dv, nm)
    d = _gemm_desc(*_batched3(a_dev, b_dev, out_dev), batched=True)
    ws = workspace.data_ptr() if workspace is not None else None
    wsb = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load().tiles_gemm_host(C.byref(d), _cfg_ptr(cfg), a_host.data_ptr(), b_host.data_ptr(),
                                  out_host.data_ptr(), chunks, ws, wsb, _stream_handle(stream)),
           "tiles_gemm_host")
    return out_host


def conv2d_host(x_host, w_host, y_host, x_dev, w_dev, y_dev, stride=(1, 1), pad=(0, 0),
                dil=(1, 1), tile_oh=16, cfg=None, workspace=None, stream=None, layout="nchw",
                chunks=4):
    """y_host = conv2d(x_host, w_host) through the device buffers x_dev, w_dev,
    y_dev: uploads, convolutions and downloads in `chunks` overlapping runs
    of images (tiles_conv2d_host).  Host tensors should be pinned."""
    for h, dv, nm in ((x_host, x_dev, "x"), (w_host, w_dev, "w"), (y_host, y_dev, "y")):
        _mirror(h, dv, nm)
    d = _conv_desc(x_dev, w_dev, stride, pad, dil, y_dev, layout)
    ws = workspace.data_ptr() if workspace is not None else None
    wsb = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load().tiles_conv2d_host(C.byref(d), tile_oh, _cfg_ptr(cfg), x_host.data_ptr(),
                                    w_host.data_ptr(), y_host.data_ptr(), chunks, ws, wsb,
                                    _stream_handle(stream)),
           "tiles_conv2d_host")
    return y_host


_OUT_HW = {}


def conv_out_hw(h, w, kh, kw, stride, pad, dil):
    """Output height and width of a convolution (tiles_conv_out_hw; the
    library's answer is kept per geometry, so repeated calls skip it)."""
    key = (h, w, kh, kw, tuple(stride), tuple(pad), tuple(dil))
    hit = _OUT_HW.get(key)
    if hit is not None:
        return hit
    d = _abi.ConvDesc()
    d.n, d.c, d.h, d.w, d.c_out, d.kh, d.kw = 1, 1, h, w, 1, kh, kw
    d.sh, d.sw = stride
    d.ph, d.pw = pad
    d.dh, d.dw = dil
    oh, ow = C.c_int32(0), C.c_int32(0)
    _check(load().tiles_conv_out_hw(C.byref(d), C.byref(oh), C.byref(ow)), "tiles_conv_out_hw")
    if len(_OUT_HW) < 4096:
        _OUT_HW[key] = (oh.value, ow.value)
    return oh.value, ow.value


def _conv_desc(x, w, stride, pad, dil, out, layout):
    for t, nm in ((x, "x"), (w, "w")):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{nm} must be a contiguous CUDA tensor")
    if layout == "nchw":
        n, c, h, wd = x.shape
    elif layout == "nhwc":
        n, h, wd, c = x.shape
    else:
        raise ValueError(f"unknown layout {layout!r}")
    co, c2, kh, kw = w.shape
    if c2 != c:
        raise ValueError("channel mismatch")
    d = _abi.ConvDesc()
    d.n, d.c, d.h, d.w = n, c, h, wd
    d.c_out, d.kh, d.kw = co, kh, kw
    d.sh, d.sw = stride
    d.ph, d.pw = pad
    d.dh, d.dw = dil
    d.in_dtype = _dtype_code(x)
    if _dtype_code(w) != d.in_dtype:
        raise TypeError("x and w must share a dtype")
    d.x_layout = _abi.LAYOUT_NHWC if layout == "nhwc" else _abi.LAYOUT_NCHW
    d.x, d.wt = x.data_ptr(), w.data_ptr()
    if out is not None:
        d.y = out.data_ptr()
        d.out_dtype = _dtype_code(out)
    return d


def conv_out_shape(x, w, stride=(1, 1), pad=(0, 0), dil=(1, 1), layout="nchw"):
    n, c, h, wd = x.shape if layout == "nchw" else (x.shape[0], x.shape[3], x.shape[1], x.shape[2])
    co, _, kh, kw = w.shape
    oh, ow = conv_out_hw(h, wd, kh, kw, stride, pad, dil)
    return (n, co, oh, ow)


def conv_workspace(x, w, stride=(1, 1), pad=(0, 0), dil=(1, 1), tile_oh=16, layout="nchw"):
    """A zeroed workspace for the TMA im2col producer of this convolution."""
    torch = _torch()
    d = _conv_desc(x, w, stride, pad, dil, None, layout)
    nbytes = int(load().tiles_conv_workspace_bytes(C.byref(d), tile_oh))
    if nbytes == 0:
        raise ValueError("invalid convolution arguments")
    return torch.zeros(nbytes, dtype=torch.uint8, device=x.device)


def conv2d_htiled(x, w, stride=(1, 1), pad=(0, 0), dil=(1, 1), tile_oh=16, out=None,
                  out_dtype=None, cfg=None, workspace=None, stream=None, layout="nchw"):
    """conv2d with OIHW weights and NCHW output, as an implicit GEMM per output
    H-tile; x is NCHW or NHWC (layout).  With a workspace of conv_workspace
    size the im2col operand is built by TMA, else gathered by threads."""
    shape = conv_out_shape(x, w, stride, pad, dil, layout)
    if out is None:
        out = _alloc_out(shape, x, out_dtype)
    if not out.is_contiguous() or tuple(out.shape) != shape:
        raise ValueError("out must be contiguous with shape (n, c_out, oh, ow)")
    d = _conv_desc(x, w, stride, pad, dil, out, layout)
    ws = workspace.data_ptr() if workspace is not None else None
    wsb = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load().tiles_conv2d_htiled(C.byref(d), tile_oh, _cfg_ptr(cfg), ws, wsb,
                                      _stream_handle(stream)), "tiles_conv2d_htiled")
    return out


def conv2d_tiled(x, w, stride=(1, 1), pad=(0, 0), dil=(1, 1), tile_oh=16, tile_ow=0, tile_n=0,
                 out=None, out_dtype=None, cfg=None, workspace=None, stream=None, layout="nchw"):
    """conv2d tiled over the batch (tile_n images, no halo), the output
    height (tile_oh rows) and the output width (tile_ow columns, the same
    slicing formulas as the rows); 0 means the whole batch or width."""
    shape = conv_out_shape(x, w, stride, pad, dil, layout)
    if out is None:
        out = _alloc_out(shape, x, out_dtype)
    if not out.is_contiguous() or tuple(out.shape) != shape:
        raise ValueError("out must be contiguous with shape (n, c_out, oh, ow)")
    d = _conv_desc(x, w, stride, pad, dil, out, layout)
    ws = workspace.data_ptr() if workspace is not None else None
    wsb = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load().tiles_conv2d_tiled(C.byref(d), tile_oh, tile_ow, tile_n, _cfg_ptr(cfg), ws,
                                     wsb, _stream_handle(stream)), "tiles_conv2d_tiled")
    return out


def _batched3(a, b, out):
    if a.dim() == 2:
        return a.unsqueeze(0), b.unsqueeze(0), out.unsqueeze(0)
    return a, b, out


def gemm_schedule(a, b, out, cfg=None, workspace=None):
    """The launch geometry a GEMM call with this workspace would use (2-D
    tensors count as a batch of one)."""
    d = _gemm_desc(*_batched3(a, b, out), batched=True)
    sch = _abi.Schedule()
    wsb = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load().tiles_gemm_schedule(C.byref(d), _cfg_ptr(cfg), wsb, C.byref(sch)),
           "tiles_gemm_schedule")
    return sch


def gemm_workspace(a, b, out, cfg=None):
    """A zeroed workspace large enough for this GEMM's schedule under cfg (the
    partial tiles of a K-split last round, when that is the schedule)."""
    torch = _torch()
    d = _gemm_desc(*_batched3(a, b, out), batched=True)
    n = int(load().tiles_gemm_workspace_bytes(C.byref(d), _cfg_ptr(cfg)))
    if n == 0:
        # The call returns 0 on invalid arguments; tiles_last_error says why.
        raise TilesError(_abi.ERR_INVALID_ARG, "tiles_gemm_workspace_bytes")
    return torch.zeros(n, dtype=torch.uint8, device=a.device)


def gemm_noalloc(a, b, out=None, out_dtype=None, cfg=None, stream=None, wait=False):
    """out[t] = a[t] @ b[t] (3-D tensors) without a workspace: for callers
    that cannot allocate device memory.  The library's static scratch takes
    the workspace's place; wait=True synchronises and reports a timeout."""
    if out is None:
        out = _alloc_out((a.shape[0], a.shape[1], b.shape[2]), a, out_dtype)
    d = _gemm_desc(a, b, out, batched=True)
    _check(load().tiles_gemm_noalloc(C.byref(d), _cfg_ptr(cfg), _stream_handle(stream),
                                     1 if wait else 0), "tiles_gemm_noalloc")
    return out


def check(workspace=None, stream=None) -> None:
    """Synchronise and raise TilesError if a kernel's bounded wait expired."""
    ws = workspace.data_ptr() if workspace is not None else None
    _check(load().tiles_check(ws, _stream_handle(stream)), "tiles_check")


def selftest_wait_timeout(workspace, limit_ns: int, stream=None) -> None:
    _check(load().tiles_selftest_wait_timeout(workspace.data_ptr(), limit_ns,
                                              _stream_handle(stream)),
           "tiles_selftest_wait_timeout")


def selftest_drop_stage(stage: int, limit_ns: int) -> None:
    """Arm a planted fault for this thread's next GEMM or TMA convolution
    launch (tiles_selftest_drop_stage); stage < 0 disarms."""
    _check(load().tiles_selftest_drop_stage(stage, limit_ns), "tiles_selftest_drop_stage")
