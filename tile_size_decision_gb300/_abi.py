"""ctypes mirror of include/tiles.h and the loader of libtiles.so.

Argument marshalling only: every step of the planner and the kernels runs in
the native library.  Loading fails loudly when the library has not been
built; there is no Python or CPU fallback.
"""

from __future__ import annotations

import ctypes as C
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libtiles.so")

# tiles_status
OK = 0
ERR_INVALID_ARG = -1
ERR_UNSUPPORTED_DTYPE = -2
ERR_MISALIGNED = -3
ERR_INFEASIBLE = -4
ERR_CUDA = -5
ERR_TIMEOUT = -6
ERR_TOO_LARGE = -7

# tiles_dtype
F16, BF16, F32 = 0, 1, 2
DTYPE_CODES = {"f16": F16, "bf16": BF16, "f32": F32}

# tiles_instr
INSTR_MMA, INSTR_WGMMA, INSTR_SIMT, INSTR_TCGEN05 = 0, 1, 2, 3
INSTR_CODES = {"mma": INSTR_MMA, "wgmma": INSTR_WGMMA, "simt": INSTR_SIMT,
               "tcgen05": INSTR_TCGEN05}

DEV_H100_PAGES, DEV_GB300 = 0, 1
MODE_PAGES, MODE_GB300 = 0, 1

FAIL_C3, FAIL_C1, FAIL_C2, FAIL_OCC = 0x1, 0x2, 0x4, 0x8
WARN_TAIL, WARN_IDLE = 0x1, 0x2
BINDINGS = {0: "", 1: "regs", 2: "smem", 3: "threads", 4: "tmem"}


class Device(C.Structure):
    _fields_ = [(n, C.c_int32) for n in (
        "smem_per_sm", "smem_per_block_max", "regs_per_sm", "max_threads_per_sm",
        "max_threads_per_block", "max_blocks_per_sm", "regs_per_thread_max",
        "reg_granularity_per_warp", "warp_size", "sm_count", "tmem_cols", "mma_flops_per_clk",
        "fill_bytes_per_clk", "kernel_regs_per_thread", "cta_pairs", "partial_bytes_per_clk",
        "handoff_clocks", "pair_launch_clocks")]


class Config(C.Structure):
    _fields_ = [(n, C.c_int32) for n in (
        "bm", "bn", "bk", "stages", "threads", "instr", "acc_bufs", "cta_group", "tail",
        "conv_weights")] + [("reserved", C.c_int32 * 2)]


TAIL_AUTO, TAIL_WHOLE, TAIL_NHALF, TAIL_KSPLIT = 0, 1, 2, 3
CONV_W_AUTO, CONV_W_SMEM, CONV_W_TMEM, CONV_W_TMEM_ROWS, CONV_W_TMEM_ROWS_DIRECT = 0, 1, 2, 3, 4


class Verdict(C.Structure):
    _fields_ = [
        ("cfg", Config),
        ("smem_per_stage", C.c_int64),
        ("smem_total", C.c_int64),
        ("accum_per_thread", C.c_int32),
        ("regs_per_thread", C.c_int32),
        ("regs_per_block", C.c_int32),
        ("blocks_by_regs", C.c_int32),
        ("blocks_by_smem", C.c_int32),
        ("blocks_by_threads", C.c_int32),
        ("blocks_by_tmem", C.c_int32),
        ("blocks_per_sm", C.c_int32),
        ("tmem_cols_alloc", C.c_int32),
        ("binding", C.c_int32),
        ("failures", C.c_uint32),
        ("c3_violations", C.c_int32),
        ("warnings", C.c_uint32),
        ("tail_split", C.c_int32),
        ("grid", C.c_int64),
        ("waves", C.c_int64),
        ("last_wave_fill", C.c_double),
        ("c0_bytes", C.c_double),
        ("est_clocks", C.c_int64),
    ]


class Problem(C.Structure):
    _fields_ = [("b", C.c_int64), ("m", C.c_int64), ("n", C.c_int64), ("k", C.c_int64),
                ("in_dtype", C.c_int32), ("out_dtype", C.c_int32), ("instr", C.c_int32),
                ("mode", C.c_int32)]


class HTile(C.Structure):
    _fields_ = [(n, C.c_int32) for n in ("in_start", "in_end", "in_span", "pt", "pb", "halo")]


class GemmDesc(C.Structure):
    _fields_ = [("m", C.c_int64), ("n", C.c_int64), ("k", C.c_int64), ("batch", C.c_int64),
                ("a", C.c_void_p), ("b", C.c_void_p), ("c", C.c_void_p),
                ("lda", C.c_int64), ("ldb", C.c_int64), ("ldc", C.c_int64),
                ("stride_a", C.c_int64), ("stride_b", C.c_int64), ("stride_c", C.c_int64),
                ("a_dtype", C.c_int32), ("b_dtype", C.c_int32), ("c_dtype", C.c_int32),
                ("pad0", C.c_int32)]


class Schedule(C.Structure):
    _fields_ = [("cfg", Config), ("tiles", C.c_int64), ("resident_groups", C.c_int64),
                ("full_units", C.c_int64), ("units", C.c_int64), ("groups", C.c_int64),
                ("tail_mode", C.c_int32), ("ksplit", C.c_int32), ("workspace_bytes", C.c_int64)]


class VariantInfo(C.Structure):
    _fields_ = [("cfg", Config)] + [(n, C.c_int32) for n in (
        "regs_per_thread", "local_bytes_per_thread", "static_smem_bytes", "dynamic_smem_bytes",
        "max_dynamic_smem_bytes", "blocks_per_sm", "resident_groups")] + \
        [("reserved", C.c_int32 * 5)]


class TuneResult(C.Structure):
    _fields_ = [("cfg", Config), ("status", C.c_int32), ("tail_mode", C.c_int32),
                ("ksplit", C.c_int32), ("us", C.c_float)]


class ConvDesc(C.Structure):
    _fields_ = [(n, C.c_int32) for n in (
        "n", "c", "h", "w", "c_out", "kh", "kw", "sh", "sw", "ph", "pw", "dh", "dw",
        "in_dtype", "out_dtype", "x_layout")] + \
        [("x", C.c_void_p), ("wt", C.c_void_p), ("y", C.c_void_p)]


LAYOUT_NCHW, LAYOUT_NHWC = 0, 1


# Every exported entry point: name -> (restype, argtypes).
SIGNATURES = {
    "tiles_status_string": (C.c_char_p, [C.c_int]),
    "tiles_last_error": (C.c_char_p, []),
    "tiles_version": (C.c_char_p, []),
    "tiles_device_preset": (C.c_int, [C.c_int, C.POINTER(Device)]),
    "tiles_device_query": (C.c_int, [C.c_int, C.POINTER(Device)]),
    "tiles_evaluate": (C.c_int, [C.POINTER(Device), C.POINTER(Config), C.c_int, C.c_int,
                                 C.POINTER(Verdict)]),
    "tiles_finish_parallelism": (C.c_int, [C.POINTER(Device), C.c_int64, C.c_int64, C.c_int64,
                                           C.POINTER(Verdict)]),
    "tiles_c0_bytes": (C.c_double, [C.c_int64, C.c_int64, C.c_int64, C.c_int64, C.c_int, C.c_int,
                                    C.c_int, C.c_int]),
    "tiles_plan": (C.c_int, [C.POINTER(Device), C.POINTER(Problem), C.POINTER(Verdict), C.c_int,
                             C.POINTER(C.c_int)]),
    "tiles_htile_rows": (C.c_int, [C.c_int] * 7 + [C.POINTER(HTile)]),
    "tiles_workspace_bytes": (C.c_size_t, []),
    "tiles_gemm": (C.c_int, [C.POINTER(GemmDesc), C.POINTER(Config), C.c_void_p, C.c_size_t,
                             C.c_void_p]),
    "tiles_gemm_batched": (C.c_int, [C.POINTER(GemmDesc), C.POINTER(Config), C.c_void_p,
                                     C.c_size_t, C.c_void_p]),
    "tiles_gemm_schedule": (C.c_int, [C.POINTER(GemmDesc), C.POINTER(Config), C.c_size_t,
                                      C.POINTER(Schedule)]),
    "tiles_gemm_workspace_bytes": (C.c_size_t, [C.POINTER(GemmDesc), C.POINTER(Config)]),
    "tiles_gemm_variant_count": (C.c_int, []),
    "tiles_gemm_variant": (C.c_int, [C.c_int, C.POINTER(Config)]),
    "tiles_gemm_variant_info": (C.c_int, [C.c_int, C.POINTER(VariantInfo)]),
    "tiles_conv2d_htiled": (C.c_int, [C.POINTER(ConvDesc), C.c_int, C.POINTER(Config),
                                      C.c_void_p, C.c_size_t, C.c_void_p]),
    "tiles_gemm_noalloc": (C.c_int, [C.POINTER(GemmDesc), C.POINTER(Config), C.c_void_p,
                                     C.c_int]),
    "tiles_gemm_host": (C.c_int, [C.POINTER(GemmDesc), C.POINTER(Config), C.c_void_p, C.c_void_p,
                                  C.c_void_p, C.c_int, C.c_void_p, C.c_size_t, C.c_void_p]),
    "tiles_conv2d_host": (C.c_int, [C.POINTER(ConvDesc), C.c_int, C.POINTER(Config), C.c_void_p,
                                    C.c_void_p, C.c_void_p, C.c_int, C.c_void_p, C.c_size_t,
                                    C.c_void_p]),
    "tiles_conv2d_tiled": (C.c_int, [C.POINTER(ConvDesc), C.c_int, C.c_int, C.c_int,
                                     C.POINTER(Config), C.c_void_p, C.c_size_t, C.c_void_p]),
    "tiles_conv_workspace_bytes": (C.c_size_t, [C.POINTER(ConvDesc), C.c_int]),
    "tiles_conv_out_hw": (C.c_int, [C.POINTER(ConvDesc), C.POINTER(C.c_int32),
                                    C.POINTER(C.c_int32)]),
    "tiles_gemm_autotune": (C.c_int, [C.POINTER(GemmDesc), C.c_int, C.c_int, C.c_void_p,
                                      C.c_size_t, C.c_void_p, C.POINTER(TuneResult), C.c_int,
                                      C.POINTER(C.c_int), C.POINTER(Config)]),
    "tiles_tuned_lookup": (C.c_int, [C.c_int, C.c_int64, C.c_int64, C.c_int64, C.c_int64,
                                     C.c_int, C.c_int, C.POINTER(Config)]),
    "tiles_tuned_save": (C.c_int, [C.c_char_p]),
    "tiles_tuned_load": (C.c_int, [C.c_char_p]),
    "tiles_tuned_clear": (C.c_int, []),
    "tiles_check": (C.c_int, [C.c_void_p, C.c_void_p]),
    "tiles_selftest_wait_timeout": (C.c_int, [C.c_void_p, C.c_int64, C.c_void_p]),
    "tiles_selftest_drop_stage": (C.c_int, [C.c_int, C.c_int64]),
}

_lib = None


def load(path: str = LIB_PATH):
    """Load libtiles.so once; raise if it is missing or lacks a symbol."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(
            f"libtiles.so not found at {path}: build it first "
            "(python -m tile_size_decision_gb300.build, or __graft_entry__.build())")
    lib = C.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


class TilesError(RuntimeError):
    def __init__(self, status: int, where: str):
        lib = load()
        name = lib.tiles_status_string(status).decode()
        msg = lib.tiles_last_error().decode()
        super().__init__(f"{where}: {name} ({status}): {msg}")
        self.status = status


def check(status: int, where: str) -> None:
    if status != OK:
        raise TilesError(status, where)
