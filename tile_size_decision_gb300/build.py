"""Build libtiles.so in-tree with nvcc for sm_103a (no cmake).

    python -m tile_size_decision_gb300.build [-v] [--force]

Each translation unit compiles in parallel into ``_build/``; the GEMM source
compiles once per (tile width, CTAs per MMA).  Objects newer than every source and header
are reused.  The shared library links the CUDA runtime statically and looks
up the driver at run time, so it loads on machines without a GPU.
"""

from __future__ import annotations

import argparse
import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libtiles.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
          "--expt-relaxed-constexpr"]
GEMM_VARIANTS = ((64, 1), (128, 1), (192, 1), (256, 1), (128, 2), (256, 2))


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found; the CUDA toolkit is required to build libtiles")
    return path


def units():
    """(source, object, extra flags) of every translation unit."""
    out = [
        ("planner.cpp", "planner.o", []),
        ("api.cu", "api.o", []),
        ("conv_sm103a.cu", "conv_sm103a.o", []),
        ("conv_tma_sm103a.cu", "conv_tma_sm103a.o", []),
        ("host_pipeline.cu", "host_pipeline.o", []),
    ]
    for bn, cg in GEMM_VARIANTS:
        out.append(("gemm_sm103a.cu", f"gemm_bn{bn}_cg{cg}.o",
                    [f"-DTILES_GEMM_BN={bn}", f"-DTILES_GEMM_CG={cg}"]))
    return out


def _headers_mtime() -> float:
    files = glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))
    return max(os.path.getmtime(f) for f in files)


def _compile(src: str, obj: str, extra: list, force: bool, verbose: bool) -> str:
    src_path = os.path.join(CSRC, src)
    obj_path = os.path.join(BUILD, obj)
    if not force and os.path.exists(obj_path):
        newest = max(os.path.getmtime(src_path), _headers_mtime())
        if os.path.getmtime(obj_path) >= newest:
            return obj_path
    cmd = [nvcc(), *ARCH, *COMMON, *extra, "-c", src_path, "-o", obj_path]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
        print(" ".join(cmd), flush=True)
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src} ({obj}):\n{res.stdout}\n{res.stderr}")
    if verbose and (res.stdout or res.stderr):
        print(res.stdout + res.stderr, flush=True)
    return obj_path


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile every unit and link libtiles.so; return its path."""
    os.makedirs(BUILD, exist_ok=True)
    jobs = min(len(units()), max(1, os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(max_workers=jobs) as ex:
        futs = [ex.submit(_compile, s, o, e, force, verbose) for s, o, e in units()]
        objs = [f.result() for f in futs]
    if force or not os.path.exists(LIB) or \
            os.path.getmtime(LIB) < max(os.path.getmtime(o) for o in objs):
        tmp = LIB + ".tmp"
        cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs,
               "-ldl", "-lpthread", "-lrt"]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
        os.replace(tmp, LIB)
    return LIB


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("-v", "--verbose", action="store_true", help="print commands and ptxas usage")
    ap.add_argument("--force", action="store_true", help="rebuild every unit")
    args = ap.parse_args(argv)
    print(build(force=args.force, verbose=args.verbose))
    return 0


if __name__ == "__main__":
    sys.exit(main())
