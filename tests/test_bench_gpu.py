"""bench.py end to end on the GPU: the line it prints for a small and a
bandwidth-bound workload carries the keys the contract asks for, with the
timed steps over rotating operand copies (no oracle sample, no extras)."""

import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("workload", ["gemm_512", "conv_htiled"])
def test_bench_line(workload):
    out = subprocess.run(
        [sys.executable, os.path.join(ROOT, "bench.py"), "--workload", workload, "--steps", "5",
         "--warmup", "3", "--no-cpu-baseline", "--autotune", "0"],
        capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "e2e", "gpu_launches", "clocks", "operand_copies"):
        assert key in line, key
    assert line["value"] > 0 and line["ms_per_step"] > 0
    assert line["steps"] == 5 and line["warmup"] == 3 and line["n_gpus"] == 1
    assert line["gpu_launches"] == 5
    assert line["operand_copies"] >= 2
    roof = line["roofline"]
    assert roof["bound"] == ("hbm" if workload.startswith("conv") else "tensor")
    assert 0 < roof["frac"] < 1.5 and roof["peak"] > 0
    e2e = line["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert line["config"]["workload"] == workload
