"""CPU oracle for the tiled GEMM, the H-tiled convolution and the tile planner.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call, link
or execute anything in this package: only the tests, the smoke check and the
benchmark's CPU-baseline leg use it.  It shares no code with the CUDA library
(no kernels, headers, helpers, tables or constants); the only module both
sides use is ``synth_inputs``, which draws and rounds random inputs and holds
none of the method's arithmetic.

Contents
  planner   constraint procedure C0-C4 and the sweep, restated from the page
            "04-tile-size-decision/tile_decision.py" (device, config and
            verdict records; functions evaluate, finish_parallelism,
            dram_traffic, sweep) and its README (C0 with the batch term b).
            The GB300 mode in ``planner_gb300`` is this library's own
            extension: parity unpinned (no page value fixes it).
  gemm      float64 GEMM C = A x B and the bound sum_k |A||B| (the tiling
            tutorial's problem statement C = A x B).
  conv      H-tile row formulas (tutorial section "H/W 维切分的通用公式") and a
            direct float64 convolution, untiled and H-tiled.
  tolerance the pass criterion |C - C_ref| <= 1e-3 * S + ulp_out(C_ref).
"""
