"""Host logic of bench.py that decides what a bench line reports (no GPU)."""

import os

import bench


def test_code_only_drops_comments_and_collapses_whitespace():
    src = "int a = 1; // one\n/* block\n comment */ int  b =\n 2;\n"
    assert bench.code_only(src) == "int a = 1; int b = 2;"


def test_source_hash_ignores_comment_edits_but_not_code_edits():
    csrc = os.path.join(os.path.dirname(bench.__file__), "tile_size_decision_gb300", "csrc")

    def read(name):
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            return f.read()

    base = bench.kernel_source_hash("gemm_4096", read)
    assert base == bench.kernel_source_hash("gemm_4096")
    commented = lambda name: read(name) + ("\n// a note\n/* another */\n" if name == "api.cu" else "")
    assert bench.kernel_source_hash("gemm_4096", commented) == base
    edited = lambda name: read(name) + ("\nstatic int unused_edit = 1;\n" if name == "api.cu" else "")
    assert bench.kernel_source_hash("gemm_4096", edited) != base
    # The convolution's figure depends on its own sources, not the GEMM's API file.
    assert bench.kernel_source_hash("conv_htiled", edited) == bench.kernel_source_hash("conv_htiled")


def test_recorded_traffic_needs_a_matching_hash(tmp_path, monkeypatch):
    rec = tmp_path / "profiles"
    rec.mkdir()
    (rec / "traffic_gemm_4096.txt").write_text(
        "# note\nsource_hash = 0000000000000000\ndram_bytes_per_launch = 123\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda wl: "0000000000000000")
    assert bench.recorded_traffic("gemm_4096") == 123
    monkeypatch.setattr(bench, "kernel_source_hash", lambda wl: "1111111111111111")
    assert bench.recorded_traffic("gemm_4096") is None
    assert bench.recorded_traffic("conv_htiled") is None


def test_clock_summary_keeps_only_the_samples_of_its_window():
    lines = [f"2026/12/02 14:41:0{i}.250, 0, {2000 - 100 * i}, 2070, 1000, 0x0, Not Active, "
             f"Not Active, {'Active' if i == 3 else 'Not Active'}, Not Active" for i in range(5)]
    rows = bench.parse_clock_rows("\n".join(lines) + "\nmalformed,row\n")
    assert len(rows) == 5
    t = [r["t"] for r in rows]
    assert all(b - a == 1.0 for a, b in zip(t, t[1:]))
    s = bench.summarize_clocks(rows, t[1], t[2])
    assert (s["samples"], s["sm_mhz"], s["sm_max_mhz"], s["reasons"]) == (2, 1850.0, 2070.0, [])
    assert bench.summarize_clocks(rows)["reasons"] == ["sw_thermal_slowdown"]
    assert bench.summarize_clocks(rows, t[4] + 1, t[4] + 2)["samples"] == 0


def test_both_arms_describe_each_workload_alike():
    # The reference arm and this library's arm build their line's config
    # from the same description of the workload.
    import synth_inputs as S
    for name, wl in S.WORKLOADS.items():
        c = bench.workload_config(wl, 2)
        assert (c["workload"], c["seed"], c["accumulate"]) == (name, wl.seed, "f32")
        assert c["parallelism"] == "replicas x2" and "tile" not in c
        assert c == bench.workload_config(wl, 2)
