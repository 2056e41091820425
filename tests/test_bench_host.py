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


def test_rotation_keeps_each_steps_inputs_out_of_l2():
    # Between two uses of one operand copy the other copies pass through L2:
    # at least twice its capacity, whatever the size of one copy.
    import synth_inputs as S
    for set_bytes in (1, 2 << 20, 77_217_792, 100_663_296, 125_536_000, 129 << 20,
                      268_435_456, 1 << 34):
        r = bench.rotation_sets(set_bytes)
        assert r >= 2
        assert (r - 1) * set_bytes >= 2 * bench.L2_BYTES or r == 2 and set_bytes >= 2 * bench.L2_BYTES
        # No more copies than that needs.
        assert r == 2 or (r - 2) * set_bytes < 2 * bench.L2_BYTES
    # The seeded workloads' copies, as the bench counts them.
    gemm = S.WORKLOADS["gemm_4096"]
    one = gemm.b * (gemm.m * gemm.k + gemm.k * gemm.n) * 2 + gemm.b * gemm.m * gemm.n * 2
    assert bench.rotation_sets(one) == 4


class _FakeJob:
    def __init__(self):
        self.calls = []
        self.sets = [0, 1, 2]

    def step(self, i, stream):
        self.calls.append(i % len(self.sets))


def test_timed_steps_continue_the_rotation_from_the_warm_up(monkeypatch):
    # timed_rotating runs steps start .. start + K - 1, so that the first
    # timed step uses the copy after the warm-up's last one.
    import types
    events = []

    class Ev:
        def __init__(self, enable_timing=False):
            self.t = None

        def record(self, stream=None):
            self.t = len(events)
            events.append(self)

        def elapsed_time(self, other):
            return 6.0

    fake_torch = types.SimpleNamespace(cuda=types.SimpleNamespace(Event=Ev, synchronize=lambda: None))
    monkeypatch.setitem(__import__("sys").modules, "torch", fake_torch)
    job = _FakeJob()
    ms, (t0, t1) = bench.timed_rotating(job, None, 4, start=5)
    assert job.calls == [2, 0, 1, 2]
    assert ms == 1.5 and t1 >= t0
