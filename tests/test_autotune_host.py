"""The tuned-configuration table on the host: file format, merge and
rejection rules of tiles_tuned_save / tiles_tuned_load (no GPU needed)."""
import pytest

import synth_inputs as S
import tile_size_decision_gb300 as T
from tile_size_decision_gb300 import _abi

HEADER = "tiles-tuned 1\n"
# sm_count batch m n k in out | bm bn bk stages threads instr acc_bufs cta_group tail | us
LINE_A = "152 1 4096 4096 4096 {f16} {f16} 256 256 64 6 192 3 2 2 3 85.600\n"
LINE_B = "148 16 2048 2048 1024 {bf16} {bf16} 128 256 64 4 192 3 2 1 1 101.250\n"


def fmt(line):
    return line.format(f16=_abi.F16, bf16=_abi.BF16)


@pytest.fixture(autouse=True)
def clean_table():
    T.load()
    T.tuned_clear()
    yield
    T.tuned_clear()


def test_load_then_lookup(tmp_path):
    p = tmp_path / "tuned.txt"
    p.write_text(HEADER + fmt(LINE_A) + "\n" + fmt(LINE_B))
    T.tuned_load(str(p))
    a = T.tuned_lookup(152, 1, 4096, 4096, 4096, S.F16, S.F16)
    assert (a.bm, a.bn, a.bk, a.stages, a.cta_group, a.tail) == (256, 256, 64, 6, 2, 3)
    b = T.tuned_lookup(148, 16, 2048, 2048, 1024, S.BF16, S.BF16)
    assert (b.bm, b.bn, b.stages, b.cta_group, b.tail) == (128, 256, 4, 1, 1)
    # Another SM count is another problem.
    assert T.tuned_lookup(148, 1, 4096, 4096, 4096, S.F16, S.F16) is None


def test_save_round_trip(tmp_path):
    src = tmp_path / "a.txt"
    src.write_text(HEADER + fmt(LINE_B) + fmt(LINE_A))
    T.tuned_load(str(src))
    out = tmp_path / "b.txt"
    T.tuned_save(str(out))
    text = out.read_text().splitlines()
    assert text[0] == HEADER.strip()
    assert sorted(text[1:]) == sorted([fmt(LINE_A).strip(), fmt(LINE_B).strip()])
    T.tuned_clear()
    assert T.tuned_lookup(152, 1, 4096, 4096, 4096, S.F16, S.F16) is None
    T.tuned_load(str(out))
    assert T.tuned_lookup(152, 1, 4096, 4096, 4096, S.F16, S.F16) is not None


@pytest.mark.parametrize("bad", [
    "152 1 4096 4096 4096 {f16} {f16} 256 256 64 7 192 3 2 2 3\n",          # missing time
    "152 1 4096 4096 4096 {f16} {f16} 256 256 64 7 192 3 2 2 3 85.6 9\n",   # extra field
    "152 0 4096 4096 4096 {f16} {f16} 256 256 64 7 192 3 2 2 3 85.6\n",     # batch 0
    "152 1 4096 4096 4096 {f16} {f16} 256 256 64 7 192 3 2 5 3 85.6\n",     # cta_group 5
    "152 1 4096 4096 4096 {f16} {f16} 256 256 64 7 192 3 2 2 9 85.6\n",     # tail 9
    "152 1 4096 4096 4096 77 {f16} 256 256 64 7 192 3 2 2 3 85.6\n",        # dtype 77
])
def test_malformed_line_merges_nothing(tmp_path, bad):
    p = tmp_path / "bad.txt"
    p.write_text(HEADER + fmt(LINE_B) + fmt(bad))
    with pytest.raises(T.TilesError) as e:
        T.tuned_load(str(p))
    assert e.value.status == -1
    assert T.tuned_lookup(148, 16, 2048, 2048, 1024, S.BF16, S.BF16) is None


def test_header_and_missing_file(tmp_path):
    p = tmp_path / "nohdr.txt"
    p.write_text(fmt(LINE_A))
    with pytest.raises(T.TilesError):
        T.tuned_load(str(p))
    with pytest.raises(T.TilesError):
        T.tuned_load(str(tmp_path / "absent.txt"))
    empty = tmp_path / "empty.txt"
    empty.write_text("")
    with pytest.raises(T.TilesError):
        T.tuned_load(str(empty))
