"""The split table's reader and writer (paged_kv_cache_forward_gb300/sweep.py) on
the CPU: parsing the committed table and writing it back gives the same rows, so
a partial re-sweep (--merge) replaces only the cells it measured."""

import os
import tempfile

from paged_kv_cache_forward_gb300 import sweep as S

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TABLE = os.path.join(ROOT, "paged_kv_cache_forward_gb300", "csrc", "lut_gb300.inc")


def _rows(path):
    return [line for line in open(path) if line.startswith("    {")]


def _first_array_rows(path):
    text = open(path).read()
    return [line for line in text[:text.index("};")].splitlines(True) if line.startswith("    {")]


def test_table_round_trip():
    cells, wide = S.read_table(TABLE), S.read_table(TABLE, S.WIDE_NAME)
    assert cells and {k[0] for k in cells} == {64, 128, 256}
    with tempfile.TemporaryDirectory() as d:
        out = os.path.join(d, "t.inc")
        S.write_table(out, cells, "test", "today", wide)
        assert _rows(out) == _rows(TABLE)
        assert S.read_table(out, S.WIDE_NAME) == wide


def test_every_head_dim_ends_with_a_catch_all():
    rows = [r.strip() for r in _first_array_rows(TABLE)]
    for d in (64, 128, 256):
        mine = [r for r in rows if r.startswith(f"{{{d}, ")]
        assert mine[-1].startswith(f"{{{d}, 1 << 30, 1 << 30, ")


def test_merge_replaces_one_cell():
    cells, wide = S.read_table(TABLE), S.read_table(TABLE, S.WIDE_NAME)
    key = (128, 4096, 8)  # (head dim, bound, decode units)
    new = (48, 4, 4, 1) if cells[key] != (48, 4, 4, 1) else (64, 4, 4, 1)
    merged = dict(cells)
    merged[key] = new
    with tempfile.TemporaryDirectory() as d:
        out = os.path.join(d, "t.inc")
        S.write_table(out, merged, "test", "today", wide)
        a, b = _rows(TABLE), _rows(out)
        diff = [(x, y) for x, y in zip(a, b) if x != y]
        assert len(a) == len(b) and len(diff) == 1
        assert diff[0][1].strip() == f"{{128, 4096, 8, {new[0]}, 4, 4, 1}},"


def test_wide_rows_are_a_second_array():
    """Cells for more than 16 query heads per KV head go to kSplitTableWide (which
    always ends with a head-dim-0 row), not into the first table."""
    cells = S.read_table(TABLE)
    wide = {(128, 8192, 2): (1024, 3, 8, 1), (128, 32768, 2): (1024, 3, 8, 1)}
    with tempfile.TemporaryDirectory() as d:
        out = os.path.join(d, "t.inc")
        S.write_table(out, cells, "test", "today", wide)
        assert S.read_table(out) == cells
        assert S.read_table(out, S.WIDE_NAME) == wide
        text = open(out).read()
        second = text[text.index(S.WIDE_NAME):]
        assert "{128, 1 << 30, 1 << 30, 1024, 3, 8, 1}," in second
        assert second.rstrip().endswith("{0, 0, 0, 0, 0, 0, 0},\n};")
