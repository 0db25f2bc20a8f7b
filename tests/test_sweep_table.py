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


def test_table_round_trip():
    cells = S.read_table(TABLE)
    assert cells and {k[0] for k in cells} == {64, 128, 256}
    with tempfile.TemporaryDirectory() as d:
        out = os.path.join(d, "t.inc")
        S.write_table(out, cells, "test", "today")
        assert _rows(out) == _rows(TABLE)


def test_every_head_dim_ends_with_a_catch_all():
    rows = [r.strip() for r in _rows(TABLE)]
    for d in (64, 128, 256):
        mine = [r for r in rows if r.startswith(f"{{{d}, ")]
        assert mine[-1].startswith(f"{{{d}, 1 << 30, 1 << 30, ")


def test_merge_replaces_one_cell():
    cells = S.read_table(TABLE)
    key = (128, 4096, 8)  # (head dim, bound, decode units)
    new = (48, 4, 4, 1) if cells[key] != (48, 4, 4, 1) else (64, 4, 4, 1)
    merged = dict(cells)
    merged[key] = new
    with tempfile.TemporaryDirectory() as d:
        out = os.path.join(d, "t.inc")
        S.write_table(out, merged, "test", "today")
        a, b = _rows(TABLE), _rows(out)
        diff = [(x, y) for x, y in zip(a, b) if x != y]
        assert len(a) == len(b) and len(diff) == 1
        assert diff[0][1].strip() == f"{{128, 4096, 8, {new[0]}, 4, 4, 1}},"
