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


def _write(cells, path):
    batches = sorted({k[1] for k in cells})
    bounds = sorted({k[0] for k in cells})
    entries = [(bd, bt) + cells[(bd, bt)] for bt in batches for bd in bounds if (bd, bt) in cells]
    fallback = max(entries, key=lambda e: (e[1], e[0]))[2:]
    S.write_table(path, entries, max(batches), fallback, "test", "today")


def test_table_round_trip():
    cells = S.read_table(TABLE)
    assert cells and max(k[1] for k in cells) == max(S.BATCHES)
    with tempfile.TemporaryDirectory() as d:
        out = os.path.join(d, "t.inc")
        _write(cells, out)
        assert _rows(out) == _rows(TABLE)


def test_merge_replaces_one_cell():
    cells = S.read_table(TABLE)
    key = (4096, 1)
    merged = dict(cells)
    merged.update({key: (0, 2, 8, 8)})
    with tempfile.TemporaryDirectory() as d:
        out = os.path.join(d, "t.inc")
        _write(merged, out)
        a, b = _rows(TABLE), _rows(out)
        diff = [(x, y) for x, y in zip(a, b) if x != y]
        assert len(a) == len(b) and len(diff) == 1 and diff[0][1].strip() == "{4096, 8, 16, 2, 8, 8},"
