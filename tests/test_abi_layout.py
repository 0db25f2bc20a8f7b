"""The ctypes structures of the Python binding against the C header: a small C
program compiled against include/pagedattn.h prints every structure's size and
each field's offset, which must match the binding's (a mismatch would pass
garbage across the boundary without any error)."""

import ctypes
import os
import shutil
import subprocess
import tempfile

import pytest

from paged_kv_cache_forward_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
STRUCTS = {"pa_dims": B.Dims, "pa_options": B.Options, "pa_plan_info": B.PlanInfo, "pa_cache_dims": B.CacheDims}


def _c_layout():
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lines = ['#include <stddef.h>', '#include <stdio.h>', '#include "pagedattn.h"', "int main(void) {"]
    for cname, py in STRUCTS.items():
        lines.append(f'    printf("{cname} size %zu\\n", sizeof({cname}));')
        for field, _ in py._fields_:
            lines.append(f'    printf("{cname} {field} %zu\\n", offsetof({cname}, {field}));')
    lines += ["    return 0;", "}"]
    with tempfile.TemporaryDirectory() as d:
        src, exe = os.path.join(d, "layout.c"), os.path.join(d, "layout")
        open(src, "w").write("\n".join(lines) + "\n")
        subprocess.run([cc, "-I", os.path.join(ROOT, "include"), src, "-o", exe], check=True)
        out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout
    return {tuple(l.split()[:2]): int(l.split()[2]) for l in out.splitlines()}


def test_binding_structs_match_the_header():
    c = _c_layout()
    for cname, py in STRUCTS.items():
        assert ctypes.sizeof(py) == c[(cname, "size")], cname
        for field, _ in py._fields_:
            assert getattr(py, field).offset == c[(cname, field)], (cname, field)
