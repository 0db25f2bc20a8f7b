"""Plants plausible mistakes in a copy of oracle.c and checks that the pins catch
each one.  A pin set that let one of these through would not be pinning the
oracle.  Each mutant is compiled to a temporary library and exercised in a child
process, so a mutant that crashes cannot take the test session down (a crash
also counts as caught)."""

import json
import os
import subprocess
import sys
import tempfile

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

# (name, original text, replacement, replace every occurrence?)
MUTANTS = [
    ("drop_scale", "scores[j] = scale * dot;", "scores[j] = dot;", False),
    ("scale_twice", "scores[j] = scale * dot;", "scores[j] = scale * scale * dot;", False),
    ("top_left_causal", "const int64_t p = L - n + i;", "const int64_t p = i;", False),
    ("no_causal_mask", "const int64_t p = L - n + i;", "const int64_t p = L - 1;", False),
    ("causal_off_by_one", "j <= p", "j < p", True),
    ("gqa_modulo", "const int64_t hk = h / group;", "const int64_t hk = h % d->num_kv_heads;", False),
    ("ignore_block_table", "int64_t page = block_table[b * d->max_pages + j / d->page_size];",
     "int64_t page = (j / d->page_size) % d->num_blocks;", False),
    ("slot_reversed", "int64_t slot = j % d->page_size;",
     "int64_t slot = d->page_size - 1 - j % d->page_size;", False),
    ("head_major_page", "return cache + ((page * d->page_size + slot) * d->num_kv_heads + hk) * d->head_dim;",
     "return cache + ((page * d->num_kv_heads + hk) * d->page_size + slot) * d->head_dim;", False),
    ("no_max_subtraction", "scores[j] = exp(scores[j] - m);", "scores[j] = exp(scores[j]);", False),
    ("v_from_k_cache", "cache_row(v_cache, d,", "cache_row(k_cache, d,", False),
    ("q_of_kv_head", "const uint16_t* qrow = q + (t * d->num_q_heads + h) * D;",
     "const uint16_t* qrow = q + (t * d->num_q_heads + hk) * D;", False),
    ("normalise_by_count", "const double w = scores[j] / l;", "const double w = scores[j] / (double)(p + 1);", False),
    ("owner_seq_off_by_one", "if (qsl[mid] <= t) lo = mid;", "if (qsl[mid] < t) lo = mid;", False),
    ("wrong_seq_row", "int64_t page = block_table[b * d->max_pages + j / d->page_size];",
     "int64_t page = block_table[j / d->page_size];", False),
    ("lse_without_max", "if (lse) *lse = m + log(l);", "if (lse) *lse = log(l);", False),
    ("lse_of_weights_sum", "if (lse) *lse = m + log(l);", "if (lse) *lse = m;", False),
    ("cache_write_page_slot_swapped", "const int64_t page = s / page_size, slot = s % page_size;",
     "const int64_t page = s % page_size, slot = s / page_size;", False),
    ("cache_write_v_from_k", "memcpy(v_cache + (page * page_size + slot) * row, v_new + t * row",
     "memcpy(v_cache + (page * page_size + slot) * row, k_new + t * row", False),
    ("cache_write_ignores_padding", "        if (s < 0) continue;\n", "", False),
]

_CHILD = r"""
import json, sys
sys.path.insert(0, sys.argv[1]); sys.path.insert(0, sys.argv[1] + '/tests')
import oracle, oracle_pins as P
lib = oracle.load(sys.argv[2])
res = {}
for pin in P.ALL_PINS:
    try:
        pin(lib)
        res[pin.__name__] = 'pass'
    except Exception as e:
        res[pin.__name__] = 'fail: ' + type(e).__name__
print(json.dumps(res))
"""


def _mutate(text: str, old: str, new: str, every: bool) -> str:
    n = text.count(old)
    assert n >= 1, f"mutation anchor not found: {old!r}"
    if not every:
        assert n == 1, f"mutation anchor not unique: {old!r}"
    return text.replace(old, new)


@pytest.fixture(scope="module")
def workdir():
    with tempfile.TemporaryDirectory() as d:
        yield d


def test_unmutated_copy_passes_every_pin(workdir):
    lib = oracle.compile_oracle(SRC, os.path.join(workdir, "orig.so"))
    out = subprocess.run([sys.executable, "-c", _CHILD, ROOT, lib], capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr
    res = json.loads(out.stdout.strip().splitlines()[-1])
    assert all(v == "pass" for v in res.values()), res


@pytest.mark.parametrize("name,old,new,every", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(workdir, name, old, new, every):
    text = open(SRC).read()
    src = os.path.join(workdir, f"{name}.c")
    with open(src, "w") as f:
        f.write(_mutate(text, old, new, every))
    lib = oracle.compile_oracle(src, os.path.join(workdir, f"{name}.so"))
    out = subprocess.run([sys.executable, "-c", _CHILD, ROOT, lib], capture_output=True, text=True, timeout=600)
    if out.returncode != 0:
        return  # the mutant crashed: caught
    res = json.loads(out.stdout.strip().splitlines()[-1])
    caught = [k for k, v in res.items() if v != "pass"]
    assert caught, f"mutant {name} passed every pin"
