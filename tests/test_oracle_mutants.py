"""Sensitivity of the pins: plant one plausible mistake at a time in a copy of the oracle source
(on the CPU), rebuild it, and check that at least one pin in test_oracle_pins.py fails for it."""
import os
import re
import subprocess
import sys

import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "hs_oracle.c")

# (name, pattern, replacement): each is a small slip someone could make writing the oracle.
MUTANTS = [
    ("no_hit_refresh", r"stamp\[slot_of\[i\]\] = step;", ";"),
    ("victim_tiebreak_reversed", r"return x->idx < y->idx \? -1 : 1;", "return x->idx < y->idx ? 1 : -1;"),
    ("victim_newest_first", r"return x->key < y->key \? -1 : 1;", "return x->key < y->key ? 1 : -1;"),
    ("evict_same_step", r"stamp\[s\] < step && !hit_slot\[s\]", "stamp[s] <= step && !hit_slot[s]"),
    ("evict_hit_slots", r"stamp\[s\] < step && !hit_slot\[s\]", "stamp[s] < step"),
    ("resident_offset_dropped", r"row\[i\] = \(int64_t\)bt\[page\] \* S \+ off;", "row[i] = (int64_t)bt[page] * S;"),
    ("hot_row_transposed", r"return \(int64_t\)hot_blocks_r\[slot / S\] \* S \+ slot % S;",
     "return (int64_t)hot_blocks_r[slot % S] * S + slot / S;"),
    ("last_occurrence_plan", r"if \(j == 0 \|\| by_id\[j\]\.key != by_id\[j - 1\]\.key\) group_first = by_id\[j\]\.idx;",
     "group_first = by_id[j].idx;"),
    ("resident_checked_after_hot", r"if \(bt\[page\] >= 0\) \{", "if (bt[page] >= 0 && find_first(by_tok, nt, id) < 0) {"),
    ("copy_from_wrong_row", r"host \+ src\[i\] \* \(int64_t\)B", "host + (src[i] + 1) * (int64_t)B"),
    ("step_order_ignored", r"if \(stamp\[s\] > step\) err_step = 1;", ";"),
    ("capacity_off_by_one", r"if \(nmiss > ncand\) err_capacity = 1;", "if (nmiss >= ncand && nmiss) err_capacity = 1;"),
    ("missing_row_not_checked", r"if \(hbt\[page\] < 0\) err_missing = 1;\n\s*else ", ""),
    ("gather_wrong_stride", r"pools\[layer_begin \+ l\] \+ \(int64_t\)r \* B", "pools[layer_begin + l] + (int64_t)r * (B - 16)"),
    ("offload_one_layer", r"for \(int32_t l = 0; l < num_layers; l\+\+\)", "for (int32_t l = 0; l < 1; l++)"),
    ("stats_hits_misses_swapped", r"out_stats\[2\] = nhit; out_stats\[3\] = nmiss;", "out_stats[2] = nmiss; out_stats[3] = nhit;"),
    ("index_share_copies_one_layer", r"for \(int32_t g = 0; g < G; g\+\+\)", "for (int32_t g = 0; g < 1; g++)"),
    ("index_share_group_offset_dropped", r"int32_t grp = layer_begin / G \+ gr;", "int32_t grp = gr;"),
]

PIN_FUNCS = [getattr(pins, n) for n in dir(pins) if n.startswith("test_")]


def _run_pins():
    """Return the names of pins that fail (parametrised pins run over their parameters)."""
    failed = []
    for f in PIN_FUNCS:
        marks = getattr(f, "pytestmark", [])
        params = [m for m in marks if m.name == "parametrize"]
        if params:
            names = [x.strip() for x in params[0].args[0].split(",")]
            calls = [dict(zip(names, v if isinstance(v, tuple) else (v,))) for v in params[0].args[1]]
        else:
            calls = [{}]
        for kw in calls:
            try:
                f(**kw)
            except Exception:
                failed.append(f.__name__)
                break
    return failed


def _child(so_path):
    """Run in a child process: route the oracle through the mutant and print the failing pins."""
    oracle.use_library(oracle.load_library(so_path))
    print("FAILED_PINS", ",".join(_run_pins()))


@pytest.mark.parametrize("name,pat,rep", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, name, pat, rep):
    src = open(SRC).read()
    mutated, n = re.subn(pat, rep, src)
    assert n >= 1, f"mutation {name} did not apply"
    c = tmp_path / "mut.c"
    so = tmp_path / "libmut.so"
    c.write_text(mutated)
    r = subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", str(c), "-o", str(so)], capture_output=True,
                       text=True)
    assert r.returncode == 0, r.stderr
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = f"import sys; sys.path.insert(0, {root!r}); from tests import test_oracle_mutants as m; m._child({str(so)!r})"
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    if r.returncode != 0:
        return  # the planted mistake made the oracle crash: caught loudly
    line = [x for x in r.stdout.splitlines() if x.startswith("FAILED_PINS")][-1]
    failed = [x for x in line.split(" ", 1)[1].split(",") if x] if " " in line else []
    assert failed, f"no pin caught the planted mistake {name}"
