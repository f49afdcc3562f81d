"""Plant plausible mistakes in a copy of the oracle and check that a pin catches each.

Every mutant is the oracle source with one textual change (a dropped term, a
wrong sign, index or operand, an off-by-one), compiled into a temporary library
on the CPU. The test passes when at least one pin in ``oracle_pins`` fails on
the mutant, which shows the pins constrain that part of the oracle.
"""
import os
import subprocess
import sys

import pytest

import oracle as O

SRC = os.path.join(os.path.dirname(O.__file__), "spin_oracle.c")
HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

MUTANTS = {
    "scores_drop_first_head": ("for (int g = 0; g < G; ++g)\n      for (int i = 0; i < OD; ++i) s +=",
                               "for (int g = 1; g < G; ++g)\n      for (int i = 0; i < OD; ++i) s +="),
    "scores_transposed_summary": ("s += bf(q[g * OD + i]) * summ[p * OD + i];",
                                  "s += bf(q[g * OD + i]) * summ[i * P % (P * OD) + p % OD];"),
    "rank_ascending": ("if (x->s > y->s) return -1;\n  if (x->s < y->s) return 1;",
                       "if (x->s > y->s) return 1;\n  if (x->s < y->s) return -1;"),
    "ties_to_higher_index": ("return (x->p > y->p) - (x->p < y->p);", "return (x->p < y->p) - (x->p > y->p);"),
    "index_divides_by_64": ("summ[p * OD + i] = s / (double)(t1 - t0);", "summ[p * OD + i] = s / (double)OPART;"),
    # the next three anchors occur in both attention routines (with and without the tail); both are mutated
    "softmax_scale_1_over_d": ("const double scale = 1.0 / sqrt((double)OD);", "const double scale = 1.0 / (double)OD;", 2),
    "attention_values_from_keys": ("u->slots + (int64_t)sel_slot[j] * OPAGE_ELEMS + OPART * OD;",
                                   "u->slots + (int64_t)sel_slot[j] * OPAGE_ELEMS;", 2),
    "attention_drops_max_shift": ("double w = exp(x[c] - m);", "double w = exp(x[c] - m) * (c == 0 ? 0.5 : 1.0);", 2),
    # (Dropping the mandatory-page exclusion alone is an equivalent mutant: hits are
    # stamped with the current step first, so they sit in the newest bucket, which
    # the cutoff never reaches because cap >= k. It is therefore not listed.)
    "evict_exactly_demand": ("if (bucket <= out->cutoff) {", "if (bucket <= out->cutoff && out->evicted < out->demand) {"),
    "hits_not_bumped": ("out->hits += 1;\n      u->last_use[s] = t;", "out->hits += 1;"),
    "cutoff_exclusive": ("if (bucket <= out->cutoff) {", "if (bucket < out->cutoff) {"),
    "cutoff_one_bucket_late": ("if (cum >= out->demand) { out->cutoff = c; break; }",
                               "if (cum > out->demand) { out->cutoff = c; break; }"),
    "bucket_newest_first": ("int32_t bucket = OBUCKETS - 1 - (age < OBUCKETS - 1 ? age : OBUCKETS - 1);\n      hist",
                            "int32_t bucket = (age < OBUCKETS - 1 ? age : OBUCKETS - 1);\n      hist"),
    "segment_never_freed": ("if (u->seg_live[s] == 0) {", "if (u->seg_live[s] == -7) {"),
    "miss_copies_wrong_page": ("host_pages + (int64_t)p * OPAGE_ELEMS,", "host_pages + (int64_t)(p / 2) * OPAGE_ELEMS,"),
    "append_tail_not_attended": ("        valid = tail_n;\n        K = tail_kv;", "        valid = 0;\n        K = tail_kv;"),
    "append_no_growth": ("  u->P += 1;\n  u->ntok = u->P * OPART;", "  u->ntok = u->P * OPART;"),
    "budget_ignored": ("out->free_before = u->budget - out->resident_before;",
                       "out->free_before = u->cap - out->resident_before;"),
    "offload_drops_tail_token": ("for (int64_t t = 0; t < ntok; ++t) {\n    int64_t p = t / OPART",
                                 "for (int64_t t = 0; t < ntok - 1; ++t) {\n    int64_t p = t / OPART"),
    "parts_valid_drops_last_token": ("  if (u->part_n) return u->part_n[p];",
                                     "  if (u->part_n) return u->part_n[p] - (u->part_n[p] > 1);"),
    "parts_index_ignores_order": ("s += bf(k[(int64_t)order[j] * OD + i]);", "s += bf(k[(int64_t)j * OD + i]);"),
    "parts_index_divides_by_64": ("summ[(int64_t)p * OD + i] = s / (double)(j1 - j0);",
                                  "summ[(int64_t)p * OD + i] = s / (double)OPART;"),
    "parts_offload_rows_reversed": ("const int64_t t = order[j], r = j - starts[p];",
                                    "const int64_t t = order[j], r = starts[p + 1] - 1 - j;"),
}


@pytest.fixture(scope="module")
def src_text():
    with open(SRC) as f:
        return f.read()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, src_text, tmp_path):
    old, new = MUTANTS[name][:2]
    count = MUTANTS[name][2] if len(MUTANTS[name]) > 2 else 1
    assert src_text.count(old) == count, f"mutation anchor for {name} does not match the oracle source"
    path = tmp_path / "mutant.c"
    path.write_text(src_text.replace(old, new))
    so = str(tmp_path / "libmutant.so")
    subprocess.run(["gcc", "-O1", "-fPIC", "-shared", "-ffp-contract=off", "-std=c11", str(path), "-o", so, "-lm"],
                   check=True, capture_output=True)
    # run the pins in a child process: a mutant may also corrupt its own memory
    code = ("import sys; sys.path[:0] = [%r, %r]\n"
            "import oracle as O, oracle_pins as pins\n"
            "lib = O.load(%r)\n"
            "for check in pins.ALL_CHECKS:\n"
            "    try:\n"
            "        check(lib)\n"
            "    except AssertionError:\n"
            "        print('CAUGHT', check.__name__); sys.exit(0)\n"
            "print('MISSED'); sys.exit(3)\n") % (ROOT, HERE, so)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "CAUGHT" in r.stdout, f"no pin caught mutant {name}: {r.stdout[-500:]} {r.stderr[-500:]}"
