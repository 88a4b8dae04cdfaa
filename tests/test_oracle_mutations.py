"""The pins must catch plausible mistakes in the oracle.  Each mutant below
is oracle.c with one slip planted (on the CPU, in a copy); it is compiled,
the oracle module is pointed at it, and a battery of the pins runs.  The
real oracle passes the battery; every mutant must fail it."""

import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
import test_oracle_pins as P

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle",
                   "oracle.c")

MUTANTS = [
    ("causal bound drops the row's own token",
     "if (b * MM3O_BLOCK + t > pos)", "if (b * MM3O_BLOCK + t >= pos)"),
    ("scale not applied", "out[b] = sm_scale * best;", "out[b] = best;"),
    ("block minimum instead of maximum",
     "if (dot > best)\n                best = dot;",
     "if (dot < best || best == -INFINITY)\n                best = dot;"),
    ("ties go to the higher id",
     "return (a->id > b->id) - (a->id < b->id);", "return (a->id < b->id) - (a->id > b->id);"),
    ("one local block too many", "(b > c - local_blocks)", "(b >= c - local_blocks)"),
    ("one init block too many", "(b < init_blocks)", "(b <= init_blocks)"),
    ("visible blocks rounded down", "nb = pos / MM3O_BLOCK + 1;", "nb = (pos + 1) / MM3O_BLOCK;"),
    ("NVFP4 nibbles swapped",
     "uint8_t nib = (d & 1) ? (c[d / 2] >> 4) : (c[d / 2] & 15);",
     "uint8_t nib = (d & 1) ? (c[d / 2] & 15) : (c[d / 2] >> 4);"),
    ("e2m1 subnormal doubled", "v = 0.5 * m;", "v = 1.0 * m;"),
    ("e4m3 ties away from even",
     "(d == bd && (c & 1) == 0 && (best & 1) == 1)", "(d == bd && (c & 1) == 1)"),
    ("sparse context misses the last token",
     "ctx += (last < pos ? last : pos) - (int64_t)b * MM3O_BLOCK + 1;",
     "ctx += (last < pos ? last : pos) - (int64_t)b * MM3O_BLOCK;"),
    ("sparse pages spaced by P, not the stride",
     "attn_table[i * attn_stride + b] *\n                                          block_page_stride + p",
     "attn_table[i * attn_stride + b] *\n                                          pages_per_block + p"),
]


def battery():
    """True when every pin of the battery holds for the oracle now loaded."""
    checks = [lambda c=c: P.test_oracle_matches_brute_force(c) for c in P.tiny_cases()[:40]]
    checks += [lambda s=s: P.test_oracle_matches_brute_force_nvfp4(s) for s in range(3)]
    checks += [P.test_planted_winners_and_scores, P.test_planted_exact_tie_goes_to_lower_id,
               P.test_select_ties_and_forced_rule, P.test_tiny_decode_by_hand,
               P.test_e2m1_values_from_the_spec, P.test_e4m3_rounding_matches_torch_in_range,
               P.test_nvfp4_subnormal_results, P.test_sparse_table_by_hand,
               P.test_sparse_table_full_selection_and_identity_layout,
               lambda: P.test_sparse_table_walk_reads_exactly_the_selected_visible_tokens(0, 2, 2),
               lambda: P.test_invariants(0)]
    for check in checks:
        try:
            check()
        except (AssertionError, ValueError):
            return False
    return True


@pytest.fixture
def use_source(tmp_path, monkeypatch):
    """Point the oracle module at a given C source (compiled into tmp_path)."""
    def load(text):
        src = tmp_path / "oracle.c"
        src.write_text(text)
        monkeypatch.setattr(oracle, "_SRC", str(src))
        monkeypatch.setattr(oracle, "_OUT_DIR", str(tmp_path / "build"))
        monkeypatch.setattr(oracle, "_LIB_PATH", str(tmp_path / "build" / "liboracle.so"))
        monkeypatch.setattr(oracle, "_lib", None)
        oracle._load()
    yield load
    oracle._lib = None  # the real library is loaded again on next use


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_real_oracle_passes_battery(use_source):
    use_source(open(SRC).read())
    assert battery()


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(use_source, name, old, new):
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation site not found: {name}"
    use_source(text.replace(old, new))
    assert not battery(), f"no pin caught: {name}"
