"""Plant plausible mistakes in a copy of the oracle and check the pins catch
each one. The copy is compiled into a temporary directory on the CPU; the real
oracle is never modified."""
import os
import subprocess

import pytest

import oracle
from tests import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (name, text in oracle.c, replacement)
MUTANTS = [
    ("drop_last_term", "for (int32_t j = 0; j < d; ++j) acc +=", "for (int32_t j = 0; j < d - 1; ++j) acc +="),
    ("drop_first_term", "for (int32_t j = 0; j < d; ++j) acc +=", "for (int32_t j = 1; j < d; ++j) acc +="),
    ("wrong_sign", "acc += (double)row[j] * (double)query[j]", "acc -= (double)row[j] * (double)query[j]"),
    ("transposed_corpus", "acc += (double)row[j] * (double)query[j]",
     "acc += (double)corpus[(int64_t)j * n + i] * (double)query[j]"),
    ("query_index", "acc += (double)row[j] * (double)query[j]", "acc += (double)row[j] * (double)query[0]"),
    ("float_accumulator", "double acc = 0.0;", "float acc = 0.0f;"),
    ("tie_higher_index", "if (x->index != y->index) return (x->index < y->index) ? -1 : 1;",
     "if (x->index != y->index) return (x->index > y->index) ? -1 : 1;"),
    ("ascending_scores", "if (x->score != y->score) return (x->score > y->score) ? -1 : 1;",
     "if (x->score != y->score) return (x->score < y->score) ? -1 : 1;"),
    ("nan_not_mapped", "if (isnan(acc)) acc = -INFINITY;", ""),
    ("output_wrong_slot", "out_idx[j] = pairs[j].index;", "out_idx[j] = pairs[j > 0 ? j - 1 : 0].index;"),
    ("i32_smallest_first", "if (x->value != y->value) return (x->value > y->value) ? -1 : 1;",
     "if (x->value != y->value) return (x->value < y->value) ? -1 : 1;"),
    ("i32_tie_higher_pos", "if (x->position != y->position) return (x->position < y->position) ? -1 : 1;",
     "if (x->position != y->position) return (x->position > y->position) ? -1 : 1;"),
    ("i32_position_shift", "pairs[i].position = i;", "pairs[i].position = i + 1;"),
    ("bf16_truncate", "bits += 0x7FFFu + lsb;", "(void)lsb;"),
    ("bf16_ties_up", "bits += 0x7FFFu + lsb;", "bits += 0x8000u;"),
    ("cos_no_query_norm", "const double denom = qnorm * sqrt(cc);", "const double denom = sqrt(cc);"),
    ("cos_squared_row_norm", "const double denom = qnorm * sqrt(cc);", "const double denom = qnorm * cc;"),
    ("cos_zero_denominator_scores_zero", "double cosv = denom > 0.0 ? dot / denom : -INFINITY;",
     "double cosv = denom > 0.0 ? dot / denom : 0.0;"),
    ("cos_row_norm_from_query", "cc += (double)row[j] * (double)row[j];",
     "cc += (double)query[j] * (double)query[j];"),
    ("cos_topk_scores_inner_product", "  if (cosine)\n", "  if (0)\n"),
    ("cos_query_norm_drops_last", "for (int32_t j = 0; j < d; ++j) qq +=", "for (int32_t j = 0; j < d - 1; ++j) qq +="),
]


@pytest.fixture(scope="module")
def source():
    with open(SRC) as f:
        return f.read()


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, source, name, old, new):
    assert source.count(old) >= 1, f"mutation site for {name} not found"
    src = tmp_path / f"{name}.c"
    src.write_text(source.replace(old, new, 1))
    lib = tmp_path / f"lib{name}.so"
    oracle.build(str(src), str(lib))
    bad = oracle.Oracle(oracle.load(str(lib)))
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(bad)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"no pin catches the planted mistake {name}"
