"""Each plausible mistake, planted in a copy of the C oracle on the CPU, must
fail at least one pin -- evidence that the pins constrain the oracle."""
import functools
import os

import pytest

import oracle
from tests import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "seg_oracle.c")

# (name, [(text in seg_oracle.c, replacement), ...])
MUTANTS = [
    ("float_sum_drops_first_row",
     [("for (int64_t r = b; r < e; ++r)\n            acc += (double)",
       "for (int64_t r = b + 1; r < e; ++r)\n            acc += (double)")]),
    ("int_sum_drops_last_row",
     [("for (int64_t r = b; r < e; ++r)\n            acc += v[",
       "for (int64_t r = b; r + 1 < e; ++r)\n            acc += v[")]),
    ("float_sum_wrong_sign", [("acc += (double)v[r * F + f];", "acc -= (double)v[r * F + f];")]),
    ("ties_to_higher_row",
     [("(op == ORC_MIN && x < best) || (op == ORC_MAX && x > best)",
       "(op == ORC_MIN && x <= best) || (op == ORC_MAX && x >= best)")]),
    ("segment_relative_arg", [("best_row = r;", "best_row = r - b;")]),
    ("wrong_column", [("float x = v[r * F + f];", "float x = v[r * F];")]),
    ("s32_compared_unsigned",
     [("    int32_t best = v[b * F + f];", "    uint32_t best = (uint32_t)v[b * F + f];"),
      ("        int32_t x = v[r * F + f];", "        uint32_t x = (uint32_t)v[r * F + f];")]),
    ("empty_float_not_zero", [("((float *)out)[o] = 0.0f;", "((float *)out)[o] = 3.0e38f;")]),
    ("empty_int_not_zero", [("((uint32_t *)out)[o] = 0u;", "((uint32_t *)out)[o] = 0xFFFFFFFFu;")]),
    ("mean_length_off_by_one", [("float len = (float)(e - b);", "float len = (float)(e - b + 1);")]),
    ("inclusive_segment_end",
     [("int64_t e = offset_at(offsets, off_dtype, s + 1);",
       "int64_t e = offset_at(offsets, off_dtype, s + 1);\n        if (e < num_values && e > b) e += 1;")]),
    ("offsets_shifted",
     [("int64_t b = offset_at(offsets, off_dtype, s);",
       "int64_t b = offset_at(offsets, off_dtype, s > 0 ? s - 1 : 0);")]),
    ("int_sum_saturates",
     [("acc += (uint32_t)v[r * F + f];",
       "{ uint32_t t = acc + (uint32_t)v[r * F + f]; acc = t < acc ? 0xFFFFFFFFu : t; }")]),
    ("float_sum_in_float", [("double acc = 0.0;", "float acc = 0.0f;")]),
]


@pytest.mark.parametrize("name,edits", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, edits):
    mutated = open(SRC).read()
    for old, new in edits:
        assert old in mutated, f"mutation anchor for {name} not found"
        mutated = mutated.replace(old, new)
    path = tmp_path / "mutant.c"
    path.write_text(mutated)
    lib = oracle.load_library(oracle.compile_source(str(path), str(tmp_path / "libmutant.so")))
    reduce = functools.partial(oracle.seg_reduce, lib=lib)
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(reduce)
        except (AssertionError, ValueError, IndexError):
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
