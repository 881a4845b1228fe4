"""Plant plausible mistakes in a copy of the oracle's C source and check that
the pins in test_oracle.py catch every one (CPU only, nothing here touches a
GPU).  A mutation the pins let through would mean the oracle is trusted on
evidence that could not have told it apart from a broken one."""
import os
import subprocess

import pytest

import oracle
from tests import test_oracle as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "pkv_oracle.c")

MUTATIONS = {
    "dropped_scale": ("x[t] = j->scale * dot;", "x[t] = dot;"),
    "exp_sign": ("x[t] = exp(x[t] - mx);", "x[t] = exp(mx - x[t]);"),
    "no_normaliser": ("const double p = x[t] / z;", "const double p = x[t];"),
    "block_slot_swapped": ("t / PKV_ORACLE_BLOCK];", "t % PKV_ORACLE_BLOCK];"),
    "head_major_layout": ("(((size_t)blk * j->num_kv_heads + hkv) * PKV_ORACLE_BLOCK",
                          "(((size_t)hkv * j->num_blocks + blk) * PKV_ORACLE_BLOCK"),
    "strided_gqa": ("const int hq = hkv * g + n;", "const int hq = n * j->num_kv_heads + hkv;"),
    "keys_from_values": ("dot += widen(j->q, qrow + i, j->dtype) * K[(size_t)t * d + i];",
                         "dot += widen(j->q, qrow + i, j->dtype) * V[(size_t)t * d + i];"),
    "prefill_sees_next_token": ("const int pos = len - n + qi;",
                                "const int pos = (len - n + qi + 1 < len) ? len - n + qi + 1 : len - 1;"),
    "prefill_misses_own_token": ("const int pos = len - n + qi;", "const int pos = len - n + qi - 1;"),
    "bf16_low_half": ("uint32_t bits = ((uint32_t)((const uint16_t *)base)[idx]) << 16;",
                      "uint32_t bits = ((uint32_t)((const uint16_t *)base)[idx]) << 15;"),
}

PIN_CALLS = [
    lambda: pins.test_two_token_closed_form(1.0),
    lambda: pins.test_two_token_closed_form(-1.0),
    lambda: pins.test_single_token_returns_value_row(),
    lambda: pins.test_equal_keys_and_zero_query_give_mean(17),
    lambda: pins.test_gqa_consecutive_grouping(),
    lambda: pins.test_matches_dense_bruteforce("f32", 4),
    lambda: pins.test_matches_dense_bruteforce("bf16", 1),
    lambda: pins.test_log_sum_exp_merge_of_partitions_equals_whole(),
    lambda: pins.test_prefill_matches_dense_causal_bruteforce(1),
    lambda: pins.test_prefill_first_query_sees_only_itself_and_last_query_is_decode(),
]


def _build_mutant(tmp_path, name):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    lib = tmp_path / f"lib_{name}.so"
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread", str(path), "-o", str(lib), "-lm"])
    return str(lib)


def _pins_fail():
    for call in PIN_CALLS:
        try:
            call()
        except (AssertionError, ValueError):
            return True
    return False


def test_unmutated_source_passes_the_same_pins(tmp_path):
    lib = tmp_path / "lib_clean.so"
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread", SRC, "-o", str(lib), "-lm"])
    with oracle.use_library(str(lib)):
        assert not _pins_fail()


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(tmp_path, name):
    with oracle.use_library(_build_mutant(tmp_path, name)):
        assert _pins_fail(), f"pins did not catch the planted mistake {name!r}"
