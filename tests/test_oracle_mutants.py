"""The oracle's pins must catch plausible mistakes.

Each case copies ``oracle/lp_oracle.c``, plants one mistake (a dropped term, a
wrong sign, an off-by-one index, a swapped operand), compiles the copy on the
CPU, swaps it in for the real oracle and reruns the pins that should notice.
A mutant that survives every named pin fails this test.
"""
import os
import subprocess

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "lp_oracle.c")

MUTANTS = [
    # (name, original text, planted mistake, pins expected to fail)
    ("bit_order", "(w >> (j % 32)) & 1u", "(w >> (31 - j % 32)) & 1u",
     ["test_golden_apply", "test_apply_matches_numpy_unpack"]),
    ("keep_is_zero", "lpo_bit(bitmask, bitmask_stride, b, j) == 0",
     "lpo_bit(bitmask, bitmask_stride, b, j) != 0", ["test_golden_apply"]),
    ("vocab_default_max", "return cols < w ? cols : w;", "return cols > w ? cols : w;",
     ["test_golden_apply"]),
    ("f16_exponent_bias", "ex - 25", "ex - 24", ["test_decode_all_half_patterns"]),
    ("round_toward_zero", "rint(x / quantum)", "trunc(x / quantum)",
     ["test_encode_round_to_nearest_even"]),
    ("greedy_last_tie", "if (best < 0 || l[j] > l[best]) best = j;",
     "if (best < 0 || l[j] >= l[best]) best = j;", ["test_golden_greedy"]),
    ("no_temperature", "z[j] = l[j] / T;", "z[j] = l[j];",
     ["test_golden_keep_sets", "test_keep_set_brute_force_tiny_vocab"]),
    ("top_k_off_by_one", "c[top_k - 1].p", "c[top_k].p",
     ["test_golden_keep_sets", "test_keep_set_brute_force_tiny_vocab"]),
    ("top_p_dropped_sum", "cum += c[i].p;", "cum = c[i].p;",
     ["test_golden_keep_sets", "test_keep_set_brute_force_tiny_vocab"]),
    ("top_p_after_crossing", "cut = i;", "cut = (i + 1 < n) ? i + 1 : i;",
     ["test_golden_keep_sets", "test_keep_set_brute_force_tiny_vocab"]),
    ("min_p_not_relative", "t_m = min_p * p_max;", "t_m = min_p;",
     ["test_golden_keep_sets"]),
    ("philox_round_const", "0xD2511F53u", "0xD2511F55u", ["test_philox_matches_pytorch_engine"]),
    ("philox_key_bump", "k1 += 0xBB67AE85u;", "k1 += 0xBB67AE84u;",
     ["test_philox_matches_pytorch_engine"]),
    ("counter_swap", "{(uint32_t)(v >> 2), (uint32_t)row,", "{(uint32_t)row, (uint32_t)(v >> 2),",
     ["test_random_word_counter_layout"]),
    ("word_pick", "return out[v & 3];", "return out[(v + 1) & 3];",
     ["test_random_word_counter_layout"]),
    ("gumbel_sign", "return -log(-log(lpo_uniform(x)));", "return log(-log(lpo_uniform(x)));",
     ["test_draw_is_exponential_race", "test_draw_distribution_goodness_of_fit"]),
    ("uniform_bits", "((double)(x >> 9) + 0.5)", "((double)(x >> 8) + 0.5)",
     ["test_uniform_and_gumbel_range"]),
    ("draw_ignores_z", "const double score = z[j] + lpo_gumbel", "const double score = 0.0 * z[j] + lpo_gumbel",
     ["test_draw_is_exponential_race"]),
    ("unsat_not_minus_one", "*id_out = -1;\n    return 0;", "*id_out = 0;\n    return 0;",
     ["test_golden_greedy"]),
    ("rows_flags_ignored", "const int masked = flags == NULL || flags[b] != 0;",
     "const int masked = 1;",
     ["test_apply_rows_hand_worked", "test_apply_rows_against_numpy_and_indices"]),
    ("rows_unflagged_report_zero", "if (has_token) has_token[b] = any;",
     "if (has_token) has_token[b] = masked ? any : 0;",
     ["test_apply_rows_hand_worked", "test_apply_rows_against_numpy_and_indices"]),
    ("rows_fill_sign", "lpo_store_fill(logits, dtype, b * logits_stride + j, -INFINITY);",
     "lpo_store_fill(logits, dtype, b * logits_stride + j, INFINITY);",
     ["test_apply_rows_hand_worked", "test_apply_rows_against_numpy_and_indices"]),
]


def _run_pin(name, monkeypatch, request):
    fn = getattr(pins, name)
    import inspect

    params = inspect.signature(fn).parameters
    kwargs = {}
    if "torch_philox" in params:
        kwargs["torch_philox"] = request.getfixturevalue("torch_philox")
    marks = getattr(fn, "pytestmark", [])
    argsets = [{}]
    for m in marks:
        if m.name == "parametrize":
            names = [n.strip() for n in m.args[0].split(",")]
            argsets = [dict(zip(names, v if isinstance(v, (tuple, list)) else (v,)))
                       for v in m.args[1]]
    for extra in argsets:
        fn(**kwargs, **extra)


torch_philox = pins.torch_philox


@pytest.mark.parametrize("name,orig,bad,catchers", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(name, orig, bad, catchers, tmp_path, monkeypatch, request):
    src = open(SRC).read()
    assert src.count(orig) >= 1, f"mutation site for {name} not found"
    mutated = src.replace(orig, bad, 1)
    csrc, so = tmp_path / "m.c", tmp_path / "libm.so"
    csrc.write_text(mutated)
    subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-o", str(so), str(csrc), "-lm"])
    monkeypatch.setattr(oracle, "_lib", oracle.load_library(str(so)))
    caught = []
    for pin in catchers:
        try:
            _run_pin(pin, monkeypatch, request)
        except (AssertionError, ValueError):
            caught.append(pin)
    assert caught, f"mutant {name} survived {catchers}"
