"""Planted mistakes in the oracle must fail at least one pin (CPU only).

Each case copies ``oracle/carat_oracle.c`` to a temporary directory, replaces
one exact snippet with a plausible mistake (an off-by-one window edge, a
dropped scale, a wrong head mapping, a missing normaliser, a wrong slot rule
...), compiles the copy, and runs every pin against it.  The test passes when
some pin rejects the broken build; it also checks that each snippet still
exists in the real source, so the cases follow the oracle when it is edited.
"""
import os

import pytest

import oracle
import oracle_pins

MUTATIONS = {
    "window_first_off_by_one": ("int64_t first = position - window + 1;",
                                "int64_t first = position - window;"),
    "window_excludes_query": ("int64_t last = position;", "int64_t last = position - 1;"),
    "dropped_scale": ("score[t - first] = scale * dot;", "score[t - first] = dot;"),
    "no_max_subtraction": ("double w = exp(score[t - first] - max_score);",
                           "double w = exp(score[t - first]);"),
    "flipped_sign": ("double w = exp(score[t - first] - max_score);",
                     "double w = exp(max_score - score[t - first]);"),
    "wrong_head_map": ("kv_heads, head_dim, h / group,", "kv_heads, head_dim, h % kv_heads,"),
    "no_normaliser": ("out_row[d] /= denom;", "out_row[d] /= 1.0;"),
    "reversed_queries": ("int64_t position = context_length + j;",
                         "int64_t position = context_length + proposal_count - 1 - j;"),
    "bf16_shift": ("uint32_t word = ((uint32_t)bits) << 16;",
                   "uint32_t word = ((uint32_t)bits) << 15;"),
    "reversed_dim": ("dot += bf16_value(q_row[d]) * hist_value(k_hist, k_row + d, kind);",
                     "dot += bf16_value(q_row[d]) * hist_value(k_hist, k_row + head_dim - 1 - d, kind);"),
    "v_from_k": ("out_row[d] += w * hist_value(v_hist, v_row + d, kind);",
                 "out_row[d] += w * hist_value(k_hist, v_row + d, kind);"),
    "slot_rule": ("return position % window;", "return (position + 1) % window;"),
    "key_count_rule": ("return context_length + proposal_count;",
                       "return context_length + proposal_count - 1;"),
    "ring_first_slot": ("int64_t first = key_count - window > 0 ? key_count - window : 0;",
                        "int64_t first = key_count - window + 1 > 0 ? key_count - window + 1 : 0;"),
    "displaced_offset": ("int64_t t = context_length - window + 1 + i;",
                         "int64_t t = context_length - window + i;"),
    "e4m3_bias": ("ldexp(1.0 + (double)m / 8.0, e - 7)", "ldexp(1.0 + (double)m / 8.0, e - 8)"),
    "e4m3_subnormal_exponent": ("ldexp((double)m / 8.0, -6)", "ldexp((double)m / 8.0, -7)"),
    "e4m3_ties_up": ("c = (lo & 1) == 0 ? lo : hi;", "c = hi;"),
    "e4m3_overflow_to_nan": ("return sign | 0x7e;", "return 0x7f;"),
    "e4m3_sign_dropped": ("return sign ? -mag : mag;", "return mag;"),
    "quantize_no_reciprocal": ("float inv = 1.0f / scale;", "float inv = scale;"),
    "f64_history_reads_bf16": ("return ((const double *)hist)[i];",
                               "return bf16_value(((const uint16_t *)hist)[i]);"),
}


def _source():
    with open(oracle.SOURCE) as f:
        return f.read()


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path):
    before, after = MUTATIONS[name]
    src = _source()
    assert src.count(before) >= 1, f"snippet for {name} no longer in the oracle source"
    mutated = src.replace(before, after)
    path = os.path.join(tmp_path, "mutant.c")
    with open(path, "w") as f:
        f.write(mutated)
    lib_path = oracle.build(source=path, library=os.path.join(tmp_path, "libmutant.so"))
    mutant = oracle.Oracle(oracle.load_library(lib_path))
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(mutant)
        except (AssertionError, ValueError, FloatingPointError) as e:  # a pin rejected it
            caught.append(pin.__name__)
    assert caught, f"no pin catches the planted mistake {name}"
