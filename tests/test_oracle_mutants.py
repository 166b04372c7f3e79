"""Plant one plausible mistake at a time in a copy of the oracle (on the CPU)
and check that the pins catch every one of them.

A mistake that no pin catches would mean the oracle is checked against less
than it seems; this test keeps the pin set honest.  The copies are compiled
into a temporary folder; the oracle's own source is never modified.
"""
import os

import pytest

from oracle import Oracle
from oracle.build import SRC, build_variant

from .oracle_pins import ALL_PINS

# (name, text in the oracle source, replacement) -- each a slip a careful
# implementer could make.
MUTANTS = [
    ("reciprocal_multiply", "float v = xf[k] / s;", "float v = xf[k] * (1.0f / s);"),
    ("scale_over_128", "amax / 127.0f", "amax / 128.0f"),
    ("ties_away_from_zero", "float r = nearbyintf(v);", "float r = roundf(v);"),
    ("truncating_quantiser", "float r = nearbyintf(v);", "float r = truncf(v);"),
    ("signed_amax", "float a = fabsf(xf[k]);", "float a = xf[k];"),
    ("zero_block_scale_zero", "(amax == 0.0f) ? 1.0f", "(amax == 0.0f) ? 0.0f"),
    ("clamp_to_126", "if (r > 127.0f) r = 127.0f;", "if (r > 126.0f) r = 126.0f;"),
    ("dot_sign", "acc += (int32_t)w[(size_t)n * K + k] * (int32_t)q[(size_t)m * K + k];",
     "acc -= (int32_t)w[(size_t)n * K + k] * (int32_t)q[(size_t)m * K + k];"),
    ("dot_block_local_index", "acc += (int32_t)w[(size_t)n * K + k] * (int32_t)q[(size_t)m * K + k];",
     "acc += (int32_t)w[(size_t)n * K + k] * (int32_t)q[(size_t)m * K + (k % 32)];"),
    ("linear_misindexed_codes", "d += (int32_t)wr[k] * (int32_t)q[k];", "d += (int32_t)wr[k] * (int32_t)q[k ^ 1];"),
    ("scales_transposed", "oracle_half_to_float(sw[(size_t)n * nb + b]) * sx[b]",
     "oracle_half_to_float(sw[(size_t)b * N + n]) * sx[b]"),
    ("dropped_accumulation", "acc = acc + t;", "acc = t;"),
    ("missing_act_scale", "float p = oracle_half_to_float(sw[(size_t)n * nb + b]) * sx[b];",
     "float p = oracle_half_to_float(sw[(size_t)n * nb + b]);"),
    ("half_bias_off_by_one", "v = ldexpf((float)(m | 0x400), e - 25);", "v = ldexpf((float)(m | 0x400), e - 24);"),
    ("half_round_truncates", "float t = nearbyintf(ldexpf(a, 10 - E));", "float t = truncf(ldexpf(a, 10 - E));"),
    ("half_overflow_threshold", "if (a >= 65520.0f)", "if (a >= 65504.0f)"),
    ("unpack_no_offset", "(int8_t)((int)(byte & 0x0f) - 8)", "(int8_t)((int)(byte & 0x0f))"),
    ("unpack_nibbles_swapped", "w[(size_t)n * K + 2 * j] = (int8_t)((int)(byte & 0x0f) - 8);",
     "w[(size_t)n * K + 2 * j] = (int8_t)((int)(byte >> 4) - 8);"),
    ("gated_branches_swapped", "double g = (double)acc[(size_t)m * 2 * N + n];",
     "double g = (double)acc[(size_t)m * 2 * N + N + n];"),
    ("silu_sign", "return g / (1.0 + exp(-g));", "return g / (1.0 + exp(g));"),
    ("gelu_cubic_coefficient", "(g + 0.044715 * g * g * g)", "(g + 0.044715 * g * g)"),
    ("gated_up_row_offset", "double u = (double)acc[(size_t)m * 2 * N + N + n];",
     "double u = (double)acc[(size_t)m * 2 * N + N + n - 1 + (n == 0)];"),
    ("rmsnorm_sum_not_mean", "ms /= (double)K;", "ms /= 1.0;"),
    ("rmsnorm_eps_outside_root", "double inv = 1.0 / sqrt(ms + (double)eps);", "double inv = 1.0 / (sqrt(ms) + (double)eps);"),
    ("rmsnorm_no_gamma", "double v = (double)r[k] * inv * (double)oracle_half_to_float(gamma[k]);",
     "double v = (double)r[k] * inv;"),
    ("rmsnorm_residual_dropped", "if (res) h = h + oracle_half_to_float(res[(size_t)m * K + k]);", "(void)res;"),
    ("rmsnorm_no_root", "double inv = 1.0 / sqrt(ms + (double)eps);", "double inv = 1.0 / (ms + (double)eps);"),
    ("attention_scale_over_d", "double scale = 1.0 / sqrt((double)D);", "double scale = 1.0 / (double)D;"),
    ("attention_group_modulo", "int g = h / G, L = lens[b];", "int g = h % Hkv, L = lens[b];"),
    ("attention_length_off_by_one", "for (int t = 0; t < L; ++t) {\n                double p", "for (int t = 0; t <= L && t < Lmax; ++t) {\n                double p"),
    ("attention_unnormalised", "(float)(o[d] / den)", "(float)(o[d])"),
    ("attention_no_max_shift", "double p = exp(s[t] - m);", "double p = exp(s[t]);"),
    ("f64_drops_weight_scale", "acc += (swd * (double)w[(size_t)n * K + k]) * (sxd * (double)q[k]);",
     "acc += ((double)w[(size_t)n * K + k]) * (sxd * (double)q[k]);"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found in the oracle"
    mutated = src.replace(old, new)
    lib = build_variant(mutated, os.path.join(str(tmp_path), f"liboracle_{name}.so"))
    orc = Oracle(lib)
    caught = []
    for pin in ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"no pin catches the planted mistake {name}"
