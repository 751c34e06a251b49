"""Plants plausible mistakes in copies of the oracle source and checks that the
pins catch every one (CPU only).  The real oracle is never modified: each
mutant is compiled from a patched copy into a temporary directory."""
import os
import subprocess

import pytest

from oracle import oracle as O
import oracle_pins as P

SRC = os.path.join(os.path.dirname(O.__file__), "pq2_oracle.c")

# (name, original text, mistaken text)
MUTANTS = [
    ("decode_offset", "& 3u) - 1;", "& 3u) - 0;"),
    ("decode_field_width", "(byte >> (2 * field))", "(byte >> (field))"),
    ("scale_big_endian", "(blk[0] | (blk[1] << 8))", "(blk[1] | (blk[0] << 8))"),
    ("code_byte_offset", "blk[2 + j]", "blk[1 + j]"),
    ("scale_reciprocal", "float s = amax / 127.0f;", "float s = amax * (1.0f / 127.0f);"),
    ("scale_128", "float s = amax / 127.0f;", "float s = amax / 128.0f;"),
    ("round_half_away", "nearbyintf(x[i] / d)", "roundf(x[i] / d)"),
    ("round_trunc", "nearbyintf(x[i] / d)", "truncf(x[i] / d)"),
    ("divide_by_reciprocal", "nearbyintf(x[i] / d)", "nearbyintf(x[i] * (1.0f / d))"),
    ("zero_group_scale_stored", "sx[m * G + g] = s;", "sx[m * G + g] = d;"),
    ("dot_sign", "acc += w * (int32_t)q[m * K + k];", "acc -= w * (int32_t)q[m * K + k];"),
    ("dot_field_order", "(int)(k % 4));\n          acc", "(int)((k / 32) % 4));\n          acc"),
    ("weight_scale_dropped", "t = t * ws;", "t = t * xs;"),
    ("last_group_dropped", "for (int64_t g = 0; g < G; ++g) {\n        int32_t dot",
     "for (int64_t g = 0; g + 1 < G; ++g) {\n        int32_t dot"),
    ("planes_transposed", "q[m * K + g * ORC_GROUP + 4 * j + s]", "q[m * K + g * ORC_GROUP + 4 * s + j]"),
    ("half_exponent_bias", "(int)expo - 25", "(int)expo - 24"),
    ("half_subnormal", "ldexp((double)frac, -24)", "ldexp((double)frac, -25)"),
    ("bf16_ties_up", "lower > 0x8000u ||", "lower >= 0x8000u ||"),
    ("widen_kind_swap", "if (kind == 0)\n        a[m * K + k] = orc_bf16_to_float",
     "if (kind == 1)\n        a[m * K + k] = orc_bf16_to_float"),
    ("fp64_term_sign", "acc64 += term;", "acc64 -= term;"),
    ("qsum_off_by_one", "for (int i = 0; i < ORC_GROUP; ++i) t +=", "for (int i = 1; i < ORC_GROUP; ++i) t +="),
    ("gated_halves_swapped", "double g = y64[m * N + n];\n      double u = y64[m * N + I + n];",
     "double u = y64[m * N + n];\n      double g = y64[m * N + I + n];"),
    ("gated_exp_sign", "g / (1.0 + exp(-g)) * u", "g / (1.0 + exp(g)) * u"),
    ("gated_sigmoid_only", "g / (1.0 + exp(-g)) * u", "1.0 / (1.0 + exp(-g)) * u"),
    ("fwht_unnormalised", "v[j] = v[j] * 0.03125f;", "v[j] = v[j] * 1.0f;"),
    ("fwht_butterfly_swapped", "v[j] = a + c;\n        v[j + h] = a - c;",
     "v[j] = a - c;\n        v[j + h] = a + c;"),
    ("sumsq_sequential", "for (int i = 0; i < len; ++i) p[i] = p[i] + p[i + len];",
     "for (int i = 1; i < 2 * len; ++i) if (len == 1024) p[0] = p[0] + p[i];"),
    ("norm_weight_no_offset", "(orc_bf16_to_float(w[j]) + 1.0f)", "(orc_bf16_to_float(w[j]) + 0.0f)"),
    ("norm_eps_dropped", "1.0f / sqrtf(mean + eps)", "1.0f / sqrtf(mean)"),
    ("norm_sign_dropped", "* (float)sign[j];", "* 1.0f;"),
    ("grouped_scale_index", "float xs = sx[m * GA + g * H + h];", "float xs = sx[m * GA + g * H];"),
    ("grouped_quant_range", "for (int i = 0; i < A; ++i) {\n        float v = fabsf(x[i]);",
     "for (int i = 0; i < ORC_GROUP && g * A + i < K; ++i) {\n        float v = fabsf(x[i]);"),
    ("grouped_dot_offset", "int64_t k = j * A + i;", "int64_t k = j * A + i + 1 - (i + 1) / A;"),
    ("grouped_weight_group", "float ws = orc_half_to_float(scales[n * G + g]);\n        for (int64_t h",
     "float ws = orc_half_to_float(scales[n * G + (g * H) % G]);\n        for (int64_t h"),
    ("ptq_trit_carry", "v = w & 0xFFu;", "v = w & 0x7Fu;"),
    ("ptq_trit_low_digit", "t = w >> 8;", "t = v % 3u;"),
    ("ptq_weight_order", "int k = 24 * lv + j;", "int k = 5 * j + lv;"),
    ("ptq_qh_order", "int k = 120 + 2 * lv + j;", "int k = 120 + 4 * j + lv;"),
    ("ptq_scale_first", "(uint16_t)(blk[26] | (blk[27] << 8))", "(uint16_t)(blk[0] | (blk[1] << 8))"),
    ("ptq_scale_big_endian", "(uint16_t)(blk[26] | (blk[27] << 8))", "(uint16_t)(blk[27] | (blk[26] << 8))"),
    ("norm_residual_dropped", "if (residual) a = a + orc_bf16_to_float", "if (0) a = a + orc_bf16_to_float"),
]


@pytest.mark.parametrize("name,orig,bad", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, name, orig, bad):
    src = open(SRC).read()
    assert src.count(orig) >= 1, f"mutation anchor not found: {name}"
    mutated = src.replace(orig, bad, 1)
    c_path = tmp_path / f"{name}.c"
    so_path = tmp_path / f"{name}.so"
    c_path.write_text(mutated)
    subprocess.run(["gcc", *O._CFLAGS, str(c_path), "-o", str(so_path), "-lm"],
                   check=True)
    lib = O.load(str(so_path))
    failed = []
    for pin in P.ALL_PINS:
        try:
            pin(lib)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin caught mutant {name}"
