"""Plant plausible mistakes in copies of the oracle and check that the pins catch each.

Each mutant is the oracle's C source with one textual change, compiled into a
temporary directory; the real oracle is never modified.  A mutant that passed
every pin would mean the pins leave that part of the oracle unchecked.

Reordering the dequant's multiplications, e.g. d*(sc*q) for (d*sc)*q, is not
a mutant: every product of an fp16 scale, a 6-bit (Q4_K) or int8 (Q6_K)
scale and a quant is exact in fp32 (21 and 23 significant bits).  Any order
gives the same bits; the pin that every weight is its exact value rounded
once to fp32 states that directly.
"""
import os

import pytest

import oracle
from tests import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "qk_oracle.c")

# (name, exact text in the oracle, replacement)
MUTANTS = [
    ("q4k_nibble_halves_swapped", "(i % 64) < 32 ? (byte & 0x0F)", "(i % 64) >= 32 ? (byte & 0x0F)"),
    ("q4k_qs_byte_index", "qs[32 * (i / 64) + (i % 32)]", "qs[(i / 2) % 128]"),
    ("q4k_scale_high_bits_wrong_byte", "*sc = (s[j + 4] & 0x0F) | ((s[j - 4] >> 6) << 4);",
     "*sc = (s[j + 4] & 0x0F) | ((s[j] >> 6) << 4);"),
    ("q4k_min_high_bits_wrong_byte", "*mn = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);",
     "*mn = (s[j + 4] >> 4) | ((s[j - 4] >> 6) << 4);"),
    ("q4k_low_scale_min_swapped", "*sc = s[j] & 63;\n        *mn = s[j + 4] & 63;",
     "*sc = s[j + 4] & 63;\n        *mn = s[j] & 63;"),
    ("q4k_min_sign", "out[i] = t - dmn;", "out[i] = t + dmn;"),
    ("q4k_min_uses_d", "const float dmn = dmin * (float)mn;", "const float dmn = d * (float)mn;"),
    ("q4k_subblock_of_64", "q4k_scale_min(s, i / 32, &sc, &mn);", "q4k_scale_min(s, i / 64, &sc, &mn);"),
    ("q6k_offset", "return (lo | (hi << 4)) - 32;", "return (lo | (hi << 4)) - 31;"),
    ("q6k_scale_index", "d * (float)sc[i / 16]", "d * (float)sc[i / 32]"),
    ("q6k_qh_shift", "(qh[32 * h + l] >> (2 * g)) & 3", "(qh[32 * h + l] >> (2 * (3 - g))) & 3"),
    ("q6k_ql_group", "ql[64 * h + 32 * (g & 1) + l]", "ql[64 * h + 32 * (g >> 1) + l]"),
    ("q6k_nibble_select", "g < 2 ? (lb & 0x0F) : (lb >> 4)", "g < 1 ? (lb & 0x0F) : (lb >> 4)"),
    ("q6k_d_offset", "oracle_half_to_float(rd16(blk + 208))", "oracle_half_to_float(rd16(blk + 206))"),
    ("half_subnormal_scale", "ldexpf((float)frac, -24)", "ldexpf((float)frac, -25)"),
    ("half_exponent_bias", "expo - 25);", "expo - 24);"),
    ("half_nan_as_inf", "if (expo == 31 && frac) {", "if (expo == 32 && frac) {"),
    ("matmul_k_misaligned", "acc += xm[k] * (double)w[k];", "acc += xm[k] * (double)w[(k + 1) % K];"),
    ("matmul_wrong_token_row", "const double *xm = xd + m * K;\n                double acc",
     "const double *xm = xd + (M - 1 - m) * K;\n                double acc"),
    ("matmul_fp32_accumulate", "double acc = 0.0;", "float acc = 0.0f;"),
    ("gateup_swapped", "g += xm[k] * (double)wg[k];\n                    u += xm[k] * (double)wu[k];",
     "g += xm[k] * (double)wu[k];\n                    u += xm[k] * (double)wg[k];"),
    ("silu_sign", "g / (1.0 + exp(-g))", "g / (1.0 + exp(g))"),
    ("swiglu_times_gate", "out[m * n_rows + r] = silu * u;", "out[m * n_rows + r] = silu * g;"),
    ("silu_of_up", "const double silu = g / (1.0 + exp(-g));", "const double silu = u / (1.0 + exp(-u));"),
    # field offsets inside a block
    ("q4k_dmin_offset", "rd16(blk + 2)", "rd16(blk)"),
    ("q4k_scales_offset", "const uint8_t *s = blk + 4;", "const uint8_t *s = blk + 3;"),
    ("q4k_quants_offset", "const uint8_t *qs = blk + 16;", "const uint8_t *qs = blk + 15;"),
    ("q6k_qh_offset", "const uint8_t *qh = blk + 128;", "const uint8_t *qh = blk + 64;"),
    ("q6k_scales_unsigned", "const int8_t *sc = (const int8_t *)(blk + 192);",
     "const uint8_t *sc = (const uint8_t *)(blk + 192);"),
    ("q6k_lane_of_16", "l = i % 32;", "l = i % 16;"),
    ("half_sign_dropped", "return sign ? -v : v;", "return v;"),
    # RMSNorm in front of a linear
    ("rms_eps_outside_sqrt", "1.0 / sqrt(ss / (double)K + eps)", "1.0 / (sqrt(ss / (double)K) + eps)"),
    ("rms_mean_of_x", "ss += v * v;", "ss += v;"),
    ("rms_sum_not_mean", "sqrt(ss / (double)K + eps)", "sqrt(ss + eps)"),
    ("rms_gamma_dropped", "* inv * (double)oracle_half_to_float(gamma[k]);", "* inv;"),
    ("rms_gamma_reversed", "oracle_half_to_float(gamma[k])", "oracle_half_to_float(gamma[K - 1 - k])"),
    ("rms_matmul_eps_ignored", "int rc = oracle_rmsnorm(x, gamma, M, K, eps, xn);\n    if (rc == 0)\n        rc = matmul_core",
     "int rc = oracle_rmsnorm(x, gamma, M, K, 0.0, xn);\n    if (rc == 0)\n        rc = matmul_core"),
    ("rms_gateup_up_as_gate", "rc = gateup_core(Wg, Wu, xn", "rc = gateup_core(Wg, Wg, xn"),
    # Q8 activations
    ("q8_divide_by_128", "volatile float db = amax / 127.0f;", "volatile float db = amax / 128.0f;"),
    ("q8_ties_to_even", "const float t = roundf(r);", "const float t = rintf(r);"),
    ("q8_truncate", "const float t = roundf(r);", "const float t = truncf(r);"),
    ("q8_amax_half_block", "for (int i = 0; i < 32; ++i) {\n                const float v = fabsf",
     "for (int i = 0; i < 16; ++i) {\n                const float v = fabsf"),
    ("q8_scale_of_64", "(double)d[(i / K) * (K / 32) + (i % K) / 32]", "(double)d[(i / K) * (K / 32) + (i % K) / 64]"),
    ("q8_amax_signed", "const float v = fabsf(oracle_half_to_float(xb[i]));",
     "const float v = oracle_half_to_float(xb[i]);"),
    # GQA attention
    ("attn_group_modulo", "const int64_t g = h / group;", "const int64_t g = h % Hkv;"),
    ("attn_sees_one_less", "const int64_t n = pos0 + i + 1;", "const int64_t n = pos0 + i + (i > 0);"),
    ("attn_sees_one_more", "const int64_t n = pos0 + i + 1;", "const int64_t n = pos0 + i + 1 + (pos0 + i + 1 < Lmax);"),
    ("attn_scale_dropped", "s[j] = scale * dot;", "s[j] = dot;"),
    ("attn_not_normalized", "const double p = s[j] / denom;", "const double p = s[j];"),
    ("attn_token_major_cache", "const uint16_t *kj = kc + (g * Lmax + j) * D;",
     "const uint16_t *kj = kc + (j * Hkv + g) * D;"),
    ("attn_values_are_keys", "const uint16_t *vj = vc + (g * Lmax + j) * D;",
     "const uint16_t *vj = kc + (g * Lmax + j) * D;"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, "mutation anchor must match exactly once: %r" % old
    msrc = tmp_path / "mutant.c"
    msrc.write_text(src.replace(old, new))
    O = oracle.Oracle(oracle.build(force=True, src=str(msrc), out=str(tmp_path / "libmutant.so")))
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(O)
        except AssertionError:
            caught.append(pin.__name__)
            break
    assert caught, "no pin catches mutant %s" % name
