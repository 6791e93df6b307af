"""The pins must catch plausible mistakes in the oracle.

Each mutant is a copy of ``oracle/bq_oracle.c`` with one planted mistake (a
wrong divisor, tie rule, sign, index, nibble order, dropped term, transposed
operand...).  It is compiled on the CPU into a temporary library and the quick
pin checks run against it; at least one of them must fail.  Each mutation
names a substring that must still occur in the source, so a rewrite of the
oracle that silently disarms a mutant fails here instead.
"""
import os

import pytest

import oracle
from oracle import build as obuild

import oracle_checks as checks

# (name, original substring, mutated substring); the first occurrence is mutated
MUTANTS = [
    ("q8_divisor", "float d32 = amax / 127.0f;", "float d32 = amax / 128.0f;"),
    ("q4_divisor", "float d32 = amax / 8.0f;", "float d32 = amax / 7.0f;"),
    ("bankers_round", "float r = roundf(w[j] / df);", "float r = rintf(w[j] / df);"),
    ("q8_clamp", "if (r < -127.0f) r = -127.0f;", "if (r < -128.0f) r = -128.0f;"),
    ("q4_clamp", "if (r > 15.0f) r = 15.0f;", "if (r > 16.0f) r = 16.0f;"),
    ("q4_pack_bias", "r = roundf(w[j] / df) + 8.0f;", "r = roundf(w[j] / df) + 7.0f;"),
    ("nibble_order_pack", "(uint8_t)(n[j] | (n[j + 16] << 4))",
     "(uint8_t)((n[j] << 4) | n[j + 16])"),
    ("nibble_order_dequant", "(j < 16) ? (byte & 0xF) : (byte >> 4)",
     "(j < 16) ? (byte >> 4) : (byte & 0xF)"),
    ("q4_dequant_bias", "return d * (double)(nib - 8);", "return d * (double)(nib - 7);"),
    ("q8_unsigned", "return d * (double)(int8_t)blk[2 + j];",
     "return d * (double)(uint8_t)blk[2 + j];"),
    ("scale_byte_order_read", "(uint16_t)(blk[0] | (blk[1] << 8))",
     "(uint16_t)(blk[1] | (blk[0] << 8))"),
    ("scale_byte_order_write", "blk[0] = (uint8_t)(dh & 0xFFu);\n    blk[1] = (uint8_t)(dh >> 8);",
     "blk[1] = (uint8_t)(dh & 0xFFu);\n    blk[0] = (uint8_t)(dh >> 8);"),
    ("signed_amax", "float a = fabsf(w[j]);", "float a = w[j];"),
    ("f16_ties_away", "if (rem > half || (rem == half && (m & 1u))) m += 1u;",
     "if (rem >= half) m += 1u;"),
    ("f16_subnormal_edge", "int qe = (e < -14) ? -24 : e - 10;",
     "int qe = (e < -15) ? -24 : e - 10;"),
    ("f16_to_f64_bias", "ldexp((double)(man + 1024), be - 25)",
     "ldexp((double)(man + 1024), be - 24)"),
    ("f16_to_f64_subnormal", "ldexp((double)man, -24)", "ldexp((double)man, -25)"),
    ("gemv_reversed_x", "(int)(k % 32)) * x[k];", "(int)(k % 32)) * x[K - 1 - k];"),
    ("gemv_dropped_term", "        for (int64_t k = 0; k < K; ++k) {",
     "        for (int64_t k = 0; k < K - 1; ++k) {"),
    ("gemv_S_signed", "sacc += fabs(p);", "sacc += p;"),
    ("dequant_transposed", "out[m * K + k] = dequant_elem(qtype, Wq + (m * nb + k / 32) * bb",
     "out[m * K + k] = dequant_elem(qtype, Wq + (k / 32 * M + m) * bb"),
    ("rms_eps_outside", "double r = 1.0 / sqrt(ss / (double)K + eps);",
     "double r = 1.0 / (sqrt(ss / (double)K) + eps);"),
    ("rms_sum_not_mean", "double r = 1.0 / sqrt(ss / (double)K + eps);",
     "double r = 1.0 / sqrt(ss / (double)(K - 1) + eps);"),
    ("rms_no_gamma", "* (gamma ? gamma[k] : 1.0)", "* 1.0"),
    ("silu_sign", "return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));"),
    ("gate_up_swapped", "y[m] = bqo_silu(gm) * um;", "y[m] = bqo_silu(um) * gm;"),
    ("bias_subtracted", "y[m] += bias[m];", "y[m] -= bias[m];"),
    ("bias_shifted_row", "y[m] += bias[m];", "y[m] += bias[m > 0 ? m - 1 : 0];"),
    ("bias_S_signed", "S[m] += fabs(bias[m]);", "S[m] += bias[m];"),
    ("f16_gemv_transposed", "bqo_f16_bits_to_f64(W[m * K + k])", "bqo_f16_bits_to_f64(W[k * M + m])"),
    ("f16_gemv_reversed_x", "(W[m * K + k]) * x[k];", "(W[m * K + k]) * x[K - 1 - k];"),
    ("f16_gemv_dropped_term", "for (int64_t k = 0; k < K; k++) {", "for (int64_t k = 1; k < K; k++) {"),
    ("f16_gemv_S_signed", "sacc += fabs(p); /* sum of |w x| */", "sacc += p; /* sum of |w x| */"),
    # Q4_K
    ("q4k_scale_mask", "*sc = s[j] & 63;", "*sc = s[j] & 31;"),
    ("q4k_min_high_bits", "*mn = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);",
     "*mn = (s[j + 4] >> 4) | ((s[j - 4] >> 6) << 4);"),
    ("q4k_nibble_order", "*q = (j & 1) ? (byte >> 4) : (byte & 0xF);",
     "*q = (j & 1) ? (byte & 0xF) : (byte >> 4);"),
    ("q4k_min_sign", "return D * (double)q - Mf;", "return D * (double)q + Mf;"),
    ("q4k_range_divisor", "scale[j] = (hi - lo) / 15.0f;", "scale[j] = (hi - lo) / 16.0f;"),
    ("q4k_super_divisor", "uint16_t dh = bqo_f32_to_f16_bits(smax / 63.0f);",
     "uint16_t dh = bqo_f32_to_f16_bits(smax / 64.0f);"),
    ("q4k_lo_unclamped", "float lo = 0.0f, hi = w[32 * j];", "float lo = w[32 * j], hi = w[32 * j];"),
    ("q4k_pair_bytes", "qs[32 * (j / 2) + i] |=", "qs[32 * (j % 4) + i] |="),
    ("q4k_sc_pack_shift", "s[j] = (uint8_t)(sc[j] | ((sc[j + 4] >> 4) << 6));",
     "s[j] = (uint8_t)(sc[j] | ((sc[j + 4] >> 3) << 6));"),
    ("q4k_dmin_bytes", "*Mf = bqo_f16_bits_to_f64((uint16_t)(sb[2] | (sb[3] << 8))) * (double)mn;",
     "*Mf = bqo_f16_bits_to_f64((uint16_t)(sb[0] | (sb[1] << 8))) * (double)mn;"),
    ("q4k_code_shift", "(w[32 * j + i] + Mf) / D", "(w[32 * j + i] - Mf) / D"),
    ("q4k_split_drops_min", "acc += D * fabs((double)q * x[k]) + Mf * fabs(x[k]);",
     "acc += D * fabs((double)q * x[k]);"),
    ("q4k_superblock_stride", "out + (m * ns + b) * 144", "out + (b * M + m) * 144"),
]


@pytest.fixture(scope="module")
def source():
    with open(obuild.SRC) as f:
        return f.read()


def test_real_oracle_passes_quick_pins():
    assert checks.run_quick(oracle.get()) == []


@pytest.mark.parametrize("name,orig,mut", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, orig, mut, source, tmp_path):
    assert orig in source, f"mutation site for {name} no longer in the oracle source"
    src = tmp_path / f"mutant_{name}.c"
    src.write_text(source.replace(orig, mut, 1))
    lib = obuild.compile_oracle(str(src), str(tmp_path / f"libmutant_{name}.so"), force=True)
    failed = checks.run_quick(oracle.Oracle(lib))
    assert failed, f"mutant {name} passed every quick pin"
    os.remove(lib)
