"""Planted mistakes in copies of the oracle must each fail at least one pin (no GPU).

Each mutant is the oracle's C source with one plausible mistake planted by a
text substitution, compiled into a temporary directory.  The real oracle is
never modified.
"""
import os
import tempfile

import pytest

import oracle
from tests import oracle_pins

MUTANTS = [
    # quantiser
    ("reciprocal_multiply", "roundf(x[i] / d)", "roundf(x[i] * (1.0f / d))"),
    ("round_half_even", "roundf(x[i] / d)", "rintf(x[i] / d)"),
    ("truncate", "(int8_t)(int)roundf(x[i] / d)", "(int8_t)(int)(x[i] / d)"),
    ("scale_128", "amax / 127.0f", "amax / 128.0f"),
    ("signed_max", "float a = fabsf(x[i]);", "float a = x[i];"),
    ("store_f32_trunc", "dh = q8o_f32_to_f16(d);", "dh = (uint16_t)(q8o_f32_to_f16(d) & 0xfffeu);"),
    # binary16
    ("f16_ties_away", "if (rest > 0x1000u || (rest == 0x1000u && (keep & 1u)))", "if (rest >= 0x1000u)"),
    ("f16_flush_subnormal", "int shift = -(e + 1);", "int shift = 40;"),
    ("f16_decode_bias", "v = ldexpf((float)(1024 + f), e - 25);", "v = ldexpf((float)(1024 + f), e - 24);"),
    ("f16_decode_subnormal", "v = ldexpf((float)f, -24);", "v = ldexpf((float)(1024 + f), -25);"),
    # dot
    ("drop_last_block", "acc += (dw * dx) * (float)isum;", "if (b + 1 < nb) acc += (dw * dx) * (float)isum;"),
    ("wrong_index", "(int32_t)blk_q(ab, i)", "(int32_t)blk_q(ab, QK - 1 - i)"),
    ("wrong_sign", "acc += (dw * dx) * (float)isum;", "acc -= (dw * dx) * (float)isum;"),
    ("missing_scale", "acc += (dw * dx) * (float)isum;", "acc += dw * (float)isum;"),
    ("transposed", "out[t * out_dim + o] = q8o_dot_row(W + o * nb * QBYTES, xq + t * nb * QBYTES, nb, &bd);",
     "out[t * out_dim + o] = q8o_dot_row(W + (o % n_tok) * nb * QBYTES, xq + (t % out_dim) * nb * QBYTES, nb, &bd);"),
    ("d_byte_order", "(uint16_t)(blk[0] | ((uint16_t)blk[1] << 8))", "(uint16_t)(blk[1] | ((uint16_t)blk[0] << 8))"),
    ("q_offset", "return (int8_t)blk[2 + i];", "return (int8_t)blk[1 + i];"),
    # routed experts
    ("moe_row_choice", "xq + (x_per_pair ? p : t) * nb * QBYTES", "xq + (x_per_pair ? t : p % n_tok) * nb * QBYTES"),
    ("moe_expert_stride", "W_experts + (uint64_t)e * expert_stride + o * nb * QBYTES", "W_experts + (uint64_t)e * out_dim * nb * QBYTES + o * nb * QBYTES"),
    ("moe_no_flag", "                    flag = 1;\n                } else {\n                    const uint8_t *w", "                    flag = 0;\n                } else {\n                    const uint8_t *w"),
    # the expert FFN around the routed product
    ("swiglu_sigmoid", "mid[i] = (float)(g / (1.0 + exp(-g)) * u);", "mid[i] = (float)(1.0 / (1.0 + exp(-g)) * u);"),
    ("swiglu_exp_sign", "mid[i] = (float)(g / (1.0 + exp(-g)) * u);", "mid[i] = (float)(g / (1.0 + exp(g)) * u);"),
    ("swiglu_swapped", "double g = gate[i], u = up[i];", "double g = up[i], u = gate[i];"),
    ("swiglu_no_up_floor", "if (u < -limit) u = -limit;", ";"),
    ("swiglu_gate_floor", "if (g > limit) g = limit;", "if (g > limit) g = limit;\n            if (g < -limit) g = -limit;"),
    ("swiglu_always_clamped", "if (limit > 0.0f) {", "if (limit >= 0.0f) {"),
    ("combine_drop_last", "for (uint32_t j = 0; j < k; ++j) {\n                uint64_t p = t * k + j;",
     "for (uint32_t j = 0; j + 1 < k; ++j) {\n                uint64_t p = t * k + j;"),
    ("combine_unweighted", "double v = (double)w[p] * (double)y[p * dim + o];", "double v = (double)y[p * dim + o];"),
    ("ffn_up_as_gate", "q8o_moe(gate, NULL, W_gate,", "q8o_moe(gate, NULL, W_up,"),
    ("ffn_down_token_rows", "midq, 1, n_tok);", "midq, 0, n_tok);"),
    ("ffn_down_gate_stride", "q8o_moe(y, y_bound, W_down, n_expert, down_stride,", "q8o_moe(y, y_bound, W_down, n_expert, gate_up_stride,"),
    ("ffn_no_bad_flag", "rc = (f1 < 0 || f2 < 0 || f3 < 0) ? -1 : (f1 | f2 | f3);", "rc = (f1 < 0 || f2 < 0 || f3 < 0) ? -1 : 0;"),
    # RMSNorm feeding the quantiser
    ("rms_sum_not_mean", "double r = 1.0 / sqrt(s / (double)dim + eps);", "double r = 1.0 / sqrt(s + eps);"),
    ("rms_no_sqrt", "double r = 1.0 / sqrt(s / (double)dim + eps);", "double r = 1.0 / (s / (double)dim + eps);"),
    ("rms_eps_outside", "double r = 1.0 / sqrt(s / (double)dim + eps);", "double r = 1.0 / sqrt(s / (double)dim) + eps;"),
    ("rms_no_gamma", "(gamma ? (double)gamma[i] : 1.0)", "1.0"),
    ("rms_quantise_x", "return q8o_quantize(xq, y, dim, n_tok);", "return q8o_quantize(xq, x, dim, n_tok);"),
    ("rms_abs_sum", "s += (double)xr[i] * (double)xr[i];", "s += fabs((double)xr[i]);"),
    # second weight format (K-quant blocks x Q8_K)
    ("q2k_scale_min_swapped", "*sc = blk[sb] & 15;\n        *m = blk[sb] >> 4;", "*sc = blk[sb] >> 4;\n        *m = blk[sb] & 15;"),
    ("q2k_field_order", "*q = (blk[16 + 32 * h + 16 * s + l] >> (2 * j)) & 3;", "*q = (blk[16 + 32 * h + 16 * s + l] >> (6 - 2 * j)) & 3;"),
    ("q2k_byte_order", "*q = (blk[16 + 32 * h + 16 * s + l] >> (2 * j)) & 3;", "*q = (blk[16 + 16 * h + 32 * s + l] >> (2 * j)) & 3;"),
    ("q2k_subblock", "int sb = 8 * h + 2 * j + s;", "int sb = 8 * h + j + 4 * s;"),
    ("q2k_d_offset", "*d = q8o_f16_to_f32(le16(blk + 80));", "*d = q8o_f16_to_f32(le16(blk + 82));"),
    ("q4k_nibbles_swapped", "*q = hi ? (byte >> 4) : (byte & 15);", "*q = hi ? (byte & 15) : (byte >> 4);"),
    ("q4k_high_scale_bits", "*sc = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);", "*sc = (s[j + 4] & 15) | ((s[j - 4] >> 4) << 4);"),
    ("q4k_min_low", "*m = s[j + 4] & 63;", "*m = s[j] & 63;"),
    ("q4k_min_high", "*m = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);", "*m = (s[j + 4] >> 4) | ((s[j - 4] >> 6) << 4);"),
    ("q4k_dmin_offset", "*dmin = q8o_f16_to_f32(le16(blk + 2));", "*dmin = q8o_f16_to_f32(le16(blk));"),
    ("kq_min_added", "w[i] = d * (double)sc * (double)q - dmin * (double)m;", "w[i] = d * (double)sc * (double)q + dmin * (double)m;"),
    ("q8k_scale_128", "float scale = amax / 127.0f;", "float scale = amax / 128.0f;"),
    ("q8k_round_even", "qb[i] = scale != 0.0f ? (int8_t)(int)roundf(xb[i] / scale) : 0;", "qb[i] = scale != 0.0f ? (int8_t)(int)rintf(xb[i] / scale) : 0;"),
    ("kq_dot_drop_block", "    for (uint64_t b = 0; b < nsb; ++b) {\n        const uint8_t *blk = w + b * bb;", "    for (uint64_t b = 0; b + 1 < nsb; ++b) {\n        const uint8_t *blk = w + b * bb;"),
    ("kq_dot_block_scale", "        double xd = (double)dx[b];", "        double xd = (double)dx[0];"),
    ("kq_moe_row", "uint64_t xr = x_per_pair ? p : p / k;", "uint64_t xr = x_per_pair ? p / k : p;"),
    ("kq_moe_stride", "W_experts + (uint64_t)e * expert_stride + o * nsb * bb", "W_experts + (uint64_t)e * out_dim * bb + o * nsb * bb"),
]


@pytest.fixture(scope="module")
def source():
    with open(oracle.SOURCE) as f:
        return f.read()


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(source, name, old, new):
    assert source.count(old) >= 1, f"mutation site for {name} not found in the oracle source"
    mutated = source.replace(old, new)
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, f"mut_{name}.c")
        lib = os.path.join(d, f"libmut_{name}.so")
        with open(src, "w") as f:
            f.write(mutated)
        oracle.compile_lib(src, lib)
        m = oracle.Oracle(lib)
        failed = []
        for pin in oracle_pins.ALL_PINS:
            try:
                pin(m)
            except AssertionError:
                failed.append(pin.__name__)
            except Exception:  # a crash on the mutant also counts as caught
                failed.append(pin.__name__ + "(error)")
        assert failed, f"planted mistake {name!r} passed every pin"
