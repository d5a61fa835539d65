"""Plant plausible mistakes in copies of the oracle; every one must trip a pin.

Each mutant is a copy of oracle/bl_oracle.c with one textual change (or a
consistent set of changes, e.g. a code table swapped in both the packer and
the decoder so that round trips still pass).  The copy is compiled on the CPU
and the whole pin suite runs against it; the test fails if a mutant passes
every pin.  Mistakes are planted only in the oracle, only on the CPU.
"""
import os
import subprocess

import pytest

import pins
from oracle import oracle as O

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "bl_oracle.c")

MUTANTS = {
    "i2s_shift_order": [("return 6 - 2 * (int)((e % 128) / 32);", "return 2 * (int)((e % 128) / 32);")],
    "i2s_byte_order": [("(e / 128) * 32 + (e % 32);", "(e / 128) * 32 + (31 - e % 32);")],
    "i2s_decode_sign": [("{-1, 0, 1, 99}", "{1, 0, -1, 99}")],
    "i2s_table_swapped_both_ways": [("{-1, 0, 1, 99}", "{1, 0, -1, 99}"),
                                    ("if (w == -1) return 0;", "if (w == -1) return 2;"),
                                    ("if (w == 1) return 2;", "if (w == 1) return 0;")],
    "i2s_scale_at_start": [("const double s = (double)read_f32_le(packed + N * (K / 4));",
                            "const double s = (double)read_f32_le(packed);")],
    "i2s_dropped_scale": [("y[r] = s * acc;", "y[r] = acc;")],
    "i2s_x_reversed": [("acc += (double)w * x[e];", "acc += (double)w * x[K - 1 - e];")],
    "i2s_int8_q_transposed": [("acc += (int64_t)q[m * K + k] * w;", "acc += (int64_t)q[k * M + m] * w;")],
    "i2s_int8_dropped_token_scale": [("y[m * nrows + r] = (double)acc * sm * sw;",
                                      "y[m * nrows + r] = (double)acc * sw;")],
    "gate_up_relu_on_up": [("const double a = g[r] > 0.0 ? g[r] : 0.0;\n      h[r] = a * a * u[r];",
                            "const double a = g[r];\n      h[r] = a * a * (u[r] > 0.0 ? u[r] : 0.0);")],
    "gate_up_not_squared": [("h[r] = a * a * u[r];", "h[r] = a * u[r];")],
    "gate_up_scales_swapped": [("int st = orc_gemv_i2s(packed_gate, x, N, K, rows, nrows, g, cg);",
                                "int st = orc_gemv_i2s(packed_up, x, N, K, rows, nrows, g, cg);"),
                               ("if (st == ORC_OK) st = orc_gemv_i2s(packed_up, x, N, K, rows, nrows, u, cu);",
                                "if (st == ORC_OK) st = orc_gemv_i2s(packed_gate, x, N, K, rows, nrows, u, cu);")],
    "norm_dropped_eps": [("inv = 1.0 / sqrt(ss / (double)K + eps);", "inv = 1.0 / sqrt(ss / (double)K);")],
    "norm_sum_not_mean": [("inv = 1.0 / sqrt(ss / (double)K + eps);", "inv = 1.0 / sqrt(ss + eps);")],
    "norm_weight_ignored": [("xn[e] = rms_w ? x[e] * inv * rms_w[e] : x[e];", "xn[e] = rms_w ? x[e] * inv : x[e];")],
    "residual_dropped": [("y[r] += residual[rows ? rows[r] : r];", "y[r] += 0.0;")],
    "tq2_decode_sign": [("{0, 1, 99, -1}", "{0, -1, 99, 1}")],
    "tq2_shift_order_both_ways": [("return tq2_value_of((blk[j / 4] >> (2 * (j % 4))) & 3);",
                                   "return tq2_value_of((blk[j / 4] >> (6 - 2 * (j % 4))) & 3);"),
                                  ("blk[j / 4] |= (uint8_t)(code << (2 * (j % 4)));",
                                   "blk[j / 4] |= (uint8_t)(code << (6 - 2 * (j % 4)));")],
    "tq2_scale_byte_order": [("(uint16_t)(blk[64] | (blk[65] << 8))", "(uint16_t)(blk[65] | (blk[64] << 8))")],
    "tq2_dropped_block_scale": [("total += d * blk;", "total += blk;")],
    "tq2_block_stride_both_ways": [("return packed + (n * (K / 256) + b) * 66;", "return packed + (n * (K / 256) + b) * 64;"),
                                   ("uint8_t* blk = out + (n * nb + b) * 66;", "uint8_t* blk = out + (n * nb + b) * 64;")],
    "tq2_int8_dropped_block_scale": [("total += d * (double)dot;", "total += (double)dot;")],
    "tq2_int8_dropped_token_scale": [("y[m * nrows + r] = sm * total;", "y[m * nrows + r] = total;")],
    "tq2_int8_q_transposed": [("dot += (int64_t)q[m * K + e] * w;", "dot += (int64_t)q[e * M + m] * w;")],
    "tq2_int8_q_block_shift": [("dot += (int64_t)q[m * K + e] * w;", "dot += (int64_t)q[m * K + (e + 1) % K] * w;")],
    "w1_bit_order_both_ways": [("word |= bit << i;", "word |= bit << (31 - i);"),
                               ("return ((word >> (k % 32)) & 1u) ? 1 : -1;", "return ((word >> (31 - k % 32)) & 1u) ? 1 : -1;")],
    "w1_zero_as_plus": [("const uint32_t bit = (v == 1) ? 1u : 0u;", "const uint32_t bit = (v >= 0) ? 1u : 0u;")],
    "w1_zero_weight": [("return ((word >> (k % 32)) & 1u) ? 1 : -1;", "return ((word >> (k % 32)) & 1u) ? 1 : 0;")],
    "w1a8_dropped_bias": [("y[m * nrows + r] = sm * acc + b;", "y[m * nrows + r] = sm * acc;")],
    "w1a8_scale_transposed": [("const double wsg = orc_fp16_to_double(ws[n * ng + g]);",
                               "const double wsg = orc_fp16_to_double(ws[g * N + n]);")],
    "act_truncate": [("float r = rintf(t);", "float r = truncf(t);")],
    "act_128": [("volatile float inv = 127.0f / amax;", "volatile float inv = 128.0f / amax;")],
    "act_scale_inverted": [("volatile float sv = amax / 127.0f;", "volatile float sv = 127.0f / amax;")],
    "fp16_subnormal": [("v = ldexp((double)m, -24);", "v = ldexp((double)m, -25);")],
    "fp16_bias": [("v = ldexp((double)(1024 + m), e - 25);", "v = ldexp((double)(1024 + m), e - 24);")],
    "bf16_subnormal": [("v = ldexp((double)m, -133);", "v = ldexp((double)m, -134);")],
    "bf16_round_ties_away": [("double r = nearbyint(ldexp(f, 8));", "double r = round(ldexp(f, 8));")],
    "i2s_code_not_centered": [("acc += (double)w * x[e];", "acc += (double)(w + 1) * x[e];")],
    "i2s_int8_code_not_centered": [("acc += (int64_t)q[m * K + k] * w;", "acc += (int64_t)q[m * K + k] * (w + 1);")],
    "gate_up_dropped_relu": [("const double a = g[r] > 0.0 ? g[r] : 0.0;", "const double a = g[r];")],
    "w1a8_dropped_token_scale": [("y[m * nrows + r] = sm * acc + b;", "y[m * nrows + r] = acc + b;")],
    "w1a8_next_group_scale": [("const double wsg = orc_fp16_to_double(ws[n * ng + g]);",
                               "const double wsg = orc_fp16_to_double(ws[n * ng + (g + 1) % ng]);")],
    "act_amax_signed": [("const float a = fabsf(v);", "const float a = v;")],
    "w1a8_cond_without_bias": [("if (cond) cond[m * nrows + r] = fabs(sm) * c + fabs(b);",
                                "if (cond) cond[m * nrows + r] = fabs(sm) * c;")],
    "gate_up_cond_first_term_dropped": [("if (cond) cond[r] = 2.0 * a * fabs(u[r]) * cg[r] + a * a * cu[r];",
                                         "if (cond) cond[r] = a * a * cu[r];")],
    "act_in_double": [("volatile float t = v * inv;", "volatile float t = (float)((double)v * (127.0 / (double)amax));")],
    "norm_not_inverted": [("inv = 1.0 / sqrt(ss / (double)K + eps);", "inv = sqrt(ss / (double)K + eps);")],
    "residual_scaled": [("y[r] += residual[rows ? rows[r] : r];", "y[r] = (y[r] + residual[rows ? rows[r] : r]) * 2.0;")],
    "w1a8_bias_scaled": [("y[m * nrows + r] = sm * acc + b;", "y[m * nrows + r] = sm * (acc + b);")],
    "fp16_sign_dropped": [("  return sign ? -v : v;\n}\n\n/* bfloat16", "  return v;\n}\n\n/* bfloat16")],
    "bf16_truncate": [("double r = nearbyint(ldexp(f, 8));", "double r = floor(ldexp(f, 8));")],
}


def _build_mutant(tmp_path, name, edits):
    src = open(SRC).read()
    for old, new in edits:
        assert src.count(old) == 1, "mutation anchor not unique/absent: %r" % old
        src = src.replace(old, new)
    c = tmp_path / (name + ".c")
    c.write_text(src)
    so = tmp_path / (name + ".so")
    subprocess.run(["gcc", "-std=c99", "-O1", "-fPIC", "-shared", "-ffp-contract=off", str(c), "-o", str(so), "-lm"],
                   check=True, capture_output=True)
    return str(so)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path, oracle_lib):
    path = _build_mutant(tmp_path, name, MUTANTS[name])
    saved = O._lib
    O._lib = O.load(path)
    failed = []
    try:
        for pin in pins.ALL_PINS:
            try:
                pin()
            except (AssertionError, O.OracleError):
                failed.append(pin.__name__)
    finally:
        O._lib = saved
    assert failed, "planted mistake %s passed every pin" % name
