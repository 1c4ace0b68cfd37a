"""Planted mistakes in the CPU oracle must fail a pin.

Each case copies ``oracle/oracle.c`` to a temporary directory, applies one
plausible mistake (a dropped term, a wrong sign, a wrong divisor, a transposed
operand, a contracted multiply-add, a wrong rounding), builds it with the same
flags, and runs every pin of ``oracle_pins`` against it: at least one pin must
fail.  The real oracle is never modified.  Runs without a GPU.
"""
import os
import shutil

import pytest

import oracle
from oracle import build as oracle_build
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle_build.__file__), "oracle.c")
HDR = os.path.join(os.path.dirname(oracle_build.__file__), "oracle.h")

MUTANTS = {
    # o1: y = relu(x + b1) * scale + b2
    "o1_sign_b2": ("tmp = tmp + b2;", "tmp = tmp - b2;"),
    "o1_drop_relu": ("tmp = oracle_relu_f32(tmp);", "(void)0;"),
    "o1_fixed_scale": ("tmp = tmp * scale;", "tmp = tmp * 0.5f;"),
    "o1_fma": ("tmp = tmp * scale;              /* step 3: * scale   -> tmp3 */\n"
               "    tmp = tmp + b2;",
               "tmp = fmaf(tmp, scale, b2);"),
    "relu_keeps_neg_zero": ("if (v > 0.0f)", "if (v >= 0.0f)"),
    "o1_bcast_row_index": ("int64_t k = per_col ? j : i * cols + j;",
                           "int64_t k = per_col ? i % cols : i * cols + j;"),
    "o1_bcast_flags_swapped": ("o1_operand(b1, bf16, b1_per_col, i, j, cols)",
                               "o1_operand(b1, bf16, b2_per_col, i, j, cols)"),
    # o2: TorchInductor example chain
    "o2_mean_divisor": ("float m = (float)(sum / (double)cols);",
                        "float m = (float)(sum / (double)(cols + 1));"),
    "o2_gamma_beta_swapped": ("d = d * gamma[j];", "d = d * beta[j];"),
    "o2_branch_uses_x_scale": ("float q = a * branch_scale;", "float q = a * x_scale;"),
    "o2_drop_x_scale": ("float t = x * x_scale;", "float t = x;"),
    "o2_drop_square": ("float p = a * a;", "float p = a;"),
    "o2_sign_mean": ("float d = s - m;", "float d = s + m;"),
    "o2_no_relu": ("float a = oracle_relu_f32(t);", "float a = t;"),
    # o3: residual + LayerNorm + GeLU
    "o3_drop_eps": ("double rstd = 1.0 / sqrt(var + (double)eps);",
                    "double rstd = 1.0 / sqrt(var);"),
    "o3_unbiased_var": ("double var = sq / (double)hidden;",
                        "double var = sq / (double)(hidden - 1);"),
    "o3_uncentred_var": ("double d = (double)v - mean;", "double d = (double)v;"),
    "o3_mean_divisor": ("double mean = sum / (double)hidden;",
                        "double mean = sum / (double)(hidden + 1);"),
    "o3_drop_rstd": ("double xhat = ((double)v - mean) * rstd;",
                     "double xhat = ((double)v - mean);"),
    "o3_w_b_swapped": ("double n = xhat * (double)load(w, j) + (double)load(b, j);",
                       "double n = xhat * (double)load(b, j) + (double)load(w, j);"),
    "o3_residual_sign": ("float v = load(x, base + j) + load(r, base + j);",
                         "float v = load(x, base + j) - load(r, base + j);"),
    "gelu_cubic_dropped": ("0.044715 * z * z * z", "0.044715 * z * z"),
    "gelu_tanh_sign": ("return 0.5 * z * (1.0 + tanh(u));",
                       "return 0.5 * z * (1.0 - tanh(u));"),
    "gelu_half_dropped": ("return 0.5 * z * (1.0 + tanh(u));",
                          "return z * (1.0 + tanh(u));"),
    "bf16_truncates": ("double k = rint(ldexp(a, -q));",
                       "double k = floor(ldexp(a, -q));"),
    "bf16_extra_bit": ("int q = e - 8;", "int q = e - 9;"),
    # o2 bf16
    "o2bf16_drop_beta": ("float o = d + widen_bf16(beta[j]);", "float o = d;"),
    # o4: LayerNorm family
    "o4_relu_dropped": ("return n > 0.0 ? n : 0.0;      /* relu", "return n;      /* relu"),
    "o4_drop_eps": ("double rstd = 1.0 / sqrt(sq / (double)hidden + (double)eps);",
                    "double rstd = 1.0 / sqrt(sq / (double)hidden);"),
    "o4_h_is_x": ("((float *)h_out)[base + j] = v;",
                  "((float *)h_out)[base + j] = load(x, base + j);"),
    "o4_residual_ignored_in_stats": ("            if (r)\n                v = v + load(r, base + j);\n            sum += (double)v;",
                                     "            sum += (double)v;"),
    # o5: row softmax
    "o5_sum_unshifted": ("sum += exp((double)load(x, base + j) - m);",
                         "sum += exp((double)load(x, base + j));"),
    "o5_divide_by_cols": ("double p = exp((double)load(x, base + j) - m) / sum;",
                          "double p = exp((double)load(x, base + j) - m) / (double)cols;"),
    # o4 extras and o6: statistics out, Philox, dropout
    "stats_mean_is_sum": ("ex->mean_out[i] = mean;", "ex->mean_out[i] = sum;"),
    "stats_rstd_is_var": ("ex->rstd_out[i] = rstd;", "ex->rstd_out[i] = 1.0 / (rstd * rstd);"),
    "philox32_multiplier": ("0xD2511F53u", "0xD2511F55u"),
    "philox32_no_key_bump": ("            k0 += W0;\n            k1 += W1;\n        }\n        uint64_t p0",
                             "        }\n        uint64_t p0"),
    "philox32_nine_rounds": ("uint32_t k0 = key[0], k1 = key[1];\n    for (int round = 0; round < 10;",
                             "uint32_t k0 = key[0], k1 = key[1];\n    for (int round = 0; round < 9;"),
    "philox32_words_swapped": ("uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;",
                               "uint32_t n0 = (uint32_t)(p1 >> 32) ^ c3 ^ k0;"),
    "philox64_hi_word": ("uint64_t n2 = (uint64_t)(p0 >> 64) ^ c3 ^ k1;",
                         "uint64_t n2 = (uint64_t)(p0 >> 64) ^ c1 ^ k1;"),
    "philox64_key_order": ("uint64_t n0 = (uint64_t)(p1 >> 64) ^ c1 ^ k0;",
                           "uint64_t n0 = (uint64_t)(p1 >> 64) ^ c1 ^ k1;"),
    "dropout_word": ("uint32_t word = w[(i % 8) / 2];", "uint32_t word = w[(i % 4)];"),
    "dropout_halves_swapped": ("uint32_t half = (i % 2) ? (word >> 16) : (word & 0xFFFFu);",
                               "uint32_t half = (i % 2) ? (word & 0xFFFFu) : (word >> 16);"),
    "dropout_counter_word": ("uint32_t ctr[4] = {0u, 0u, (uint32_t)g, (uint32_t)(g >> 32)};",
                             "uint32_t ctr[4] = {(uint32_t)g, 0u, 0u, (uint32_t)(g >> 32)};"),
    "dropout_block_of_four": ("uint64_t g = offset + (uint64_t)i / 8u;",
                              "uint64_t g = offset + (uint64_t)i / 4u;"),
    "dropout_strict_threshold": ("return u >= p;", "return u > p;"),
    "dropout_scale_of_u": ("float u = (float)half * 0x1p-16f;", "float u = (float)half * 0x1p-15f;"),
    "dropout_scale_inverted": ("g = g / (1.0 - (double)ex->p);", "g = g * (1.0 - (double)ex->p);"),
    "dropout_dropped_kept": ("                else\n                    g = g * 0.0;",
                             "                else\n                    g = g * 1.0;"),
    "o5m_mask_off_by_one": ("if (last + 1 < end)\n                end = last + 1;",
                            "if (last < end)\n                end = last;"),
    "o5m_period_ignored": ("int64_t last = i % period + offset;", "int64_t last = i + offset;"),
    "o5m_offset_ignored": ("int64_t last = i % period + offset;", "int64_t last = i % period;"),
    "o5m_scale_dropped": ("float v = load(x, k) * scale;", "float v = load(x, k);"),
    "o5m_masked_not_zero": ("            double p = 0.0;\n            if (j < end)",
                            "            double p = 1e-30;\n            if (j < end)"),
    "o5m_max_over_row": ("        double m = -INFINITY;\n        for (int64_t j = 0; j < end; ++j) {\n            double v = (double)o5m_value",
                         "        double m = -INFINITY;\n        for (int64_t j = 0; j < cols; ++j) {\n            double v = (double)o5m_value"),
    "o5_min_not_max": ("if (v > m)\n                m = v;", "if (v < m || m == -INFINITY)\n                m = v;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_fails_a_pin(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert old in src, f"mutation site for {name} not found"
    mutated = src.replace(old, new)
    shutil.copy(HDR, tmp_path / "oracle.h")
    (tmp_path / "oracle.c").write_text(mutated)
    so = oracle_build.build(src=str(tmp_path / "oracle.c"),
                            out=str(tmp_path / f"liboracle_{name}.so"))
    lib = oracle.load(so)
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(lib)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
