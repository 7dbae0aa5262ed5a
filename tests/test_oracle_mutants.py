"""The pins are strong enough: a copy of oracle.c with one plausible mistake
planted in it (on the CPU, in a temporary build) must fail at least one pin."""
import os
import subprocess
import sys
import tempfile

import pytest

import oracle
import oracle_pins

# (name, original text, mutated text) -- each original occurs exactly once.
MUTANTS = [
    ("dropped_beta_term", "r = r + be * decode_c(c_dtype, C, i * ldc + j);\n            acc[j] = r;",
     "r = r + 0.0 * decode_c(c_dtype, C, i * ldc + j);\n            acc[j] = r;"),
    ("sampled_dropped_beta", "r = r + be * decode_c(c_dtype, C, i * ldc + j);\n        R[s] = r;",
     "r = r + 0.0 * decode_c(c_dtype, C, i * ldc + j);\n        R[s] = r;"),
    ("dropped_alpha", "double r = use_ab ? al * acc[j] : 0.0;",
     "double r = use_ab ? acc[j] : 0.0;"),
    ("sign_of_product", "acc[j] = acc[j] + p;", "acc[j] = acc[j] - p;"),
    ("k_loop_short", "for (int64_t k = 0; k < K; ++k) {\n                const double a",
     "for (int64_t k = 0; k < K - 1; ++k) {\n                const double a"),
    ("transA_swapped", "return is_n(transA) ? i * lda + k : k * lda + i;",
     "return is_n(transA) ? k * lda + i : i * lda + k;"),
    ("transB_swapped", "return is_n(transB) ? k * ldb + j : j * ldb + k;",
     "return is_n(transB) ? j * ldb + k : k * ldb + j;"),
    ("ldb_used_for_a", "decode_in(ab_dtype, A, a_off(transA, i, k, lda));",
     "decode_in(ab_dtype, A, a_off(transA, i, k, ldb));"),
    ("ldc_ignored", "decode_c(c_dtype, C, i * ldc + j);\n            acc[j] = r;",
     "decode_c(c_dtype, C, i * N + j);\n            acc[j] = r;"),
    ("f16_bias_off_by_one", "v = ldexp((double)(1024 + m), e - 25);",
     "v = ldexp((double)(1024 + m), e - 24);"),
    ("f16_subnormal_scale", "v = ldexp((double)m, -24);", "v = ldexp((double)m, -25);"),
    ("bf16_mantissa_width", "v = ldexp((double)(128 + m), e - 134);",
     "v = ldexp((double)(256 + m), e - 135);"),
    ("ties_away_from_zero", "return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;",
     "return fl + 1.0;"),
    ("truncating_rounder", "if (frac > 0.5) return fl + 1.0;", "if (frac > 2.0) return fl + 1.0;"),
    ("overflow_threshold", "if (efield >= (1 << ebits) - 1) return sign | exp_all_ones;",
     "if (efield > (1 << ebits) - 1) return sign | exp_all_ones;"),
    ("subnormal_floor", "int ulp_exp = (e < emin ? emin : e) - mbits;",
     "int ulp_exp = e - mbits;"),
    ("abs_sum_signed", "sabs[j] = sabs[j] + fabs(p);", "sabs[j] = sabs[j] + p;"),
    ("sampled_transB", "decode_in(ab_dtype, B, b_off(transB, k, j, ldb));\n                acc = acc + p;",
     "decode_in(ab_dtype, B, b_off('N', k, j, ldb));\n                acc = acc + p;"),
    ("epilogue_bias_dropped",
     "if (bias != NULL) x = x + decode_c(bias_dtype, bias, j);\n            R[i * N + j]",
     "if (bias != NULL) x = x + 0.0 * decode_c(bias_dtype, bias, j);\n            R[i * N + j]"),
    ("epilogue_bias_by_row",
     "if (bias != NULL) x = x + decode_c(bias_dtype, bias, j);\n            R[i * N + j]",
     "if (bias != NULL) x = x + decode_c(bias_dtype, bias, i);\n            R[i * N + j]"),
    ("sampled_bias_by_row", "if (bias != NULL) x = x + decode_c(bias_dtype, bias, cols[s]);",
     "if (bias != NULL) x = x + decode_c(bias_dtype, bias, rows[s]);"),
    ("gelu_missing_half", "return 0.5 * x * erfc(-x / sqrt(2.0));",
     "return x * erfc(-x / sqrt(2.0));"),
    ("gelu_wrong_scale", "return 0.5 * x * erfc(-x / sqrt(2.0));",
     "return 0.5 * x * erfc(-x / 2.0);"),
    ("gelu_cancelling_form", "return 0.5 * x * erfc(-x / sqrt(2.0));",
     "return 0.5 * x * (1.0 + erf(x / sqrt(2.0)));"),
    ("silu_sign", "return x / (1.0 + exp(-x));", "return x / (1.0 + exp(x));"),
    ("relu_leaky", "return isnan(x) ? x : (x > 0.0 ? x : 0.0);",
     "return isnan(x) ? x : (x > 0.0 ? x : 0.01 * x);"),
    ("activation_after_bias_skipped", "        R[i * N + j] = oracle_activation(act, x);",
     "        R[i * N + j] = x;"),
    ("tf32_keeps_11_bits", "return oracle_decode_f32(u & 0xFFFFE000u);",
     "return oracle_decode_f32(u & 0xFFFFF000u);"),
    ("tf32_rounds_up", "return oracle_decode_f32(u & 0xFFFFE000u);",
     "return oracle_decode_f32((u + 0x1000u) & 0xFFFFE000u);"),
    ("tf32_not_truncated", "if (dt == OR_F32) return oracle_decode_tf32(((const uint32_t*)p)[idx]);",
     "if (dt == OR_F32) return oracle_decode_f32(((const uint32_t*)p)[idx]);"),
    ("softmax_no_max_shift", "y[j] = exp(y[j] - m);", "y[j] = exp(y[j]);"),
    ("softmax_not_normalised", "for (int64_t j = 0; j < cols; ++j) y[j] = y[j] / s;",
     "for (int64_t j = 0; j < cols; ++j) y[j] = y[j] / (s + 1e-3);"),
    ("softmax_min_not_max", "else if (x > m) m = x;", "else if (x < m || m == -INFINITY) m = x;"),
    ("softmax_sum_skips_first", "s = s + y[j];", "if (j > 0) s = s + y[j];"),
    ("softmax_row_pitch_ignored", "const double x = decode_c(x_dtype, X, i * ldx + j);",
     "const double x = decode_c(x_dtype, X, i * cols + j);"),
    ("softmax_f32_as_tf32", "const double x = decode_c(x_dtype, X, i * ldx + j);",
     "const double x = decode_in(x_dtype, X, i * ldx + j);"),
    ("softmax_selected_rows_ignored", "const int64_t i = row_ids ? row_ids[t] : t;",
     "const int64_t i = t;"),
    ("softmax_masked_row_zero", "for (int64_t j = 0; j < cols; ++j) y[j] = y[j] / s;",
     "for (int64_t j = 0; j < cols; ++j) y[j] = (s > 0.0) ? y[j] / s : 0.0;"),
    ("conv_filter_flipped", "decode_in(x_dtype, Wt, ((k * R + r) * S + s) * C + c);",
     "decode_in(x_dtype, Wt, ((k * R + (R - 1 - r)) * S + s) * C + c);"),
    ("conv_pad_sign", "const int64_t h = p * stride_h - pad_h + r * dil_h;",
     "const int64_t h = p * stride_h + pad_h + r * dil_h;"),
    ("conv_stride_ignored", "const int64_t w = q * stride_w - pad_w + s * dil_w;",
     "const int64_t w = q - pad_w + s * dil_w;"),
    ("conv_dilation_ignored", "const int64_t h = p * stride_h - pad_h + r * dil_h;",
     "const int64_t h = p * stride_h - pad_h + r;"),
    ("conv_channels_reversed", "decode_in(x_dtype, X, ((n * H + h) * W + w) * C + c);",
     "decode_in(x_dtype, X, ((n * H + h) * W + w) * C + (C - 1 - c));"),
    ("conv_out_size", "return span < 0 ? 0 : span / stride + 1;", "return span < 0 ? 0 : (span + stride - 1) / stride + 1;"),
    ("conv_beta_dropped", "if (be != 0.0) y = y + be * decode_c(y_dtype, Yin, m * K + k);", "(void)Yin;"),
    ("conv_no_padding_check", "if (w < 0 || w >= W) continue;", "if (w < 0) continue;"),
    ("beta_read_when_zero", "if (be != 0.0) r = r + be * decode_c(c_dtype, C, i * ldc + j);\n            acc[j] = r;",
     "r = r + be * decode_c(c_dtype, C, i * ldc + j);\n            acc[j] = r;"),
    ("ln_unbiased_variance", "const double var = sq / (double)N;",
     "const double var = sq / (double)(N - 1);"),
    ("ln_eps_outside_sqrt", "const double inv = 1.0 / sqrt(var + eps);",
     "const double inv = 1.0 / (sqrt(var) + eps);"),
    ("ln_h_not_rounded", "h[j] = round_to_type(c_dtype, x);", "h[j] = x;"),
    ("ln_bias_dropped", "if (bias != NULL) x = x + decode_c(bias_dtype, bias, j);\n            h[j]",
     "(void)bias;\n            h[j]"),
    ("ln_gamma_shift_swapped", "Y[s * N + j] = (h[j] - mu) * inv * g + t;",
     "Y[s * N + j] = (h[j] - mu) * inv * t + g;"),
    ("ln_variance_about_zero", "sq = sq + (h[j] - mu) * (h[j] - mu);", "sq = sq + h[j] * h[j];"),
    ("ln_row_ids_ignored", "rr[s * N + j] = row_ids != NULL ? row_ids[s] : s;", "rr[s * N + j] = s;"),
    ("ln_gamma_first_only", "const double g = gamma != NULL ? decode_c(ln_dtype, gamma, j) : 1.0;",
     "const double g = gamma != NULL ? decode_c(ln_dtype, gamma, 0) : 1.0;"),
    ("ln_mean_over_n_minus_1", "const double mu = sum / (double)N;",
     "const double mu = sum / (double)(N > 1 ? N - 1 : 1);"),
]


@pytest.fixture(scope="module")
def source():
    return open(oracle.SRC).read()


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(source, name, old, new):
    assert source.count(old) == 1, f"mutation site for {name} not unique/found"
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "mutant.c")
        with open(src, "w") as f:
            f.write(source.replace(old, new))
        lib = oracle.compile_source(src, os.path.join(d, "libmutant.so"))
        # The battery runs in a child process: a mutant may crash (e.g. read
        # through a NULL C), which counts as caught.
        here = os.path.dirname(os.path.abspath(__file__))
        code = (
            "import sys; sys.path[:0] = [%r, %r]\n"
            "import oracle, oracle_pins\n"
            "o = oracle.Oracle(%r)\n"
            "for pin in oracle_pins.ALL_PINS:\n"
            "    try:\n"
            "        pin(o)\n"
            "    except (AssertionError, ValueError):\n"
            "        print('caught by', pin.__name__); sys.exit(3)\n"
            "sys.exit(0)\n" % (here, os.path.dirname(here), lib))
        res = subprocess.run([sys.executable, "-c", code], capture_output=True,
                             text=True, timeout=600)
        assert res.returncode != 0, f"mutant {name} passed every pin"
