"""Planted mistakes in a copy of the oracle source must each fail a pin (CPU).

Every mutant below is a plausible slip (a dropped term, a wrong sign, index
or operand).  The source copy is compiled into a temporary directory, the
oracle module is pointed at it, and at least one check of oracle_checks must
raise.  The in-tree oracle is never modified.
"""
import os

import pytest

import oracle
import oracle_checks

SRC = os.path.join(os.path.dirname(oracle.__file__), "flux_attn_oracle.c")

MUTANTS = {
    "rms_drop_eps": ("sqrt(ss / d + eps)", "sqrt(ss / d)"),
    "rms_sum_not_mean": ("sqrt(ss / d + eps)", "sqrt(ss + eps)"),
    "rms_drop_weight": ("y[i] = x[i] * inv * w[i]", "y[i] = x[i] * inv"),
    "rope_sign": ("y[off + 2 * j] = x0 * c - x1 * s", "y[off + 2 * j] = x0 * c + x1 * s"),
    "rope_freq_exponent": ("pow(theta, -2.0 * j / da)", "pow(theta, -1.0 * j / da)"),
    "rope_axis_offset": ("    off += da;", "    off += 0;"),
    "rope_axis_order": ("(double)pos3[a]", "(double)pos3[2 - a]"),
    "softmax_no_scale": ("double inv_sqrt_d = 1.0 / sqrt((double)d);", "double inv_sqrt_d = 1.0;"),
    "softmax_no_normalise": ("double p = srow[m] / l;", "double p = srow[m];"),
    "pv_wrong_operand": ("o[i] += p * vh[(int64_t)m * d + i]", "o[i] += p * kh[(int64_t)m * d + i]"),
    "qk_transposed_index": ("s += qh[i] * kh[(int64_t)m * d + i]", "s += qh[i] * kh[(int64_t)i * d + m % d]"),
    "e4m3_truncate": ("double m = nearbyint((2.0 * fr - 1.0) * 8.0);", "double m = floor((2.0 * fr - 1.0) * 8.0);"),
    "e4m3_saturate_nan": ("if (a >= 448.0) return (uint8_t)(sign | 0x7E);", "if (a >= 448.0) return (uint8_t)(sign | 0x7F);"),
    "e4m3_subnormal_shift": ("double q = nearbyint(ldexp(a, 9));", "double q = nearbyint(ldexp(a, 8));"),
    "fp8_scale_240": ("amax > 0.0 ? amax / 448.0 : 1.0", "amax > 0.0 ? amax / 240.0 : 1.0"),
    "fp8_scale_first": ("oracle_e4m3_encode(amax > 0.0 ? (448.0 * a[i]) / amax : a[i])", "oracle_e4m3_encode(a[i] / scale)"),
    "fp8_signed_amax": ("if (fabs(a[i]) > amax) amax = fabs(a[i]);", "if (a[i] > amax) amax = a[i];"),
    "qkv_drop_bias": ("y[o] = acc + (bias ? (double)bias[o] : 0.0);", "y[o] = acc;"),
    "qkv_swap_q_k": ("rmsnorm_row(q, y + (int64_t)h * d, d, wq, eps);", "rmsnorm_row(q, y + (int64_t)(H + h) * d, d, wq, eps);"),
    "qkv_x_row_of_token": ("xr[c] = bf16_to_f64(x[m * D + c]);", "xr[c] = bf16_to_f64(x[n * D + c]);"),
    "qkv_q_weights_everywhere": ("bf16_to_f64(w[(int64_t)o * D + c])", "bf16_to_f64(w[(int64_t)(o % (H * d)) * D + c])"),
    "vc_error_k_only": ("e += dk * dk + dv * dv;", "e += dk * dk;"),
    "vc_error_of_value_not_residual": ("double dv = vx[m * d + i] - vq[m * d + i];", "double dv = vx[m * d + i];"),
    "vc_smallest_errors": ("if (x->e > y->e) return -1;\n  if (x->e < y->e) return 1;",
                           "if (x->e < y->e) return -1;\n  if (x->e > y->e) return 1;"),
    "vc_ties_higher_index": ("return (x->m > y->m) - (x->m < y->m);", "return (x->m < y->m) - (x->m > y->m);"),
    "vc_count_floor": ("double r = ceil(rho * (double)N);", "double r = floor(rho * (double)N);"),
    "vc_repair_v_only": ("memcpy(kh + sel[r] * d, kx + sel[r] * d, sizeof(double) * d);", "(void)0;"),
    "sol_pool_sum_not_mean": ("      qb[blk * d + i] /= cnt[blk];\n", "      (void)0;\n"),
    "sol_no_block_size_weight": ("sc[j] = s * scale + log(cnt[j]);", "sc[j] = s * scale;"),
    "sol_threshold_not_per_block": ("mass[i * nb + j] >= tau / (double)nb", "mass[i * nb + j] >= tau"),
    "sol_no_best_block": ("mass[i * nb + j] >= tau / (double)nb || j == best", "mass[i * nb + j] >= tau / (double)nb"),
    "sol_row_mask_of_key_block": ("keep_row[m / 128]) continue;\n    double s = 0.0;", "keep_row[0]) continue;\n    double s = 0.0;"),
    "qkv_v_normalised": ("for (int i = 0; i < d; ++i) v[i] = y[(int64_t)(2 * H + h) * d + i];", "rmsnorm_row(v, y + (int64_t)(2 * H + h) * d, d, wk, eps);"),
}


@pytest.fixture(scope="module")
def source():
    with open(SRC) as f:
        return f.read()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, source, tmp_path):
    old, new = MUTANTS[name]
    assert source.count(old) == 1, "mutation anchor not unique: %r" % old
    path = tmp_path / ("mut_%s.c" % name)
    path.write_text(source.replace(old, new))
    lib = oracle.compile_source(str(path), str(tmp_path / ("mut_%s.so" % name)))
    oracle.use_library(lib)
    failed = []
    try:
        for check in oracle_checks.ALL_CHECKS:
            try:
                check()
            except (AssertionError, ValueError):
                failed.append(check.__name__)
    finally:
        oracle.use_library(None)
    assert failed, "mutant %s passed every pin" % name
