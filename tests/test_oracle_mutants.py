"""Plant plausible mistakes in a copy of the oracle; the pins must catch each one.

Every mutant is a one-line textual change to a temporary copy of
oracle/softmax_oracle.c, compiled on the CPU; the real oracle is untouched.
"""
import os

import pytest

import oracle
from tests import pins

MUTANTS = {
    "sum_without_max": ("s += exp(x[j] - m);", "s += exp(x[j]);"),
    "no_max_subtraction": ("exp(x[j] - m)", "exp(x[j])"),
    "wrong_sign": ("y[j] = exp(x[j] - m) / s;", "y[j] = exp(m - x[j]) / s;"),
    "min_instead_of_max": ("if (x[j] > m) m = x[j];", "if (x[j] < m) m = x[j];"),
    "sum_skips_first": ("for (int64_t j = 0; j < n; ++j)\n        s +=",
                        "for (int64_t j = 1; j < n; ++j)\n        s +="),
    "sum_skips_last": ("for (int64_t j = 0; j < n; ++j)\n        s +=",
                       "for (int64_t j = 0; j + 1 < n; ++j)\n        s +="),
    "multiply_by_sum": ("exp(x[j] - m) / s;", "exp(x[j] - m) * s;"),
    "input_stride_N": ("i * jb->ld_in + j", "i * jb->N + j"),
    "output_stride_N": ("jb->out, i * jb->ld_out + j", "jb->out, i * jb->N + j"),
    "truncating_cast": ("nearbyint(ldexp(a, -qe))", "floor(ldexp(a, -qe))"),
    "bf16_seven_bits": ("round_to_format(y, 8, -126, 127, 8)", "round_to_format(y, 7, -126, 127, 8)"),
    "bf16_via_float": ("round_to_format(y, 8, -126, 127, 8)",
                       "round_to_format((double)(float)y, 8, -126, 127, 8)"),
    "f16_via_float": ("round_to_format(y, 11, -14, 15, 5)",
                      "round_to_format((double)(float)y, 11, -14, 15, 5)"),
    "no_subnormal_clamp": ("(e < emin ? emin : e) - mbits", "e - mbits"),
    "f16_bias_off_by_one": ("e - 25);", "e - 24);"),
    "bf16_decode_shift": ("(uint32_t)h << 16;", "(uint32_t)h << 15;"),
    "f32_output_truncated": ("float f = (float)y;", "float f = (float)(y * (1.0 - 0x1p-30));"),
    "masked_as_zero": ("decode(jb->in, i * jb->ld_in + j, jb->dtype) : -INFINITY;",
                       "decode(jb->in, i * jb->ld_in + j, jb->dtype) : 0.0;"),
    "causal_off_by_one": ("v = i % jb->causal_period + 1;", "v = i % jb->causal_period;"),
    "rmsnorm_no_residual": ("decode(x, i * ld_x + j, dtype) + decode(r, i * ld_r + j, dtype), dtype)",
                            "decode(x, i * ld_x + j, dtype), dtype)"),
    "rmsnorm_unrounded_sum": ("h[j] = to_dtype(decode(x, i * ld_x + j, dtype) + decode(r, i * ld_r + j, dtype), dtype);",
                              "h[j] = decode(x, i * ld_x + j, dtype) + decode(r, i * ld_r + j, dtype);"),
    "rmsnorm_sum_not_mean": ("ms /= (double)N;", "ms /= 1.0;"),
    "rmsnorm_eps_outside": ("sqrt(ms + eps);", "sqrt(ms) + eps;"),
    "rmsnorm_weight_index": ("decode(w, j, dtype)", "decode(w, N - 1 - j, dtype)"),
    "backward_drops_dot": ("encode(dx, i * ld_dx + j, dtype, yj * (gj - dot));",
                           "encode(dx, i * ld_dx + j, dtype, yj * gj);"),
    "backward_sign": ("encode(dx, i * ld_dx + j, dtype, yj * (gj - dot));",
                      "encode(dx, i * ld_dx + j, dtype, yj * (dot - gj));"),
    "backward_dot_skips_last": ("for (int64_t j = 0; j < N; ++j)\n            dot +=",
                                "for (int64_t j = 0; j + 1 < N; ++j)\n            dot +="),
}


def _battery_fails(orc):
    failures = []
    for check in pins.ALL_CHECKS:
        try:
            check(orc)
        except AssertionError:
            failures.append(check.__name__)
        except Exception as e:  # a crash also counts as detection
            failures.append("%s (%s)" % (check.__name__, type(e).__name__))
    return failures


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(oracle.SOURCE).read()
    assert old in src, "mutation %s no longer applies" % name
    path = tmp_path / ("%s.c" % name)
    path.write_text(src.replace(old, new))
    lib = oracle.compile_library(str(path), str(tmp_path / ("lib%s.so" % name)))
    failures = _battery_fails(oracle.Oracle(lib))
    assert failures, "mutant %s passed every pin" % name
