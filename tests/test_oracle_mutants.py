"""Each plausible mistake planted in a copy of the oracle fails some pin.

The mistakes are planted on the CPU, in a temporary copy of the oracle's C
source; the real oracle is untouched.  A mutant that every pin accepted would
mean the pins cannot see that class of bug.
"""
import os
import subprocess
import sys

import pytest

import oracle
from tests import oracle_pins

# (name, text in gemm_oracle.c, replacement, occurrence index)
MUTANTS = [
    ("b_layout_swapped", "j * ldb + k : k * ldb + j", "k * ldb + j : j * ldb + k", 0),
    ("beta_term_dropped", "cterm = beta * load_fp(out_dtype, C, i * ldc + j);", "cterm = 0.0 * beta;", 0),
    ("alpha_scales_c", "*ref = alpha * sum + cterm + bterm;", "*ref = alpha * (sum + cterm) + bterm;", 0),
    ("alpha_scales_bias", "*ref = alpha * sum + cterm + bterm;", "*ref = alpha * (sum + bterm) + cterm;", 0),
    ("bias_dropped", "*ref = alpha * sum + cterm + bterm;", "*ref = alpha * sum + cterm;", 0),
    ("bias_indexed_by_row", "load_fp(out_dtype, bias, j)", "load_fp(out_dtype, bias, i)", 0),
    ("i8_bias_dropped", "if (bias) r +=", "if (0) r +=", 0),
    ("a_layout_swapped", "? k * lda + i : i * lda + k", "? i * lda + k : k * lda + i", 0),
    ("sum_rows_skips_last", "for (int64_t i = 0; i < rows; ++i) {", "for (int64_t i = 0; i + 1 < rows; ++i) {", 0),
    ("k_loop_short_fp", "for (int64_t k = 0; k < K; ++k) {", "for (int64_t k = 0; k + 1 < K; ++k) {", 0),
    ("k_loop_short_i8", "for (int64_t k = 0; k < K; ++k) {", "for (int64_t k = 0; k + 1 < K; ++k) {", 1),
    ("product_sign", "sum += a * b;", "sum -= a * b;", 0),
    ("bf16_decode_shift", "((uint32_t)h) << 16", "((uint32_t)h) << 15", 0),
    ("round_ties_away", "nearbyint(scaled)", "round(scaled)", 0),
    ("i8_beta_dropped", "if (beta != 0) r +=", "if (0) r +=", 0),
    ("bound_without_alpha", "rel * fabs(alpha) * abs_sum", "rel * abs_sum", 0),
    ("ulp_one_bit_off", "ldexp(1.0, exp2 - 7)", "ldexp(1.0, exp2 - 8)", 0),
    ("f16_bias", "e - 25);", "e - 24);", 0),
    ("beta_zero_reads_c", "if (beta != 0.0) cterm", "if (1) cterm", 0),
    ("alpha_zero_reads_ab", "if (alpha != 0.0) {", "if (1) {", 0),
    ("lda_ignored", "a_index(layout_a, i, k, lda)", "a_index(layout_a, i, k, K)", 0),
    ("i8_lda_ignored", "a_index(layout_a, i, k, lda)", "a_index(layout_a, i, k, K)", 1),
    ("spmv_x_by_position", "(double)x[column_indices[p]];  /* exact */", "(double)x[p % cols];", 0),
    ("spmv_row_end_inclusive", "p < row_offsets[i + 1]; ++p) {\n                double prod",
     "p <= row_offsets[i + 1] && p < row_offsets[rows]; ++p) {\n                double prod", 0),
    ("spmv_skips_first", "p = row_offsets[i]; p < row_offsets[i + 1]; ++p) {\n                double prod",
     "p = row_offsets[i] + 1; p < row_offsets[i + 1]; ++p) {\n                double prod", 0),
    ("spmv_beta_dropped", "double yterm = beta != 0.0 ? beta * (double)y[i] : 0.0;", "double yterm = 0.0;", 0),
    ("spmv_alpha_on_y", "ref[i] = alpha * sum + yterm;", "ref[i] = alpha * (sum + yterm);", 0),
    ("spmv_beta_zero_reads_y", "double yterm = beta != 0.0 ?", "double yterm = 1 ?", 0),
    ("spmv_no_column_check", "column_indices[p] >= cols) return -1;", "column_indices[p] > cols) return -1;", 0),
    ("sampled_fp_rows_cols_swapped", "rows[s], cols[s], &ref[s]", "cols[s], rows[s], &ref[s]", 0),
    ("sampled_i8_rows_cols_swapped", "NULL, rows[s], cols[s]);", "NULL, cols[s], rows[s]);", 0),
    ("sampled_fp_ldc_one", "beta, C, ldc, NULL, rows[s]", "beta, C, 1, NULL, rows[s]", 0),
    ("sampled_i8_ldc_one", "beta, C, ldc,\n                            NULL, rows[s]",
     "beta, C, 1,\n                            NULL, rows[s]", 0),
    ("sampled_fp_lda_ignored", "OR_ROW_MAJOR, layout_b, K, alpha, A, lda, B, ldb,\n                   beta",
     "OR_ROW_MAJOR, layout_b, K, alpha, A, K, B, ldb,\n                   beta", 0),
    ("f16_round_ties_away", "ldexp(nearbyint(ldexp(ax, -q)), q)", "ldexp(round(ldexp(ax, -q)), q)", 0),
    ("f16_subnormal_quantum", "int q = exp2 < -14 ? -24 : exp2 - 10;", "int q = exp2 < -15 ? -25 : exp2 - 10;", 0),
    ("f16_no_overflow", "if (r > 65504.0) return sign | 0x7c00;", "if (isinf(r)) return sign | 0x7c00;", 0),
    ("ulp_f16_one_bit_off", "ldexp(1.0, exp2 - 10)", "ldexp(1.0, exp2 - 11)", 0),
    ("ulp_f16_subnormal", "exp2 < -14 ? ldexp(1.0, -24)", "exp2 < -14 ? ldexp(1.0, -25)", 0),
    ("tf32_term_dropped", "in_dtype == OR_TF32 ? ldexp(1.0, -9) + ldexp(1.0, -20) + 1e-4 : 1e-4",
     "1e-4", 0),
    ("tf32_read_as_16_bit", "    case OR_F32:\n    case OR_TF32: return (double)((const float*)p)[idx];",
     "    case OR_F32: return (double)((const float*)p)[idx];\n"
     "    case OR_TF32: return decode_bf16(((const uint16_t*)p)[idx]);", 0),
]


def _replace_nth(text, old, new, n):
    idx = -1
    for _ in range(n + 1):
        idx = text.index(old, idx + 1)
    return text[:idx] + new + text[idx + len(old):]


_RUNNER = """
import sys
sys.path.insert(0, {root!r})
import oracle
from tests import oracle_pins
plain = oracle.Oracle({plain!r})
counting = oracle.Oracle({counting!r})
failures = []
for pin in oracle_pins.ALL_PINS:
    try:
        pin(plain)
    except Exception:
        failures.append(pin.__name__)
try:
    oracle_pins.pin_mac_count(counting)
except Exception:
    failures.append("pin_mac_count")
print("FAILED_PINS", failures)
sys.exit(1 if failures else 0)
"""


@pytest.mark.parametrize("name,old,new,nth", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new, nth, tmp_path):
    src = open(oracle.SOURCE).read()
    mutated = _replace_nth(src, old, new, nth)
    assert mutated != src
    path = tmp_path / f"{name}.c"
    path.write_text(mutated)
    plain = str(tmp_path / f"lib{name}.so")
    counting = str(tmp_path / f"lib{name}_count.so")
    oracle.build_variant(str(path), plain)
    oracle.build_variant(str(path), counting, ("ORACLE_COUNT_MACS",))
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    # a child process, so that a mutant that crashes (e.g. reads C through a
    # null pointer when beta == 0) also counts as caught
    proc = subprocess.run([sys.executable, "-c", _RUNNER.format(root=root, plain=plain,
                                                                counting=counting)],
                          capture_output=True, text=True, timeout=600,
                          env={**os.environ, "OMP_NUM_THREADS": "2"})
    assert proc.returncode != 0, f"mutant {name} passed every pin"
