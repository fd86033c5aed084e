"""Plant plausible slips in a copy of the oracle (on the CPU) and check that
the pins in test_oracle_pins.py catch every one of them."""
import os

import pytest

import oracle
import test_oracle_pins as pins

# (description, text in oracle.c, replacement, pins expected to catch it)
MUTATIONS = [
    ("sum subtracts", "acc += prod;", "acc -= prod;",
     [pins.test_spmv_equals_dense_product_exactly]),
    ("beta term dropped", "y += by;", "y += 0;",
     [pins.test_spmv_equals_dense_product_exactly]),
    ("x indexed by nonzero", "(long double)x[col_idx[k]]", "(long double)x[k % n]",
     [pins.test_spmv_unit_vectors_give_columns]),
    ("row end off by one", "for (int32_t k = row_ptr[i]; k < row_ptr[i + 1]; ++k) {\n            long double prod = (long double)vals[k] * (long double)x[col_idx[k]];\n            acc += prod;\n            mag += prod < 0 ? -prod : prod;\n        }\n        long double y = a * acc;\n        long double by = 0.0L;\n        if (beta != 0.0) {\n            by = b * (long double)y_old[i];\n            y += by;\n        }\n        y_out[t] = (double)y;",
     "for (int32_t k = row_ptr[i]; k + 1 < row_ptr[i + 1]; ++k) {\n            long double prod = (long double)vals[k] * (long double)x[col_idx[k]];\n            acc += prod;\n            mag += prod < 0 ? -prod : prod;\n        }\n        long double y = a * acc;\n        long double by = 0.0L;\n        if (beta != 0.0) {\n            by = b * (long double)y_old[i];\n            y += by;\n        }\n        y_out[t] = (double)y;",
     [pins.test_laplacian_times_ones_closed_form]),
    ("merge ties go to the nonzero", "(int64_t)row_ptr[i + 1] + i < d", "(int64_t)row_ptr[i + 1] + i + 1 < d",
     [pins.test_partition_matches_literal_merge_walk_exhaustively]),
    ("merge uses row start", "(int64_t)row_ptr[i + 1] + i < d", "(int64_t)row_ptr[i] + i < d",
     [pins.test_partition_matches_literal_merge_walk_exhaustively]),
    ("length class off by one", "while (k < 31 && (len >> k) != 0) ++k;", "while (k < 31 && (len >> (k + 1)) != 0) ++k;",
     [pins.test_length_class_boundaries]),
    ("rgcsr row-major instead of interleaved", "rg_col[base + (int64_t)k * G] = col_idx[row_ptr[i] + k];\n            rg_val[base + (int64_t)k * G] = vals[row_ptr[i] + k];\n        }\n    }\n    return 0;\n}\n\nint oracle_rgcsr_pack_f32",
     "rg_col[group_ptr[i / G] + (i % G) * (group_ptr[i / G + 1] - group_ptr[i / G]) / G + k] = col_idx[row_ptr[i] + k];\n            rg_val[group_ptr[i / G] + (i % G) * (group_ptr[i / G + 1] - group_ptr[i / G]) / G + k] = vals[row_ptr[i] + k];\n        }\n    }\n    return 0;\n}\n\nint oracle_rgcsr_pack_f32",
     [pins.test_rgcsr_pack_decodes_back_to_csr]),
    ("long-row bin excludes its bound", "if (len < min_len) continue;", "if (len <= min_len) continue;",
     [pins.test_long_rows_worked_example]),
    ("segment count rounds wrongly", "segs += ((int64_t)len + seg_nnz - 1) / seg_nnz;",
     "segs += (int64_t)len / seg_nnz + 1;", [pins.test_long_rows_worked_example]),
    ("window sort ascending", "if (best < 0 || len > best_len) {", "if (best < 0 || len < best_len) {",
     [pins.test_window_sort_worked_example]),
    ("window sort ties by last index", "if (best < 0 || len > best_len) {", "if (best < 0 || len >= best_len) {",
     [pins.test_window_sort_worked_example]),
    ("spmm reads X column-major", "(long double)X[(int64_t)col_idx[q] * ldx + t]", "(long double)X[(int64_t)t * ldx + col_idx[q] % ldx]",
     [pins.test_spmm_equals_dense_product_exactly]),
    ("spmm drops the beta term", "                    y += by;                                                                              \\", "                    y += 0;                                                                               \\",
     [pins.test_spmm_equals_dense_product_exactly]),
    ("transpose lists a column's rows in decreasing order",
     "        for (int32_t i = 0; i < m; ++i)                                                                   \\\n            for (int32_t q = row_ptr[i];",
     "        for (int32_t i = m - 1; i >= 0; --i)                                                              \\\n            for (int32_t q = row_ptr[i];",
     [pins.test_transpose_worked_example]),
    ("transpose keeps the row index of the column", "                t_idx[pos] = i;  ", "                t_idx[pos] = col_idx[q];  ",
     [pins.test_transpose_worked_example]),
    ("transposed product uses y index for x", "long double prod = (long double)vals[q] * (long double)x[i];", "long double prod = (long double)vals[q] * (long double)x[col_idx[q] % m];",
     [pins.test_spmv_transposed_equals_dense_product_exactly]),
    ("spgemm drops the last product of a row of B", "for (int32_t r = b_ptr[q]; r < b_ptr[q + 1]; ++r) {", "for (int32_t r = b_ptr[q]; r + 1 < b_ptr[q + 1]; ++r) {",
     [pins.test_spgemm_equals_dense_product_exactly]),
    ("spgemm keeps only entries whose sum is nonzero", "                if (mark[j]) {  ", "                if (mark[j] && acc[j] != 0.0L) {",
     [pins.test_spgemm_equals_dense_product_exactly]),
    ("spgemm carries a row's sums into the next row", "                    acc[j] = 0.0L;  ", "                    acc[j] += 0.0L; ",
     [pins.test_spgemm_equals_dense_product_exactly, pins.test_spgemm_with_identity_and_permutation]),
]


def _run_pin(fn):
    """Run a pin over its parametrisations; True if any of them fails."""
    import inspect
    params = inspect.signature(fn).parameters
    cases = [{}]
    if "dtype" in params:
        cases = [dict(dtype=d, shape=s) for d in ("f64",) for s in [(7, 3), (33, 64)]]
    elif "nx" in params:
        cases = [dict(nx=5, ny=9)]
    elif "G" in params:
        cases = [dict(G=4)]
    elif "k" in params:
        cases = [dict(k=3)]
    for kw in cases:
        try:
            fn(**kw)
        except AssertionError:
            return True
    return False


@pytest.mark.parametrize("desc,old,new,catchers", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_slip(tmp_path, desc, old, new, catchers):
    src = oracle.source_text()
    assert src.count(old) >= 1, f"mutation anchor not found: {desc}"
    mutated = src.replace(old, new, 1)
    path = oracle.compile_variant(mutated, str(tmp_path / "mutant.so"))
    with oracle.use_library(path):
        caught = any(_run_pin(fn) for fn in catchers)
    assert caught, f"planted slip not caught: {desc}"
    # the unmodified oracle passes the same pins
    assert not any(_run_pin(fn) for fn in catchers)
