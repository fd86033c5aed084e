// SpMM straight from CSR for matrices whose rows are all short (a warp per
// 32 consecutive rows, lanes sharing X rows); used by api.cu.
#pragma once

#include "internal.cuh"

namespace lbcsr {

// rows longer than this keep SpMM on the merge-path partition
constexpr int32_t kRowSpmmMaxLen = 64;

// rows of at least this many nonzeros go to the long-row SpMM kernel when
// the matrix has rows longer than kRowSpmmMaxLen
constexpr int32_t kSpmmLongMin = kRowSpmmMaxLen + 1;
// ... and only when they are rare: at most one per kSpmmRowsPerLongRow rows.
// (Measured on GB300: 65 long rows in 8.4 M, k = 8: 2178 -> 1609 us; 93,535
// long rows in 4.2 M, k = 32: 3092 -> 7273 us, so such matrices keep the
// merge-path SpMM.)
constexpr int64_t kSpmmRowsPerLongRow = 4096;

struct RowSpmmArgs {
    int32_t m, k;
    const int32_t *row_ptr, *col_idx;
    const void *vals;
    const void *X;
    int64_t ldx;
    void *Y;
    int64_t ldy;
    double alpha, beta;
    // long rows (num_long == 0: none): rows of length >= long_min, ascending,
    // their first segments of kLongSegmentNnz nonzeros, per segment a partial
    // of up to 32 values, per row an arrival counter (zero between products)
    int32_t long_min;
    int32_t num_long;
    int64_t num_segs;
    const int32_t *long_rows;
    const int64_t *seg_begin;
    void *seg_partial;
    int32_t *arrivals;
};

// The long rows alone (any k, any X and Y layout): a warp per segment of
// kLongSegmentNnz nonzeros of the listed rows, in slices of 32 columns;
// seg_partial holds 32 values per segment.  Used next to the Row-grouped
// SpMM, whose copy leaves the long rows out.
struct LongSpmmArgs {
    int32_t k;
    const int32_t *row_ptr, *col_idx;
    const void *vals;
    const void *X;
    int64_t ldx;
    void *Y;
    int64_t ldy;
    double alpha, beta;
    int32_t num_long;
    int64_t num_segs;
    const int32_t *long_rows;
    const int64_t *seg_begin;
    void *seg_partial;
    int32_t *arrivals;
};
cudaError_t launch_long_spmm(spmv_dtype_t dtype, const LongSpmmArgs &a, cudaStream_t stream);

// k a multiple of the values per 16 bytes; X, Y 16-byte aligned row by row
bool row_spmm_supported(spmv_dtype_t dtype, int32_t k, const void *X, int64_t ldx, const void *Y, int64_t ldy);
cudaError_t launch_row_spmm(spmv_dtype_t dtype, const RowSpmmArgs &a, cudaStream_t stream);

}  // namespace lbcsr
