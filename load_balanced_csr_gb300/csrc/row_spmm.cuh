// SpMM straight from CSR for matrices whose rows are all short (a warp per
// 32 consecutive rows, lanes sharing X rows); used by api.cu.
#pragma once

#include "internal.cuh"

namespace lbcsr {

// rows longer than this keep SpMM on the merge-path partition
constexpr int32_t kRowSpmmMaxLen = 64;

struct RowSpmmArgs {
    int32_t m, k;
    const int32_t *row_ptr, *col_idx;
    const void *vals;
    const void *X;
    int64_t ldx;
    void *Y;
    int64_t ldy;
    double alpha, beta;
};

// k a multiple of the values per 16 bytes; X, Y 16-byte aligned row by row
bool row_spmm_supported(spmv_dtype_t dtype, int32_t k, const void *X, int64_t ldx, const void *Y, int64_t ldy);
cudaError_t launch_row_spmm(spmv_dtype_t dtype, const RowSpmmArgs &a, cudaStream_t stream);

}  // namespace lbcsr
