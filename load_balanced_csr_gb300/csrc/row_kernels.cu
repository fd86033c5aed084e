// Row-mapped SpMV kernels.
//
// Thread per row: the thread-mapped schedule of "A GPU load-balancing
// programming model" (section 4.2, Listing 2: tiles handed to threads in a
// grid-stride loop, a tile's atoms walked in order) and the "scalar CSR"
// kernel of the Row-grouped CSR page (section 3).  Neighbouring threads read
// neighbouring rows, so the loads of a warp are not coalesced unless rows are
// very short; the plan uses it for short, even rows and for n == 1.
// Accumulation is sequential per row, so its rounding error grows with the
// row length; the plan does not choose it for long rows.
#include "internal.cuh"

namespace lbcsr {

namespace {

template <typename V>
__global__ void __launch_bounds__(256)
thread_per_row_kernel(int32_t m, const int32_t *__restrict__ rp, const int32_t *__restrict__ col,
                      const V *__restrict__ val, const V *__restrict__ x, V *__restrict__ y, V alpha,
                      V beta) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t row = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; row < m; row += stride) {
        const int32_t b = rp[row], e = rp[row + 1];
        V acc = V(0);
        for (int32_t k = b; k < e; ++k) acc += ld_stream(val + k) * ld_gather(x + ld_stream(col + k));
        V res = alpha * acc;
        if (beta != V(0)) res += beta * y[row];
        y[row] = res;
    }
}

}  // namespace

int device_sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return 148;
    return sms;
}

cudaError_t launch_thread_per_row(spmv_dtype_t dtype, int32_t m, const int32_t *row_ptr,
                                  const int32_t *col_idx, const void *vals, const void *x, void *y,
                                  double alpha, double beta, cudaStream_t stream) {
    if (m <= 0) return cudaSuccess;
    const int64_t want = ((int64_t)m + 255) / 256;
    const int64_t cap = (int64_t)device_sm_count() * 8;
    const int blocks = (int)(want < cap ? want : cap);
    if (dtype == SPMV_F64)
        thread_per_row_kernel<double><<<blocks, 256, 0, stream>>>(
            m, row_ptr, col_idx, static_cast<const double *>(vals), static_cast<const double *>(x),
            static_cast<double *>(y), alpha, beta);
    else
        thread_per_row_kernel<float><<<blocks, 256, 0, stream>>>(
            m, row_ptr, col_idx, static_cast<const float *>(vals), static_cast<const float *>(x),
            static_cast<float *>(y), (float)alpha, (float)beta);
    return cudaGetLastError();
}

}  // namespace lbcsr
