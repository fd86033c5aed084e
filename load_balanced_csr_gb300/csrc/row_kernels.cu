// Row-mapped SpMV kernels.
//
// Thread per row: the thread-mapped schedule of "A GPU load-balancing
// programming model" (section 4.2, Listing 2: tiles handed to threads in a
// grid-stride loop, a tile's atoms walked in order) and the "scalar CSR"
// kernel of the Row-grouped CSR page (section 3).  Neighbouring threads read
// neighbouring rows, so the loads of a warp are not coalesced unless rows are
// very short; the plan uses it for short, even rows and for n == 1, and for
// the rows that are not long when long rows have their own kernel.
//
// The kernel keeps U partial sums per row (nonzero k goes to sum k mod U)
// and adds them as a tree at the end: U independent chains give the loads
// and FMAs room to overlap, and the rounding error grows with length / U
// instead of length.
#include "internal.cuh"

namespace lbcsr {

namespace {

template <typename V>
__device__ __forceinline__ V finish(V s, V alpha, V beta, const V *y, int64_t row) {
    V r = alpha * s;
    if (beta != V(0)) r = fma(beta, y[row], r);
    return r;
}

template <typename V, int U>
__device__ __forceinline__ V tree_sum(const V (&a)[U]) {
    V t[U];
#pragma unroll
    for (int u = 0; u < U; ++u) t[u] = a[u];
#pragma unroll
    for (int w = 1; w < U; w <<= 1)
#pragma unroll
        for (int u = 0; u + w < U; u += 2 * w) t[u] += t[u + w];
    return t[0];
}

template <typename V>
__global__ void __launch_bounds__(256)
thread_per_row_kernel(int32_t m, const int32_t *__restrict__ rp, const int32_t *__restrict__ col,
                      const V *__restrict__ val, const V *__restrict__ x, V *__restrict__ y, V alpha,
                      V beta, int32_t skip_min_len, int32_t n, int32_t *error) {
    constexpr int U = 4;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t row = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; row < m; row += stride) {
        const int32_t b = rp[row], e = rp[row + 1];
        if (skip_min_len > 0 && e - b >= skip_min_len) continue;
        V acc[U];
#pragma unroll
        for (int u = 0; u < U; ++u) acc[u] = V(0);
        int32_t k = b;
        for (; k + U <= e; k += U) {
            int c[U];
            V v[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                c[u] = ld_stream(col + k + u);
                v[u] = ld_stream(val + k + u);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) acc[u] = fma(v[u], ld_gather(x + debug_col(c[u], n, error)), acc[u]);
        }
#pragma unroll
        for (int u = 0; u < U - 1; ++u)
            if (k + u < e)
                acc[u] = fma(ld_stream(val + k + u), ld_gather(x + debug_col(ld_stream(col + k + u), n, error)), acc[u]);
        y[row] = finish(tree_sum(acc), alpha, beta, y, row);
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

// The unified L1 / shared-memory storage of an SM is split by a carve-out.
// A kernel that gathers x at random needs L1 room for the lines of its
// gathers in flight: with the storage given to shared memory, the gathers
// stall (measured on GB300: a gather loop with 203 KB of shared memory
// reserved per SM ran 3.2x slower than with none).  This gives the smallest
// carve-out, in percent of the SM's shared memory, that still holds `ctas`
// CTAs of `smem_per_cta` bytes; the rest stays L1.
int carveout_percent(int ctas, size_t smem_per_cta) {
    int dev = 0, max_sm = 0, reserved = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (cudaDeviceGetAttribute(&max_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
        max_sm <= 0)
        return -1;
    if (cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess) reserved = 0;
    const long long need = (long long)ctas * ((long long)smem_per_cta + reserved);
    long long pct = (need * 100 + max_sm - 1) / max_sm;
    return (int)(pct < 0 ? 0 : pct > 100 ? 100 : pct);
}

cudaError_t launch_thread_per_row(spmv_dtype_t dtype, int32_t m, int32_t n, const int32_t *row_ptr,
                                  const int32_t *col_idx, const void *vals, const void *x, void *y,
                                  double alpha, double beta, int32_t skip_min_len, int32_t *error,
                                  cudaStream_t stream) {
    if (m <= 0) return cudaSuccess;
    const int64_t want = ((int64_t)m + 255) / 256;
    const int64_t cap = (int64_t)device_sm_count() * 8;
    const int blocks = (int)(want < cap ? want : cap);
    if (dtype == SPMV_F64)
        thread_per_row_kernel<double><<<blocks, 256, 0, stream>>>(
            m, row_ptr, col_idx, static_cast<const double *>(vals), static_cast<const double *>(x),
            static_cast<double *>(y), alpha, beta, skip_min_len, n, error);
    else
        thread_per_row_kernel<float><<<blocks, 256, 0, stream>>>(
            m, row_ptr, col_idx, static_cast<const float *>(vals), static_cast<const float *>(x),
            static_cast<float *>(y), (float)alpha, (float)beta, skip_min_len, n, error);
    return cudaGetLastError();
}

}  // namespace lbcsr
