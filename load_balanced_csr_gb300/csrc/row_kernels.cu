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
// Row-grouped CSR ("New Row-grouped CSR format for storing the sparse
// matrices on GPU with implementation in CUDA", section 3): also one thread
// per row, but over the plan's interleaved copy of A, in which the k-th
// nonzeros of G neighbouring rows are adjacent -- every load of a warp is
// one contiguous 128- or 256-byte line.  Each thread reads its own row
// length, so the group's padding is never loaded.
//
// Both kernels keep several partial sums per row (nonzero k goes to sum
// k mod U) and add them as a tree at the end: U independent chains give the
// loads and FMAs room to overlap, and the rounding error grows with
// length / U instead of length.
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
                      V beta, int32_t skip_min_len) {
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
            for (int u = 0; u < U; ++u) acc[u] = fma(v[u], ld_gather(x + c[u]), acc[u]);
        }
#pragma unroll
        for (int u = 0; u < U - 1; ++u)
            if (k + u < e) acc[u] = fma(ld_stream(val + k + u), ld_gather(x + ld_stream(col + k + u)), acc[u]);
        y[row] = finish(tree_sum(acc), alpha, beta, y, row);
    }
}

// U nonzeros of a row per batch; the next batch's columns and values are
// loaded before the current batch's x gathers, so two batches are in flight.
template <typename V, int U>
__global__ void __launch_bounds__(256)
rgcsr_spmv_kernel(int32_t m, int g_log2, const int64_t *__restrict__ gp, const int32_t *__restrict__ row_len,
                  const int32_t *__restrict__ rg_col, const V *__restrict__ rg_val, const V *__restrict__ x,
                  V *__restrict__ y, V alpha, V beta) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= m) return;
    const int len = ld_stream(row_len + i);
    if (len < 0) return;  // a long row: the long-row kernel writes it
    const int G = 1 << g_log2;
    const int32_t *cp = rg_col + gp[i >> g_log2] + (i & (G - 1));
    const V *vp = rg_val + (cp - rg_col);
    V acc[U];
#pragma unroll
    for (int u = 0; u < U; ++u) acc[u] = V(0);
    const int full = len / U;  // whole batches
    int c[U];
    V v[U];
    if (full > 0) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            c[u] = ld_stream(cp + (int64_t)u * G);
            v[u] = ld_stream(vp + (int64_t)u * G);
        }
    }
    for (int b = 0; b < full; ++b) {
        int cn[U];
        V vn[U];
        const int64_t nk = (int64_t)(b + 1) * U * G;
        if (b + 1 < full) {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                cn[u] = ld_stream(cp + nk + (int64_t)u * G);
                vn[u] = ld_stream(vp + nk + (int64_t)u * G);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) acc[u] = fma(v[u], ld_gather(x + c[u]), acc[u]);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            c[u] = cn[u];
            v[u] = vn[u];
        }
    }
    const int64_t tk = (int64_t)full * U * G;
#pragma unroll
    for (int u = 0; u < U - 1; ++u)
        if (full * U + u < len)
            acc[u] = fma(ld_stream(vp + tk + (int64_t)u * G), ld_gather(x + ld_stream(cp + tk + (int64_t)u * G)), acc[u]);
    y[i] = finish(tree_sum(acc), alpha, beta, y, i);
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
                                  double alpha, double beta, int32_t skip_min_len, cudaStream_t stream) {
    if (m <= 0) return cudaSuccess;
    const int64_t want = ((int64_t)m + 255) / 256;
    const int64_t cap = (int64_t)device_sm_count() * 8;
    const int blocks = (int)(want < cap ? want : cap);
    if (dtype == SPMV_F64)
        thread_per_row_kernel<double><<<blocks, 256, 0, stream>>>(
            m, row_ptr, col_idx, static_cast<const double *>(vals), static_cast<const double *>(x),
            static_cast<double *>(y), alpha, beta, skip_min_len);
    else
        thread_per_row_kernel<float><<<blocks, 256, 0, stream>>>(
            m, row_ptr, col_idx, static_cast<const float *>(vals), static_cast<const float *>(x),
            static_cast<float *>(y), (float)alpha, (float)beta, skip_min_len);
    return cudaGetLastError();
}

cudaError_t launch_rgcsr_spmv(spmv_dtype_t dtype, int32_t m, int g_log2, const int64_t *group_ptr,
                              const int32_t *row_len, const int32_t *rg_col, const void *rg_val,
                              const void *x, void *y, double alpha, double beta, cudaStream_t stream) {
    if (m <= 0) return cudaSuccess;
    const unsigned blocks = (unsigned)(((int64_t)m + 255) / 256);
    if (dtype == SPMV_F64)
        rgcsr_spmv_kernel<double, 4><<<blocks, 256, 0, stream>>>(
            m, g_log2, group_ptr, row_len, rg_col, static_cast<const double *>(rg_val),
            static_cast<const double *>(x), static_cast<double *>(y), alpha, beta);
    else
        rgcsr_spmv_kernel<float, 8><<<blocks, 256, 0, stream>>>(
            m, g_log2, group_ptr, row_len, rg_col, static_cast<const float *>(rg_val),
            static_cast<const float *>(x), static_cast<float *>(y), (float)alpha, (float)beta);
    return cudaGetLastError();
}

}  // namespace lbcsr
