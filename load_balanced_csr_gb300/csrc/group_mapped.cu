// Group-mapped SpMV: the group-level load balancing of "A GPU
// load-balancing programming model" (section 5.2.3).  A group -- here a
// CTA of kGmThreads threads -- takes an equal share of tiles (rows), counts
// each tile's atoms (nonzeros) into a prefix-sum array in shared memory,
// and its threads then take the group's atoms in a range loop strided by
// the group size, so that consecutive threads read consecutive nonzeros
// whatever the row lengths.
//
// The page's threads find an atom's tile by a binary search in the
// prefix-sum array and add its product into y.  Here the products of a
// chunk of kGmChunk atoms go to shared memory instead, and each thread then
// adds up its own row's products in order: no atomics, and the same sums
// every time.  (The thread of a row knows where its atoms sit from the
// prefix-sum array, so no search is needed.)  Rows longer than a chunk are
// summed over several chunks; the imbalance between groups is left to the
// hardware scheduler, as on the page.
#include "internal.cuh"

namespace lbcsr {

namespace {

constexpr int kGmThreads = 256;  // rows per group, threads per group
constexpr int kGmChunk = 2048;   // atoms staged per round
constexpr int kGmItems = kGmChunk / kGmThreads;

template <typename V>
__global__ void __launch_bounds__(kGmThreads)
group_mapped_kernel(int32_t m, const int32_t *__restrict__ rp, const int32_t *__restrict__ col,
                    const V *__restrict__ val, const V *__restrict__ x, V *__restrict__ y, V alpha, V beta,
                    int32_t n, int32_t *error) {
    __shared__ int pre[kGmThreads + 1];
    __shared__ int s_warp[kGmThreads / 32];
    __shared__ V prod[kGmChunk];
    const int t = threadIdx.x;
    const int lane = t & 31, warp = t >> 5;
    const long long r = (long long)blockIdx.x * kGmThreads + t;
    const long long r0 = (long long)blockIdx.x * kGmThreads;
    const int len = r < m ? rp[r + 1] - rp[r] : 0;

    // exclusive prefix sum of the group's row lengths (the group's atoms
    // are contiguous, so they fit int32 like nnz)
    int incl = len;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int w = lane < kGmThreads / 32 ? s_warp[lane] : 0;
        int wi = w;
#pragma unroll
        for (int off = 1; off < kGmThreads / 32; off <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, wi, off);
            if (lane >= off) wi += v;
        }
        if (lane < kGmThreads / 32) s_warp[lane] = wi - w;
    }
    __syncthreads();
    const int start = s_warp[warp] + incl - len;  // my row's first atom
    pre[t] = start;
    if (t == kGmThreads - 1) pre[kGmThreads] = start + len;
    __syncthreads();
    const int total = pre[kGmThreads];
    const long long base = r0 < m ? rp[r0] : 0;  // the group's first nonzero

    // four partial sums used in turn (kept in registers by rotating them)
    V s0 = V(0), s1 = V(0), s2 = V(0), s3 = V(0);
    for (int c0 = 0; c0 < total; c0 += kGmChunk) {
        const int cn = min(kGmChunk, total - c0);
        // the range loop: atom c0 + t + i * kGmThreads for this thread
        int cc[kGmItems];
        V vv[kGmItems];
#pragma unroll
        for (int i = 0; i < kGmItems; ++i) {
            const int a = t + i * kGmThreads;
            cc[i] = a < cn ? ld_stream(col + base + c0 + a) : 0;
            vv[i] = a < cn ? ld_stream(val + base + c0 + a) : V(0);
        }
#pragma unroll
        for (int i = 0; i < kGmItems; ++i) {
            const int a = t + i * kGmThreads;
            if (a < cn) prod[a] = vv[i] * ld_gather(x + debug_col(cc[i], n, error));
        }
        __syncthreads();
        // my row's atoms in this chunk, in order
        const int lo = max(start, c0) - c0, hi = min(start + len, c0 + cn) - c0;
        for (int a = lo; a < hi; ++a) {
            const V v = s0 + prod[a];
            s0 = s1;
            s1 = s2;
            s2 = s3;
            s3 = v;
        }
        __syncthreads();
    }
    if (r < m) {
        V res = alpha * ((s0 + s1) + (s2 + s3));
        if (beta != V(0)) res = fma(beta, y[r], res);
        y[r] = res;
    }
}

}  // namespace

cudaError_t launch_group_mapped(spmv_dtype_t dtype, int32_t m, int32_t n, const int32_t *row_ptr,
                                const int32_t *col_idx, const void *vals, const void *x, void *y, double alpha,
                                double beta, int32_t *error, cudaStream_t stream) {
    if (m <= 0) return cudaSuccess;
    const unsigned groups = (unsigned)(((int64_t)m + kGmThreads - 1) / kGmThreads);
    if (dtype == SPMV_F64)
        group_mapped_kernel<double><<<groups, kGmThreads, 0, stream>>>(
            m, row_ptr, col_idx, static_cast<const double *>(vals), static_cast<const double *>(x),
            static_cast<double *>(y), alpha, beta, n, error);
    else
        group_mapped_kernel<float><<<groups, kGmThreads, 0, stream>>>(
            m, row_ptr, col_idx, static_cast<const float *>(vals), static_cast<const float *>(x),
            static_cast<float *>(y), (float)alpha, (float)beta, n, error);
    return cudaGetLastError();
}

}  // namespace lbcsr
