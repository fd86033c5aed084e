// Long rows: one warp per segment of kLongSegmentNnz nonzeros.
//
// "A GPU load-balancing programming model" (section 5.2.2) leaves the
// imbalance of a row-mapped schedule to the hardware scheduler; OpSparse
// ("OpSparse: a highly optimized framework for sparse general matrix
// multiplication on GPUs", section 5.1) gives its longest rows their own,
// wider kernels and launches them first.  Here every row the plan lists as
// long is cut into segments of equal size; a row of up to one segment gets
// one warp (warp per row), a longer row as many warps as it has segments,
// spread over CTAs (CTA per row and the multi-CTA split in one scheme).
//
// A warp reads its segment with lane-strided loads (each warp load is one
// contiguous 128-byte line of col_idx and of vals) and keeps 8 partial sums
// per lane, then adds them as a tree and across lanes with a shuffle tree.
// A one-segment row is written directly.  Otherwise the warp stores its
// partial and counts in on the row's arrival counter; the segment that
// arrives last adds the row's partials in segment order (a fixed tree, so
// the result does not depend on which warp came last) and writes y.
#include "internal.cuh"

namespace lbcsr {

namespace {

constexpr int kLongThreads = 256;
constexpr int kLongWarps = kLongThreads / 32;
constexpr int kLongU = 8;

template <typename V>
__global__ void __launch_bounds__(kLongThreads)
long_rows_kernel(const int32_t *__restrict__ rp, const int32_t *__restrict__ col, const V *__restrict__ val,
                 const V *__restrict__ x, V *__restrict__ y, V alpha, V beta,
                 const int32_t *__restrict__ long_rows, const int64_t *__restrict__ seg_begin, int32_t num_long,
                 int64_t num_segs, V *__restrict__ seg_partial, int32_t *__restrict__ arrivals, int32_t n,
                 int32_t *error) {
    const int lane = threadIdx.x & 31;
    const int64_t s = (int64_t)blockIdx.x * kLongWarps + (threadIdx.x >> 5);
    if (s >= num_segs) return;
    // the long row holding segment s: the last r with seg_begin[r] <= s
    int lo = 0, hi = num_long - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (seg_begin[mid] <= s) lo = mid;
        else hi = mid - 1;
    }
    const int32_t row = long_rows[lo];
    const int64_t first = seg_begin[lo];
    const int64_t nsegs = seg_begin[lo + 1] - first;
    const int32_t rb = rp[row], re = rp[row + 1];
    const int32_t b = rb + (int32_t)((s - first) * kLongSegmentNnz);
    const int32_t e = min(b + kLongSegmentNnz, re);

    V acc[kLongU];
#pragma unroll
    for (int u = 0; u < kLongU; ++u) acc[u] = V(0);
    int32_t k = b + lane;
    for (; k + (kLongU - 1) * 32 < e; k += kLongU * 32) {
        int c[kLongU];
        V v[kLongU];
#pragma unroll
        for (int u = 0; u < kLongU; ++u) {
            c[u] = ld_stream(col + k + u * 32);
            v[u] = ld_stream(val + k + u * 32);
        }
#pragma unroll
        for (int u = 0; u < kLongU; ++u) acc[u] = fma(v[u], ld_gather(x + debug_col(c[u], n, error)), acc[u]);
    }
#pragma unroll
    for (int u = 0; u < kLongU - 1; ++u)
        if (k + u * 32 < e)
            acc[u] = fma(ld_stream(val + k + u * 32), ld_gather(x + debug_col(ld_stream(col + k + u * 32), n, error)),
                         acc[u]);
#pragma unroll
    for (int w = 1; w < kLongU; w <<= 1)
#pragma unroll
        for (int u = 0; u + w < kLongU; u += 2 * w) acc[u] += acc[u + w];
    V sum = acc[0];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);

    if (nsegs == 1) {
        if (lane == 0) {
            V r = alpha * sum;
            if (beta != V(0)) r = fma(beta, y[row], r);
            y[row] = r;
        }
        return;
    }
    int last = 0;
    if (lane == 0) {
        seg_partial[s] = sum;
        __threadfence();
        last = atomicAdd(arrivals + lo, 1) == (int)(nsegs - 1);
        if (last) __threadfence();
    }
    if (!__shfl_sync(0xffffffffu, last, 0)) return;
    V t = V(0);
    for (int64_t q = first + lane; q < first + nsegs; q += 32) t += __ldcg(seg_partial + q);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
    if (lane == 0) {
        V r = alpha * t;
        if (beta != V(0)) r = fma(beta, y[row], r);
        y[row] = r;
        arrivals[lo] = 0;  // ready for the next product
    }
}

}  // namespace

cudaError_t launch_long_rows_spmv(spmv_dtype_t dtype, const LongRowsArgs &a, cudaStream_t stream) {
    if (a.num_long <= 0 || a.num_segs <= 0) return cudaSuccess;
    const unsigned blocks = (unsigned)((a.num_segs + kLongWarps - 1) / kLongWarps);
    if (dtype == SPMV_F64)
        long_rows_kernel<double><<<blocks, kLongThreads, 0, stream>>>(
            a.row_ptr, a.col_idx, static_cast<const double *>(a.vals), static_cast<const double *>(a.x),
            static_cast<double *>(a.y), a.alpha, a.beta, a.long_rows, a.seg_begin, a.num_long, a.num_segs,
            static_cast<double *>(a.seg_partial), a.arrivals, a.n, a.error);
    else
        long_rows_kernel<float><<<blocks, kLongThreads, 0, stream>>>(
            a.row_ptr, a.col_idx, static_cast<const float *>(a.vals), static_cast<const float *>(a.x),
            static_cast<float *>(a.y), (float)a.alpha, (float)a.beta, a.long_rows, a.seg_begin, a.num_long,
            a.num_segs, static_cast<float *>(a.seg_partial), a.arrivals, a.n, a.error);
    return cudaGetLastError();
}

}  // namespace lbcsr
