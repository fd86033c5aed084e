// Plan-time analysis kernels: row-length statistics and the merge-path
// partition.
//
// Statistics follow OpSparse's row binning ("OpSparse: a highly optimized
// framework for sparse general matrix multiplication on GPUs", section 5.1,
// Algorithm 1): each CTA counts its rows per length class and tracks the
// longest row with shared-memory atomics only; per-CTA results go to the
// workspace and a second single-CTA kernel adds them up in a fixed order,
// so no global atomics are involved and the result is deterministic.
//
// The partition is the merge-path split of "A GPU load-balancing
// programming model" (section 5.2.1): the m row ends and the nnz nonzeros
// are m + nnz equal units of work, taken in merge order (a row end before
// the nonzero at the same index), and tile p starts after p*T units.  After
// d units, the row ends taken are those with row_ptr[r+1] + r < d, a
// strictly increasing sequence in r, so each split is one binary search.
#include <climits>

#include "internal.cuh"

namespace lbcsr {

namespace {

__device__ __forceinline__ int length_class(int len) {
    return len <= 0 ? 0 : 32 - __clz(len);  // 0 for empty, else bit length
}

__global__ void __launch_bounds__(kStatsThreads)
row_stats_kernel(int32_t m, int32_t n, int32_t nnz, const int32_t *__restrict__ row_ptr,
                 const int32_t *__restrict__ col_idx, int64_t nnz_per_cta,
                 StatsPartial *__restrict__ partials) {
    __shared__ int s_hist[32];
    __shared__ int s_min, s_max, s_empty, s_flags, s_bw;
    __shared__ int s_wmax[kStatsThreads / 32];
    __shared__ long long s_rg[4];
    const int tid = threadIdx.x;
    if (tid < 32) s_hist[tid] = 0;
    if (tid < 4) s_rg[tid] = 0;
    if (tid == 0) {
        s_min = INT_MAX;
        s_max = 0;
        s_empty = 0;
        s_flags = 0;
        s_bw = 0;
    }
    __syncthreads();

    const int64_t r0 = (int64_t)blockIdx.x * kStatsRowsPerCta;
    for (int64_t base = r0; base < r0 + kStatsRowsPerCta && base < m; base += kStatsThreads) {
        const int64_t i = base + tid;
        int len = 0;
        if (i < m) {
            const int a = row_ptr[i];
            const int b = row_ptr[i + 1];
            if (i == 0 && a != 0) atomicOr(&s_flags, 1);
            len = b - a;
            if (len < 0) {
                atomicOr(&s_flags, 2);
                len = 0;
            }
            atomicAdd(&s_hist[length_class(len)], 1);
            atomicMin(&s_min, len);
            atomicMax(&s_max, len);
            if (len == 0) atomicAdd(&s_empty, 1);
            // distance of the row's outermost stored entries from the diagonal
            // (read only when the row's range lies inside col_idx)
            if (len > 0 && a >= 0 && b <= nnz) {
                const long long d0 = (long long)col_idx[a] - i, d1 = (long long)col_idx[b - 1] - i;
                const long long d = max(d0 < 0 ? -d0 : d0, d1 < 0 ? -d1 : d1);
                atomicMax(&s_bw, (int)min(d, (long long)INT_MAX));
            }
        }
        // Row-grouped CSR storage: groups of G = 32, 64, 128, 256 rows, each
        // padded to its longest row (rows past m count as empty).
        const int wmax = __reduce_max_sync(0xffffffffu, len);
        if ((tid & 31) == 0) s_wmax[tid >> 5] = wmax;
        __syncthreads();
        if (tid == 0) {
            long long g32 = 0, g64 = 0, g128 = 0;
            int all = 0;
            for (int w = 0; w < kStatsThreads / 32; w += 4) {
                const int a0 = s_wmax[w], a1 = s_wmax[w + 1], a2 = s_wmax[w + 2], a3 = s_wmax[w + 3];
                g32 += 32LL * (a0 + a1 + a2 + a3);
                g64 += 64LL * (max(a0, a1) + max(a2, a3));
                g128 += 128LL * max(max(a0, a1), max(a2, a3));
                all = max(all, max(max(a0, a1), max(a2, a3)));
            }
            s_rg[0] += g32;
            s_rg[1] += g64;
            s_rg[2] += g128;
            s_rg[3] += 256LL * all;
        }
        __syncthreads();
    }
    // row_ptr[m] must equal nnz: checked by the CTA holding the last row.
    if (tid == 0 && (m == 0 ? blockIdx.x == 0 : (m - 1) / kStatsRowsPerCta == (int64_t)blockIdx.x)) {
        if (row_ptr[m] != nnz) atomicOr(&s_flags, 4);
        if (m == 0 && row_ptr[0] != 0) atomicOr(&s_flags, 1);
    }
    // every column index in [0, n)
    const int64_t c0 = (int64_t)blockIdx.x * nnz_per_cta;
    const int64_t c1 = min(c0 + nnz_per_cta, (int64_t)nnz);
    int bad = 0;
    for (int64_t k = c0 + tid; k < c1; k += kStatsThreads) {
        const int c = col_idx[k];
        bad |= (c < 0) | (c >= n);
    }
    if (__syncthreads_or(bad) && tid == 0) s_flags |= 8;
    __syncthreads();

    StatsPartial *out = partials + blockIdx.x;
    if (tid < 32) out->hist[tid] = s_hist[tid];
    if (tid < 4) out->rg_slots[tid] = s_rg[tid];
    if (tid == 0) {
        const int64_t r1 = min(r0 + kStatsRowsPerCta, (int64_t)m);
        out->sum_len = r1 > r0 ? (long long)row_ptr[r1] - row_ptr[r0] : 0;
        out->min_len = s_min;
        out->max_len = s_max;
        out->n_empty = s_empty;
        out->flags = s_flags;
        out->bandwidth = s_bw;
    }
}

// One CTA adds the per-CTA partials up: warp w reduces fields w, w + 32,
// ... (0-31 the classes, 32-35 the Row-grouped slots, 36 the length sum,
// 37 min, 38 max, 39 empty rows, 40 flags, 41 bandwidth), its lanes
// striding over the partials.  Integer sums, minima and maxima do not
// depend on the order.
constexpr int kStatsFields = 42;

__device__ __forceinline__ long long stats_field(const StatsPartial &q, int f) {
    if (f < 32) return q.hist[f];
    if (f < 36) return q.rg_slots[f - 32];
    switch (f) {
    case 36: return q.sum_len;
    case 37: return q.min_len;
    case 38: return q.max_len;
    case 39: return q.n_empty;
    case 40: return q.flags;
    default: return q.bandwidth;
    }
}

__global__ void __launch_bounds__(1024)
stats_reduce_kernel(int num, const StatsPartial *__restrict__ partials, int32_t m,
                    spmv_row_stats_t *__restrict__ out) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int f = warp; f < kStatsFields; f += 32) {
        const bool is_min = f == 37, is_max = f == 38 || f == 41, is_or = f == 40;
        long long v = is_min ? (long long)INT_MAX : 0;
        for (int b = lane; b < num; b += 32) {
            const long long q = stats_field(partials[b], f);
            v = is_min ? min(v, q) : is_max ? max(v, q) : is_or ? (v | q) : v + q;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const long long q = __shfl_xor_sync(0xffffffffu, v, off);
            v = is_min ? min(v, q) : is_max ? max(v, q) : is_or ? (v | q) : v + q;
        }
        if (lane != 0) continue;
        if (f < 32) out->hist[f] = v;
        else if (f < 36) out->rg_slots[f - 32] = v;
        else if (f == 36) out->sum_len = v;
        else if (f == 37) out->min_len = m > 0 ? (int)v : 0;
        else if (f == 38) out->max_len = (int)v;
        else if (f == 39) out->n_empty = (int)v;
        else if (f == 40) out->flags = (int)v;
        else {
            out->bandwidth = m > 0 ? (int)v : 0;
            out->reserved = 0;
        }
    }
}

__global__ void __launch_bounds__(256)
merge_path_partition_kernel(int32_t m, int32_t nnz, const int32_t *__restrict__ row_ptr,
                            int64_t items_per_tile, int64_t num_tiles, int2 *__restrict__ part) {
    const int64_t p = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (p > num_tiles) return;
    const int64_t total = (int64_t)m + nnz;
    const int64_t d = min(p * items_per_tile, total);
    // i(d) = #{ r : row_ptr[r+1] + r < d } lies in [max(0, d - nnz), min(d, m)]
    int64_t lo = max((int64_t)0, d - nnz);
    int64_t hi = min(d, (int64_t)m);
    while (lo < hi) {
        const int64_t mid = (lo + hi) >> 1;
        if ((int64_t)row_ptr[mid + 1] + mid < d) lo = mid + 1;
        else hi = mid;
    }
    part[p] = make_int2((int)lo, (int)(d - lo));
}

}  // namespace

int stats_num_ctas(int32_t m, int32_t nnz) {
    const int64_t by_rows = ((int64_t)m + kStatsRowsPerCta - 1) / kStatsRowsPerCta;
    const int64_t by_nnz = ((int64_t)nnz + kStatsMinNnzPerCta - 1) / kStatsMinNnzPerCta;
    int64_t b = by_rows > by_nnz ? by_rows : by_nnz;
    return (int)(b < 1 ? 1 : b);
}

cudaError_t launch_row_stats(int32_t m, int32_t n, int32_t nnz, const int32_t *row_ptr,
                             const int32_t *col_idx, StatsPartial *partials, int num_ctas,
                             spmv_row_stats_t *out, cudaStream_t stream) {
    const int64_t nnz_per_cta = ((int64_t)nnz + num_ctas - 1) / num_ctas;
    row_stats_kernel<<<num_ctas, kStatsThreads, 0, stream>>>(m, n, nnz, row_ptr, col_idx, nnz_per_cta,
                                                             partials);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    stats_reduce_kernel<<<1, 1024, 0, stream>>>(num_ctas, partials, m, out);
    return cudaGetLastError();
}

cudaError_t launch_merge_path_partition(int32_t m, int32_t nnz, const int32_t *row_ptr,
                                        int64_t items_per_tile, int64_t num_tiles, int2 *part,
                                        cudaStream_t stream) {
    const int64_t threads = num_tiles + 1;
    const int blocks = (int)((threads + 255) / 256);
    merge_path_partition_kernel<<<blocks, 256, 0, stream>>>(m, nnz, row_ptr, items_per_tile, num_tiles,
                                                            part);
    return cudaGetLastError();
}

}  // namespace lbcsr
