// Plan-time builders for the row-mapped kernels: a device-wide prefix sum,
// the list of long rows, and the Row-grouped CSR copy of A.
//
// Long rows follow OpSparse's binning ("OpSparse: a highly optimized
// framework for sparse general matrix multiplication on GPUs", section 5.1,
// Algorithms 1 and 2): a first pass counts, a prefix sum turns the counts
// into offsets, a second pass writes each row id to its place.  OpSparse
// places rows with shared-memory atomics, so the order inside a bin is
// arbitrary; here each CTA ranks its rows with a prefix sum instead, which
// keeps the list in ascending row order (the same plan every time).
//
// Row-grouped CSR ("New Row-grouped CSR format for storing the sparse
// matrices on GPU with implementation in CUDA", section 3, Figure 5): rows
// are taken in groups of G; the k-th nonzeros of a group's rows are stored
// next to each other, and every row of the group is padded to the group's
// longest row.  The group offsets are the prefix sum of G * longest row.
// The page names that padding as the format's weakness (section 4); the
// window-sorted variant lists the rows of each window of kSortWindow rows
// by decreasing length first, so that a group's rows have nearly equal
// lengths.
#include "internal.cuh"

namespace lbcsr {

namespace {

constexpr int kScanThreads = 256;
constexpr int kScanPerThread = 4;
constexpr int kScanTile = kScanThreads * kScanPerThread;  // values per CTA

// Exclusive scan of one value per thread across the CTA; *total gets the sum.
__device__ long long cta_exclusive_scan(long long v, long long *total) {
    __shared__ long long s_warp[kScanThreads / 32];
    __shared__ long long s_total;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    long long incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const long long t = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += t;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const long long w = lane < kScanThreads / 32 ? s_warp[lane] : 0;
        long long wi = w;
#pragma unroll
        for (int off = 1; off < kScanThreads / 32; off <<= 1) {
            const long long t = __shfl_up_sync(0xffffffffu, wi, off);
            if (lane >= off) wi += t;
        }
        if (lane < kScanThreads / 32) s_warp[lane] = wi - w;
        if (lane == kScanThreads / 32 - 1) s_total = wi;
    }
    __syncthreads();
    const long long r = s_warp[warp] + incl - v;
    *total = s_total;
    __syncthreads();  // the shared words may be reused by the next call
    return r;
}

__global__ void __launch_bounds__(kScanThreads)
scan_reduce_kernel(const int64_t *__restrict__ in, int64_t n, int64_t *__restrict__ tile_sums) {
    const int64_t b = (int64_t)blockIdx.x * kScanTile;
    long long s = 0;
#pragma unroll
    for (int q = 0; q < kScanPerThread; ++q) {
        const int64_t i = b + (int64_t)q * kScanThreads + threadIdx.x;
        if (i < n) s += in[i];
    }
    long long total;
    cta_exclusive_scan(s, &total);
    if (threadIdx.x == 0) tile_sums[blockIdx.x] = total;
}

// One CTA: tile_sums[0..nt) -> exclusive offsets, tile_sums[nt] = total.
__global__ void __launch_bounds__(kScanThreads)
scan_tiles_kernel(int64_t *__restrict__ tile_sums, int64_t nt) {
    long long carry = 0;
    for (int64_t b = 0; b < nt; b += kScanThreads) {
        const int64_t i = b + threadIdx.x;
        const long long v = i < nt ? tile_sums[i] : 0;
        long long total;
        const long long ex = cta_exclusive_scan(v, &total);
        if (i < nt) tile_sums[i] = carry + ex;
        carry += total;
    }
    if (threadIdx.x == 0) tile_sums[nt] = carry;
}

__global__ void __launch_bounds__(kScanThreads)
scan_apply_kernel(const int64_t *__restrict__ in, int64_t n, const int64_t *__restrict__ tile_off,
                  int64_t *__restrict__ out) {
    // each thread takes kScanPerThread consecutive values
    const int64_t b = (int64_t)blockIdx.x * kScanTile + (int64_t)threadIdx.x * kScanPerThread;
    long long v[kScanPerThread];
    long long s = 0;
#pragma unroll
    for (int q = 0; q < kScanPerThread; ++q) {
        v[q] = b + q < n ? in[b + q] : 0;
        s += v[q];
    }
    long long total;
    long long run = tile_off[blockIdx.x] + cta_exclusive_scan(s, &total);
#pragma unroll
    for (int q = 0; q < kScanPerThread; ++q) {
        if (b + q < n) out[b + q] = run;
        run += v[q];
    }
    if (blockIdx.x == gridDim.x - 1 && threadIdx.x == 0) out[n] = tile_off[gridDim.x];
}

__device__ __forceinline__ long long segments_of(int len) {
    return ((long long)len + kLongSegmentNnz - 1) / kLongSegmentNnz;
}

// Pass 1: per chunk of rows, the number of long rows and of their segments.
__global__ void __launch_bounds__(kScanThreads)
long_rows_count_kernel(int32_t m, const int32_t *__restrict__ rp, int32_t min_len, int64_t *__restrict__ chunk_rows,
                       int64_t *__restrict__ chunk_segs) {
    const int64_t r0 = (int64_t)blockIdx.x * kStatsRowsPerCta;
    long long rows = 0, segs = 0;
    for (int64_t i = r0 + threadIdx.x; i < r0 + kStatsRowsPerCta && i < m; i += kScanThreads) {
        const int len = rp[i + 1] - rp[i];
        if (len >= min_len) {
            rows += 1;
            segs += segments_of(len);
        }
    }
    long long tr, ts;
    cta_exclusive_scan(rows, &tr);
    cta_exclusive_scan(segs, &ts);
    if (threadIdx.x == 0) {
        chunk_rows[blockIdx.x] = tr;
        chunk_segs[blockIdx.x] = ts;
    }
}

// Pass 2: the chunk's long rows in ascending order at their offsets, with
// the index of each row's first segment.  seg_begin[num_long] = total is
// written by the chunk holding the last long row (or by chunk 0 when
// there are none).
__global__ void __launch_bounds__(kScanThreads)
long_rows_scatter_kernel(int32_t m, const int32_t *__restrict__ rp, int32_t min_len,
                         const int64_t *__restrict__ chunk_row_off, const int64_t *__restrict__ chunk_seg_off,
                         int num_chunks, int32_t *__restrict__ long_rows, int64_t *__restrict__ seg_begin) {
    const int64_t r0 = (int64_t)blockIdx.x * kStatsRowsPerCta;
    long long row_base = chunk_row_off[blockIdx.x];
    long long seg_base = chunk_seg_off[blockIdx.x];
    for (int64_t base = r0; base < r0 + kStatsRowsPerCta && base < m; base += kScanThreads) {
        const int64_t i = base + threadIdx.x;
        int len = 0;
        bool is_long = false;
        if (i < m) {
            len = rp[i + 1] - rp[i];
            is_long = len >= min_len;
        }
        long long nr, ns;
        const long long rank = cta_exclusive_scan(is_long ? 1 : 0, &nr);
        const long long sfirst = cta_exclusive_scan(is_long ? segments_of(len) : 0, &ns);
        if (is_long) {
            long_rows[row_base + rank] = (int32_t)i;
            seg_begin[row_base + rank] = seg_base + sfirst;
        }
        row_base += nr;
        seg_base += ns;
    }
    if (threadIdx.x == 0 && blockIdx.x == num_chunks - 1) seg_begin[row_base] = seg_base;
}

// Row lengths for the Row-grouped layout and each group's padded size.  A
// CTA covers 256 rows, i.e. 256 / G whole groups (G = 32 .. 256).
__global__ void __launch_bounds__(256)
rgcsr_lengths_kernel(int32_t m, const int32_t *__restrict__ rp, int g_log2, int32_t long_min,
                     int32_t *__restrict__ row_len, int64_t *__restrict__ gsize) {
    __shared__ int s_wmax[8];
    const int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x;
    int eff = 0;
    if (i < m) {
        const int len = rp[i + 1] - rp[i];
        const bool is_long = long_min > 0 && len >= long_min;
        row_len[i] = is_long ? -1 : len;
        eff = is_long ? 0 : len;
    }
    const int wmax = __reduce_max_sync(0xffffffffu, eff);
    if ((threadIdx.x & 31) == 0) s_wmax[threadIdx.x >> 5] = wmax;
    __syncthreads();
    const int G = 1 << g_log2;
    const int groups_here = 256 >> g_log2;
    if ((int)threadIdx.x < groups_here) {
        const int wpg = G >> 5;  // warps per group
        int mx = 0;
        for (int w = 0; w < wpg; ++w) mx = max(mx, s_wmax[threadIdx.x * wpg + w]);
        const int64_t g = ((int64_t)blockIdx.x * 256 >> g_log2) + threadIdx.x;
        const int64_t ngroups = ((int64_t)m + G - 1) >> g_log2;
        if (g < ngroups) gsize[g] = (int64_t)G * mx;
    }
}

// Window-sorted order: one CTA per window of kSortWindow rows sorts the keys
// (length descending, row ascending; long rows count as length -1) with a
// bitonic network in shared memory.  Keys are unique (they hold the row), so
// the order is the same every time.  Position p gets perm[p], its length
// eff_len[p], and the first position of every group of 32 -- the group's
// longest row, as lengths fall inside a window -- sets the group's size.
__global__ void __launch_bounds__(kSortWindow)
window_sort_kernel(int32_t m, const int32_t *__restrict__ rp, int32_t long_min, int32_t *__restrict__ perm,
                   int32_t *__restrict__ eff_len, int64_t *__restrict__ gsize) {
    __shared__ unsigned long long keys[kSortWindow];
    const int t = threadIdx.x;
    const int64_t r = (int64_t)blockIdx.x * kSortWindow + t;
    unsigned long long key = ~0ull;  // past the last row: sorts last
    if (r < m) {
        const int len = rp[r + 1] - rp[r];
        const int eff = long_min > 0 && len >= long_min ? -1 : len;
        key = ((unsigned long long)(0x7fffffffLL - eff) << 32) | (unsigned long long)(uint32_t)r;
    }
    keys[t] = key;
    __syncthreads();
    for (int k = 2; k <= kSortWindow; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            const int partner = t ^ j;
            if (partner > t) {
                const unsigned long long a = keys[t], b = keys[partner];
                const bool ascending = (t & k) == 0;
                if ((a > b) == ascending) {
                    keys[t] = b;
                    keys[partner] = a;
                }
            }
            __syncthreads();
        }
    }
    if (r < m) {  // positions of this window are its rows' slots
        const unsigned long long kk = keys[t];
        const int eff = (int)(0x7fffffffLL - (long long)(kk >> 32));
        perm[r] = (int32_t)(kk & 0xffffffffull);
        eff_len[r] = eff;
        if ((t & 31) == 0) gsize[r >> 5] = 32LL * (eff > 0 ? eff : 0);
    }
}

// The interleaved copy: element k of the row at position i goes to
// group_ptr[i / G] + k*G + (i mod G); the row is perm[i] (i itself when perm
// is null).  One thread per position; at every k the threads of a warp
// write neighbouring slots.
template <typename V>
__global__ void __launch_bounds__(256)
rgcsr_pack_kernel(int32_t m, const int32_t *__restrict__ rp, const int32_t *__restrict__ col,
                  const V *__restrict__ val, int g_log2, const int64_t *__restrict__ gp,
                  const int32_t *__restrict__ row_len, const int32_t *__restrict__ perm, int32_t *__restrict__ rg_col,
                  V *__restrict__ rg_val, bool pack_cols) {
    const int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x;
    if (i >= m) return;
    const int len = row_len[i];
    if (len <= 0) return;
    const int G = 1 << g_log2;
    const int64_t base = gp[i >> g_log2] + (i & (G - 1));
    const int32_t b = rp[perm ? perm[i] : i];
    for (int k = 0; k < len; ++k) {
        if (pack_cols) rg_col[base + (int64_t)k * G] = col[b + k];
        rg_val[base + (int64_t)k * G] = val[b + k];
    }
}

}  // namespace

int64_t scan_scratch_elems(int64_t n) { return (n + kScanTile - 1) / kScanTile + 1; }

cudaError_t launch_exclusive_scan(const int64_t *in, int64_t n, int64_t *out, int64_t *scratch,
                                  cudaStream_t stream) {
    if (n <= 0) return cudaMemsetAsync(out, 0, sizeof(int64_t), stream);
    const int64_t nt = (n + kScanTile - 1) / kScanTile;
    scan_reduce_kernel<<<(unsigned)nt, kScanThreads, 0, stream>>>(in, n, scratch);
    scan_tiles_kernel<<<1, kScanThreads, 0, stream>>>(scratch, nt);
    scan_apply_kernel<<<(unsigned)nt, kScanThreads, 0, stream>>>(in, n, scratch, out);
    return cudaGetLastError();
}

int long_rows_num_chunks(int32_t m) {
    const int c = (int)(((int64_t)m + kStatsRowsPerCta - 1) / kStatsRowsPerCta);
    return c < 1 ? 1 : c;
}

cudaError_t launch_long_rows_count(int32_t m, const int32_t *row_ptr, int32_t min_len, int64_t *chunk_rows,
                                   int64_t *chunk_segs, cudaStream_t stream) {
    long_rows_count_kernel<<<long_rows_num_chunks(m), kScanThreads, 0, stream>>>(m, row_ptr, min_len, chunk_rows,
                                                                                  chunk_segs);
    return cudaGetLastError();
}

cudaError_t launch_long_rows_scatter(int32_t m, const int32_t *row_ptr, int32_t min_len,
                                     const int64_t *chunk_row_off, const int64_t *chunk_seg_off,
                                     int32_t *long_rows, int64_t *seg_begin, cudaStream_t stream) {
    const int nc = long_rows_num_chunks(m);
    long_rows_scatter_kernel<<<nc, kScanThreads, 0, stream>>>(m, row_ptr, min_len, chunk_row_off, chunk_seg_off,
                                                              nc, long_rows, seg_begin);
    return cudaGetLastError();
}

cudaError_t launch_rgcsr_lengths(int32_t m, const int32_t *row_ptr, int g_log2, int32_t long_min,
                                 int32_t *row_len, int64_t *gsize, cudaStream_t stream) {
    if (m <= 0) return cudaSuccess;
    const unsigned blocks = (unsigned)(((int64_t)m + 255) / 256);
    rgcsr_lengths_kernel<<<blocks, 256, 0, stream>>>(m, row_ptr, g_log2, long_min, row_len, gsize);
    return cudaGetLastError();
}

cudaError_t launch_window_sort(int32_t m, const int32_t *row_ptr, int32_t long_min, int32_t *perm,
                               int32_t *eff_len, int64_t *gsize, cudaStream_t stream) {
    if (m <= 0) return cudaSuccess;
    const unsigned blocks = (unsigned)(((int64_t)m + kSortWindow - 1) / kSortWindow);
    window_sort_kernel<<<blocks, kSortWindow, 0, stream>>>(m, row_ptr, long_min, perm, eff_len, gsize);
    return cudaGetLastError();
}

cudaError_t launch_rgcsr_pack(spmv_dtype_t dtype, int32_t m, const int32_t *row_ptr, const int32_t *col_idx,
                              const void *vals, int g_log2, const int64_t *group_ptr, const int32_t *row_len,
                              const int32_t *perm, int32_t *rg_col, void *rg_val, bool pack_cols,
                              cudaStream_t stream) {
    if (m <= 0) return cudaSuccess;
    const unsigned blocks = (unsigned)(((int64_t)m + 255) / 256);
    if (dtype == SPMV_F64)
        rgcsr_pack_kernel<double><<<blocks, 256, 0, stream>>>(m, row_ptr, col_idx, static_cast<const double *>(vals),
                                                              g_log2, group_ptr, row_len, perm, rg_col,
                                                              static_cast<double *>(rg_val), pack_cols);
    else
        rgcsr_pack_kernel<float><<<blocks, 256, 0, stream>>>(m, row_ptr, col_idx, static_cast<const float *>(vals),
                                                             g_log2, group_ptr, row_len, perm, rg_col,
                                                             static_cast<float *>(rg_val), pack_cols);
    return cudaGetLastError();
}

}  // namespace lbcsr
