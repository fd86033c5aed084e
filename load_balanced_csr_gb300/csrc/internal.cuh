// Internal declarations shared by the library's translation units.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "spmv.h"

namespace lbcsr {

// ---------------------------------------------------------------- loads
// Matrix arrays (col_idx, vals, row_ptr) are read once per product: stream
// them with the evict-first hint so that they do not push x out of L2.
template <typename T>
__device__ __forceinline__ T ld_stream(const T *p) {
    return __ldcs(p);
}
// x is gathered through the read-only (non-coherent) path.
template <typename T>
__device__ __forceinline__ T ld_gather(const T *p) {
    return __ldg(p);
}

// Debug build (-DSPMV_DEBUG): every column index an SpMV kernel gathers x
// with is checked against [0, n).  One outside it sets kErrIndex in the
// plan's error word and reads x[0] instead, so the gather stays inside x and
// nothing traps.  Plan creation validates every index; this catches arrays
// changed after it (the plan borrows them unmodified).  Without SPMV_DEBUG
// the check compiles to nothing.
constexpr int32_t kErrIndex = 4;
#ifdef SPMV_DEBUG
__device__ __forceinline__ int debug_col(int c, int n, int32_t *error) {
    if ((unsigned)c < (unsigned)n) return c;
    if (error) atomicOr(error, kErrIndex);
    return 0;
}
#else
__device__ __forceinline__ int debug_col(int c, int, int32_t *) { return c; }
#endif

// ---------------------------------------------------------------- statistics
constexpr int kStatsThreads = 256;
constexpr int kStatsRowsPerCta = 4096;  // multiple of 256: Row-grouped groups never straddle CTAs
constexpr int kStatsMinNnzPerCta = 65536;

// Per-CTA partial statistics (workspace), reduced by a second kernel.
struct StatsPartial {
    int32_t hist[32];
    long long rg_slots[4];
    long long sum_len;
    int32_t min_len;
    int32_t max_len;
    int32_t n_empty;
    int32_t flags;
    int32_t bandwidth;
};

int stats_num_ctas(int32_t m, int32_t nnz);
cudaError_t launch_row_stats(int32_t m, int32_t n, int32_t nnz, const int32_t *row_ptr,
                             const int32_t *col_idx, StatsPartial *partials, int num_ctas,
                             spmv_row_stats_t *out, cudaStream_t stream);

// ---------------------------------------------------------------- merge path
cudaError_t launch_merge_path_partition(int32_t m, int32_t nnz, const int32_t *row_ptr,
                                        int64_t items_per_tile, int64_t num_tiles, int2 *part,
                                        cudaStream_t stream);

struct MergePathArgs {
    int32_t m;
    int32_t n = 0;  // columns (the debug build checks gathers against it)
    int32_t nnz;
    const int32_t *row_ptr;
    const int32_t *col_idx;
    const void *vals;
    const void *x;
    void *y;
    double alpha;
    double beta;
    const int2 *part;      // num_tiles + 1 splits
    int64_t num_tiles;
    void *tail_partial;    // [warps] value type: partial of the row open at a warp's run end
    void *head_partial;    // [warps] value type: partial of a cut row finished in a warp's run
    int32_t *arrivals;     // [warps] zero between executions (warps <= num_tiles)
    int32_t *error = nullptr;  // device word: bit 0 set if a copy never completed
    int64_t max_warps = 0;     // > 0: at most this many warps (tail/head/arrivals hold that many)
};

bool merge_path_supported(int items_per_thread);
int merge_path_threads();                       // threads per merge-path tile
int merge_path_min_items();                     // smallest supported items per thread
int merge_path_choose_items(spmv_dtype_t dtype, int32_t n, const spmv_row_stats_t &stats);
cudaError_t launch_merge_path_spmv(spmv_dtype_t dtype, int items_per_thread, const MergePathArgs &a,
                                   cudaStream_t stream);
// Warps the merge-path kernel runs for num_tiles tiles (each owns a run of
// tiles); `aligned`: the kernel variant for 16-byte aligned arrays.  -1 on a
// CUDA error.
int64_t merge_path_num_warps(spmv_dtype_t dtype, int items_per_thread, bool aligned, int64_t num_tiles);

// ---------------------------------------------------------------- plan-time layouts
// Exclusive prefix sum of n int64 values: out[0..n] (out[n] = total).
// scratch holds scan_scratch_elems(n) int64.
int64_t scan_scratch_elems(int64_t n);
cudaError_t launch_exclusive_scan(const int64_t *in, int64_t n, int64_t *out, int64_t *scratch,
                                  cudaStream_t stream);

// Long rows (length >= min_len), after OpSparse's two-pass binning: pass 1
// counts per chunk of kStatsRowsPerCta rows the long rows and their
// segments of kLongSegmentNnz nonzeros; after prefix sums over the chunks,
// pass 2 writes the row ids in ascending order and each row's first segment.
constexpr int kLongSegmentNnz = 4096;
int long_rows_num_chunks(int32_t m);
cudaError_t launch_long_rows_count(int32_t m, const int32_t *row_ptr, int32_t min_len, int64_t *chunk_rows,
                                   int64_t *chunk_segs, cudaStream_t stream);
cudaError_t launch_long_rows_scatter(int32_t m, const int32_t *row_ptr, int32_t min_len,
                                     const int64_t *chunk_row_off, const int64_t *chunk_seg_off,
                                     int32_t *long_rows, int64_t *seg_begin, cudaStream_t stream);

// Row-grouped CSR layout: row_len[i] (-1 for rows of length >= long_min when
// long_min > 0: those rows are left to the long-row kernel), group sizes
// gsize[g] = G * (longest remaining row of group g); after a prefix sum,
// group_ptr; then the interleaved copy (pads must be zero beforehand).
cudaError_t launch_rgcsr_lengths(int32_t m, const int32_t *row_ptr, int g_log2, int32_t long_min,
                                 int32_t *row_len, int64_t *gsize, cudaStream_t stream);
// Window-sorted order (windows of kSortWindow rows, groups of 32): perm[p]
// is the row at position p, eff_len[p] its length (-1 for a long row),
// gsize[g] = 32 * longest row of group g.
constexpr int kSortWindow = 1024;
cudaError_t launch_window_sort(int32_t m, const int32_t *row_ptr, int32_t long_min, int32_t *perm,
                               int32_t *eff_len, int64_t *gsize, cudaStream_t stream);
// perm: the row at each position (null: position = row).
cudaError_t launch_rgcsr_pack(spmv_dtype_t dtype, int32_t m, const int32_t *row_ptr, const int32_t *col_idx,
                              const void *vals, int g_log2, const int64_t *group_ptr, const int32_t *row_len,
                              const int32_t *perm, int32_t *rg_col, void *rg_val, bool pack_cols,
                              cudaStream_t stream);

// ---------------------------------------------------------------- row kernels
// Group-mapped schedule: a CTA per 256 rows, atoms staged by chunks.
cudaError_t launch_group_mapped(spmv_dtype_t dtype, int32_t m, int32_t n, const int32_t *row_ptr,
                                const int32_t *col_idx, const void *vals, const void *x, void *y, double alpha,
                                double beta, int32_t *error, cudaStream_t stream);

// Thread per row; rows of length >= skip_min_len (when > 0) are skipped.
cudaError_t launch_thread_per_row(spmv_dtype_t dtype, int32_t m, int32_t n, const int32_t *row_ptr,
                                  const int32_t *col_idx, const void *vals, const void *x, void *y,
                                  double alpha, double beta, int32_t skip_min_len, int32_t *error,
                                  cudaStream_t stream);

// Row-grouped CSR, thread per row (rows with row_len < 0 are skipped).
// rg_col and rg_val must be 128-byte aligned (the plan allocates them).
// perm (G = 32 only): the row at each position, null for the natural order.
cudaError_t launch_rgcsr_spmv(spmv_dtype_t dtype, int32_t m, int32_t n, int g_log2, const int64_t *group_ptr,
                              const int32_t *row_len, const int32_t *perm, const int32_t *rg_col,
                              const void *rg_val, const void *x, void *y, double alpha, double beta,
                              int32_t *error, cudaStream_t stream);

// Long rows: one warp per segment of kLongSegmentNnz nonzeros; rows with
// several segments are finished by the last segment to arrive.
struct LongRowsArgs {
    int32_t n = 0;             // columns (the debug build checks gathers against it)
    int32_t *error = nullptr;  // the plan's error word (debug build)
    const int32_t *row_ptr;
    const int32_t *col_idx;
    const void *vals;
    const void *x;
    void *y;
    double alpha;
    double beta;
    const int32_t *long_rows;  // [num_long] ascending
    const int64_t *seg_begin;  // [num_long + 1]
    int32_t num_long;
    int64_t num_segs;
    void *seg_partial;         // [num_segs] value type
    int32_t *arrivals;         // [num_long] zero between products
};
cudaError_t launch_long_rows_spmv(spmv_dtype_t dtype, const LongRowsArgs &a, cudaStream_t stream);

// ---------------------------------------------------------------- SpMM
// Y = alpha*A*X + beta*Y, X n-by-k and Y m-by-k row-major (ldx, ldy >= k),
// on the merge-path partition of the plan.  Columns go in slices of
// kSpmmBlocks * 32 per launch.  Scratch: tail and head partials of
// [num_warps][kSpmmBlocks * 32] values each, arrivals[num_warps] (zero
// between products).
constexpr int kSpmmBlocks = 4;
constexpr int kSpmmWarpsPerSm = 32;
int spmm_warps(int64_t num_tiles);
struct SpmmArgs {
    int32_t m, nnz, k;
    const int32_t *row_ptr;
    const int32_t *col_idx;
    const void *vals;
    const void *X;
    int64_t ldx;
    void *Y;
    int64_t ldy;
    double alpha, beta;
    const int2 *part;
    int64_t num_tiles, tile, num_warps;
    void *tail, *head;
    int32_t *arrivals;
};
cudaError_t launch_spmm(spmv_dtype_t dtype, const SpmmArgs &a, cudaStream_t stream);

// SpMM over a Row-grouped copy with groups of 32 and no long rows (thread
// per row, X rows gathered with 16-byte loads when aligned).
struct RgSpmmArgs {
    int32_t m, k;
    const int64_t *group_ptr;
    const int32_t *row_len;
    const int32_t *perm;  // null: natural order
    const int32_t *rg_col;
    const void *rg_val;
    const void *X;
    int64_t ldx;
    void *Y;
    int64_t ldy;
    double alpha, beta;
};
cudaError_t launch_rg_spmm(spmv_dtype_t dtype, const RgSpmmArgs &a, cudaStream_t stream);

// ---------------------------------------------------------------- transpose
// A^T in CSR form: t_ptr[n+1], t_idx[nnz] (rows, increasing in each
// column), t_vals[nnz], t_src[nnz] (position in A).  scratch:
// transpose_scratch_bytes(n, nnz) bytes, 256-byte aligned.
int64_t transpose_scratch_bytes(int32_t n, int32_t nnz);
cudaError_t launch_transpose(spmv_dtype_t dtype, int32_t m, int32_t n, int32_t nnz, const int32_t *row_ptr,
                             const int32_t *col_idx, const void *vals, void *scratch, int32_t *t_ptr,
                             int32_t *t_idx, void *t_vals, int32_t *t_src, cudaStream_t stream);
// t_vals[p] = vals[t_src[p]] (and t_idx[p] = row_of[t_src[p]] when t_idx).
cudaError_t launch_transpose_values(spmv_dtype_t dtype, int32_t nnz, const int32_t *t_src, const int32_t *row_of,
                                    const void *vals, int32_t *t_idx, void *t_vals, cudaStream_t stream);

int device_sm_count();
// Smallest shared-memory carve-out (percent) holding `ctas` CTAs of
// `smem_per_cta` bytes per SM (-1 if the device cannot be queried).
int carveout_percent(int ctas, size_t smem_per_cta);

}  // namespace lbcsr
