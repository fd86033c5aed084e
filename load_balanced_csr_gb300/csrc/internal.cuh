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
    void *tail_partial;    // [num_tiles] value type: partial of the row open at a tile's end
    void *head_partial;    // [num_tiles] value type: partial of a split row finished in a tile
    int32_t *arrivals;     // [num_tiles] zero between executions
    int32_t *error = nullptr;  // device word: bit 0 set if a copy never completed
};

bool merge_path_supported(int items_per_thread);
int merge_path_threads();                       // threads per merge-path tile
int merge_path_min_items();                     // smallest supported items per thread
int merge_path_choose_items(spmv_dtype_t dtype, int32_t n, const spmv_row_stats_t &stats);
cudaError_t launch_merge_path_spmv(spmv_dtype_t dtype, int items_per_thread, const MergePathArgs &a,
                                   cudaStream_t stream);

// ---------------------------------------------------------------- row kernels
cudaError_t launch_thread_per_row(spmv_dtype_t dtype, int32_t m, const int32_t *row_ptr,
                                  const int32_t *col_idx, const void *vals, const void *x, void *y,
                                  double alpha, double beta, cudaStream_t stream);

int device_sm_count();

}  // namespace lbcsr
