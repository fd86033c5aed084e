// One-shot merge-path product that allocates no memory.
//
// Some callers cannot allocate device memory at the point where they need a
// product: for example a service that reserves the whole device for its own
// memory pool at start-up (a cudaMalloc then fails, or fragments the pool),
// or a latency-critical loop where a cudaMalloc would implicitly synchronise
// the device and stall the work already queued on other streams.  For them,
// spmv_execute_noalloc runs the merge-path product with its scratch (tile
// splits, cut-row partial sums, arrival counters, a failure word) in a
// fixed-size array in the library's own device memory, declared below.  The
// array is part of the loaded module: every GPU that loads the library holds
// it until the process exits.  Every call shares it, so calls that overlap
// on the GPU (on two streams, or two host threads) race and give wrong
// results.
#include <cstring>

#include "internal.cuh"

namespace lbcsr {
namespace {

// Tiles of 384 units (12 items per lane, the merge-path kernel's choice for
// matrices with scattered columns), for m + nnz <= 2^28 rows plus nonzeros.
constexpr int kNoAllocItemsPerLane = 12;
constexpr int64_t kNoAllocMaxUnits = int64_t(1) << 28;
constexpr int64_t kNoAllocTile = 32 * kNoAllocItemsPerLane;
constexpr int64_t kNoAllocMaxTiles = (kNoAllocMaxUnits + kNoAllocTile - 1) / kNoAllocTile;
// The kernel's cut-row partials and arrival counters are per warp (at most
// one warp per tile, and no more than the GPU holds at once).
constexpr int64_t kNoAllocMaxWarps = 16384;

struct NoAllocLayout {
    int2 part[kNoAllocMaxTiles + 1];
    double tail[kNoAllocMaxWarps];
    double head[kNoAllocMaxWarps];
    int32_t error;                       // cleared with the counters
    int32_t arrivals[kNoAllocMaxWarps];  // zero between products
};

// Scratch of spmv_execute_noalloc (about 6 MB).  Host code must not pass
// this name to a kernel: on the host it is only a stand-in for the symbol.
// The device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[sizeof(NoAllocLayout)];

// The scratch's device address on the current device and context.  Looked
// up on every call: once the module is loaded this is a host-side table
// lookup, and it stays right after a device reset or under another context
// (a cached address would not).  The first lookup on a device loads the
// module there, which is why the first call should come before any stream
// capture.
NoAllocLayout *scratch_address() {
    void *addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess) return nullptr;
    return static_cast<NoAllocLayout *>(addr);
}

}  // namespace
}  // namespace lbcsr

using namespace lbcsr;

extern "C" spmv_status_t spmv_execute_noalloc(int32_t m, int32_t n, int32_t nnz, const int32_t *row_ptr,
                                              const int32_t *col_idx, const void *vals, spmv_dtype_t dtype,
                                              double alpha, const void *x, double beta, void *y,
                                              spmv_stream_t stream_handle) {
    if (m < 0 || n < 0 || nnz < 0) return SPMV_ERR_INVALID_ARG;
    if ((int64_t)m + (int64_t)nnz > kNoAllocMaxUnits) return SPMV_ERR_INVALID_ARG;  // beyond the fixed scratch
    if (dtype != SPMV_F32 && dtype != SPMV_F64) return SPMV_ERR_INVALID_ARG;
    if (m == 0) return SPMV_OK;
    if (!row_ptr || !y) return SPMV_ERR_INVALID_ARG;
    if (nnz > 0 && (!col_idx || !vals || !x)) return SPMV_ERR_INVALID_ARG;

    const int64_t P = ((int64_t)m + nnz + kNoAllocTile - 1) / kNoAllocTile;
    NoAllocLayout *s = scratch_address();
    if (!s) return SPMV_ERR_CUDA;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_handle);

    // the failure word and the arrival counters must start at zero (the
    // kernel leaves the counters at zero, but a call that was interrupted
    // may not have)
    const int64_t warps = P < kNoAllocMaxWarps ? P : kNoAllocMaxWarps;
    if (cudaMemsetAsync(&s->error, 0, sizeof(int32_t) * (size_t)(1 + warps), stream) != cudaSuccess)
        return SPMV_ERR_CUDA;
    if (launch_merge_path_partition(m, nnz, row_ptr, kNoAllocTile, P, s->part, stream) != cudaSuccess)
        return SPMV_ERR_CUDA;
    MergePathArgs a;
    a.m = m;
    a.n = n;
    a.nnz = nnz;
    a.row_ptr = row_ptr;
    a.col_idx = col_idx;
    a.vals = vals;
    a.x = x;
    a.y = y;
    a.alpha = alpha;
    a.beta = beta;
    a.part = s->part;
    a.num_tiles = P;
    a.tail_partial = s->tail;
    a.head_partial = s->head;
    a.arrivals = s->arrivals;
    a.error = &s->error;
    a.max_warps = kNoAllocMaxWarps;
    if (launch_merge_path_spmv(dtype, kNoAllocItemsPerLane, a, stream) != cudaSuccess) return SPMV_ERR_CUDA;
    return SPMV_OK;
}

extern "C" spmv_status_t spmv_noalloc_device_status(int32_t *flags) {
    if (!flags) return SPMV_ERR_INVALID_ARG;
    NoAllocLayout *s = scratch_address();
    if (!s) return SPMV_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return SPMV_ERR_CUDA;
    if (cudaMemcpy(flags, &s->error, sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess) return SPMV_ERR_CUDA;
    return SPMV_OK;
}
