// One-shot merge-path product that allocates no memory.
//
// Some callers cannot allocate device memory at the point where they need a
// product: for example a service that reserves the whole device for its own
// memory pool at start-up (a cudaMalloc then fails, or fragments the pool),
// or a latency-critical loop where a cudaMalloc would implicitly synchronise
// the device and stall the work already queued on other streams.  For them,
// spmv_execute_noalloc runs the merge-path product with its scratch (tile
// splits, cut-row partial sums, arrival counters) in a fixed-size array in
// the library's own device memory, declared below.  The array is part of the
// loaded module: every GPU that loads the library holds it until the process
// exits.  Every call shares it, so calls that overlap on the GPU (on two
// streams, or two host threads) race and give wrong results.
#include <cstring>

#include "internal.cuh"

namespace lbcsr {
namespace {

// Tiles of 1,024 units (32 items per lane), up to this many of them:
// m + nnz <= 262,144 * 1,024 = 268,435,456 rows plus nonzeros.
constexpr int kNoAllocItemsPerLane = 32;
constexpr int64_t kNoAllocMaxTiles = 262144;

struct NoAllocLayout {
    int2 part[kNoAllocMaxTiles + 1];
    double tail[kNoAllocMaxTiles];
    double head[kNoAllocMaxTiles];
    int32_t arrivals[kNoAllocMaxTiles];
};

// Scratch of spmv_execute_noalloc (about 7.3 MB).  Host code must not pass
// this name to a kernel: on the host it is only a stand-in for the symbol.
// The device address comes from cudaGetSymbolAddress, once per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[sizeof(NoAllocLayout)];

constexpr int kMaxDevices = 64;
void *g_scratch_addr[kMaxDevices] = {};

}  // namespace
}  // namespace lbcsr

using namespace lbcsr;

extern "C" spmv_status_t spmv_execute_noalloc(int32_t m, int32_t n, int32_t nnz, const int32_t *row_ptr,
                                              const int32_t *col_idx, const void *vals, spmv_dtype_t dtype,
                                              double alpha, const void *x, double beta, void *y,
                                              spmv_stream_t stream_handle) {
    if (m < 0 || n < 0 || nnz < 0) return SPMV_ERR_INVALID_ARG;
    if ((int64_t)m + (int64_t)nnz >= (1LL << 31)) return SPMV_ERR_INVALID_ARG;
    if (dtype != SPMV_F32 && dtype != SPMV_F64) return SPMV_ERR_INVALID_ARG;
    if (m == 0) return SPMV_OK;
    if (!row_ptr || !y) return SPMV_ERR_INVALID_ARG;
    if (nnz > 0 && (!col_idx || !vals || !x)) return SPMV_ERR_INVALID_ARG;

    const int ipt = kNoAllocItemsPerLane;
    const int64_t T = (int64_t)merge_path_threads() * ipt;
    const int64_t P = ((int64_t)m + nnz + T - 1) / T;
    if (P > kNoAllocMaxTiles) return SPMV_ERR_INVALID_ARG;  // beyond the fixed scratch

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SPMV_ERR_CUDA;
    if (!g_scratch_addr[dev]) {
        // first call on this device: look up the array's device address
        void *addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || !addr) return SPMV_ERR_CUDA;
        g_scratch_addr[dev] = addr;
    }
    NoAllocLayout *s = static_cast<NoAllocLayout *>(g_scratch_addr[dev]);
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_handle);

    // arrival counters must start at zero (the kernel leaves them at zero,
    // but a call that was interrupted may not have)
    if (cudaMemsetAsync(s->arrivals, 0, sizeof(int32_t) * (size_t)P, stream) != cudaSuccess) return SPMV_ERR_CUDA;
    if (launch_merge_path_partition(m, nnz, row_ptr, T, P, s->part, stream) != cudaSuccess) return SPMV_ERR_CUDA;
    MergePathArgs a;
    a.m = m;
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
    if (launch_merge_path_spmv(dtype, ipt, a, stream) != cudaSuccess) return SPMV_ERR_CUDA;
    return SPMV_OK;
}
