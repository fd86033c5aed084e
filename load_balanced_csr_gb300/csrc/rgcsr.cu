// Row-grouped CSR SpMV ("New Row-grouped CSR format for storing the sparse
// matrices on GPU with implementation in CUDA", section 3): one thread per
// row over the plan's interleaved copy of A, in which the k-th nonzeros of a
// group's G rows are adjacent.
//
// The page's kernel reads the copy straight from global memory, a warp at a
// time (section 3, coalescing with G >= 32).  Here every group's slots are
// one contiguous, aligned block of the copy, so a CTA of G threads has the
// Tensor Memory Accelerator bring it into shared memory in chunks of
// `levels` rows of slots (one bulk copy each for columns and values, the
// next chunk in flight while the current one is used), and the threads read
// their slots there.  The copy's padding is loaded with the rest of the
// block but never used: each thread stops at its own row length.  Since a
// warp's threads hold neighbouring rows, their x gathers at one level touch
// neighbouring columns whenever the matrix is banded.
//
// With G = 32 (the default: it pads least) a group is exactly one warp's
// rows -- in the natural order or, for the window-sorted copy, the rows the
// plan lists at the group's 32 positions -- so warps work independently, as in the merge-path kernel: each warp
// owns a contiguous run of groups and its own two-stage copy pipeline, and
// never waits for another warp.  Larger groups take a CTA of G threads per
// group, which must meet at a barrier before each stage is refilled; CTAs
// are persistent and take groups b, b + grid, ... in order.
//
// Each thread keeps U partial sums (level k goes to sum k mod U) and adds
// them as a tree, so the rounding error grows with length / U.
#include <atomic>

#include "internal.cuh"
#include "tma.cuh"

namespace lbcsr {

namespace {

using namespace tma;

constexpr int kRgStages = 2;
constexpr int kRgStageTarget = 16384;  // bytes of slots per stage (at most)

template <typename V>
struct RgParams {
    int32_t m;
    int32_t n;  // columns (the debug build checks the gathers against it)
    int g_log2;
    long long ngroups;
    const int64_t *gp;
    const int32_t *row_len;
    const int32_t *perm;  // row at each position (null: the natural order; G = 32 only)
    const int32_t *rg_col;
    const V *rg_val;
    const V *x;
    V *y;
    V alpha;
    V beta;
    int levels;       // slot rows per chunk, a multiple of U
    int32_t *error;   // bit 0 set if a copy never completed
    long long num_warps;  // warp kernel: warps with a run of groups
};

template <typename V>
__host__ __device__ constexpr int rg_unroll() {
    return sizeof(V) == 8 ? 4 : 8;
}

// levels per chunk for group size G: as many as fit the stage target, a
// multiple of U, at least U
template <typename V>
int rg_levels(int G) {
    constexpr int U = rg_unroll<V>();
    int l = kRgStageTarget / (G * (int)(sizeof(int) + sizeof(V)));
    l = l / U * U;
    return l < U ? U : l;
}

template <typename V>
__host__ __device__ inline size_t rg_stage_bytes(int G, int levels) {
    return (size_t)levels * G * (sizeof(int) + sizeof(V));
}

// Chunks of a group with L levels (an empty group still has one, to write y).
__device__ __forceinline__ int rg_chunks(long long L, int levels) {
    return L > 0 ? (int)((L + levels - 1) / levels) : 1;
}

template <typename V>
__device__ __forceinline__ void rg_issue(const RgParams<V> &p, unsigned char *stage, uint64_t *bar, long long g,
                                         int c, uint64_t pol) {
    const int G = 1 << p.g_log2;
    const long long base = p.gp[g];
    const long long L = (p.gp[g + 1] - base) >> p.g_log2;
    const long long lev0 = (long long)c * p.levels;
    const long long nlev = L - lev0 < p.levels ? L - lev0 : p.levels;
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (nlev <= 0) {
        mbar_expect_tx(bar, 0);
        return;
    }
    const uint32_t n = (uint32_t)(nlev * G);
    mbar_expect_tx(bar, n * (uint32_t)(sizeof(int) + sizeof(V)));
    const long long s0 = base + lev0 * G;
    bulk_copy(stage, p.rg_col + s0, n * (uint32_t)sizeof(int), bar, pol);
    bulk_copy(stage + (size_t)p.levels * G * sizeof(int), p.rg_val + s0, n * (uint32_t)sizeof(V), bar, pol);
}

template <typename V>
__global__ void __launch_bounds__(256)
rgcsr_tma_kernel(const RgParams<V> p) {
    constexpr int U = rg_unroll<V>();
    extern __shared__ __align__(128) unsigned char dsm[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(dsm);
    unsigned char *stages = dsm + 128;
    const int G = 1 << p.g_log2;
    const int t = threadIdx.x;
    const size_t sbytes = rg_stage_bytes<V>(G, p.levels);
    const long long gstride = gridDim.x;
    const uint64_t stream_pol = l2_policy_evict_first();
    const uint64_t x_pol = l2_policy_evict_last();

    if (t == 0) {
        for (int s = 0; s < kRgStages; ++s) mbar_init(bars + s);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    // issue cursor (thread 0): the item kRgStages ahead of the one in use
    long long ig = blockIdx.x;
    int ic = 0;
    if (t == 0) {
        for (int s = 0; s < kRgStages && ig < p.ngroups; ++s) {
            rg_issue(p, stages + s * sbytes, bars + s, ig, ic, stream_pol);
            const long long L = (p.gp[ig + 1] - p.gp[ig]) >> p.g_log2;
            if (++ic == rg_chunks(L, p.levels)) {
                ic = 0;
                ig += gstride;
            }
        }
    }

    V acc[U];
    int len = -1;
    long long it = 0;
    for (long long g = blockIdx.x; g < p.ngroups; g += gstride) {
        const long long L = (p.gp[g + 1] - p.gp[g]) >> p.g_log2;
        const int nch = rg_chunks(L, p.levels);
        const long long row = (g << p.g_log2) + t;
        len = row < p.m ? p.row_len[row] : -1;
#pragma unroll
        for (int u = 0; u < U; ++u) acc[u] = V(0);
        for (int c = 0; c < nch; ++c, ++it) {
            const int s = (int)(it % kRgStages);
            const uint32_t parity = (uint32_t)((it / kRgStages) & 1);
            const bool ok = __syncthreads_and(mbar_wait_bounded(bars + s, parity));
            if (!ok) {  // a copy never completed: report it and stop this CTA
                if (t == 0) {
                    if (p.error) atomicOr(p.error, 1);
                    // let the copies still in flight land before the CTA exits
                    for (long long j = it; j < it + kRgStages; ++j)
                        mbar_wait_bounded(bars + j % kRgStages, (uint32_t)((j / kRgStages) & 1));
                }
                return;
            }
            const unsigned char *stage = stages + s * sbytes;
            const int *scol = reinterpret_cast<const int *>(stage);
            const V *sval = reinterpret_cast<const V *>(stage + (size_t)p.levels * G * sizeof(int));
            const int lev0 = c * p.levels;
            const int mine = min(p.levels, len - lev0);  // this row's levels in the chunk
            int k = 0;
            for (; k + U <= mine; k += U) {
                V xv[U];
#pragma unroll
                for (int u = 0; u < U; ++u) xv[u] = gather_keep(p.x + debug_col(scol[(k + u) * G + t], p.n, p.error), x_pol);
#pragma unroll
                for (int u = 0; u < U; ++u) acc[u] = fma(sval[(k + u) * G + t], xv[u], acc[u]);
            }
#pragma unroll
            for (int u = 0; u < U - 1; ++u)
                if (k + u < mine) acc[u] = fma(sval[(k + u) * G + t], gather_keep(p.x + debug_col(scol[(k + u) * G + t], p.n, p.error), x_pol), acc[u]);
            __syncthreads();  // the stage is free
            if (t == 0 && ig < p.ngroups) {
                rg_issue(p, stages + s * sbytes, bars + s, ig, ic, stream_pol);
                const long long Li = (p.gp[ig + 1] - p.gp[ig]) >> p.g_log2;
                if (++ic == rg_chunks(Li, p.levels)) {
                    ic = 0;
                    ig += gstride;
                }
            }
        }
        if (len >= 0) {
#pragma unroll
            for (int w = 1; w < U; w <<= 1)
#pragma unroll
                for (int u = 0; u + w < U; u += 2 * w) acc[u] += acc[u + w];
            V r = p.alpha * acc[0];
            if (p.beta != V(0)) r = fma(p.beta, p.y[row], r);
            store_stream(p.y + row, r, stream_pol);
        }
    }
}

// ---------------------------------------------------------------- G = 32: one warp per group
constexpr int kWarpStages = 2;
constexpr int kWarpStageTarget = 4096;  // bytes of slots per stage (at most); 16 fp32 levels
constexpr int kWarpThreads = 256;

template <typename V>
int rg_warp_levels() {
    constexpr int U = rg_unroll<V>();
    int l = kWarpStageTarget / (32 * (int)(sizeof(int) + sizeof(V)));
    l = l / U * U;
    return l < U ? U : l;
}

// A warp's region: barriers (padded to 128 bytes), then its stages.
template <typename V>
size_t rg_warp_region(int levels) {
    return 128 + kWarpStages * rg_stage_bytes<V>(32, levels);
}

// Copy chunk c of the group whose slots are [b, e) into a stage.
template <typename V>
__device__ __forceinline__ void rg_issue_slots(const RgParams<V> &p, unsigned char *stage, uint64_t *bar,
                                               long long b, long long e, int c, uint64_t pol) {
    const int G = 1 << p.g_log2;
    const long long L = (e - b) >> p.g_log2;
    const long long lev0 = (long long)c * p.levels;
    const long long nlev = L - lev0 < p.levels ? L - lev0 : p.levels;
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (nlev <= 0) {
        mbar_expect_tx(bar, 0);
        return;
    }
    const uint32_t n = (uint32_t)(nlev * G);
    mbar_expect_tx(bar, n * (uint32_t)(sizeof(int) + sizeof(V)));
    const long long s0 = b + lev0 * G;
    bulk_copy(stage, p.rg_col + s0, n * (uint32_t)sizeof(int), bar, pol);
    bulk_copy(stage + (size_t)p.levels * G * sizeof(int), p.rg_val + s0, n * (uint32_t)sizeof(V), bar, pol);
}

// Everything a group needs besides its slots -- its slot range, and per lane
// the length, row and old y of the lane's position -- is loaded one group
// ahead, so that no dependent global load sits between two groups (groups
// of short rows hold only a few dozen nonzeros).
template <typename V>
__global__ void __launch_bounds__(kWarpThreads)
rgcsr_warp_kernel(const RgParams<V> p) {
    constexpr int U = rg_unroll<V>();
    extern __shared__ __align__(128) unsigned char dsm[];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const long long me = (long long)blockIdx.x * (kWarpThreads / 32) + warp;
    if (me >= p.num_warps) return;  // warps never wait for each other
    const long long ng = p.ngroups;
    const long long g_begin = me * ng / p.num_warps;
    const long long g_end = (me + 1) * ng / p.num_warps;
    const size_t sbytes = rg_stage_bytes<V>(32, p.levels);
    unsigned char *region = dsm + (size_t)warp * (128 + kWarpStages * sbytes);
    uint64_t *bars = reinterpret_cast<uint64_t *>(region);
    unsigned char *stages = region + 128;
    const uint64_t stream_pol = l2_policy_evict_first();
    const uint64_t x_pol = l2_policy_evict_last();
    const bool with_y = p.beta != V(0);
    if (lane == 0) {
        for (int s = 0; s < kWarpStages; ++s) mbar_init(bars + s);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();

    // issue cursor (lane 0): chunk ic of group ig, slots [ib, ie); the end of
    // group ig + 1 is already loaded
    long long ig = g_begin, ib = 0, ie = 0, ie_next = 0;
    int ic = 0;
    if (lane == 0) {
        ib = p.gp[ig];
        ie = p.gp[ig + 1];
        ie_next = ig + 2 <= ng ? p.gp[ig + 2] : ie;
        for (int s = 0; s < kWarpStages && ig < g_end; ++s) {
            rg_issue_slots(p, stages + s * sbytes, bars + s, ib, ie, ic, stream_pol);
            if (++ic == rg_chunks((ie - ib) >> 5, p.levels)) {
                ic = 0;
                ++ig;
                ib = ie;
                ie = ie_next;
                ie_next = ig + 2 <= ng ? p.gp[ig + 2] : ie;
            }
        }
    }

    // compute cursor: group g, slots [gb, ge), the next group's end ge_next
    long long gb = p.gp[g_begin], ge = p.gp[g_begin + 1];
    long long ge_next = g_begin + 2 <= ng ? p.gp[g_begin + 2] : ge;
    int len_n = -1;
    long long row_n = 0;
    V yo_n = V(0);
    {
        const long long q = g_begin * 32 + lane;
        if (q < p.m) {
            len_n = p.row_len[q];
            row_n = p.perm ? p.perm[q] : q;
            if (with_y && len_n >= 0) yo_n = p.y[row_n];
        }
    }
    long long it = 0;
    for (long long g = g_begin; g < g_end; ++g) {
        const int nch = rg_chunks((ge - gb) >> 5, p.levels);
        const int len = len_n;
        const long long row = row_n;  // the row at this lane's position
        const V yo = yo_n;
        long long ge_nn = ge_next;
        len_n = -1;
        if (g + 1 < g_end) {
            const long long q = (g + 1) * 32 + lane;
            if (q < p.m) {
                len_n = p.row_len[q];
                row_n = p.perm ? p.perm[q] : q;
                if (with_y && len_n >= 0) yo_n = p.y[row_n];
            }
            if (g + 3 <= ng) ge_nn = p.gp[g + 3];
        }
        V acc[U];
#pragma unroll
        for (int u = 0; u < U; ++u) acc[u] = V(0);
        for (int c = 0; c < nch; ++c, ++it) {
            const int s = (int)(it % kWarpStages);
            const uint32_t parity = (uint32_t)((it / kWarpStages) & 1);
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(bars + s, parity))) {
                // a copy never completed: report it and stop this warp
                if (lane == 0) {
                    if (p.error) atomicOr(p.error, 1);
                    for (long long j = it; j < it + kWarpStages; ++j)
                        mbar_wait_bounded(bars + j % kWarpStages, (uint32_t)((j / kWarpStages) & 1));
                }
                return;
            }
            const unsigned char *stage = stages + s * sbytes;
            const int *scol = reinterpret_cast<const int *>(stage);
            const V *sval = reinterpret_cast<const V *>(stage + (size_t)p.levels * 32 * sizeof(int));
            const int mine = min(p.levels, len - c * p.levels);
            int k = 0;
            for (; k + U <= mine; k += U) {
                V xv[U];
#pragma unroll
                for (int u = 0; u < U; ++u) xv[u] = gather_keep(p.x + debug_col(scol[(k + u) * 32 + lane], p.n, p.error), x_pol);
#pragma unroll
                for (int u = 0; u < U; ++u) acc[u] = fma(sval[(k + u) * 32 + lane], xv[u], acc[u]);
            }
#pragma unroll
            for (int u = 0; u < U - 1; ++u)
                if (k + u < mine)
                    acc[u] = fma(sval[(k + u) * 32 + lane], gather_keep(p.x + debug_col(scol[(k + u) * 32 + lane], p.n, p.error), x_pol), acc[u]);
            __syncwarp();  // the stage is free
            if (lane == 0 && ig < g_end) {
                rg_issue_slots(p, stages + s * sbytes, bars + s, ib, ie, ic, stream_pol);
                if (++ic == rg_chunks((ie - ib) >> 5, p.levels)) {
                    ic = 0;
                    ++ig;
                    ib = ie;
                    ie = ie_next;
                    ie_next = ig + 2 <= ng ? p.gp[ig + 2] : ie;
                }
            }
        }
        if (len >= 0) {
#pragma unroll
            for (int w = 1; w < U; w <<= 1)
#pragma unroll
                for (int u = 0; u + w < U; u += 2 * w) acc[u] += acc[u + w];
            V r = p.alpha * acc[0];
            if (with_y) r = fma(p.beta, yo, r);
            store_stream(p.y + row, r, stream_pol);
        }
        gb = ge;
        ge = ge_next;
        ge_next = ge_nn;
    }
}

// Per-device launch settings, 0 (false) until first computed.  Host threads
// may fill an entry at the same time: they compute the same value.
std::atomic<int> g_rg_warp_ctas_per_sm[2][64];  // occupancy of the warp kernel per (type, device)

template <typename V>
cudaError_t launch_rg_warp(RgParams<V> p, cudaStream_t stream) {
    p.levels = rg_warp_levels<V>();
    const size_t smem = (kWarpThreads / 32) * rg_warp_region<V>(p.levels);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::atomic<int> &cached = g_rg_warp_ctas_per_sm[sizeof(V) == 8][dev & 63];
    int per_sm = cached.load(std::memory_order_acquire);
    if (per_sm == 0) {
        e = cudaFuncSetAttribute(rgcsr_warp_kernel<V>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        int nb = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, rgcsr_warp_kernel<V>, kWarpThreads, smem);
        if (e != cudaSuccess) return e;
        per_sm = nb > 0 ? nb : 1;
        cached.store(per_sm, std::memory_order_release);
    }
    const long long max_warps = (long long)per_sm * device_sm_count() * (kWarpThreads / 32);
    p.num_warps = p.ngroups < max_warps ? p.ngroups : max_warps;
    const unsigned grid = (unsigned)((p.num_warps + kWarpThreads / 32 - 1) / (kWarpThreads / 32));
    rgcsr_warp_kernel<V><<<grid, kWarpThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- G > 32: one CTA per group
std::atomic<int> g_rg_ctas_per_sm[2][9][64];  // occupancy per (type, log2 G, device)
std::atomic<bool> g_rg_smem_set[2][64];         // kernel's shared-memory limit raised (per type, device)

template <typename V>
size_t rg_smem(int G) {
    return 128 + kRgStages * rg_stage_bytes<V>(G, rg_levels<V>(G));
}

template <typename V>
cudaError_t launch_rg(int32_t m, int32_t n, int g_log2, const int64_t *group_ptr, const int32_t *row_len, const int32_t *perm,
                      const int32_t *rg_col, const void *rg_val, const void *x, void *y, double alpha, double beta,
                      int32_t *error, cudaStream_t stream) {
    const int G = 1 << g_log2;
    if (perm && G != 32) return cudaErrorInvalidValue;
    RgParams<V> p;
    p.m = m;
    p.n = n;
    p.g_log2 = g_log2;
    p.ngroups = ((long long)m + G - 1) >> g_log2;
    p.gp = group_ptr;
    p.row_len = row_len;
    p.perm = perm;
    p.rg_col = rg_col;
    p.rg_val = static_cast<const V *>(rg_val);
    p.x = static_cast<const V *>(x);
    p.y = static_cast<V *>(y);
    p.alpha = (V)alpha;
    p.beta = (V)beta;
    p.levels = rg_levels<V>(G);
    p.error = error;
    p.num_warps = 0;
    if (G == 32) return launch_rg_warp<V>(p, stream);
    const size_t smem = rg_smem<V>(G);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (!g_rg_smem_set[sizeof(V) == 8][dev & 63].load(std::memory_order_acquire)) {
        // one limit for every group size: the largest they need
        size_t most = 0;
        for (int gl = 5; gl <= 8; ++gl) most = rg_smem<V>(1 << gl) > most ? rg_smem<V>(1 << gl) : most;
        e = cudaFuncSetAttribute(rgcsr_tma_kernel<V>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)most);
        if (e != cudaSuccess) return e;
        g_rg_smem_set[sizeof(V) == 8][dev & 63].store(true, std::memory_order_release);
    }
    std::atomic<int> &cached_g = g_rg_ctas_per_sm[sizeof(V) == 8][g_log2][dev & 63];
    int per_sm = cached_g.load(std::memory_order_acquire);
    if (per_sm == 0) {
        int nb = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, rgcsr_tma_kernel<V>, G, smem);
        if (e != cudaSuccess) return e;
        per_sm = nb > 0 ? nb : 1;
        cached_g.store(per_sm, std::memory_order_release);
    }
    const long long cap = (long long)per_sm * device_sm_count();
    const unsigned grid = (unsigned)(p.ngroups < cap ? p.ngroups : cap);
    rgcsr_tma_kernel<V><<<grid, G, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rgcsr_spmv(spmv_dtype_t dtype, int32_t m, int32_t n, int g_log2, const int64_t *group_ptr,
                              const int32_t *row_len, const int32_t *perm, const int32_t *rg_col,
                              const void *rg_val, const void *x, void *y, double alpha, double beta,
                              int32_t *error, cudaStream_t stream) {
    if (m <= 0) return cudaSuccess;
    if (dtype == SPMV_F64)
        return launch_rg<double>(m, n, g_log2, group_ptr, row_len, perm, rg_col, rg_val, x, y, alpha, beta, error,
                                 stream);
    return launch_rg<float>(m, n, g_log2, group_ptr, row_len, perm, rg_col, rg_val, x, y, alpha, beta, error, stream);
}

}  // namespace lbcsr
