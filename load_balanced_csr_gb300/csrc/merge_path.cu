// Merge-path CSR SpMV on warp-sized tiles, with a fused carry-out fix-up.
//
// Schedule: "A GPU load-balancing programming model" (Osama, Porumbescu,
// Owens), section 5.2.1 -- every row end and every nonzero is one unit of
// work, the m + nnz units are split into equal tiles of T units, and each
// worker finds where its share starts by a search over (row ends, nonzero
// indices).  The plan computes the tile splits once (plan_kernels.cu).
//
// Here a tile belongs to one warp (T = 32 * IPL units) and the warps of a
// CTA never wait for each other, so a stalled warp never holds up its
// neighbours.  For each tile the warp:
//
//  1. copies the tile's col_idx, vals and row ends row_ptr[i0+1 .. i1] into
//     its own shared-memory region with 16-byte cp.async copies;
//  2. marks in a bitmap, for every row that has a nonzero in the tile, the
//     position of its last one;
//  3. splits the tile's nonzeros over the 32 lanes in runs of Q = the odd
//     number nearest above nnz/32 (odd, so the lanes' shared-memory reads
//     hit distinct banks); each lane first gathers x for its whole run into
//     registers through the read-only path, so all of its gathers are in
//     flight at once;
//  4. then adds its run up in order (one fused multiply-add per nonzero)
//     and, where the bitmap marks a row's last nonzero, closes the row and
//     keeps its sum in that nonzero's slot (no other lane reads it).  Row
//     ends cost no floating-point work, so every lane of every warp-wide FMA
//     does useful work -- this matters on GB300, whose fp64 unit runs 2 lanes
//     per clock per SM and charges a warp instruction the same for 1 or 32
//     lanes;
//  5. a segmented warp scan adds the sum carried into each lane's first
//     closed row (it stops once every open segment has reached its start);
//  6. writes the rows that start and end in the tile to y, coalesced.  A
//     row with no nonzero in the tile contributes 0.
//
// Rows cut by a tile boundary ("partial tiles" in the section) are finished
// without a second kernel and without any waiting: each tile holding part of
// such a row stores its partial sum, then counts itself in on the row's
// arrival counter; the tile that arrives last (the counter says how many to
// expect: the tiles from the one holding the row's first nonzero to the one
// holding its end) adds the partials in tile order with a tree and writes y.
// The order of the sum does not depend on which tile arrives last, so
// results are deterministic.  (The CUB implementation the paper compares
// with runs a separate fix-up step for these rows.)
#include <climits>

#include "internal.cuh"

namespace lbcsr {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

template <typename V>
struct MPParams {
    int32_t m;
    int32_t nnz;
    const int32_t *row_ptr;
    const int32_t *col_idx;
    const V *vals;
    const V *x;
    V *y;
    V alpha;
    V beta;
    int mode;  // bit0: alpha != 1, bit1: beta != 0
    const int2 *part;
    long long num_tiles;
    V *tail_partial;
    V *head_partial;
    int32_t *arrivals;
};

// Per-warp shared memory for a tile with n nonzeros and r row ends
// (n + r <= T), laid out as
//   col[ns] | val[ns] | row_end[r] | bitmap[(n + 31) / 32 + 2]
// with ns = (sh + n + 4) & ~3 <= n + 7 slots.  The size grows with n, so
// it is largest for n = T, r = 0:
template <typename V, int IPL>
__host__ __device__ constexpr int warp_region_bytes() {
    constexpr int T = 32 * IPL;
    constexpr int per_nnz = sizeof(int) + sizeof(V);
    return ((per_nnz * (T + 8) + 4 * (T / 32 + 8)) + 15) & ~15;
}

// ---------------------------------------------------------------- cp.async
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_small(uint32_t dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], %2;" ::"r"(dst), "l"(src), "n"(N) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Copy elements [b, e) of a global array into shared memory (element b at
// dst), b a multiple of 4.  VEC: 16-byte chunks (the array is 16-byte
// aligned) and element-sized copies for the last partial chunk only.
template <typename E, bool VEC>
__device__ __forceinline__ void warp_copy(E *dst, const E *src, int b, int e, int lane) {
    const int n = e - b;
    if (n <= 0) return;
    const uint32_t d = smem_addr(dst);
    if (VEC) {
        constexpr int EPC = 16 / sizeof(E);
        const int nfull = n / EPC;
        for (int c = lane; c < nfull; c += 32) cp_async16(d + 16u * c, src + b + c * EPC);
        const int done = nfull * EPC;
        if (lane < n - done) cp_async_small<sizeof(E)>(d + sizeof(E) * (done + lane), src + b + done + lane);
    } else {
        for (int q = lane; q < n; q += 32) cp_async_small<sizeof(E)>(d + sizeof(E) * q, src + b + q);
    }
}

template <typename V>
__device__ __forceinline__ V finish_row(V s, V alpha, V beta, int mode, const V *y, int row) {
    switch (mode) {
    case 0: return s;
    case 1: return alpha * s;
    case 2: return fma(beta, y[row], s);
    default: return fma(beta, y[row], alpha * s);
    }
}

// Cut rows: store this tile's partial, count in; the last to arrive adds all
// partials (tiles first..last-1 as tails, tile last as head) and writes y.
// Called by the whole warp; `lane_with_value` holds the partial.
template <typename V>
__device__ void cut_row(const MPParams<V> &p, int lane, int lane_with_value, V partial, bool as_head, long long me,
                        int row, long long first, long long last) {
    int finisher = 0;
    if (lane == lane_with_value) {
        if (as_head) p.head_partial[me] = partial;
        else p.tail_partial[me] = partial;
        __threadfence();
        const int before = atomicAdd(p.arrivals + last, 1);
        finisher = before == (int)(last - first);
        if (finisher) __threadfence();
    }
    if (!__shfl_sync(0xffffffffu, finisher, lane_with_value)) return;
    V s = V(0);
    for (long long t = first + lane; t < last; t += 32) s += __ldcg(p.tail_partial + t);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0) {
        s += __ldcg(p.head_partial + last);
        p.y[row] = finish_row(s, p.alpha, p.beta, p.mode, p.y, row);
        p.arrivals[last] = 0;  // ready for the next product
    }
}

template <typename V, int IPL, bool VEC>
__global__ void __launch_bounds__(kThreads)
merge_path_spmv_kernel(const MPParams<V> p) {
    constexpr bool F64 = sizeof(V) == 8;
    constexpr int T = 32 * IPL;
    extern __shared__ __align__(16) unsigned char dsm[];

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const long long tile = (long long)blockIdx.x * kWarps + warp;
    if (tile >= p.num_tiles) return;  // warps never wait for each other

    const int2 c0 = p.part[tile];
    const int2 c1 = p.part[tile + 1];
    const int i0 = c0.x, j0 = c0.y, i1 = c1.x, j1 = c1.y;
    const int nrows = i1 - i0;
    const int nnzt = j1 - j0;
    const int base = j0 & ~3;  // staged nonzero g sits at index g - base
    const int sh = j0 - base;  // tile nonzero k sits at index k + sh
    const int ns = (sh + nnzt + 4) & ~3;

    unsigned char *region = dsm + warp * warp_region_bytes<V, IPL>();
    int *s_col = reinterpret_cast<int *>(region);
    V *s_val = reinterpret_cast<V *>(s_col + ns);
    int *s_re = reinterpret_cast<int *>(s_val + ns);  // absolute row ends
    unsigned *s_bm = reinterpret_cast<unsigned *>(s_re + nrows);
    const int nwords = (nnzt + 31) >> 5;

    // ---- 1. stage
    warp_copy<int, VEC>(s_col, p.col_idx, base, j1, lane);
    warp_copy<V, VEC>(s_val, p.vals, base, j1, lane);
    for (int w = lane; w < nwords + 2; w += 32) s_bm[w] = 0u;  // two spare words
    for (int r = lane; r < nrows; r += 32) s_re[r] = ld_stream(p.row_ptr + i0 + 1 + r);
    cp_async_wait_all();
    __syncwarp();

    // ---- 2. mark each row's last nonzero in the tile
    for (int r = lane; r < nrows; r += 32) {
        const int e = s_re[r] - j0;
        const int ep = r == 0 ? 0 : s_re[r - 1] - j0;
        if (e > ep) atomicOr(s_bm + ((e - 1) >> 5), 1u << ((e - 1) & 31));
    }

    __syncwarp();

    // ---- 3. this lane's run of nonzeros [k0, k0 + q) and its x values
    int Q = (nnzt + 31) >> 5;
    Q |= 1;  // odd stride: lanes read distinct banks
    const int k0 = min(lane * Q, nnzt);
    const int run = min(Q, nnzt - k0);
    V xr[IPL + 1];
#pragma unroll
    for (int i = 0; i <= IPL; ++i) xr[i] = i < run ? ld_gather(p.x + s_col[k0 + i + sh]) : V(0);
    // bits of this run: bit i set when nonzero k0 + i is a row's last one
    const unsigned long long two = ((unsigned long long)s_bm[(k0 >> 5) + 1] << 32) | s_bm[k0 >> 5];
    unsigned long long bits = two >> (k0 & 31);

    // ---- 4. add the run up, closing rows where the bitmap says
    V acc = V(0);
    V first_val = V(0);
    int first_pos = -1;
#pragma unroll
    for (int i = 0; i <= IPL; ++i) {
        if (i < run) {
            const int k = k0 + i;
            acc = fma(s_val[k + sh], xr[i], acc);
            if (bits & 1ull) {
                if (first_pos < 0) {
                    first_val = acc;
                    first_pos = k;
                } else {
                    s_val[k + sh] = acc;
                }
                acc = V(0);
            }
            bits >>= 1;
        }
    }

    // ---- 5. segmented inclusive scan of (row closed, running sum)
    V v = acc;
    int f = first_pos >= 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        if (!__any_sync(0xffffffffu, !f && lane >= off)) break;
        const V pv = __shfl_up_sync(0xffffffffu, v, off);
        const int pf = __shfl_up_sync(0xffffffffu, f, off);
        if (lane >= off && !f) {
            v = pv + v;
            f = pf;
        }
    }
    V carry_in = __shfl_up_sync(0xffffffffu, v, 1);
    if (lane == 0) carry_in = V(0);
    if (first_pos >= 0) s_val[first_pos + sh] = carry_in + first_val;
    __syncwarp();

    // ---- 6. rows that start and end in this tile
    const int32_t rp_i0 = p.row_ptr[i0];
    const bool head_cut = nrows > 0 && rp_i0 < j0;
    V head_val = V(0);
    for (int q = lane; q < nrows; q += 32) {
        const int e = s_re[q] - j0;
        const int ep = q == 0 ? 0 : s_re[q - 1] - j0;
        const V s = e > ep ? s_val[e - 1 + sh] : V(0);
        if (q == 0 && head_cut) {
            head_val = s;
        } else {
            const int row = i0 + q;
            p.y[row] = finish_row(s, p.alpha, p.beta, p.mode, p.y, row);
        }
    }
    if (head_cut)
        cut_row<V>(p, lane, 0, head_val, true, tile, i0, ((long long)rp_i0 + i0) / T, tile);

    // ---- the row open at the tile's end
    if (i1 < p.m) {
        const int32_t rp_i1 = nrows > 0 ? s_re[nrows - 1] : rp_i0;
        if (j1 > max(rp_i1, j0)) {  // it has nonzeros in this tile
            const long long first = ((long long)rp_i1 + i1) / T;
            const long long last = ((long long)p.row_ptr[i1 + 1] + i1) / T;
            cut_row<V>(p, lane, 31, v, false, tile, i1, first, last);
        }
    }
}

template <typename V, int IPL, bool VEC>
cudaError_t launch_typed(const MergePathArgs &a, cudaStream_t stream) {
    if (a.num_tiles <= 0) return cudaSuccess;
    constexpr size_t smem = (size_t)kWarps * warp_region_bytes<V, IPL>();
    static unsigned long long configured = 0;  // one bit per device
    int dev = 0;
    cudaGetDevice(&dev);
    if (!((configured >> (dev & 63)) & 1ull)) {
        cudaError_t e = cudaFuncSetAttribute(merge_path_spmv_kernel<V, IPL, VEC>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        configured |= 1ull << (dev & 63);
    }
    MPParams<V> p;
    p.m = a.m;
    p.nnz = a.nnz;
    p.row_ptr = a.row_ptr;
    p.col_idx = a.col_idx;
    p.vals = static_cast<const V *>(a.vals);
    p.x = static_cast<const V *>(a.x);
    p.y = static_cast<V *>(a.y);
    p.alpha = static_cast<V>(a.alpha);
    p.beta = static_cast<V>(a.beta);
    p.mode = (p.alpha != V(1) ? 1 : 0) | (p.beta != V(0) ? 2 : 0);
    p.part = a.part;
    p.num_tiles = a.num_tiles;
    p.tail_partial = static_cast<V *>(a.tail_partial);
    p.head_partial = static_cast<V *>(a.head_partial);
    p.arrivals = a.arrivals;
    const long long grid = (a.num_tiles + kWarps - 1) / kWarps;
    merge_path_spmv_kernel<V, IPL, VEC><<<(unsigned)grid, kThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

template <typename V, bool VEC>
cudaError_t launch_ipl(int ipl, const MergePathArgs &a, cudaStream_t stream) {
    switch (ipl) {
    case 8: return launch_typed<V, 8, VEC>(a, stream);
    case 12: return launch_typed<V, 12, VEC>(a, stream);
    case 16: return launch_typed<V, 16, VEC>(a, stream);
    case 24: return launch_typed<V, 24, VEC>(a, stream);
    case 32: return launch_typed<V, 32, VEC>(a, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

bool merge_path_supported(int ipl) { return ipl == 8 || ipl == 12 || ipl == 16 || ipl == 24 || ipl == 32; }

int merge_path_threads() { return 32; }

int merge_path_default_items(spmv_dtype_t dtype) { return dtype == SPMV_F64 ? 8 : 16; }

cudaError_t launch_merge_path_spmv(spmv_dtype_t dtype, int ipl, const MergePathArgs &a, cudaStream_t stream) {
    // 16-byte copies need col_idx and vals 16-byte aligned
    const bool vec = (reinterpret_cast<uintptr_t>(a.col_idx) % 16 == 0) &&
                     (reinterpret_cast<uintptr_t>(a.vals) % 16 == 0);
    if (dtype == SPMV_F64)
        return vec ? launch_ipl<double, true>(ipl, a, stream) : launch_ipl<double, false>(ipl, a, stream);
    return vec ? launch_ipl<float, true>(ipl, a, stream) : launch_ipl<float, false>(ipl, a, stream);
}

}  // namespace lbcsr
