// Merge-path CSR SpMV with a fused carry-out fix-up.
//
// Schedule: "A GPU load-balancing programming model" (Osama, Porumbescu,
// Owens), section 5.2.1 -- every row end and every nonzero is one unit of
// work, the m + nnz units are split into equal tiles of T units, and each
// worker finds where its share starts by a search over (row ends, nonzero
// indices).  The plan computes the tile splits once (plan_kernels.cu); each
// CTA takes one tile:
//
//  1. stage the tile in shared memory: the row ends row_ptr[i0+1 .. i1]
//     (relative to the tile's first nonzero j0, with a sentinel), and for the
//     nonzeros j in [j0, j1) either the products vals[j]*x[col[j]] (fp32) or
//     the values and the gathered x[col[j]] (fp64).  col_idx and vals are
//     read with 16-byte loads, all issued before the x gathers;
//  2. the tile's nonzeros are split evenly over the threads (a thread's share
//     differs from another's by at most one), and each thread walks its
//     share: a nonzero adds to the running sum; after it, every row that
//     ends there is closed.  Row ends cost no floating-point work, so every
//     lane of every warp-wide add or FMA does useful work.  This matters on
//     GB300: its fp64 unit runs 2 lanes per clock per SM and a warp
//     instruction costs it the same whether 1 or 32 lanes are active;
//  3. a segmented scan over the threads adds the sum carried into each
//     thread's first closed row (it stops as soon as every open segment has
//     reached its start, so short rows cost one step);
//  4. a closed row's sum is kept in the slot of its last nonzero, which no
//     other thread reads; rows are then written to y once, coalesced.
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
    V *tail_partial;
    V *head_partial;
    int32_t *arrivals;
};

// Shared memory of one tile (n = nonzeros, r = row ends, n + r <= T):
//   fp32: prod[n + 4] | row_end[r + 1]
//   fp64: val[n + 4] | xg[n + 4] | row_end[r + 1]
// With sh <= 3 and n + r <= T this stays below the bound used here.
template <typename V, int IPT>
constexpr size_t tile_smem_bytes() {
    constexpr int T = kThreads * IPT;
    return (sizeof(V) == 8 ? 16 : 4) * (size_t)(T + 8) + 64;
}

// First row in [lo, hi) whose end is after position k (s_re ascends; the
// sentinel s_re[hi] is larger than any position).
__device__ __forceinline__ int rows_ending_by(const int *s_re, int lo, int hi, int k) {
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (s_re[mid] <= k) lo = mid + 1;
        else hi = mid;
    }
    return lo;
}

template <typename V>
struct TileSmem {
    V warp_sum[kWarps];
    int warp_flag[kWarps];
    V warp_prefix[kWarps];
    V red[kWarps];
    long long run_first[2];
    long long run_last[2];
    int run_row[2];
    int run_finish[2];
};

template <typename V>
__device__ __forceinline__ V finish_row(V s, V alpha, V beta, int mode, const V *y, int row) {
    switch (mode) {
    case 0: return s;
    case 1: return alpha * s;
    case 2: return fma(beta, y[row], s);
    default: return fma(beta, y[row], alpha * s);
    }
}

// Sum of the partials of one cut row, by the tile that arrived last.
template <typename V>
__device__ void finish_cut_row(V *red, int32_t row, long long first_tile, long long last_tile,
                               const MPParams<V> &p) {
    const int tid = threadIdx.x;
    V s = V(0);
    for (long long t = first_tile + tid; t < last_tile; t += kThreads) s += __ldcg(p.tail_partial + t);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if ((tid & 31) == 0) red[tid >> 5] = s;
    __syncthreads();
    if (tid == 0) {
        V total = red[0];
#pragma unroll
        for (int w = 1; w < kWarps; ++w) total += red[w];
        total += __ldcg(p.head_partial + last_tile);
        p.y[row] = finish_row(total, p.alpha, p.beta, p.mode, p.y, row);
        p.arrivals[last_tile] = 0;  // ready for the next product
    }
    __syncthreads();
}

template <typename V, int IPT, bool VEC>
__global__ void __launch_bounds__(kThreads)
merge_path_spmv_kernel(const MPParams<V> p) {
    constexpr bool F64 = sizeof(V) == 8;
    constexpr int T = kThreads * IPT;
    extern __shared__ __align__(16) unsigned char dsm[];
    __shared__ TileSmem<V> sm;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const long long tile = blockIdx.x;

    const int2 c0 = p.part[tile];
    const int2 c1 = p.part[tile + 1];
    const int i0 = c0.x, j0 = c0.y, i1 = c1.x, j1 = c1.y;
    const int nrows = i1 - i0;
    const int nnzt = j1 - j0;
    const int base = VEC ? (j0 & ~3) : j0;  // staged nonzero g sits at index g - base
    const int sh = j0 - base;               // tile nonzero k sits at index k + sh
    const int nslots = (sh + nnzt + 4) & ~3;
    V *s_a = reinterpret_cast<V *>(dsm);                  // fp32 products / fp64 values
    V *s_b = F64 ? s_a + nslots : s_a;                    // fp64 gathered x
    int *s_re = reinterpret_cast<int *>(F64 ? s_b + nslots : s_a + nslots);

    // ---- 1. stage
    for (int r = tid; r < nrows; r += kThreads) s_re[r] = ld_stream(p.row_ptr + i0 + 1 + r) - j0;
    if (tid == 0) s_re[nrows] = INT_MAX;
    if (VEC) {
        constexpr int CH = ((T + 6) / 4 + kThreads - 1) / kThreads;
        const int nch = (j1 - base + 3) >> 2;
        int4 cc[CH];
        V vv[CH][4];
#pragma unroll
        for (int u = 0; u < CH; ++u) {
            const int c = tid + u * kThreads;
            const int g = base + 4 * c;
            if (c < nch && g + 4 <= p.nnz) {
                cc[u] = ld_stream(reinterpret_cast<const int4 *>(p.col_idx + g));
                if constexpr (F64) {
                    const double2 v01 = ld_stream(reinterpret_cast<const double2 *>(p.vals + g));
                    const double2 v23 = ld_stream(reinterpret_cast<const double2 *>(p.vals + g) + 1);
                    vv[u][0] = v01.x; vv[u][1] = v01.y; vv[u][2] = v23.x; vv[u][3] = v23.y;
                } else {
                    const float4 v = ld_stream(reinterpret_cast<const float4 *>(p.vals + g));
                    vv[u][0] = v.x; vv[u][1] = v.y; vv[u][2] = v.z; vv[u][3] = v.w;
                }
            } else if (c < nch) {  // the array's last, partial chunk
                int ci[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const bool ok = g + e < j1;
                    ci[e] = ok ? ld_stream(p.col_idx + g + e) : 0;
                    vv[u][e] = ok ? ld_stream(p.vals + g + e) : V(0);
                }
                cc[u] = make_int4(ci[0], ci[1], ci[2], ci[3]);
            }
        }
#pragma unroll
        for (int u = 0; u < CH; ++u) {
            const int c = tid + u * kThreads;
            if (c < nch) {
                const int g = base + 4 * c;
                const int ci[4] = {cc[u].x, cc[u].y, cc[u].z, cc[u].w};
                V xv[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) xv[e] = (g + e >= j0 && g + e < j1) ? ld_gather(p.x + ci[e]) : V(0);
                if constexpr (F64) {
                    reinterpret_cast<double2 *>(s_a)[2 * c] = make_double2(vv[u][0], vv[u][1]);
                    reinterpret_cast<double2 *>(s_a)[2 * c + 1] = make_double2(vv[u][2], vv[u][3]);
                    reinterpret_cast<double2 *>(s_b)[2 * c] = make_double2(xv[0], xv[1]);
                    reinterpret_cast<double2 *>(s_b)[2 * c + 1] = make_double2(xv[2], xv[3]);
                } else {
                    reinterpret_cast<float4 *>(s_a)[c] =
                        make_float4(vv[u][0] * xv[0], vv[u][1] * xv[1], vv[u][2] * xv[2], vv[u][3] * xv[3]);
                }
            }
        }
    } else {
        for (int k = tid; k < nnzt; k += kThreads) {
            const V xv = ld_gather(p.x + ld_stream(p.col_idx + j0 + k));
            const V v = ld_stream(p.vals + j0 + k);
            if constexpr (F64) {
                s_a[k] = v;
                s_b[k] = xv;
            } else {
                s_a[k] = v * xv;
            }
        }
    }
    __syncthreads();

    // ---- 2. this thread's nonzeros [k0, k1) and the first row it meets
    const int k0 = (tid * nnzt) >> 8;
    const int k1 = ((tid + 1) * nnzt) >> 8;
    // Rows ending at or before k0 were closed by earlier threads; thread 0
    // closes the rows that end before the tile's first nonzero (the first of
    // them takes the carry into the tile, which is zero here).
    int r = rows_ending_by(s_re, 0, nrows, k0);
    int re = s_re[r];
    V acc = V(0);
    V first_val = V(0);
    int first_pos = INT_MIN;  // slot of the first closed row's last nonzero
    bool ended = tid == 0 && r > 0;
    if (ended) first_pos = -1;
    for (int k = k0; k < k1; ++k) {
        if constexpr (F64) acc = fma(s_a[k + sh], s_b[k + sh], acc);
        else acc += s_a[k + sh];
        if (re == k + 1) {  // row r ends after nonzero k; empty rows may follow it
            if (!ended) {
                ended = true;
                first_val = acc;
                first_pos = k;
            } else {
                s_a[k + sh] = acc;  // only this thread touches slot k
            }
            acc = V(0);
            ++r;
            re = s_re[r];
            if (re == k + 1) {  // skip the empty rows in one search
                r = rows_ending_by(s_re, r, nrows, k + 1);
                re = s_re[r];
            }
        }
    }

    // ---- 3. segmented inclusive scan of (row closed, running sum)
    V v = acc;
    int f = ended;
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
    if (lane == 31) {
        sm.warp_sum[warp] = v;
        sm.warp_flag[warp] = f;
    }
    __syncthreads();
    if (warp == 0) {  // segmented exclusive scan over the warps' totals
        V ws = lane < kWarps ? sm.warp_sum[lane] : V(0);
        int wf = lane < kWarps ? sm.warp_flag[lane] : 1;
#pragma unroll
        for (int off = 1; off < kWarps; off <<= 1) {
            if (!__any_sync(0xffffffffu, !wf && lane >= off && lane < kWarps)) break;
            const V pv = __shfl_up_sync(0xffffffffu, ws, off);
            const int pf = __shfl_up_sync(0xffffffffu, wf, off);
            if (lane >= off && !wf) {
                ws = pv + ws;
                wf = pf;
            }
        }
        const V ex = __shfl_up_sync(0xffffffffu, ws, 1);
        if (lane < kWarps) sm.warp_prefix[lane] = lane == 0 ? V(0) : ex;
    }
    __syncthreads();
    const V wprefix = sm.warp_prefix[warp];
    V incl = v;
    if (warp > 0 && __any_sync(0xffffffffu, !f)) {
        if (!f) incl = wprefix + v;
    }
    V carry_in = __shfl_up_sync(0xffffffffu, incl, 1);
    if (lane == 0) carry_in = wprefix;
    if (first_pos >= 0) s_a[first_pos + sh] = carry_in + first_val;
    __syncthreads();

    // ---- 4. rows that start and end in this tile: the sum sits in the slot
    // of the row's last nonzero in the tile (no nonzero here: the sum is 0)
    const int32_t rp_i0 = p.row_ptr[i0];
    const bool head_cut = nrows > 0 && rp_i0 < j0;
    for (int q = tid; q < nrows; q += kThreads) {
        const int e = s_re[q];
        const int ep = q == 0 ? 0 : s_re[q - 1];
        const V s = e > ep ? s_a[e - 1 + sh] : V(0);
        if (q == 0 && head_cut) {
            sm.run_finish[0] = 0;
            const long long first = ((long long)rp_i0 + i0) / T;
            p.head_partial[tile] = s;
            __threadfence();
            const int before = atomicAdd(p.arrivals + tile, 1);
            if (before == (int)(tile - first)) {
                __threadfence();
                sm.run_finish[0] = 1;
                sm.run_row[0] = i0;
                sm.run_first[0] = first;
                sm.run_last[0] = tile;
            }
        } else {
            const int row = i0 + q;
            p.y[row] = finish_row(s, p.alpha, p.beta, p.mode, p.y, row);
        }
    }
    if (tid == 0 && !head_cut) sm.run_finish[0] = 0;

    // ---- the row open at the tile's end
    if (tid == kThreads - 1) {
        sm.run_finish[1] = 0;
        if (i1 < p.m) {
            const int32_t rp_i1 = nrows > 0 ? s_re[nrows - 1] + j0 : rp_i0;
            if (j1 > max(rp_i1, j0)) {  // the open row has nonzeros in this tile
                const long long first = ((long long)rp_i1 + i1) / T;
                const long long last = ((long long)p.row_ptr[i1 + 1] + i1) / T;
                p.tail_partial[tile] = incl;
                __threadfence();
                const int before = atomicAdd(p.arrivals + last, 1);
                if (before == (int)(last - first)) {
                    __threadfence();
                    sm.run_finish[1] = 1;
                    sm.run_row[1] = i1;
                    sm.run_first[1] = first;
                    sm.run_last[1] = last;
                }
            }
        }
    }
    __syncthreads();
    if (sm.run_finish[0]) finish_cut_row<V>(sm.red, sm.run_row[0], sm.run_first[0], sm.run_last[0], p);
    if (sm.run_finish[1]) finish_cut_row<V>(sm.red, sm.run_row[1], sm.run_first[1], sm.run_last[1], p);
}

template <typename V, int IPT, bool VEC>
cudaError_t launch_typed(const MergePathArgs &a, cudaStream_t stream) {
    if (a.num_tiles <= 0) return cudaSuccess;
    constexpr size_t smem = tile_smem_bytes<V, IPT>();
    static unsigned long long configured = 0;  // one bit per device
    int dev = 0;
    cudaGetDevice(&dev);
    if (!((configured >> (dev & 63)) & 1ull)) {
        cudaError_t e = cudaFuncSetAttribute(merge_path_spmv_kernel<V, IPT, VEC>,
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
    p.tail_partial = static_cast<V *>(a.tail_partial);
    p.head_partial = static_cast<V *>(a.head_partial);
    p.arrivals = a.arrivals;
    merge_path_spmv_kernel<V, IPT, VEC><<<(unsigned)a.num_tiles, kThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

template <typename V, bool VEC>
cudaError_t launch_ipt(int ipt, const MergePathArgs &a, cudaStream_t stream) {
    switch (ipt) {
    case 5: return launch_typed<V, 5, VEC>(a, stream);
    case 7: return launch_typed<V, 7, VEC>(a, stream);
    case 9: return launch_typed<V, 9, VEC>(a, stream);
    case 11: return launch_typed<V, 11, VEC>(a, stream);
    case 13: return launch_typed<V, 13, VEC>(a, stream);
    case 15: return launch_typed<V, 15, VEC>(a, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

bool merge_path_supported(int ipt) {
    return ipt == 5 || ipt == 7 || ipt == 9 || ipt == 11 || ipt == 13 || ipt == 15;
}

int merge_path_threads() { return kThreads; }

cudaError_t launch_merge_path_spmv(spmv_dtype_t dtype, int ipt, const MergePathArgs &a, cudaStream_t stream) {
    // 16-byte staging needs col_idx and vals 16-byte aligned
    const bool vec = (reinterpret_cast<uintptr_t>(a.col_idx) % 16 == 0) &&
                     (reinterpret_cast<uintptr_t>(a.vals) % 16 == 0);
    if (dtype == SPMV_F64)
        return vec ? launch_ipt<double, true>(ipt, a, stream) : launch_ipt<double, false>(ipt, a, stream);
    return vec ? launch_ipt<float, true>(ipt, a, stream) : launch_ipt<float, false>(ipt, a, stream);
}

}  // namespace lbcsr
