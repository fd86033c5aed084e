// Merge-path CSR SpMV with a fused carry-out fix-up.
//
// Schedule: "A GPU load-balancing programming model" (Osama, Porumbescu,
// Owens), section 5.2.1 -- every row end and every nonzero is one unit of
// work, the m + nnz units are split into equal tiles of T units, and each
// worker finds where its share starts by a search over (row ends, nonzero
// indices).  The plan computes the tile splits once (plan_kernels.cu); this
// kernel does the rest inside each CTA:
//
//  1. stage the tile in shared memory: the row ends row_ptr[i0+1 .. i1], and
//     for the nonzeros j in [j0, j1) either the products vals[j]*x[col[j]]
//     (fp32) or the values and the gathered x[col[j]] side by side (fp64, so
//     that the walk can use one fused multiply-add per nonzero).  col_idx and
//     vals are read with 16-byte loads, all issued before the x gathers;
//  2. each thread takes IPT consecutive units, finds its start by a binary
//     search in shared memory, and walks them: a nonzero adds to the running
//     sum, a row end closes the row;
//  3. a segmented scan over the threads adds the sum carried into each
//     thread's first finished row.  It stops as soon as every open segment
//     has reached its start, so short rows cost one step;
//  4. rows that start and end in the tile are written to y once, coalesced.
//
// GB300 runs fp64 arithmetic at 2 lanes per clock per SM, so the fp64 path
// counts its floating-point instructions: one FMA per nonzero, 0-2 per row
// (alpha = 1 and beta = 0 need none), and a few per thread for carries.
//
// Rows cut by a tile boundary ("partial tiles" in the section) are finished
// without a second kernel and without any waiting: each tile holding part of
// such a row stores its partial sum, then counts itself in on the row's
// arrival counter; the tile that arrives last (the counter says how many to
// expect: the tiles from the one holding the row's first nonzero to the one
// holding its end) adds the partials in index order with a tree and writes
// y.  The order of the sum does not depend on which tile arrives last, so
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

template <typename V>
__device__ __forceinline__ V finish_row(V s, V alpha, V beta, int mode, const V *y, int row) {
    switch (mode) {
    case 0: return s;
    case 1: return alpha * s;
    case 2: return fma(beta, y[row], s);
    default: return fma(beta, y[row], alpha * s);
    }
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

template <typename V, int IPT>
constexpr size_t dyn_smem_bytes() {
    constexpr int T = kThreads * IPT;
    return sizeof(V) * (T + 4) * (sizeof(V) == 8 ? 2 : 1) + sizeof(int) * T;
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
    V *s_a = reinterpret_cast<V *>(dsm);                            // fp32 products / fp64 values
    V *s_b = F64 ? s_a + (T + 4) : s_a;                              // fp64 gathered x
    int *s_re = reinterpret_cast<int *>(dsm + sizeof(V) * (T + 4) * (F64 ? 2 : 1));
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
    const int nitems = nrows + nnzt;
    const int base = VEC ? (j0 & ~3) : j0;  // staged element g sits at s_*[g - base]
    const int sh = j0 - base;

    // ---- 1. stage
    for (int r = tid; r < nrows; r += kThreads) s_re[r] = ld_stream(p.row_ptr + i0 + 1 + r);
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
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (g + e >= j0 && g + e < j1) {
                        const V xv = ld_gather(p.x + ci[e]);
                        if constexpr (F64) {
                            s_a[g + e - base] = vv[u][e];
                            s_b[g + e - base] = xv;
                        } else {
                            s_a[g + e - base] = vv[u][e] * xv;
                        }
                    }
                }
            }
        }
    } else {
#pragma unroll
        for (int it = 0; it < IPT; ++it) {
            const int k = tid + it * kThreads;
            if (k < nnzt) {
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
    }
    __syncthreads();

    // ---- 2. thread split and walk: units [dt, dt + IPT) of the tile
    const int dt = min(tid * IPT, nitems);
    int lo = max(0, dt - nnzt), hi = min(dt, nrows);
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (s_re[mid] - j0 + mid < dt) lo = mid + 1;
        else hi = mid;
    }
    const int r_first = lo;
    int r = lo;
    int k = dt - lo;
    int re = r < nrows ? s_re[r] - j0 : INT_MAX;
    V acc = V(0);
    V out[IPT];
    unsigned ends = 0;
#pragma unroll
    for (int it = 0; it < IPT; ++it) {
        const bool valid = dt + it < nitems;
        if (valid && k >= re) {  // row r has no nonzero left: its end is next
            out[it] = acc;
            acc = V(0);
            ends |= 1u << it;
            ++r;
            re = r < nrows ? s_re[r] - j0 : INT_MAX;
        } else if (valid) {
            if constexpr (F64) acc = fma(s_a[k + sh], s_b[k + sh], acc);
            else acc += s_a[k + sh];
            ++k;
        }
    }

    // ---- 3. segmented inclusive scan of (row end seen, running sum)
    V v = acc;
    int f = ends != 0;
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
    __syncthreads();  // also: every thread is done reading the staged tile
    if (tid == 0) {
        V run = V(0);
        for (int w = 0; w < kWarps; ++w) {
            sm.warp_prefix[w] = run;
            run = sm.warp_flag[w] ? sm.warp_sum[w] : run + sm.warp_sum[w];
        }
    }
    __syncthreads();
    const V wprefix = sm.warp_prefix[warp];
    V incl = v;
    if (warp > 0 && __any_sync(0xffffffffu, !f)) {
        if (!f) incl = wprefix + v;
    }
    V carry_in = __shfl_up_sync(0xffffffffu, incl, 1);
    if (lane == 0) carry_in = wprefix;
    {
        bool first = true;
        int rr = r_first;
#pragma unroll
        for (int it = 0; it < IPT; ++it) {
            if ((ends >> it) & 1u) {
                V s = out[it];
                if (first) s = carry_in + s;
                first = false;
                s_a[rr++] = s;
            }
        }
    }
    __syncthreads();

    // ---- 4. rows that start and end in this tile
    const int32_t rp_i0 = p.row_ptr[i0];
    const bool head_cut = nrows > 0 && rp_i0 < j0;
    for (int q = tid + (head_cut ? 1 : 0); q < nrows; q += kThreads) {
        const int row = i0 + q;
        p.y[row] = finish_row(s_a[q], p.alpha, p.beta, p.mode, p.y, row);
    }

    // ---- cut rows: store partials and count arrivals
    if (tid == 0) {
        sm.run_finish[0] = 0;
        if (head_cut) {
            const long long first = ((long long)rp_i0 + i0) / T;
            p.head_partial[tile] = s_a[0];
            __threadfence();
            const int before = atomicAdd(p.arrivals + tile, 1);
            if (before == (int)(tile - first)) {
                __threadfence();
                sm.run_finish[0] = 1;
                sm.run_row[0] = i0;
                sm.run_first[0] = first;
                sm.run_last[0] = tile;
            }
        }
    }
    if (tid == kThreads - 1) {
        sm.run_finish[1] = 0;
        if (i1 < p.m) {
            const int32_t rp_i1 = nrows > 0 ? s_re[nrows - 1] : rp_i0;
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
    constexpr size_t smem = dyn_smem_bytes<V, IPT>();
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
