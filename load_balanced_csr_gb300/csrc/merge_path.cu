// Merge-path CSR SpMV with a fused carry-out fix-up.
//
// Schedule: "A GPU load-balancing programming model" (Osama, Porumbescu,
// Owens), section 5.2.1 -- every row end and every nonzero is one unit of
// work, the m + nnz units are split into equal tiles of T units, and each
// worker finds where its share starts by a search over (row ends, nonzero
// indices).  The plan computes the tile splits once (plan_kernels.cu); this
// kernel does the rest of the section's two steps inside each CTA:
//
//  1. stage the tile: row ends row_ptr[i0+1 .. i1] and the products
//     vals[j] * x[col_idx[j]] for j in [j0, j1) go to shared memory, loaded
//     with coalesced streaming loads (x through the read-only path);
//  2. each thread takes IPT consecutive units, finds its start by a binary
//     search in shared memory, and walks them: a nonzero adds its product to
//     the running sum, a row end closes the row;
//  3. a segmented scan over the threads (warp shuffles, then across warps)
//     adds the sums carried into each thread's first finished row;
//  4. rows that start and end in the tile are written to y once, coalesced.
//
// Rows cut by a tile boundary ("partial tiles" in the section) are fixed up
// without a second kernel and without any waiting: each tile that holds
// part of such a row stores its partial sum, then counts itself in on the
// row's arrival counter; the tile that arrives last (the counter tells it
// how many participants to expect: the tiles from the one holding the
// row's first nonzero to the one holding its end) adds all partials in
// index order with a tree reduction and writes y.  The order of the sum does
// not depend on which tile arrives last, so results are deterministic.
// The paper's CUB comparison needs a separate fix-up step for these rows.
#include <climits>

#include "internal.cuh"

namespace lbcsr {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

template <typename V, int IPT>
struct alignas(16) MergeSmem {
    static constexpr int T = kThreads * IPT;
    int32_t row_end[T];   // row_ptr[i0 + 1 + r], absolute
    V val[T];             // products; after the walk, finished row sums
    V warp_sum[kWarps];
    int warp_flag[kWarps];
    V red[kWarps];
    int64_t run_first[2];
    int64_t run_last[2];
    int32_t run_row[2];
    int32_t run_finish[2];
};

// Sum of the partials of one cut row, by the tile that arrived last.
template <typename V>
__device__ void finish_cut_row(V *smem_red, int32_t row, int64_t first_tile, int64_t last_tile,
                               const V *tail_partial, const V *head_partial, V *y, V alpha, V beta,
                               int32_t *arrivals) {
    const int tid = threadIdx.x;
    V s = V(0);
    for (int64_t t = first_tile + tid; t < last_tile; t += kThreads) s += __ldcg(tail_partial + t);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if ((tid & 31) == 0) smem_red[tid >> 5] = s;
    __syncthreads();
    if (tid == 0) {
        V total = smem_red[0];
#pragma unroll
        for (int w = 1; w < kWarps; ++w) total += smem_red[w];
        total += __ldcg(head_partial + last_tile);
        V res = alpha * total;
        if (beta != V(0)) res += beta * y[row];
        y[row] = res;
        arrivals[last_tile] = 0;  // ready for the next product
    }
    __syncthreads();
}

template <typename V, int IPT>
__global__ void __launch_bounds__(kThreads)
merge_path_spmv_kernel(const MergePathArgs a) {
    constexpr int T = kThreads * IPT;
    __shared__ MergeSmem<V, IPT> sm;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int64_t tile = blockIdx.x;

    const int32_t *__restrict__ rp = a.row_ptr;
    const int32_t *__restrict__ col = a.col_idx;
    const V *__restrict__ val = static_cast<const V *>(a.vals);
    const V *__restrict__ x = static_cast<const V *>(a.x);
    V *__restrict__ y = static_cast<V *>(a.y);
    const V alpha = static_cast<V>(a.alpha);
    const V beta = static_cast<V>(a.beta);

    const int2 c0 = a.part[tile];
    const int2 c1 = a.part[tile + 1];
    const int i0 = c0.x, j0 = c0.y, i1 = c1.x, j1 = c1.y;
    const int nrows = i1 - i0;
    const int nnzt = j1 - j0;
    const int nitems = nrows + nnzt;

    // ---- 1. stage row ends and products
#pragma unroll
    for (int it = 0; it < IPT; ++it) {
        const int r = tid + it * kThreads;
        if (r < nrows) sm.row_end[r] = ld_stream(rp + i0 + 1 + r);
    }
    {
        int c[IPT];
#pragma unroll
        for (int it = 0; it < IPT; ++it) {
            const int k = tid + it * kThreads;
            c[it] = k < nnzt ? ld_stream(col + j0 + k) : 0;
        }
        V xv[IPT];
#pragma unroll
        for (int it = 0; it < IPT; ++it) {
            const int k = tid + it * kThreads;
            xv[it] = k < nnzt ? ld_gather(x + c[it]) : V(0);
        }
#pragma unroll
        for (int it = 0; it < IPT; ++it) {
            const int k = tid + it * kThreads;
            if (k < nnzt) sm.val[k] = ld_stream(val + j0 + k) * xv[it];
        }
    }
    __syncthreads();

    // ---- 2. thread split: units [dt, dt + IPT) of the tile
    const int dt = min(tid * IPT, nitems);
    int lo = max(0, dt - nnzt), hi = min(dt, nrows);
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (sm.row_end[mid] - j0 + mid < dt) lo = mid + 1;
        else hi = mid;
    }
    const int r_first = lo;
    int r = lo;
    int k = dt - lo;
    int re = r < nrows ? sm.row_end[r] - j0 : INT_MAX;
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
            re = r < nrows ? sm.row_end[r] - j0 : INT_MAX;
        } else if (valid) {
            acc += sm.val[k];
            ++k;
        }
    }

    // ---- 3. segmented inclusive scan of (has row end, running sum) over threads
    V v = acc;
    int f = ends != 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const V pv = __shfl_up_sync(0xffffffffu, v, off);
        const int pf = __shfl_up_sync(0xffffffffu, f, off);
        if (lane >= off) {
            if (!f) v = pv + v;
            f |= pf;
        }
    }
    if (lane == 31) {
        sm.warp_sum[warp] = v;
        sm.warp_flag[warp] = f;
    }
    __syncthreads();  // also: every thread is done reading sm.val
    V wprefix = V(0);
    for (int w = 0; w < warp; ++w) wprefix = sm.warp_flag[w] ? sm.warp_sum[w] : wprefix + sm.warp_sum[w];
    const V incl = f ? v : wprefix + v;
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
                sm.val[rr++] = s;
            }
        }
    }
    __syncthreads();

    // ---- 4. rows that start and end in this tile
    const int32_t rp_i0 = rp[i0];
    const bool head_cut = nrows > 0 && rp_i0 < j0;
    for (int q = tid; q < nrows; q += kThreads) {
        if (q == 0 && head_cut) continue;
        const int row = i0 + q;
        V res = alpha * sm.val[q];
        if (beta != V(0)) res += beta * y[row];
        y[row] = res;
    }

    // ---- cut rows: store partials and count arrivals
    V *tail_partial = static_cast<V *>(a.tail_partial);
    V *head_partial = static_cast<V *>(a.head_partial);
    if (tid == 0) {
        sm.run_finish[0] = 0;
        if (head_cut) {
            const int64_t first = ((int64_t)rp_i0 + i0) / T;
            head_partial[tile] = sm.val[0];
            __threadfence();
            const int before = atomicAdd(a.arrivals + tile, 1);
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
        if (i1 < a.m) {
            const int32_t rp_i1 = nrows > 0 ? sm.row_end[nrows - 1] : rp_i0;
            if (j1 > max(rp_i1, j0)) {  // the open row has nonzeros in this tile
                const int64_t first = ((int64_t)rp_i1 + i1) / T;
                const int64_t last = ((int64_t)rp[i1 + 1] + i1) / T;
                tail_partial[tile] = incl;
                __threadfence();
                const int before = atomicAdd(a.arrivals + last, 1);
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
#pragma unroll
    for (int s = 0; s < 2; ++s) {
        if (sm.run_finish[s])
            finish_cut_row<V>(sm.red, sm.run_row[s], sm.run_first[s], sm.run_last[s], tail_partial,
                              head_partial, y, alpha, beta, a.arrivals);
    }
}

template <typename V, int IPT>
cudaError_t launch_typed(const MergePathArgs &a, cudaStream_t stream) {
    if (a.num_tiles <= 0) return cudaSuccess;
    merge_path_spmv_kernel<V, IPT><<<(unsigned)a.num_tiles, kThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

template <typename V>
cudaError_t launch_ipt(int ipt, const MergePathArgs &a, cudaStream_t stream) {
    switch (ipt) {
    case 5: return launch_typed<V, 5>(a, stream);
    case 7: return launch_typed<V, 7>(a, stream);
    case 9: return launch_typed<V, 9>(a, stream);
    case 11: return launch_typed<V, 11>(a, stream);
    case 13: return launch_typed<V, 13>(a, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

bool merge_path_supported(int ipt) {
    return ipt == 5 || ipt == 7 || ipt == 9 || ipt == 11 || ipt == 13;
}

int merge_path_threads() { return kThreads; }

cudaError_t launch_merge_path_spmv(spmv_dtype_t dtype, int ipt, const MergePathArgs &a,
                                   cudaStream_t stream) {
    return dtype == SPMV_F64 ? launch_ipt<double>(ipt, a, stream) : launch_ipt<float>(ipt, a, stream);
}

}  // namespace lbcsr
