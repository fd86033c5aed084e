// Sparse times dense: Y = alpha * A * X + beta * Y for k right-hand sides,
// X (n-by-k) and Y (m-by-k) row-major.  "A GPU load-balancing programming
// model" (section 4.3, Listing 4) writes SpMM as the SpMV row loop with an
// inner loop over the columns of X; its merge-path schedule (section 5.2.1)
// balances the rows.
//
// Each warp takes the same share of the merge path as in the SpMV kernel
// (the plan's partition: a contiguous run of row ends and nonzeros, cut
// into equal tiles) and walks its run in merge order; its lanes span 32
// columns of X and Y (up to kSpmmBlocks * 32 per launch), so every X row it
// gathers and every Y row it writes is one coalesced access.  Columns and
// values arrive 32 nonzeros at a time (lane q loads nonzero q, the walk
// takes them from the lanes by shuffles), row ends 32 rows at a time, and
// the X rows of the next few nonzeros are loaded before they are needed.
//
// A row cut between warps is finished as in the SpMV kernel: each warp
// holding part of it stores its k partial sums, counts in on the row's
// arrival counter, and the last to arrive adds the partials in warp order
// and writes the row of Y.
#include "internal.cuh"
#include "tma.cuh"

namespace lbcsr {

namespace {

using namespace tma;

constexpr int kSpmmThreads = 256;
constexpr int kSpmmAhead = 4;  // nonzeros whose X rows are loaded ahead

template <typename V>
struct SpmmParams {
    int32_t m, nnz, k;
    const int32_t *row_ptr;
    const int32_t *col_idx;
    const V *vals;
    const V *X;
    long long ldx;
    V *Y;
    long long ldy;
    V alpha, beta;
    const int2 *part;
    long long P, W, T;
    V *tail, *head;  // [W][kSpmmBlocks * 32]
    int32_t *arrivals;
};

__device__ __forceinline__ long long spmm_warp_of_unit(long long d, long long T, long long P, long long W) {
    const long long t = d / T;
    return ((t + 1) * W - 1) / P;  // warp w owns tiles [w*P/W, (w+1)*P/W)
}

template <typename V, int KB>
__device__ __forceinline__ void spmm_store_row(const SpmmParams<V> &p, long long row, const V (&acc)[KB], int lane,
                                               uint64_t pol) {
#pragma unroll
    for (int b = 0; b < KB; ++b) {
        const int c = b * 32 + lane;
        if (c < p.k) {
            V r = p.alpha * acc[b];
            if (p.beta != V(0)) r = fma(p.beta, p.Y[row * p.ldy + c], r);
            store_stream(p.Y + row * p.ldy + c, r, pol);
        }
    }
}

// A row cut between warps first..last: store this warp's partials, count
// in; the last to arrive adds them in warp order (blocks of 16 warps, then
// the blocks) and writes the row.
template <typename V, int KB>
__device__ void spmm_cut_row(const SpmmParams<V> &p, int lane, const V (&part)[KB], bool as_head, long long me,
                             long long row, long long first, long long last, uint64_t pol) {
    constexpr int KW = KB * 32;
    V *mine = (as_head ? p.head : p.tail) + me * KW;
#pragma unroll
    for (int b = 0; b < KB; ++b) mine[b * 32 + lane] = part[b];
    __threadfence();
    __syncwarp();
    int finisher = 0;
    if (lane == 0) {
        finisher = atomicAdd(p.arrivals + last, 1) == (int)(last - first);
        if (finisher) __threadfence();
    }
    if (!__shfl_sync(0xffffffffu, finisher, 0)) return;
    V sum[KB];
#pragma unroll
    for (int b = 0; b < KB; ++b) {
        const int c = b * 32 + lane;
        V total = V(0);
        for (long long w0 = first; w0 < last; w0 += 16) {
            V blk = V(0);
            for (long long w = w0; w < last && w < w0 + 16; ++w) blk += __ldcg(p.tail + w * KW + c);
            total += blk;
        }
        sum[b] = total + __ldcg(p.head + last * KW + c);
    }
    spmm_store_row<V, KB>(p, row, sum, lane, pol);
    if (lane == 0) p.arrivals[last] = 0;  // ready for the next product
}

template <typename V, int KB>
__global__ void __launch_bounds__(kSpmmThreads)
spmm_kernel(const SpmmParams<V> p) {
    const int lane = threadIdx.x & 31;
    const long long me = (long long)blockIdx.x * (kSpmmThreads / 32) + (threadIdx.x >> 5);
    if (me >= p.W) return;
    const uint64_t stream_pol = l2_policy_evict_first();
    // the warp's run: units [d_s, d_e) of the merge path
    const int2 s = p.part[me * p.P / p.W];
    const int2 e = p.part[(me + 1) * p.P / p.W];
    const long long i_s = s.x, j_s = s.y, i_e = e.x, j_e = e.y;

    V acc[KB];
#pragma unroll
    for (int b = 0; b < KB; ++b) acc[b] = V(0);
    bool head = i_s < p.m && p.row_ptr[i_s] < j_s;  // the first row began in an earlier warp

    long long r = i_s;       // current row
    long long rb = -(1ll << 40);  // first row whose end the lanes hold (none yet)
    int re_lane = 0;         // lane q: row_ptr[rb + 1 + q]
    long long jb = j_s;      // first nonzero the lanes hold
    int col_lane = 0;
    V val_lane = V(0);
    auto row_end = [&](long long row) -> long long {
        if (row < rb || row >= rb + 32) {  // refill: rows row .. row + 31
            rb = row;
            const long long q = rb + 1 + lane;
            re_lane = q <= p.m ? p.row_ptr[q] : p.nnz;
        }
        return __shfl_sync(0xffffffffu, re_lane, (int)(row - rb));
    };
    // finish every row that ends before nonzero j (or, at the run's end,
    // every row of the run)
    auto close_rows = [&](long long j) {
        while (r < i_e) {
            const long long re = row_end(r);
            if (re > j) break;
            if (head) {
                head = false;
                const long long first = spmm_warp_of_unit((long long)p.row_ptr[r] + r, p.T, p.P, p.W);
                spmm_cut_row<V, KB>(p, lane, acc, true, me, r, first, me, stream_pol);
            } else {
                spmm_store_row<V, KB>(p, r, acc, lane, stream_pol);
            }
#pragma unroll
            for (int b = 0; b < KB; ++b) acc[b] = V(0);
            ++r;
        }
    };

    for (long long j0 = j_s; j0 < j_e; j0 += 32) {
        const int nb = (int)(j_e - j0 < 32 ? j_e - j0 : 32);
        jb = j0;
        col_lane = lane < nb ? ld_stream(p.col_idx + jb + lane) : 0;
        val_lane = lane < nb ? ld_stream(p.vals + jb + lane) : V(0);
        for (int q0 = 0; q0 < nb; q0 += kSpmmAhead) {
            V xv[kSpmmAhead][KB];
            V vv[kSpmmAhead];
#pragma unroll
            for (int a = 0; a < kSpmmAhead; ++a) {
                const int q = q0 + a;
                const int c = __shfl_sync(0xffffffffu, col_lane, q & 31);
                vv[a] = __shfl_sync(0xffffffffu, val_lane, q & 31);
#pragma unroll
                for (int b = 0; b < KB; ++b) {
                    const int t = b * 32 + lane;
                    xv[a][b] = q < nb && t < p.k ? ld_gather(p.X + (long long)c * p.ldx + t) : V(0);
                }
            }
#pragma unroll
            for (int a = 0; a < kSpmmAhead; ++a) {
                const int q = q0 + a;
                if (q < nb) {
                    close_rows(jb + q);
#pragma unroll
                    for (int b = 0; b < KB; ++b) acc[b] = fma(vv[a], xv[a][b], acc[b]);
                }
            }
        }
    }
    close_rows(j_e);  // rows that end after the run's last nonzero (empty rows too)
    // the row open at the run's end, if it has nonzeros in this run
    if (i_e < p.m) {
        const long long rp_e = p.row_ptr[i_e];
        if (j_e > (rp_e > j_s ? rp_e : j_s)) {
            const long long first = spmm_warp_of_unit(rp_e + i_e, p.T, p.P, p.W);
            const long long last = spmm_warp_of_unit((long long)p.row_ptr[i_e + 1] + i_e, p.T, p.P, p.W);
            spmm_cut_row<V, KB>(p, lane, acc, false, me, i_e, first, last, stream_pol);
        }
    }
}

template <typename V, int KB>
cudaError_t launch_kb(const SpmmArgs &a, int32_t k, const void *X, void *Y, cudaStream_t stream) {
    SpmmParams<V> p;
    p.m = a.m;
    p.nnz = a.nnz;
    p.k = k;
    p.row_ptr = a.row_ptr;
    p.col_idx = a.col_idx;
    p.vals = static_cast<const V *>(a.vals);
    p.X = static_cast<const V *>(X);
    p.ldx = a.ldx;
    p.Y = static_cast<V *>(Y);
    p.ldy = a.ldy;
    p.alpha = (V)a.alpha;
    p.beta = (V)a.beta;
    p.part = a.part;
    p.P = a.num_tiles;
    p.W = a.num_warps;
    p.T = a.tile;
    p.tail = static_cast<V *>(a.tail);
    p.head = static_cast<V *>(a.head);
    p.arrivals = a.arrivals;
    const unsigned grid = (unsigned)((p.W + kSpmmThreads / 32 - 1) / (kSpmmThreads / 32));
    spmm_kernel<V, KB><<<grid, kSpmmThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

template <typename V>
cudaError_t launch_typed(const SpmmArgs &a, cudaStream_t stream) {
    // columns in slices of kSpmmBlocks * 32, one launch each
    for (int32_t c0 = 0; c0 < a.k; c0 += kSpmmBlocks * 32) {
        const int32_t kc = a.k - c0 < kSpmmBlocks * 32 ? a.k - c0 : kSpmmBlocks * 32;
        const void *X = static_cast<const V *>(a.X) + c0;
        void *Y = static_cast<V *>(a.Y) + c0;
        cudaError_t e;
        if (kc <= 32) e = launch_kb<V, 1>(a, kc, X, Y, stream);
        else if (kc <= 64) e = launch_kb<V, 2>(a, kc, X, Y, stream);
        else e = launch_kb<V, 4>(a, kc, X, Y, stream);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

int spmm_warps(int64_t num_tiles) {
    const int64_t cap = (int64_t)device_sm_count() * kSpmmWarpsPerSm;
    return (int)(num_tiles < cap ? num_tiles : cap);
}

cudaError_t launch_spmm(spmv_dtype_t dtype, const SpmmArgs &a, cudaStream_t stream) {
    if (a.m <= 0 || a.k <= 0) return cudaSuccess;
    return dtype == SPMV_F64 ? launch_typed<double>(a, stream) : launch_typed<float>(a, stream);
}

}  // namespace lbcsr
