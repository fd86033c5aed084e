// Sparse times dense: Y = alpha * A * X + beta * Y for k right-hand sides,
// X (n-by-k) and Y (m-by-k) row-major.  "A GPU load-balancing programming
// model" (section 4.3, Listing 4) writes SpMM as the SpMV row loop with an
// inner loop over the columns of X; its merge-path schedule (section 5.2.1)
// balances the rows.
//
// Each warp takes the same share of the merge path as in the SpMV kernel
// (the plan's partition: a contiguous run of row ends and nonzeros, cut
// into equal tiles).  A lane holds VW consecutive columns of a row: VW = 4
// (fp32) or 2 (fp64), one 16-byte load per X row and lane, when X's layout
// allows it, else 1.  The rows that lie wholly inside the run are summed by
// sub-warps of k' lanes (k' = k / VW rounded up to a power of two, at most
// 32): 32 / k' rows at once, each sub-warp walking its row's nonzeros with
// its lanes over the columns; with k' = 32 a sub-warp is the whole warp,
// which takes 32 * VW columns at a time (up to kSpmmBlocks * 32 per
// launch).  The rows cut by the run's ends are summed by the whole warp,
// with several of the row's nonzeros per step when k' is small.  Every X
// row gathered and every Y row written is one coalesced access.
//
// Wider lanes pay on matrices whose X rows are gathered at random: the
// kernel is bound by the latency of those gathers, and a 16-byte load
// keeps four times the bytes of a 4-byte one in flight for the same
// registers of column indices and values.
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

// VW consecutive values of an X row (16-byte aligned when VW > 1).
template <typename V, int VW>
__device__ __forceinline__ void ld_x(const V *p, V (&o)[VW]) {
    if constexpr (VW == 1) {
        o[0] = ld_gather(p);
    } else if constexpr (sizeof(V) == 4 && VW == 4) {
        const float4 t = __ldg(reinterpret_cast<const float4 *>(p));
        o[0] = t.x, o[1] = t.y, o[2] = t.z, o[3] = t.w;
    } else if constexpr (sizeof(V) == 4 && VW == 2) {
        const float2 t = __ldg(reinterpret_cast<const float2 *>(p));
        o[0] = t.x, o[1] = t.y;
    } else {
        static_assert(sizeof(V) == 8 && VW == 2, "16-byte lanes");
        const double2 t = __ldg(reinterpret_cast<const double2 *>(p));
        o[0] = t.x, o[1] = t.y;
    }
}

// Column of value v of block b held by a lane serving column group tcol.
template <int KP, int VW>
__device__ __forceinline__ int spmm_col(int b, int tcol, int v) {
    return (b * KP + tcol) * VW + v;
}

// Lanes of slot 0 write the row.
template <typename V, int KB, int KP, int VW>
__device__ __forceinline__ void spmm_store_row(const SpmmParams<V> &p, long long row, const V (&acc)[KB * VW],
                                               int lane, uint64_t pol) {
    if (lane >= KP) return;
#pragma unroll
    for (int b = 0; b < KB; ++b)
#pragma unroll
        for (int v = 0; v < VW; ++v) {
            const int c = spmm_col<KP, VW>(b, lane, v);
            if (c < p.k) {
                V r = p.alpha * acc[b * VW + v];
                if (p.beta != V(0)) r = fma(p.beta, p.Y[row * p.ldy + c], r);
                store_stream(p.Y + row * p.ldy + c, r, pol);
            }
        }
}

// A row cut between warps first..last: store this warp's partials, count
// in; the last to arrive adds them in warp order (blocks of 16 warps, then
// the blocks) and writes the row.
template <typename V, int KB, int KP, int VW>
__device__ void spmm_cut_row(const SpmmParams<V> &p, int lane, const V (&part)[KB * VW], bool as_head, long long me,
                             long long row, long long first, long long last, uint64_t pol) {
    constexpr int KW = kSpmmBlocks * 32;  // scratch row of a warp
    static_assert(KB * KP * VW <= KW, "a launch's columns fit a scratch row");
    V *mine = (as_head ? p.head : p.tail) + me * KW;
    if (lane < KP) {
#pragma unroll
        for (int b = 0; b < KB; ++b)
#pragma unroll
            for (int v = 0; v < VW; ++v) mine[spmm_col<KP, VW>(b, lane, v)] = part[b * VW + v];
    }
    __threadfence();
    __syncwarp();
    int finisher = 0;
    if (lane == 0) {
        finisher = atomicAdd(p.arrivals + last, 1) == (int)(last - first);
        if (finisher) __threadfence();
    }
    if (!__shfl_sync(0xffffffffu, finisher, 0)) return;
    V sum[KB * VW];
#pragma unroll
    for (int b = 0; b < KB; ++b)
#pragma unroll
        for (int v = 0; v < VW; ++v) {
            const int c = spmm_col<KP, VW>(b, lane % KP, v);
            V total = V(0);
            for (long long w0 = first; w0 < last; w0 += 16) {
                V blk = V(0);
                for (long long w = w0; w < last && w < w0 + 16; ++w) blk += __ldcg(p.tail + w * KW + c);
                total += blk;
            }
            sum[b * VW + v] = total + __ldcg(p.head + last * KW + c);
        }
    spmm_store_row<V, KB, KP, VW>(p, row, sum, lane, pol);
    if (lane == 0) p.arrivals[last] = 0;  // ready for the next product
}

#ifndef LBCSR_SPMM_WARP_U
#define LBCSR_SPMM_WARP_U 8
#endif
#ifndef LBCSR_SPMM_WARP_U4
#define LBCSR_SPMM_WARP_U4 4
#endif
#ifndef LBCSR_SPMM_WARP_UV
#define LBCSR_SPMM_WARP_UV 8
#endif
#ifndef LBCSR_SPMM_WARP_UV32
#define LBCSR_SPMM_WARP_UV32 4
#endif
// Nonzeros [j, stop) of one row summed by the whole warp: S = 32 / KP
// nonzeros per warp step (lane l serves slot l / KP, columns of group
// l % KP), the slots added by xor-shuffles at the end; every lane gets the
// row's sums.
template <typename V, int KB, int KP, int VW>
__device__ __forceinline__ void spmm_warp_row(const SpmmParams<V> &p, long long j, long long stop, int lane,
                                              V (&acc)[KB * VW]) {
    constexpr int S = 32 / KP;
    // warp steps of loads in flight: 8, or 4 where a step already loads 64
    // bytes or more per lane (k = 128: power law 6.63 -> 6.36 ms, skew
    // 23.4 -> 22.0 ms with one value per lane, 24.3 -> 20.2 ms with two)
    constexpr int U = VW == 1 ? (KB >= 4 ? LBCSR_SPMM_WARP_U4 : LBCSR_SPMM_WARP_U)
                              : (KP == 32 ? LBCSR_SPMM_WARP_UV32 : LBCSR_SPMM_WARP_UV);
    const int slot = lane / KP;
    const int tcol = lane % KP;
#pragma unroll
    for (int b = 0; b < KB * VW; ++b) acc[b] = V(0);
    for (; j < stop; j += (long long)U * S) {
        int cc[U];
        V vv[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const long long q = j + (long long)u * S + slot;
            cc[u] = q < stop ? ld_stream(p.col_idx + q) : -1;
            vv[u] = q < stop ? ld_stream(p.vals + q) : V(0);
        }
        V xv[U][KB * VW];
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
            for (int b = 0; b < KB; ++b) {
                const int c = spmm_col<KP, VW>(b, tcol, 0);
                V t[VW];
                if (cc[u] >= 0 && c < p.k) {
                    ld_x<V, VW>(p.X + (long long)cc[u] * p.ldx + c, t);
                } else {
#pragma unroll
                    for (int v = 0; v < VW; ++v) t[v] = V(0);
                }
#pragma unroll
                for (int v = 0; v < VW; ++v) xv[u][b * VW + v] = t[v];
            }
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
            for (int b = 0; b < KB * VW; ++b) acc[b] = fma(vv[u], xv[u][b], acc[b]);
    }
#pragma unroll
    for (int off = KP; off < 32; off <<= 1)
#pragma unroll
        for (int b = 0; b < KB * VW; ++b) acc[b] += __shfl_xor_sync(0xffffffffu, acc[b], off);
}

// The rows that lie wholly inside a warp's run, [r0, r1), summed by
// sub-warps of KP lanes (KB == 1), lanes over columns: S rows are in flight
// at once, which matters for short rows.  A row longer than kSpmmSubRowMax
// would hold up the warp: the whole warp sums it.
constexpr int kSpmmSubRowMax = 64;

#ifndef LBCSR_SPMM_SUB_U
#define LBCSR_SPMM_SUB_U 8
#endif
#ifndef LBCSR_SPMM_SUB_UV
#define LBCSR_SPMM_SUB_UV 8
#endif
// Each sub-warp walks its own rows, r0 + s, r0 + s + S, ..., one after the
// other: a sub-warp that finishes a short row starts its next row at once
// instead of waiting for the longest row of a group (power-law rows are
// heavy-tailed).  The next row's bounds are loaded one row ahead.  Rows
// longer than kSpmmSubRowMax are skipped here and summed by the whole warp
// afterwards, in row order.  With one value per lane, nonzero q of a row
// goes to sum (q - row start) mod U, and the U sums are added pairwise at
// the row's end; with VW values per lane, to sum (q - row start) mod 2.
template <typename V, int KP, int VW>
__device__ __forceinline__ void spmm_subwarp_rows(const SpmmParams<V> &p, long long r0, long long r1, int lane,
                                                  uint64_t pol) {
    constexpr int S = 32 / KP;
    constexpr int U = VW == 1 ? LBCSR_SPMM_SUB_U : LBCSR_SPMM_SUB_UV;  // nonzeros in flight per row
    static_assert(U == 2 || U == 4 || U == 8 || U == 16, "two, four, eight or sixteen nonzeros");
    constexpr int NA = VW == 1 ? U : 2;  // sums per column
    const int sub = lane / KP;
    const int tcol = lane % KP;
    const int c0 = spmm_col<KP, VW>(0, tcol, 0);
    const bool col_ok = c0 < p.k;
    // this sub-warp's current short row [q, e) and the next row's bounds
    long long r = r0 + sub;
    long long q = 0, e = 0;
    if (r < r1) {
        q = p.row_ptr[r];
        e = p.row_ptr[r + 1];
    }
    while (r < r1 && e - q > kSpmmSubRowMax) {  // skip long rows
        r += S;
        if (r < r1) {
            q = p.row_ptr[r];
            e = p.row_ptr[r + 1];
        }
    }
    long long nq = 0, ne = 0;
    if (r + S < r1) {
        nq = p.row_ptr[r + S];
        ne = p.row_ptr[r + S + 1];
    }
    V acc[NA][VW];
#pragma unroll
    for (int a = 0; a < NA; ++a)
#pragma unroll
        for (int v = 0; v < VW; ++v) acc[a][v] = V(0);
    while (__any_sync(0xffffffffu, r < r1)) {
        const bool live = r < r1;
        int cc[U];
        V vv[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            cc[u] = live && q + u < e ? ld_stream(p.col_idx + q + u) : -1;
            vv[u] = live && q + u < e ? ld_stream(p.vals + q + u) : V(0);
        }
        V xv[U][VW];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (cc[u] >= 0 && col_ok) {
                ld_x<V, VW>(p.X + (long long)cc[u] * p.ldx + c0, xv[u]);
            } else {
#pragma unroll
                for (int v = 0; v < VW; ++v) xv[u][v] = V(0);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
            for (int v = 0; v < VW; ++v) acc[u % NA][v] = fma(vv[u], xv[u][v], acc[u % NA][v]);
        q += U;
        if (live && q >= e) {  // the row is done: write it, move to the next short row
#pragma unroll
            for (int w = NA / 2; w > 0; w >>= 1)
#pragma unroll
                for (int a = 0; a < w; ++a)
#pragma unroll
                    for (int v = 0; v < VW; ++v) acc[a][v] = acc[a][v] + acc[a + w][v];
#pragma unroll
            for (int v = 0; v < VW; ++v) {
                const int c = c0 + v;
                if (c < p.k) {
                    V y = p.alpha * acc[0][v];
                    if (p.beta != V(0)) y = fma(p.beta, p.Y[r * p.ldy + c], y);
                    store_stream(p.Y + r * p.ldy + c, y, pol);
                }
            }
#pragma unroll
            for (int a = 0; a < NA; ++a)
#pragma unroll
                for (int v = 0; v < VW; ++v) acc[a][v] = V(0);
            r += S;
            q = nq;
            e = ne;
            while (r < r1 && e - q > kSpmmSubRowMax) {
                r += S;
                if (r < r1) {
                    q = p.row_ptr[r];
                    e = p.row_ptr[r + 1];
                }
            }
            if (r + S < r1) {
                nq = p.row_ptr[r + S];
                ne = p.row_ptr[r + S + 1];
            }
        }
    }
    // the run's long rows, one by one, by the whole warp
    for (long long base = r0; base < r1; base += 32) {
        const long long rl = base + lane;
        const bool is_long = rl < r1 && (long long)p.row_ptr[rl + 1] - p.row_ptr[rl] > kSpmmSubRowMax;
        unsigned longs = __ballot_sync(0xffffffffu, is_long);
        while (longs) {
            const int l = __ffs(longs) - 1;
            longs &= longs - 1;
            const long long row = base + l;
            V a[VW];
            spmm_warp_row<V, 1, KP, VW>(p, p.row_ptr[row], p.row_ptr[row + 1], lane, a);
            spmm_store_row<V, 1, KP, VW>(p, row, a, lane, pol);
        }
    }
}

template <typename V, int KB, int KP, int VW>
__global__ void __launch_bounds__(kSpmmThreads)
spmm_kernel(const SpmmParams<V> p) {
    const int lane = threadIdx.x & 31;
    const long long me = (long long)blockIdx.x * (kSpmmThreads / 32) + (threadIdx.x >> 5);
    if (me >= p.W) return;
    const uint64_t stream_pol = l2_policy_evict_first();
    // the warp's run: units [d_s, d_e) of the merge path
    const int2 s0 = p.part[me * p.P / p.W];
    const int2 e0 = p.part[(me + 1) * p.P / p.W];
    const long long i_s = s0.x, j_s = s0.y, i_e = e0.x, j_e = e0.y;
    V acc[KB * VW];
    long long r0 = i_s;
    // the row open at the run's start, if it began in an earlier warp
    if (i_s < p.m && p.row_ptr[i_s] < j_s) {
        if (i_s < i_e) {  // it ends in this run: finish it with the earlier warps' partials
            spmm_warp_row<V, KB, KP, VW>(p, j_s, p.row_ptr[i_s + 1], lane, acc);
            const long long first = spmm_warp_of_unit((long long)p.row_ptr[i_s] + i_s, p.T, p.P, p.W);
            spmm_cut_row<V, KB, KP, VW>(p, lane, acc, true, me, i_s, first, me, stream_pol);
            r0 = i_s + 1;
        }
        // else: the whole run lies inside that row -- the tail below
    }
    // the rows wholly inside the run
    if (KB == 1 && KP < 32) {
        spmm_subwarp_rows<V, KP, VW>(p, r0, i_e, lane, stream_pol);
    } else {
        for (long long r = r0; r < i_e; ++r) {
            spmm_warp_row<V, KB, KP, VW>(p, p.row_ptr[r], p.row_ptr[r + 1], lane, acc);
            spmm_store_row<V, KB, KP, VW>(p, r, acc, lane, stream_pol);
        }
    }
    // the row open at the run's end, if it has nonzeros in this run
    if (i_e < p.m) {
        const long long rp_e = p.row_ptr[i_e];
        const long long from = rp_e > j_s ? rp_e : j_s;
        if (j_e > from) {
            spmm_warp_row<V, KB, KP, VW>(p, from, j_e, lane, acc);
            const long long first = spmm_warp_of_unit(rp_e + i_e, p.T, p.P, p.W);
            const long long last = spmm_warp_of_unit((long long)p.row_ptr[i_e + 1] + i_e, p.T, p.P, p.W);
            spmm_cut_row<V, KB, KP, VW>(p, lane, acc, false, me, i_e, first, last, stream_pol);
        }
    }
}

template <typename V, int VW>
cudaError_t launch_slice(const SpmmParams<V> &p, cudaStream_t stream) {
    const unsigned grid = (unsigned)((p.W + kSpmmThreads / 32 - 1) / (kSpmmThreads / 32));
    // k' = lanes per row: the columns' VW-groups rounded up to a power of two
    const int groups = (p.k + VW - 1) / VW;
    constexpr int kMaxBlocks = kSpmmBlocks / VW;  // a launch's columns fit a scratch row
    if (groups > 32) {  // whole warps over blocks of 32 * VW columns
        if constexpr (kMaxBlocks >= 4) {
            if (groups > 64) spmm_kernel<V, 4, 32, VW><<<grid, kSpmmThreads, 0, stream>>>(p);
            else spmm_kernel<V, 2, 32, VW><<<grid, kSpmmThreads, 0, stream>>>(p);
        } else if constexpr (kMaxBlocks >= 2) {
            spmm_kernel<V, 2, 32, VW><<<grid, kSpmmThreads, 0, stream>>>(p);
        } else {
            return cudaErrorInvalidValue;  // not reached: a slice has at most 32 * VW columns here
        }
    } else if (groups > 16) spmm_kernel<V, 1, 32, VW><<<grid, kSpmmThreads, 0, stream>>>(p);
    else if (groups > 8) spmm_kernel<V, 1, 16, VW><<<grid, kSpmmThreads, 0, stream>>>(p);
    else if (groups > 4) spmm_kernel<V, 1, 8, VW><<<grid, kSpmmThreads, 0, stream>>>(p);
    else if (groups > 2) spmm_kernel<V, 1, 4, VW><<<grid, kSpmmThreads, 0, stream>>>(p);
    else if (groups > 1) spmm_kernel<V, 1, 2, VW><<<grid, kSpmmThreads, 0, stream>>>(p);
    else spmm_kernel<V, 1, 1, VW><<<grid, kSpmmThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

// Values per lane: 16 bytes when every X row's k values split into
// 16-byte aligned loads (X aligned, ldx and k multiples of VW), else 1.  Y
// is read and written one value per access either way.  fp32 rows wider
// than 64 columns keep one value per lane: a warp then spans the row either
// way, and four blocks of 32 lanes measured faster (power law, k = 128:
// 6.36 against 6.84 ms).  LBCSR_SPMM_VEC=0 turns the wide lanes off at
// build time, for tuning.
#ifndef LBCSR_SPMM_VEC
#define LBCSR_SPMM_VEC 1
#endif
template <typename V>
int spmm_vec_width(const SpmmArgs &a) {
    constexpr int VW = 16 / sizeof(V);
    const bool fits = reinterpret_cast<uintptr_t>(a.X) % 16 == 0 && a.ldx % VW == 0 && a.k % VW == 0;
    const bool narrow = sizeof(V) == 8 || a.k <= 16 * VW;
    return LBCSR_SPMM_VEC && fits && narrow ? VW : 1;
}

template <typename V>
cudaError_t launch_typed(const SpmmArgs &a, cudaStream_t stream) {
    const int vw = spmm_vec_width<V>(a);
    SpmmParams<V> p;
    p.m = a.m;
    p.nnz = a.nnz;
    p.row_ptr = a.row_ptr;
    p.col_idx = a.col_idx;
    p.vals = static_cast<const V *>(a.vals);
    p.ldx = a.ldx;
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
    // columns in slices of kSpmmBlocks * 32, one launch each
    for (int32_t c0 = 0; c0 < a.k; c0 += kSpmmBlocks * 32) {
        p.k = a.k - c0 < kSpmmBlocks * 32 ? a.k - c0 : kSpmmBlocks * 32;
        p.X = static_cast<const V *>(a.X) + c0;
        p.Y = static_cast<V *>(a.Y) + c0;
        cudaError_t e = vw == 1 ? launch_slice<V, 1>(p, stream) : launch_slice<V, 16 / sizeof(V)>(p, stream);
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
