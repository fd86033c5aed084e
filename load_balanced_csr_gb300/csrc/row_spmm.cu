// SpMM for matrices whose rows are all short: Y = alpha * A * X + beta * Y
// straight from CSR, a warp per 32 consecutive rows, in the row loop of
// "A GPU load-balancing programming model" (section 4.3, Listing 4: the
// SpMV row loop with an inner loop over the columns of X).  With short
// rows a warp's rows need about the same number of steps, so the rows
// balance without a schedule.
//
// Level l of the warp is the l-th nonzero of each of its rows.  LPR lanes
// share one X row slice of KC values (LPR x 16 bytes), so that one load
// instruction of the warp covers 32 / LPR rows and as many lines; each lane
// loads its own row's nonzero of a level and the lanes that serve a row take
// its column and value by shuffles.  A lane keeps KC sums.  Wider X is taken
// in slices of 32 (fp32) or 16 (fp64) columns, then of the powers of two
// that remain.
//
// Rows of at least long_min nonzeros, when the plan lists them, are left to
// a warp-per-segment kernel (long_spmm_kernel) and skipped here.
#include <climits>
#include <type_traits>

#include "internal.cuh"
#include "row_spmm.cuh"

namespace lbcsr {

namespace {

template <typename V, int KC>
__global__ void __launch_bounds__(256)
row_spmm_lines_kernel(int32_t m, const int32_t *__restrict__ rp, const int32_t *__restrict__ col,
                      const V *__restrict__ val, const V *__restrict__ X, long long ldx, V *__restrict__ Y,
                      long long ldy, V alpha, V beta, int32_t skip_len) {
    constexpr int W = 16 / sizeof(V);  // values per 16-byte load
    constexpr int LPR = KC / W;        // lanes per X row
    constexpr int RPI = 32 / LPR;      // rows per load instruction
    constexpr int J = LPR;             // load instructions per level
    using V4 = typename std::conditional<sizeof(V) == 4, float4, double2>::type;
    const int64_t p0 = ((int64_t)blockIdx.x * 8 + (threadIdx.x >> 5)) * 32;
    if (p0 >= m) return;
    const int lane = threadIdx.x & 31, sub = lane / LPR, cc = lane % LPR;
    const int64_t row_own = p0 + lane;
    const int start_own = row_own < m ? __ldg(rp + row_own) : 0;
    const int len_row = row_own < m ? __ldg(rp + row_own + 1) - start_own : 0;
    const int len_own = len_row < skip_len ? len_row : 0;  // long rows are the long-row kernel's
    const int levels = __reduce_max_sync(0xffffffffu, len_own);
    int lens[J];
#pragma unroll
    for (int j = 0; j < J; ++j) lens[j] = __shfl_sync(0xffffffffu, len_own, j * RPI + sub);
    const unsigned mine_short = __ballot_sync(0xffffffffu, len_row < skip_len);
    V acc[J][W];
#pragma unroll
    for (int j = 0; j < J; ++j)
#pragma unroll
        for (int w = 0; w < W; ++w) acc[j][w] = V(0);
    int c_own = len_own > 0 ? ld_stream(col + start_own) : 0;
    V v_own = len_own > 0 ? ld_stream(val + start_own) : V(0);
    for (int l = 0; l < levels; ++l) {
        int cn = 0;
        V vn = V(0);
        if (l + 1 < len_own) {  // the next level's nonzero while this one's X rows are gathered
            cn = ld_stream(col + start_own + l + 1);
            vn = ld_stream(val + start_own + l + 1);
        }
#pragma unroll
        for (int j = 0; j < J; ++j) {
            const int c = __shfl_sync(0xffffffffu, c_own, j * RPI + sub);
            const V v = __shfl_sync(0xffffffffu, v_own, j * RPI + sub);
            if (l < lens[j]) {
                const V4 q = __ldg(reinterpret_cast<const V4 *>(X + (int64_t)c * ldx + cc * W));
                const V *f = reinterpret_cast<const V *>(&q);
#pragma unroll
                for (int w = 0; w < W; ++w) acc[j][w] = fma(v, f[w], acc[j][w]);
            }
        }
        c_own = cn;
        v_own = vn;
    }
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const int64_t row = p0 + j * RPI + sub;
        if (row >= m || !((mine_short >> (j * RPI + sub)) & 1u)) continue;
        V *yr = Y + row * ldy + cc * W;
        V r[W];
        if (alpha != V(1)) {
#pragma unroll
            for (int w = 0; w < W; ++w) r[w] = alpha * acc[j][w];
        } else {
#pragma unroll
            for (int w = 0; w < W; ++w) r[w] = acc[j][w];
        }
        if (beta != V(0)) {
            const V4 o = *reinterpret_cast<const V4 *>(yr);
            const V *f = reinterpret_cast<const V *>(&o);
#pragma unroll
            for (int w = 0; w < W; ++w) r[w] = fma(beta, f[w], r[w]);
        }
        V4 out;
        V *fo = reinterpret_cast<V *>(&out);
#pragma unroll
        for (int w = 0; w < W; ++w) fo[w] = r[w];
        *reinterpret_cast<V4 *>(yr) = out;
    }
}

// Long rows (len >= skip_len): a warp per segment of kLongSegmentNnz
// nonzeros, as the long-row SpMV kernel, with the warp's lanes spread over
// a slice of kc <= 32 columns: each lane holds VW consecutive columns (one
// 16-byte load per X row when X's layout allows it, else one value), KQ
// lanes (kc / VW rounded up to a power of two) per nonzero, 32 / KQ
// nonzeros at a time, so that one load instruction reads the X row slices
// of 32 / KQ nonzeros, each one contiguous run.  The segment's columns and
// values are loaded 32 at a time, coalesced, and shared by shuffles.  Slots
// are added by xor shuffles at the end.  A one-segment row is written
// directly; a longer row's segment partials (kc values each) are added in
// segment order by the segment that arrives last, which then writes the row
// of Y.
template <typename V, int VW>
__device__ __forceinline__ void ld_row_slice(const V *p, V (&o)[VW]) {
    if constexpr (VW == 1) {
        o[0] = ld_gather(p);
    } else if constexpr (sizeof(V) == 4) {
        static_assert(VW == 4, "16-byte loads");
        const float4 t = __ldg(reinterpret_cast<const float4 *>(p));
        o[0] = t.x, o[1] = t.y, o[2] = t.z, o[3] = t.w;
    } else {
        static_assert(VW == 2, "16-byte loads");
        const double2 t = __ldg(reinterpret_cast<const double2 *>(p));
        o[0] = t.x, o[1] = t.y;
    }
}

template <typename V, int KQ, int VW>
__global__ void __launch_bounds__(256)
long_spmm_kernel(const int32_t *__restrict__ rp, const int32_t *__restrict__ col, const V *__restrict__ val,
                 int32_t kc, const V *__restrict__ X, long long ldx, V *__restrict__ Y, long long ldy, V alpha,
                 V beta, const int32_t *__restrict__ long_rows, const int64_t *__restrict__ seg_begin,
                 int32_t num_long, int64_t num_segs, V *__restrict__ seg_partial, int32_t *__restrict__ arrivals) {
    constexpr int S = 32 / KQ;  // nonzeros per step
    static_assert(KQ * VW <= 32, "a segment partial holds at most 32 values");
    const int lane = threadIdx.x & 31, slot = lane / KQ, cq = lane % KQ;
    const int64_t sg = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (sg >= num_segs) return;
    int lo = 0, hi = num_long - 1;  // the long row holding segment sg
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (seg_begin[mid] <= sg) lo = mid;
        else hi = mid - 1;
    }
    const int32_t row = long_rows[lo];
    const int64_t first = seg_begin[lo];
    const int64_t nsegs = seg_begin[lo + 1] - first;
    const int32_t rb = rp[row], re = rp[row + 1];
    const int32_t b = rb + (int32_t)((sg - first) * kLongSegmentNnz);
    const int32_t e = min(b + kLongSegmentNnz, re);
    const int c0 = cq * VW;  // this lane's first column
    const bool use = c0 < kc;
    const V *xb = X + c0;
    V acc[VW];
#pragma unroll
    for (int v = 0; v < VW; ++v) acc[v] = V(0);
    // batches of 32 nonzeros: all of a batch's X row slices are requested
    // before any is used, and the next batch's columns and values load
    // meanwhile
    int c_n = b + lane < e ? ld_stream(col + b + lane) : 0;
    V v_n = b + lane < e ? ld_stream(val + b + lane) : V(0);
    for (int32_t k0 = b; k0 < e; k0 += 32) {
        const int n = min(32, e - k0);
        const int c_l = c_n;
        const V v_l = v_n;
        const int32_t k1 = k0 + 32;
        c_n = k1 + lane < e ? ld_stream(col + k1 + lane) : 0;
        v_n = k1 + lane < e ? ld_stream(val + k1 + lane) : V(0);
        V xr[KQ][VW], vs[KQ];
#pragma unroll
        for (int u = 0; u < KQ; ++u) {  // KQ steps of S nonzeros
            const int src = u * S + slot;
            const int c = __shfl_sync(0xffffffffu, c_l, src);
            const V v = __shfl_sync(0xffffffffu, v_l, src);
            const bool ok = src < n && use;
            vs[u] = ok ? v : V(0);
            if (ok) {
                ld_row_slice<V, VW>(xb + (int64_t)c * ldx, xr[u]);
            } else {
#pragma unroll
                for (int q = 0; q < VW; ++q) xr[u][q] = V(0);
            }
        }
#pragma unroll
        for (int u = 0; u < KQ; ++u)
#pragma unroll
            for (int q = 0; q < VW; ++q) acc[q] = fma(vs[u], xr[u][q], acc[q]);
    }
#pragma unroll
    for (int off = KQ; off < 32; off <<= 1)
#pragma unroll
        for (int q = 0; q < VW; ++q) acc[q] += __shfl_xor_sync(0xffffffffu, acc[q], off);
    V *yr = Y + (int64_t)row * ldy + c0;
    if (nsegs == 1) {
        if (slot == 0 && use) {
#pragma unroll
            for (int q = 0; q < VW; ++q) {
                V r = alpha * acc[q];
                if (beta != V(0)) r = fma(beta, yr[q], r);
                yr[q] = r;
            }
        }
        return;
    }
    if (slot == 0 && use) {
#pragma unroll
        for (int q = 0; q < VW; ++q) seg_partial[sg * 32 + c0 + q] = acc[q];
    }
    __threadfence();
    __syncwarp();
    int last = 0;
    if (lane == 0) {
        last = atomicAdd(arrivals + lo, 1) == (int)(nsegs - 1);
        if (last) __threadfence();
    }
    if (!__shfl_sync(0xffffffffu, last, 0)) return;
    if (slot == 0 && use) {
#pragma unroll
        for (int q = 0; q < VW; ++q) {
            V t = V(0);
            for (int64_t g = first; g < first + nsegs; ++g) t += __ldcg(seg_partial + g * 32 + c0 + q);
            V r = alpha * t;
            if (beta != V(0)) r = fma(beta, yr[q], r);
            yr[q] = r;
        }
    }
    if (lane == 0) arrivals[lo] = 0;  // ready for the next product
}

// The long-row kernel for one slice of kc <= 32 columns: 16-byte lanes when
// wide is set (X 16-byte aligned, kc and ldx multiples of the values per 16
// bytes), else one value per lane.
template <typename V>
cudaError_t launch_long_slice(const LongSpmmArgs &a, int32_t kc, const V *X, V *Y, bool wide, cudaStream_t stream) {
    constexpr int W = 16 / sizeof(V);
    const unsigned blocks = (unsigned)((a.num_segs + 7) / 8);
    const int groups = wide ? (kc + W - 1) / W : kc;
    const int kq = groups <= 1 ? 1 : groups <= 2 ? 2 : groups <= 4 ? 4 : groups <= 8 ? 8 : groups <= 16 ? 16 : 32;
#define LONG_SPMM(KQ, VW)                                                                                      \
    long_spmm_kernel<V, KQ, VW><<<blocks, 256, 0, stream>>>(                                                    \
        a.row_ptr, a.col_idx, static_cast<const V *>(a.vals), kc, X, a.ldx, Y, a.ldy, (V)a.alpha, (V)a.beta,    \
        a.long_rows, a.seg_begin, a.num_long, a.num_segs, static_cast<V *>(a.seg_partial), a.arrivals)
    if (wide) {
        switch (kq) {
        case 1: LONG_SPMM(1, W); break;
        case 2: LONG_SPMM(2, W); break;
        case 4: LONG_SPMM(4, W); break;
        case 8: LONG_SPMM(8, W); break;
        default:
            if constexpr (W == 2) LONG_SPMM(16, W);
            else return cudaErrorInvalidValue;  // not reached: kc <= 32 takes at most 8 lanes of four
        }
    } else {
        switch (kq) {
        case 1: LONG_SPMM(1, 1); break;
        case 2: LONG_SPMM(2, 1); break;
        case 4: LONG_SPMM(4, 1); break;
        case 8: LONG_SPMM(8, 1); break;
        case 16: LONG_SPMM(16, 1); break;
        default: LONG_SPMM(32, 1); break;
        }
    }
#undef LONG_SPMM
    return cudaGetLastError();
}

// LBCSR_LONG_SPMM_VEC=0 keeps one value per lane in the long-row SpMM
// kernel (tuning).
#ifndef LBCSR_LONG_SPMM_VEC
#define LBCSR_LONG_SPMM_VEC 1
#endif

template <typename V, int KC>
cudaError_t launch_slice(const RowSpmmArgs &a, const V *X, V *Y, cudaStream_t stream) {
    if (a.num_long > 0 && a.num_segs > 0) {
        // this path's X is 16-byte aligned, and KC and ldx are multiples of
        // the values per 16 bytes (row_spmm_supported)
        LongSpmmArgs l{};
        l.k = KC;
        l.row_ptr = a.row_ptr;
        l.col_idx = a.col_idx;
        l.vals = a.vals;
        l.ldx = a.ldx;
        l.ldy = a.ldy;
        l.alpha = a.alpha;
        l.beta = a.beta;
        l.long_rows = a.long_rows;
        l.seg_begin = a.seg_begin;
        l.num_long = a.num_long;
        l.num_segs = a.num_segs;
        l.seg_partial = a.seg_partial;
        l.arrivals = a.arrivals;
        const cudaError_t e = launch_long_slice<V>(l, KC, X, Y, LBCSR_LONG_SPMM_VEC != 0, stream);
        if (e != cudaSuccess) return e;
    }
    const int64_t warps = ((int64_t)a.m + 31) / 32;
    row_spmm_lines_kernel<V, KC><<<(unsigned)((warps + 7) / 8), 256, 0, stream>>>(
        a.m, a.row_ptr, a.col_idx, static_cast<const V *>(a.vals), X, a.ldx, Y, a.ldy, (V)a.alpha, (V)a.beta,
        a.num_long > 0 ? a.long_min : INT32_MAX);
    return cudaGetLastError();
}

template <typename V>
cudaError_t launch_typed(const RowSpmmArgs &a, cudaStream_t stream) {
    constexpr int W = 16 / sizeof(V);
    constexpr int KMAX = sizeof(V) == 8 ? 16 : 32;
    int32_t c0 = 0;
    while (c0 < a.k) {
        const int32_t rest = a.k - c0;
        int kc = KMAX;
        while (kc > rest) kc >>= 1;  // rest is a multiple of W, so kc stays >= W
        const V *X = static_cast<const V *>(a.X) + c0;
        V *Y = static_cast<V *>(a.Y) + c0;
        cudaError_t e;
        if (kc == KMAX) e = launch_slice<V, KMAX>(a, X, Y, stream);
        else if (kc >= 4 * W) e = launch_slice<V, 4 * W>(a, X, Y, stream);
        else if (kc >= 2 * W) e = launch_slice<V, 2 * W>(a, X, Y, stream);
        else e = launch_slice<V, W>(a, X, Y, stream);
        if (e != cudaSuccess) return e;
        c0 += kc;
    }
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_long_spmm(spmv_dtype_t dtype, const LongSpmmArgs &a, cudaStream_t stream) {
    if (a.num_long <= 0 || a.num_segs <= 0 || a.k <= 0) return cudaSuccess;
    const int64_t s = dtype == SPMV_F64 ? 8 : 4;
    const int64_t w = 16 / s;
    for (int32_t c0 = 0; c0 < a.k; c0 += 32) {
        const int32_t kc = a.k - c0 < 32 ? a.k - c0 : 32;
        const bool wide = LBCSR_LONG_SPMM_VEC && reinterpret_cast<uintptr_t>(a.X) % 16 == 0 && a.ldx % w == 0 &&
                          kc % w == 0;
        const cudaError_t e =
            dtype == SPMV_F64
                ? launch_long_slice<double>(a, kc, static_cast<const double *>(a.X) + c0,
                                            static_cast<double *>(a.Y) + c0, wide, stream)
                : launch_long_slice<float>(a, kc, static_cast<const float *>(a.X) + c0, static_cast<float *>(a.Y) + c0,
                                           wide, stream);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

bool row_spmm_supported(spmv_dtype_t dtype, int32_t k, const void *X, int64_t ldx, const void *Y, int64_t ldy) {
    const int64_t s = dtype == SPMV_F64 ? 8 : 4;
    const int64_t w = 16 / s;
    return k > 0 && k % w == 0 && reinterpret_cast<uintptr_t>(X) % 16 == 0 && reinterpret_cast<uintptr_t>(Y) % 16 == 0 &&
           (ldx * s) % 16 == 0 && (ldy * s) % 16 == 0;
}

cudaError_t launch_row_spmm(spmv_dtype_t dtype, const RowSpmmArgs &a, cudaStream_t stream) {
    if (a.m <= 0 || a.k <= 0) return cudaSuccess;
    return dtype == SPMV_F64 ? launch_typed<double>(a, stream) : launch_typed<float>(a, stream);
}

}  // namespace lbcsr
