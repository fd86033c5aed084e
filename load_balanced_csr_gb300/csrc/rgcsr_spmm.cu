// SpMM over the Row-grouped copy: Y = alpha * A * X + beta * Y for plans
// that hold the interleaved copy of A in groups of 32 rows ("New
// Row-grouped CSR format for storing the sparse matrices on GPU with
// implementation in CUDA", section 3); long rows, which the copy leaves
// out, are the long-row SpMM kernel's.  One thread per
// row, as in the Row-grouped SpMV kernel: at each level the warp reads its
// 32 rows' slots as one contiguous line, and every thread gathers its X row
// -- KC consecutive values, with 16-byte loads when X allows -- and keeps
// KC sums in registers.  Wider X is taken in slices of KC columns.  When a
// slice spans several 16-byte loads and X and Y are aligned, lanes share
// X rows instead (rg_spmm_lines_kernel), so that a load instruction touches
// a few lines, not 32.
#include <type_traits>

#include "internal.cuh"
#include "tma.cuh"

namespace lbcsr {

namespace {

using namespace tma;

constexpr int kLinesMinLanes = 4;  // lanes per X row from which rg_spmm_lines_kernel is used

template <typename V, int KC, bool VEC>
__global__ void __launch_bounds__(256)
rg_spmm_kernel(int32_t m, int32_t k, const int64_t *__restrict__ gp, const int32_t *__restrict__ row_len,
               const int32_t *__restrict__ perm, const int32_t *__restrict__ rg_col, const V *__restrict__ rg_val,
               const V *__restrict__ X, long long ldx, V *__restrict__ Y, long long ldy, V alpha, V beta) {
    constexpr int W = 16 / sizeof(V);  // values per 16-byte load
    const long long pos = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (pos >= m) return;
    const int len = ld_stream(row_len + pos);
    const long long row = perm ? perm[pos] : pos;
    const long long base = gp[pos >> 5] + (pos & 31);
    const uint64_t pol = l2_policy_evict_first();
    V acc[KC];
#pragma unroll
    for (int t = 0; t < KC; ++t) acc[t] = V(0);
    int c = len > 0 ? ld_stream(rg_col + base) : 0;
    V v = len > 0 ? ld_stream(rg_val + base) : V(0);
    for (int l = 0; l < len; ++l) {
        // the next level's slot while this one's X row is gathered
        int cn = 0;
        V vn = V(0);
        if (l + 1 < len) {
            cn = ld_stream(rg_col + base + (long long)(l + 1) * 32);
            vn = ld_stream(rg_val + base + (long long)(l + 1) * 32);
        }
        const V *xr = X + (long long)c * ldx;
        if (VEC) {
#pragma unroll
            for (int t = 0; t < KC; t += W) {
                if (sizeof(V) == 4) {
                    const float4 q = __ldg(reinterpret_cast<const float4 *>(xr + t));
                    acc[t] = fma(v, (V)q.x, acc[t]);
                    acc[t + 1] = fma(v, (V)q.y, acc[t + 1]);
                    acc[t + 2] = fma(v, (V)q.z, acc[t + 2]);
                    acc[t + 3] = fma(v, (V)q.w, acc[t + 3]);
                } else {
                    const double2 q = __ldg(reinterpret_cast<const double2 *>(xr + t));
                    acc[t] = fma(v, (V)q.x, acc[t]);
                    acc[t + 1] = fma(v, (V)q.y, acc[t + 1]);
                }
            }
        } else {
#pragma unroll
            for (int t = 0; t < KC; ++t)
                if (t < k) acc[t] = fma(v, ld_gather(xr + t), acc[t]);
        }
        c = cn;
        v = vn;
    }
    if (len < 0) return;  // (no long rows in plans that use this kernel)
    V *yr = Y + row * ldy;
#pragma unroll
    for (int t = 0; t < KC; ++t) {
        if (t < k) {
            V r = alpha * acc[t];
            if (beta != V(0)) r = fma(beta, yr[t], r);
            store_stream(yr + t, r, pol);
        }
    }
}

// The same product with the lanes of a warp sharing X rows: a warp per
// group of 32 rows; LPR = KC / (values per 16 bytes) lanes read one X row
// slice (LPR x 16 bytes), so one load instruction of the warp covers
// 32 / LPR rows and as many lines instead of 32.  Each lane loads its own
// row's slot of a level (one coalesced line per level) and the lanes that
// serve a row take its column and value by shuffles; a lane keeps KC sums
// (LPR rows x the values of one 16-byte load).  A row's levels past its
// own length are skipped, as in the thread-per-row kernel.  Needs X and Y
// 16-byte aligned row by row and k == KC.
template <typename V, int KC>
__global__ void __launch_bounds__(256)
rg_spmm_lines_kernel(int32_t m, int64_t ngroups, const int64_t *__restrict__ gp, const int32_t *__restrict__ row_len,
                     const int32_t *__restrict__ perm, const int32_t *__restrict__ rg_col,
                     const V *__restrict__ rg_val, const V *__restrict__ X, long long ldx, V *__restrict__ Y,
                     long long ldy, V alpha, V beta) {
    constexpr int W = 16 / sizeof(V);  // values per 16-byte load
    constexpr int LPR = KC / W;        // lanes per X row
    constexpr int RPI = 32 / LPR;      // rows per load instruction
    constexpr int J = LPR;             // load instructions per level
    using V4 = typename std::conditional<sizeof(V) == 4, float4, double2>::type;
    const int64_t g = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (g >= ngroups) return;
    const int lane = threadIdx.x & 31, sub = lane / LPR, cc = lane % LPR;
    const int64_t p0 = g * 32;
    const int len_own = p0 + lane < m ? ld_stream(row_len + p0 + lane) : 0;
    int lens[J];
#pragma unroll
    for (int j = 0; j < J; ++j) lens[j] = __shfl_sync(0xffffffffu, len_own, j * RPI + sub);
    const int64_t b0 = gp[g];
    const int levels = (int)((gp[g + 1] - b0) >> 5);
    V acc[J][W];
#pragma unroll
    for (int j = 0; j < J; ++j)
#pragma unroll
        for (int w = 0; w < W; ++w) acc[j][w] = V(0);
    int c_own = levels > 0 ? ld_stream(rg_col + b0 + lane) : 0;
    V v_own = levels > 0 ? ld_stream(rg_val + b0 + lane) : V(0);
    for (int l = 0; l < levels; ++l) {
        int cn = 0;
        V vn = V(0);
        if (l + 1 < levels) {  // the next level's slots while this one's X rows are gathered
            cn = ld_stream(rg_col + b0 + (int64_t)(l + 1) * 32 + lane);
            vn = ld_stream(rg_val + b0 + (int64_t)(l + 1) * 32 + lane);
        }
#pragma unroll
        for (int j = 0; j < J; ++j) {
            const int c = __shfl_sync(0xffffffffu, c_own, j * RPI + sub);
            const V v = __shfl_sync(0xffffffffu, v_own, j * RPI + sub);
            if (l < lens[j]) {
                const V4 q = __ldg(reinterpret_cast<const V4 *>(X + (int64_t)c * ldx + cc * W));
                if (sizeof(V) == 4) {
                    const float *f = reinterpret_cast<const float *>(&q);
#pragma unroll
                    for (int w = 0; w < W; ++w) acc[j][w] = fma(v, (V)f[w], acc[j][w]);
                } else {
                    const double *f = reinterpret_cast<const double *>(&q);
#pragma unroll
                    for (int w = 0; w < W; ++w) acc[j][w] = fma(v, (V)f[w], acc[j][w]);
                }
            }
        }
        c_own = cn;
        v_own = vn;
    }
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const int64_t pos = p0 + j * RPI + sub;
        if (pos >= m || lens[j] < 0) continue;  // (a long row is the long-row kernel's)
        const int64_t row = perm ? perm[pos] : pos;
        V *yr = Y + row * ldy + cc * W;
        V r[W];
#pragma unroll
        for (int w = 0; w < W; ++w) r[w] = alpha * acc[j][w];
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

template <typename V, int KC>
cudaError_t launch_kc(const RgSpmmArgs &a, int32_t k, const V *X, V *Y, cudaStream_t stream) {
    const unsigned blocks = (unsigned)(((int64_t)a.m + 255) / 256);
    // 16-byte loads need X 16-byte aligned row by row and a full slice
    const bool vec = k == KC && reinterpret_cast<uintptr_t>(X) % 16 == 0 && (a.ldx * (int64_t)sizeof(V)) % 16 == 0;
    constexpr int LPR = KC * (int)sizeof(V) / 16;
    // lanes share X rows from 4 lanes per row up (at 2, fp32 k = 8, the
    // thread-per-row kernel was faster: 174 against 195 us on the stencil)
    if (LPR >= kLinesMinLanes && vec && reinterpret_cast<uintptr_t>(Y) % 16 == 0 &&
        (a.ldy * (int64_t)sizeof(V)) % 16 == 0) {
        const int64_t ngroups = ((int64_t)a.m + 31) / 32;
        rg_spmm_lines_kernel<V, LPR >= kLinesMinLanes ? KC : kLinesMinLanes * 16 / (int)sizeof(V)><<<(unsigned)((ngroups + 7) / 8), 256, 0, stream>>>(
            a.m, ngroups, a.group_ptr, a.row_len, a.perm, a.rg_col, static_cast<const V *>(a.rg_val), X, a.ldx, Y,
            a.ldy, (V)a.alpha, (V)a.beta);
        return cudaGetLastError();
    }
    if (vec)
        rg_spmm_kernel<V, KC, true><<<blocks, 256, 0, stream>>>(
            a.m, k, a.group_ptr, a.row_len, a.perm, a.rg_col, static_cast<const V *>(a.rg_val), X, a.ldx, Y, a.ldy,
            (V)a.alpha, (V)a.beta);
    else
        rg_spmm_kernel<V, KC, false><<<blocks, 256, 0, stream>>>(
            a.m, k, a.group_ptr, a.row_len, a.perm, a.rg_col, static_cast<const V *>(a.rg_val), X, a.ldx, Y, a.ldy,
            (V)a.alpha, (V)a.beta);
    return cudaGetLastError();
}

template <typename V>
cudaError_t launch_rg_typed(const RgSpmmArgs &a, cudaStream_t stream) {
    constexpr int KMAX = sizeof(V) == 8 ? 16 : 32;  // columns per slice (registers)
    for (int32_t c0 = 0; c0 < a.k; c0 += KMAX) {
        const int32_t kc = a.k - c0 < KMAX ? a.k - c0 : KMAX;
        const V *X = static_cast<const V *>(a.X) + c0;
        V *Y = static_cast<V *>(a.Y) + c0;
        cudaError_t e;
        if (kc <= 4) e = launch_kc<V, 4>(a, kc, X, Y, stream);
        else if (kc <= 8) e = launch_kc<V, 8>(a, kc, X, Y, stream);
        else if (kc <= 16) e = launch_kc<V, 16>(a, kc, X, Y, stream);
        else e = launch_kc<V, KMAX>(a, kc, X, Y, stream);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_rg_spmm(spmv_dtype_t dtype, const RgSpmmArgs &a, cudaStream_t stream) {
    if (a.m <= 0 || a.k <= 0) return cudaSuccess;
    return dtype == SPMV_F64 ? launch_rg_typed<double>(a, stream) : launch_rg_typed<float>(a, stream);
}

}  // namespace lbcsr
