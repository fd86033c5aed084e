// SpMM over the Row-grouped copy: Y = alpha * A * X + beta * Y for plans
// that hold the interleaved copy of A in groups of 32 rows ("New
// Row-grouped CSR format for storing the sparse matrices on GPU with
// implementation in CUDA", section 3) and no long rows.  One thread per
// row, as in the Row-grouped SpMV kernel: at each level the warp reads its
// 32 rows' slots as one contiguous line, and every thread gathers its X row
// -- KC consecutive values, with 16-byte loads when X allows -- and keeps
// KC sums in registers.  Wider X is taken in slices of KC columns.
#include "internal.cuh"
#include "tma.cuh"

namespace lbcsr {

namespace {

using namespace tma;

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

template <typename V, int KC>
cudaError_t launch_kc(const RgSpmmArgs &a, int32_t k, const V *X, V *Y, cudaStream_t stream) {
    const unsigned blocks = (unsigned)(((int64_t)a.m + 255) / 256);
    // 16-byte loads need X 16-byte aligned row by row and a full slice
    const bool vec = k == KC && reinterpret_cast<uintptr_t>(X) % 16 == 0 && (a.ldx * (int64_t)sizeof(V)) % 16 == 0;
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
