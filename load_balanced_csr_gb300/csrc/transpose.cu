// The transpose of A in CSR form, built on the GPU by the plan, for the
// transposed product A^T x.  "A GPU load-balancing programming model"
// (section 4.1) names CSC among the formats its abstraction covers; A^T in
// CSR form is A in CSC form.  The transposed product then runs through the
// same plan machinery (statistics, kernel choice, schedule) as A x.
//
// The entries of A are sorted by column with a stable least-significant-
// digit radix sort (8 bits per pass, as many passes as the column count
// needs): each pass counts the digits of every tile of 4096 entries, a
// prefix sum over (digit, tile) gives every tile its place per digit, and
// each warp of a tile writes its entries in order, ranked among equal
// digits with __match_any_sync.  Stable passes keep A's order inside a
// column, so each column lists its rows in increasing order -- the same
// result every time.
#include <climits>

#include "internal.cuh"

namespace lbcsr {

namespace {

constexpr int kRadixThreads = 256;
constexpr int kRadixWarps = kRadixThreads / 32;
constexpr int kRadixPerWarp = 512;  // 16 rows of 32 entries
constexpr int kRadixTile = kRadixWarps * kRadixPerWarp;
constexpr int kRadixBins = 256;

__device__ __forceinline__ int digit_of(int key, int shift) { return (int)(((unsigned)key >> shift) & 0xffu); }

// hist[bin * tiles + tile] = number of entries of the tile with that digit
__global__ void __launch_bounds__(kRadixThreads)
radix_hist_kernel(const int32_t *__restrict__ keys, int64_t n, int shift, int64_t tiles, int64_t *__restrict__ hist) {
    __shared__ int h[kRadixBins];
    for (int b = threadIdx.x; b < kRadixBins; b += kRadixThreads) h[b] = 0;
    __syncthreads();
    const int64_t t0 = (int64_t)blockIdx.x * kRadixTile;
    for (int i = threadIdx.x; i < kRadixTile; i += kRadixThreads) {
        const int64_t q = t0 + i;
        if (q < n) atomicAdd(&h[digit_of(keys[q], shift)], 1);
    }
    __syncthreads();
    for (int b = threadIdx.x; b < kRadixBins; b += kRadixThreads) hist[(int64_t)b * tiles + blockIdx.x] = h[b];
}

// Stable scatter of one pass.  off[bin * tiles + tile]: where the tile's
// entries with that digit start.  src_idx == nullptr: the payload is the
// entry's own position.
__global__ void __launch_bounds__(kRadixThreads)
radix_scatter_kernel(const int32_t *__restrict__ keys, const int32_t *__restrict__ src_idx, int64_t n, int shift,
                     int64_t tiles, const int64_t *__restrict__ off, int32_t *__restrict__ out_keys,
                     int32_t *__restrict__ out_idx) {
    __shared__ int base[kRadixWarps][kRadixBins];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t w0 = (int64_t)blockIdx.x * kRadixTile + (int64_t)warp * kRadixPerWarp;
    for (int b = lane; b < kRadixBins; b += 32) base[warp][b] = 0;
    __syncwarp();
    // this warp's digit counts
    for (int r = 0; r < kRadixPerWarp; r += 32) {
        const int64_t q = w0 + r + lane;
        const bool in = q < n;
        const int d = in ? digit_of(keys[q], shift) : kRadixBins;  // past the end: a digit of its own
        const unsigned peers = __match_any_sync(0xffffffffu, d);
        if (in && lane == __ffs(peers) - 1) base[warp][d] += __popc(peers);
    }
    __syncthreads();
    // where each warp's entries of each digit start: the tile's offset plus
    // the earlier warps' counts
    for (int b = threadIdx.x; b < kRadixBins; b += kRadixThreads) {
        long long run = off[(int64_t)b * tiles + blockIdx.x];
        for (int w = 0; w < kRadixWarps; ++w) {
            const int c = base[w][b];
            base[w][b] = (int)run;  // positions fit int32: n < 2^31
            run += c;
        }
    }
    __syncthreads();
    // the entries, in order, each after the earlier ones with its digit
    const unsigned lt = (1u << lane) - 1u;
    for (int r = 0; r < kRadixPerWarp; r += 32) {
        const int64_t q = w0 + r + lane;
        const bool in = q < n;
        const int key = in ? keys[q] : 0;
        const int d = in ? digit_of(key, shift) : kRadixBins;
        const unsigned peers = __match_any_sync(0xffffffffu, d);
        if (in) {
            const int pos = base[warp][d] + __popc(peers & lt);
            out_keys[pos] = key;
            out_idx[pos] = src_idx ? src_idx[q] : (int32_t)q;
        }
        __syncwarp();
        if (in && lane == __ffs(peers) - 1) base[warp][d] += __popc(peers);
        __syncwarp();
    }
}

// row_of[q]: the row holding entry q (the last row whose start is <= q
// among the rows that are not empty), by binary search.
__global__ void __launch_bounds__(256)
entry_rows_kernel(int32_t m, int32_t nnz, const int32_t *__restrict__ rp, int32_t *__restrict__ row_of) {
    const int64_t q = (int64_t)blockIdx.x * 256 + threadIdx.x;
    if (q >= nnz) return;
    int lo = 0, hi = m - 1;  // the largest r with rp[r] <= q and rp[r + 1] > q
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (rp[mid] <= q) lo = mid;
        else hi = mid - 1;
    }
    row_of[q] = lo;
}

__global__ void __launch_bounds__(256)
column_counts_kernel(int32_t nnz, const int32_t *__restrict__ col, int64_t *__restrict__ counts) {
    const int64_t q = (int64_t)blockIdx.x * 256 + threadIdx.x;
    if (q < nnz) atomicAdd(reinterpret_cast<unsigned long long *>(counts + col[q]), 1ull);
}

__global__ void __launch_bounds__(256)
narrow_kernel(int64_t n, const int64_t *__restrict__ in, int32_t *__restrict__ out) {
    const int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x;
    if (i < n) out[i] = (int32_t)in[i];
}

template <typename V>
__global__ void __launch_bounds__(256)
gather_transposed_kernel(int32_t nnz, const int32_t *__restrict__ src, const int32_t *__restrict__ row_of,
                         const V *__restrict__ vals, int32_t *__restrict__ t_idx, V *__restrict__ t_vals) {
    const int64_t p = (int64_t)blockIdx.x * 256 + threadIdx.x;
    if (p >= nnz) return;
    const int32_t q = src[p];
    if (t_idx) t_idx[p] = row_of[q];
    t_vals[p] = vals[q];
}

unsigned blocks_for(int64_t n) { return (unsigned)((n + 255) / 256); }

}  // namespace

namespace {
// The scratch layout of launch_transpose, in order, each piece rounded up
// to 256 bytes.
int64_t round256(int64_t b) { return (b + 255) / 256 * 256; }
}  // namespace

int64_t transpose_scratch_bytes(int32_t n, int32_t nnz) {
    const int64_t tiles = ((int64_t)nnz + kRadixTile - 1) / kRadixTile;
    const int64_t hist_n = (int64_t)kRadixBins * (tiles > 0 ? tiles : 1);
    const int64_t scan_n = hist_n > (int64_t)n ? hist_n : (int64_t)n;
    return 5 * round256(4 * (int64_t)nnz) + round256(8 * hist_n) + round256(8 * (hist_n + 1)) +
           2 * round256(8 * ((int64_t)n + 1)) + round256(8 * scan_scratch_elems(scan_n));
}

cudaError_t launch_transpose(spmv_dtype_t dtype, int32_t m, int32_t n, int32_t nnz, const int32_t *row_ptr,
                             const int32_t *col_idx, const void *vals, void *scratch, int32_t *t_ptr,
                             int32_t *t_idx, void *t_vals, int32_t *t_src, cudaStream_t stream) {
    const int64_t tiles = ((int64_t)nnz + kRadixTile - 1) / kRadixTile;
    const int64_t hist_n = (int64_t)kRadixBins * (tiles > 0 ? tiles : 1);
    const int64_t scan_n = hist_n > (int64_t)n ? hist_n : (int64_t)n;
    char *s = static_cast<char *>(scratch);
    auto take = [&](size_t bytes) {
        char *r = s;
        s += (bytes + 255) / 256 * 256;
        return r;
    };
    int32_t *keys_a = reinterpret_cast<int32_t *>(take(4 * (size_t)nnz));
    int32_t *keys_b = reinterpret_cast<int32_t *>(take(4 * (size_t)nnz));
    int32_t *idx_a = reinterpret_cast<int32_t *>(take(4 * (size_t)nnz));
    int32_t *idx_b = reinterpret_cast<int32_t *>(take(4 * (size_t)nnz));
    int32_t *row_of = reinterpret_cast<int32_t *>(take(4 * (size_t)nnz));
    int64_t *hist = reinterpret_cast<int64_t *>(take(8 * (size_t)hist_n));
    int64_t *off = reinterpret_cast<int64_t *>(take(8 * (size_t)(hist_n + 1)));
    int64_t *counts = reinterpret_cast<int64_t *>(take(8 * ((size_t)n + 1)));
    int64_t *cptr = reinterpret_cast<int64_t *>(take(8 * ((size_t)n + 1)));
    int64_t *scan_scratch = reinterpret_cast<int64_t *>(take(8 * (size_t)scan_scratch_elems(scan_n)));

    cudaError_t e = cudaSuccess;
    // column pointers: counts, prefix sum
    e = cudaMemsetAsync(counts, 0, 8 * ((size_t)n + 1), stream);
    if (e == cudaSuccess && nnz > 0) {
        column_counts_kernel<<<blocks_for(nnz), 256, 0, stream>>>(nnz, col_idx, counts);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = launch_exclusive_scan(counts, n, cptr, scan_scratch, stream);
    if (e == cudaSuccess) {
        narrow_kernel<<<blocks_for((int64_t)n + 1), 256, 0, stream>>>((int64_t)n + 1, cptr, t_ptr);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess || nnz == 0) return e;
    // stable radix sort of the entries by column
    int bits = 0;
    while (bits < 31 && ((int64_t)1 << bits) < (int64_t)n) ++bits;
    const int passes = bits == 0 ? 1 : (bits + 7) / 8;
    const int32_t *kin = col_idx;
    const int32_t *iin = nullptr;
    int32_t *kout = keys_a, *iout = idx_a;
    for (int pass = 0; pass < passes && e == cudaSuccess; ++pass) {
        const int shift = 8 * pass;
        radix_hist_kernel<<<(unsigned)tiles, kRadixThreads, 0, stream>>>(kin, nnz, shift, tiles, hist);
        e = cudaGetLastError();
        if (e == cudaSuccess) e = launch_exclusive_scan(hist, hist_n, off, scan_scratch, stream);
        if (e == cudaSuccess) {
            radix_scatter_kernel<<<(unsigned)tiles, kRadixThreads, 0, stream>>>(kin, iin, nnz, shift, tiles, off, kout,
                                                                                iout);
            e = cudaGetLastError();
        }
        kin = kout;
        iin = iout;
        kout = kout == keys_a ? keys_b : keys_a;
        iout = iout == idx_a ? idx_b : idx_a;
    }
    if (e != cudaSuccess) return e;
    // the transposed arrays
    entry_rows_kernel<<<blocks_for(nnz), 256, 0, stream>>>(m, nnz, row_ptr, row_of);
    e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaMemcpyAsync(t_src, iin, 4 * (size_t)nnz, cudaMemcpyDeviceToDevice, stream);
    if (e == cudaSuccess) e = launch_transpose_values(dtype, nnz, t_src, row_of, vals, t_idx, t_vals, stream);
    return e;
}

cudaError_t launch_transpose_values(spmv_dtype_t dtype, int32_t nnz, const int32_t *t_src, const int32_t *row_of,
                                    const void *vals, int32_t *t_idx, void *t_vals, cudaStream_t stream) {
    if (nnz <= 0) return cudaSuccess;
    if (dtype == SPMV_F64)
        gather_transposed_kernel<double><<<blocks_for(nnz), 256, 0, stream>>>(
            nnz, t_src, row_of, static_cast<const double *>(vals), t_idx, static_cast<double *>(t_vals));
    else
        gather_transposed_kernel<float><<<blocks_for(nnz), 256, 0, stream>>>(
            nnz, t_src, row_of, static_cast<const float *>(vals), t_idx, static_cast<float *>(t_vals));
    return cudaGetLastError();
}

}  // namespace lbcsr
