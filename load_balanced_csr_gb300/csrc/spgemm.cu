// Sparse times sparse: C = A * B in CSR form, after OpSparse ("OpSparse: a
// highly optimized framework for sparse general matrix multiplication on
// GPUs"): the Gustavson row-by-row product, rows binned by their work
// (section 5.1: the number of products a row of C needs, counted first,
// rows placed into bins by two passes), a symbolic phase that sizes every
// row of C with hash tables in shared memory, one allocation of C by the
// caller, and a numeric phase that accumulates into the same tables and
// writes each row in increasing column order.
//
// Bins (products per row): <= 16 -- a thread per row keeping the row's
// columns in a sorted list in shared memory (no hashing, no sort, products
// added in order); <= 128 and <= 512 -- a warp per row with a hash table of
// 256 or 1024 slots; <= 1024, <= 2048, <= 4096 -- 128 or 256 threads per row
// with 2048, 4096 or 8192 slots; more -- a dense row of C in global memory
// (values and a bit per column), each row's products cut into equal pieces
// of at most 32768, a CTA per piece.
// The numeric phase re-bins the rows between those bounds by the entries the
// symbolic phase found, so that its tables fit the row, not its products.
// Tables use multiplicative hashing and linear probing and stay at most
// half full; the thread that claims a slot appends it to a list, so that
// after a row only the claimed slots are read (sorted by column by buckets,
// or a bitonic network) and cleared.
// Values in hash tables are added with atomics, so their summation order
// (and the last bits of a sum) may differ from run to run; the pattern of C
// does not.
#include <climits>

#include "spgemm.cuh"

namespace lbcsr {

namespace {

constexpr int kSgBins = kSpgemmBins;
constexpr int kSgChunk = 4096;  // rows per classification CTA

__host__ __device__ __forceinline__ int sg_bin(long long f) {
    return f <= 16 ? 0 : f <= 128 ? 1 : f <= 512 ? 2 : f <= 1024 ? 3 : f <= 2048 ? 4 : f <= 4096 ? 5 : 6;
}

// products[i] = sum over row i of A of the lengths of the rows of B it picks
__global__ void __launch_bounds__(256)
sg_products_kernel(int32_t m, const int32_t *__restrict__ a_ptr, const int32_t *__restrict__ a_col,
                   const int32_t *__restrict__ b_ptr, int64_t *__restrict__ products) {
    const long long i = ((long long)blockIdx.x * 256 + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (i >= m) return;
    long long s = 0;
    for (int p = a_ptr[i] + lane; p < a_ptr[i + 1]; p += 32) {
        const int q = a_col[p];
        s += b_ptr[q + 1] - b_ptr[q];
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0) products[i] = s;
}

// exclusive scan of one value per thread of a 256-thread CTA
__device__ long long sg_cta_scan(long long v, long long *total) {
    __shared__ long long s_w[8];
    __shared__ long long s_t;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    long long incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const long long t = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += t;
    }
    if (lane == 31) s_w[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const long long w = lane < 8 ? s_w[lane] : 0;
        long long wi = w;
#pragma unroll
        for (int off = 1; off < 8; off <<= 1) {
            const long long t = __shfl_up_sync(0xffffffffu, wi, off);
            if (lane >= off) wi += t;
        }
        if (lane < 8) s_w[lane] = wi - w;
        if (lane == 7) s_t = wi;
    }
    __syncthreads();
    const long long r = s_w[warp] + incl - v;
    *total = s_t;
    __syncthreads();
    return r;
}

// pass 1 of the binning: counts[b * chunks + c] = rows of chunk c in bin b
__global__ void __launch_bounds__(256)
sg_bin_count_kernel(int32_t m, const int64_t *__restrict__ products, int64_t chunks, int64_t *__restrict__ counts) {
    const long long r0 = (long long)blockIdx.x * kSgChunk;
    long long c[kSgBins];
#pragma unroll
    for (int b = 0; b < kSgBins; ++b) c[b] = 0;
    for (long long i = r0 + threadIdx.x; i < r0 + kSgChunk && i < m; i += 256) {
        const int bin = sg_bin(products[i]);
#pragma unroll
        for (int b = 0; b < kSgBins; ++b) c[b] += bin == b;
    }
#pragma unroll
    for (int b = 0; b < kSgBins; ++b) {
        long long t;
        sg_cta_scan(c[b], &t);
        if (threadIdx.x == 0) counts[(long long)b * chunks + blockIdx.x] = t;
    }
}

// pass 2: each chunk's rows of each bin at their places, in row order
__global__ void __launch_bounds__(256)
sg_bin_scatter_kernel(int32_t m, const int64_t *__restrict__ products, int64_t chunks,
                      const int64_t *__restrict__ offsets, int32_t *__restrict__ rows) {
    const long long r0 = (long long)blockIdx.x * kSgChunk;
    long long base[kSgBins];
#pragma unroll
    for (int b = 0; b < kSgBins; ++b) base[b] = offsets[(long long)b * chunks + blockIdx.x];
    for (long long i0 = r0; i0 < r0 + kSgChunk && i0 < m; i0 += 256) {
        const long long i = i0 + threadIdx.x;
        const int bin = i < m ? sg_bin(products[i]) : -1;
#pragma unroll
        for (int b = 0; b < kSgBins; ++b) {
            long long t;
            const long long rank = sg_cta_scan(bin == b ? 1 : 0, &t);
            if (bin == b) rows[base[b] + rank] = (int32_t)i;
            base[b] += t;
        }
    }
}

// Group-wide barrier: a warp (G = 32), the CTA (G = block size), or a
// named barrier per group of G threads.
template <int G, int GROUPS>
__device__ __forceinline__ void sg_sync(int grp) {
    if (G == 32) __syncwarp();
    else if (GROUPS == 1) __syncthreads();
    else asm volatile("bar.sync %0, %1;" ::"r"(grp + 1), "r"(G) : "memory");
}

// Bitonic sort by key, ascending, of n (a power of two) (key, payload)
// pairs by the G threads of a group.
template <int G, int GROUPS>
__device__ __forceinline__ void sg_sort(int *key, int *pay, int n, int t, int grp) {
    for (int k = 2; k <= n; k <<= 1)
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = t; i < n; i += G) {
                const int l = i ^ j;
                if (l > i) {
                    const bool up = (i & k) == 0;
                    const int ki = key[i], kl = key[l];
                    if ((ki > kl) == up) {
                        key[i] = kl;
                        key[l] = ki;
                        const int p = pay[i];
                        pay[i] = pay[l];
                        pay[l] = p;
                    }
                }
            }
            sg_sync<G, GROUPS>(grp);
        }
}

struct SgCsr {
    const int32_t *a_ptr, *a_col, *b_ptr, *b_col;
};

// The smallest rows (<= kSgListMax products): a thread per row.  The row's
// columns are kept in increasing order in a list in shared memory (slot j
// of thread t at j * blockDim + t), each product added to its column's
// entry in the order of the row's products, new columns inserted in place.
constexpr int kSgListMax = 16;

template <typename V, bool VALUES>
__global__ void __launch_bounds__(256)
sg_list_kernel(SgCsr mat, const V *__restrict__ a_val, const V *__restrict__ b_val, const int32_t *__restrict__ rows,
               int64_t nrows, int64_t *__restrict__ row_nnz, const int64_t *__restrict__ c_ptr,
               int32_t *__restrict__ c_col, V *__restrict__ c_val, int32_t *error) {
    __shared__ int sk[kSgListMax * 256];
    __shared__ V sv[VALUES ? kSgListMax * 256 : 1];
    const int t = threadIdx.x;
    for (long long w = (long long)blockIdx.x * 256 + t; w < nrows; w += (long long)gridDim.x * 256) {
        const int i = rows[w];
        int len = 0;
        for (int p = mat.a_ptr[i]; p < mat.a_ptr[i + 1]; ++p) {
            const int q = mat.a_col[p];
            const V av = VALUES ? a_val[p] : V(0);
            for (int r = mat.b_ptr[q]; r < mat.b_ptr[q + 1]; ++r) {
                const int c = mat.b_col[r];
                int pos = len;
                while (pos > 0 && sk[(pos - 1) * 256 + t] > c) --pos;
                if (pos > 0 && sk[(pos - 1) * 256 + t] == c) {
                    if (VALUES) sv[(pos - 1) * 256 + t] += av * b_val[r];
                    continue;
                }
                if (len == kSgListMax) {  // more products than the bin allows
                    atomicOr(error, 2);
                    continue;
                }
                for (int j = len; j > pos; --j) {
                    sk[j * 256 + t] = sk[(j - 1) * 256 + t];
                    if (VALUES) sv[j * 256 + t] = sv[(j - 1) * 256 + t];
                }
                sk[pos * 256 + t] = c;
                if (VALUES) sv[pos * 256 + t] = av * b_val[r];
                ++len;
            }
        }
        if (!VALUES) {
            row_nnz[i] = len;
        } else {
            const long long o = c_ptr[i], room = c_ptr[i + 1] - o;
            if (len != room) atomicOr(error, 2);
            for (int j = 0; j < len && j < room; ++j) {
                c_col[o + j] = sk[j * 256 + t];
                c_val[o + j] = sv[j * 256 + t];
            }
        }
    }
}

// The products of row i, by the G threads of a group (t = 0 .. G-1): the
// threads take the row's entries of A (consecutive entries go to different
// warps of the group), each walks a row of B of at most kSgAlone entries
// by itself, and longer rows of B are walked by the whole warp, one after
// the other.  fn(column, a * b) is called once per product.
constexpr int kSgAlone = 8;
constexpr int kSgCtaWalk = 1024;  // dense bin: rows of B walked by the whole CTA

template <int G, bool VALUES, typename V, typename Fn>
__device__ __forceinline__ void sg_walk_row(const SgCsr &mat, const V *__restrict__ a_val,
                                            const V *__restrict__ b_val, int i, int t, Fn &fn) {
    constexpr int W = G / 32;
    const int lane = t & 31, wg = t >> 5;
    const int a1 = mat.a_ptr[i + 1];
    for (int p0 = mat.a_ptr[i]; p0 < a1; p0 += G) {
        const int p = p0 + lane * W + wg;
        int b0 = 0, b1 = 0;
        V av = V(0);
        if (p < a1) {
            const int q = mat.a_col[p];
            b0 = mat.b_ptr[q];
            b1 = mat.b_ptr[q + 1];
            if (VALUES) av = a_val[p];
        }
        const bool alone = b1 - b0 <= kSgAlone;
        if (alone)
            for (int r = b0; r < b1; ++r) fn(mat.b_col[r], VALUES ? av * b_val[r] : V(0));
        for (unsigned todo = __ballot_sync(0xffffffffu, !alone); todo; todo &= todo - 1) {
            const int src = __ffs(todo) - 1;
            const int r0 = __shfl_sync(0xffffffffu, b0, src), r1 = __shfl_sync(0xffffffffu, b1, src);
            const V sav = __shfl_sync(0xffffffffu, av, src);
            for (int r = r0 + lane; r < r1; r += 32) fn(mat.b_col[r], VALUES ? sav * b_val[r] : V(0));
        }
    }
}

// Reductions and an exclusive scan over a group of G threads: a warp
// (G = 32), or the whole CTA (G > 32, one group per CTA; s_a and s_b hold
// one value per warp).
template <int G>
__device__ __forceinline__ void sg_group_minmax(unsigned &lo, unsigned &hi, unsigned *s_a, unsigned *s_b) {
    lo = __reduce_min_sync(0xffffffffu, lo);
    hi = __reduce_max_sync(0xffffffffu, hi);
    if (G == 32) return;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) {
        s_a[warp] = lo;
        s_b[warp] = hi;
    }
    __syncthreads();
#pragma unroll
    for (int q = 0; q < G / 32; ++q) {
        lo = min(lo, s_a[q]);
        hi = max(hi, s_b[q]);
    }
    __syncthreads();
}

// exclusive prefix sum of v over the group, and the group's largest v
template <int G>
__device__ __forceinline__ int sg_group_scan(int v, int &maxv, int *s_a, int *s_b) {
    const int lane = threadIdx.x & 31, warp = (threadIdx.x % G) >> 5;
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += u;
    }
    maxv = __reduce_max_sync(0xffffffffu, v);
    if (G == 32) return incl - v;
    if (lane == 31) s_a[warp] = incl;
    if (lane == 0) s_b[warp] = maxv;
    __syncthreads();
    int before = 0;
#pragma unroll
    for (int q = 0; q < G / 32; ++q) {
        if (q < warp) before += s_a[q];
        maxv = max(maxv, s_b[q]);
    }
    __syncthreads();
    return before + incl - v;
}

// Hash-table bins.  Symbolic (VALUES false: count the row's columns) or
// numeric (VALUES true: accumulate, then write the row sorted by column).
// A group of G threads per row, GROUPS groups per CTA, each with a table of
// TS slots (keys, and values when VALUES), a list of the slots claimed (at
// most TS / 2) and, for the sort, the sorted keys and slots and a bucket
// histogram of G counters.
//
// The sort: the group finds the row's smallest and largest column, counts
// the claimed keys into G buckets by where they fall in that range, and,
// after a prefix sum of the counts, scatters them to their buckets; each
// thread then sorts its own bucket by insertion (a few keys for columns
// spread over the range).  When a bucket would hold more than
// kSgBucketMax keys (columns clustered in a narrow part of the range) the
// group sorts with the bitonic network instead.
constexpr int kSgBucketMax = 48;

template <int TS, int G, bool VALUES>
__host__ __device__ constexpr size_t sg_group_smem(size_t vs) {
    return (size_t)TS * sizeof(int) + (size_t)(TS / 2) * sizeof(int) * (VALUES ? 3 : 1) +
           (VALUES ? G * sizeof(int) + TS * vs : 0);
}

template <typename V, int TS, int G, int GROUPS, bool VALUES>
__global__ void __launch_bounds__(G * GROUPS)
sg_hash_kernel(SgCsr mat, const V *__restrict__ a_val, const V *__restrict__ b_val, const int32_t *__restrict__ rows,
               int64_t nrows, int64_t *__restrict__ row_nnz, const int64_t *__restrict__ c_ptr,
               int32_t *__restrict__ c_col, V *__restrict__ c_val, int32_t *error) {
    constexpr int HALF = TS / 2;
    constexpr int kLog2TS = TS == 256 ? 8 : TS == 1024 ? 10 : TS == 2048 ? 11 : TS == 4096 ? 12 : 13;
    static_assert(1 << kLog2TS == TS, "table sizes are 256, 1024, 2048, 4096 or 8192");
    static_assert(G == 32 || GROUPS == 1, "groups wider than a warp fill the CTA");
    extern __shared__ __align__(16) unsigned char sg_smem[];
    __shared__ int s_count[GROUPS];
    __shared__ unsigned s_ua[8], s_ub[8];
    __shared__ int s_ia[8], s_ib[8];
    const int t = threadIdx.x % G;
    const int grp = threadIdx.x / G;
    // per group: vals [TS] (first, for alignment), keys [TS], slots [HALF],
    // sorted keys [HALF], sorted slots [HALF], bucket counters [G]
    unsigned char *base = sg_smem + (size_t)grp * sg_group_smem<TS, G, VALUES>(sizeof(V));
    V *vals = VALUES ? reinterpret_cast<V *>(base) : nullptr;
    int *keys = reinterpret_cast<int *>(base + (VALUES ? TS * sizeof(V) : 0));
    int *slot = keys + TS;
    int *skey = slot + HALF;
    int *sslot = skey + HALF;
    int *hist = sslot + HALF;
    int *count = s_count + grp;
    for (int s = t; s < TS; s += G) {
        keys[s] = -1;
        if (VALUES) vals[s] = V(0);
    }
    if (t == 0) *count = 0;
    __syncthreads();
    const long long stride = (long long)gridDim.x * GROUPS;
    // (the loop bound keeps every group of a CTA in the loop together)
    for (long long w = (long long)blockIdx.x * GROUPS + grp; w - grp < nrows; w += stride) {
        const bool live = w < nrows;
        const int i = live ? rows[w] : 0;
        if (live) {
            auto insert = [&](int c, V v) {
                // multiplicative (Fibonacci) hashing: the top bits of the product mix
                // every bit of the column; low bits would depend on its low bits only
                unsigned h = ((unsigned)c * 2654435761u) >> (32 - kLog2TS);
                for (int probe = 0; probe < TS; ++probe) {
                    const int old = atomicCAS(keys + h, -1, c);
                    if (old == -1) {
                        const int j = atomicAdd(count, 1);
                        if (j < HALF) slot[j] = (int)h;
                        else atomicOr(error, 2);
                    }
                    if (old == -1 || old == c) {
                        if (VALUES) atomicAdd(vals + h, v);
                        return;
                    }
                    h = (h + 1) & (TS - 1);
                }
                atomicOr(error, 2);
            };
            sg_walk_row<G, VALUES>(mat, a_val, b_val, i, t, insert);
        }
        sg_sync<G, GROUPS>(grp);
        const int claimed = *count;
        const int cnt = claimed < HALF ? claimed : HALF;
        if (!VALUES) {
            if (live && t == 0) row_nnz[i] = claimed;
        } else {
            // the row's column range, then a histogram over G buckets of it
            unsigned lo = 0xffffffffu, hi = 0u;
            for (int j = t; j < cnt; j += G) {
                const unsigned c = (unsigned)keys[slot[j]];
                lo = min(lo, c);
                hi = max(hi, c);
            }
            sg_group_minmax<G>(lo, hi, s_ua, s_ub);
            const unsigned long long span = cnt > 0 ? (unsigned long long)(hi - lo) + 1ull : 1ull;
            hist[t] = 0;
            sg_sync<G, GROUPS>(grp);
            for (int j = t; j < cnt; j += G) {
                const unsigned c = (unsigned)keys[slot[j]];
                atomicAdd(hist + (int)((unsigned long long)(c - lo) * G / span), 1);
            }
            sg_sync<G, GROUPS>(grp);
            const int mine = hist[t];
            int biggest;
            const int start = sg_group_scan<G>(mine, biggest, s_ia, s_ib);
            if (biggest <= kSgBucketMax) {
                hist[t] = start;  // the bucket's cursor
                sg_sync<G, GROUPS>(grp);
                for (int j = t; j < cnt; j += G) {
                    const int sl = slot[j];
                    const unsigned c = (unsigned)keys[sl];
                    const int pos = atomicAdd(hist + (int)((unsigned long long)(c - lo) * G / span), 1);
                    skey[pos] = (int)c;
                    sslot[pos] = sl;
                }
                sg_sync<G, GROUPS>(grp);
                for (int a = start + 1; a < start + mine; ++a) {  // insertion sort of my bucket
                    const int key = skey[a], sl = sslot[a];
                    int z = a - 1;
                    while (z >= start && skey[z] > key) {
                        skey[z + 1] = skey[z];
                        sslot[z + 1] = sslot[z];
                        --z;
                    }
                    skey[z + 1] = key;
                    sslot[z + 1] = sl;
                }
            } else {  // clustered columns: the bitonic network
                int pw = 1;
                while (pw < cnt) pw <<= 1;
                for (int j = t; j < pw; j += G) {
                    skey[j] = j < cnt ? keys[slot[j]] : INT_MAX;
                    sslot[j] = j < cnt ? slot[j] : 0;
                }
                sg_sync<G, GROUPS>(grp);
                sg_sort<G, GROUPS>(skey, sslot, pw, t, grp);
            }
            sg_sync<G, GROUPS>(grp);
            if (live) {
                const long long o = c_ptr[i], room = c_ptr[i + 1] - o;
                if (t == 0 && claimed != room) atomicOr(error, 2);
                for (int j = t; j < cnt && j < room; j += G) {
                    c_col[o + j] = skey[j];
                    c_val[o + j] = vals[sslot[j]];
                }
            }
            sg_sync<G, GROUPS>(grp);
        }
        // clear the claimed slots only
        for (int j = t; j < cnt; j += G) {
            keys[slot[j]] = -1;
            if (VALUES) vals[slot[j]] = V(0);
        }
        sg_sync<G, GROUPS>(grp);
        if (t == 0) *count = 0;
        sg_sync<G, GROUPS>(grp);
    }
}

// The dense bin (rows of more than 4096 products), balanced over the
// products as the merge-path schedule balances SpMV over rows and
// nonzeros.  Entry space: the entries of A of the dense rows, row after row
// (dense row j owns entries e_off[j] .. e_off[j+1]-1); pp[e] = the products
// of the entries before e (an exclusive prefix sum of the lengths of the
// rows of B they pick).  Each dense row's products are cut into pieces of
// at most kSgPiece, a CTA per piece; the rows of a wave share nothing, each
// has a slot: a dense row of C in global memory (values and a bit per
// column), into which the pieces add with reductions (no value returned,
// nothing waited for).  A second kernel then reads each row of the wave
// back in column order -- the symbolic phase counts it, the numeric phase
// writes it -- and clears what was used.
constexpr int64_t kSgPiece = 32768;
constexpr int kSgWordsPerThread = 16;                        // words of bits per thread when reading rows back
constexpr int64_t kSgSegCols = 256 * kSgWordsPerThread * 32;  // columns per segment (131072)

// alen[j] = length of dense row j of A
__global__ void __launch_bounds__(256)
sg_dense_alen_kernel(int64_t nrows, const int32_t *__restrict__ drows, const int32_t *__restrict__ a_ptr,
                     int64_t *__restrict__ alen) {
    const int64_t j = (int64_t)blockIdx.x * 256 + threadIdx.x;
    if (j < nrows) alen[j] = a_ptr[drows[j] + 1] - a_ptr[drows[j]];
}

// blen[e] = length of the row of B that entry e picks (a CTA per dense row)
__global__ void __launch_bounds__(256)
sg_dense_blen_kernel(const int32_t *__restrict__ drows, const int64_t *__restrict__ e_off,
                     const int32_t *__restrict__ a_ptr, const int32_t *__restrict__ a_col,
                     const int32_t *__restrict__ b_ptr, int64_t *__restrict__ blen) {
    const int64_t j = blockIdx.x;
    const int32_t p0 = a_ptr[drows[j]];
    const int64_t e0 = e_off[j], e1 = e_off[j + 1];
    for (int64_t e = e0 + threadIdx.x; e < e1; e += 256) {
        const int q = a_col[p0 + (e - e0)];
        blen[e] = b_ptr[q + 1] - b_ptr[q];
    }
}

// rowp[j] = pp[e_off[j]], j = 0 .. nrows
__global__ void __launch_bounds__(256)
sg_dense_rowp_kernel(int64_t nrows, const int64_t *__restrict__ e_off, const int64_t *__restrict__ pp,
                     int64_t *__restrict__ rowp) {
    const int64_t j = (int64_t)blockIdx.x * 256 + threadIdx.x;
    if (j <= nrows) rowp[j] = pp[e_off[j]];
}

// piece_e[c] = the entry holding the piece's first product: the last e in
// [0, E) with pp[e] <= piece_k0[c]
__global__ void __launch_bounds__(256)
sg_dense_locate_kernel(int64_t pieces, const int64_t *__restrict__ piece_k0, const int64_t *__restrict__ pp,
                       int64_t entries, int64_t *__restrict__ piece_e) {
    const int64_t c = (int64_t)blockIdx.x * 256 + threadIdx.x;
    if (c >= pieces) return;
    const int64_t k = piece_k0[c];
    int64_t lo = 0, hi = entries;  // pp[lo] <= k < pp[hi]
    while (hi - lo > 1) {
        const int64_t mid = lo + (hi - lo) / 2;
        if (pp[mid] <= k) lo = mid;
        else hi = mid;
    }
    piece_e[c] = lo;
}

struct SgDense {
    const int32_t *drows;  // dense rows of C (rows of A)
    const int64_t *e_off, *pp, *piece_k0, *piece_e;
    const int32_t *piece_row;
    int32_t n;
    int64_t words;         // words of bits per row, a multiple of kSgWordsPerThread
    unsigned *bits;
    void *vals;
    int64_t segs;          // segments per row
    int64_t *seg_cnt;      // [dense rows * segs]  columns per segment (symbolic)
    const int64_t *seg_off;// [dense rows * segs + 1]  their exclusive prefix sum
};

// One piece per CTA: products [piece_k0[c], piece_k0[c+1]) of dense row
// piece_row[c], added into the slot of that row (its index within the
// wave that starts at row j0).  Threads take entries (consecutive entries
// to different warps); a thread walks a range of at most kSgAlone
// products of a row of B by itself, the warp longer ones, the CTA ranges
// longer than kSgCtaWalk.
template <typename V, bool VALUES>
__global__ void __launch_bounds__(256)
sg_dense_accumulate_kernel(SgCsr mat, const V *__restrict__ a_val, const V *__restrict__ b_val, SgDense d,
                           int64_t c_begin, int64_t j0) {
    __shared__ int s_qn, s_q0[256], s_q1[256];
    __shared__ V s_qa[256];
    const int t = threadIdx.x, lane = t & 31;
    const int64_t c = c_begin + blockIdx.x;
    const int64_t j = d.piece_row[c];
    const int64_t slot = j - j0;
    const int64_t words = d.words;
    unsigned *bits = d.bits + slot * words;
    V *dense = VALUES ? static_cast<V *>(d.vals) + slot * d.n : nullptr;
    const int64_t k0 = d.piece_k0[c], k1 = d.piece_k0[c + 1];
    const int64_t e_row = d.e_off[j], e_end = d.e_off[j + 1];
    const int32_t p_row = mat.a_ptr[d.drows[j]];
    auto add = [&](int col, V v) {
        atomicOr(bits + (col >> 5), 1u << (col & 31));
        if (VALUES) atomicAdd(dense + col, v);
    };
    if (t == 0) s_qn = 0;
    __syncthreads();
    for (int64_t eb = d.piece_e[c]; eb < e_end && d.pp[eb] < k1; eb += 256) {
        const int64_t e = eb + lane * 8 + (t >> 5);
        int b0 = 0, b1 = 0;
        V av = V(0);
        if (e < e_end) {
            const int64_t pe = d.pp[e], pn = d.pp[e + 1];
            if (pe < k1 && pn > k0) {
                const int32_t p = p_row + (int32_t)(e - e_row);
                const int q = mat.a_col[p];
                const int rb = mat.b_ptr[q];
                b0 = rb + (int)((pe < k0 ? k0 : pe) - pe);
                b1 = rb + (int)((pn > k1 ? k1 : pn) - pe);
                if (VALUES) av = a_val[p];
            }
        }
        const int len = b1 - b0;
        const bool alone = len <= kSgAlone, by_cta = len > kSgCtaWalk;
        if (alone)
            for (int r = b0; r < b1; ++r) add(mat.b_col[r], VALUES ? av * b_val[r] : V(0));
        if (by_cta) {
            const int jq = atomicAdd(&s_qn, 1);
            s_q0[jq] = b0;
            s_q1[jq] = b1;
            s_qa[jq] = av;
        }
        for (unsigned todo = __ballot_sync(0xffffffffu, !alone && !by_cta); todo; todo &= todo - 1) {
            const int src = __ffs(todo) - 1;
            const int r0 = __shfl_sync(0xffffffffu, b0, src), r1 = __shfl_sync(0xffffffffu, b1, src);
            const V sav = __shfl_sync(0xffffffffu, av, src);
            for (int r = r0 + lane; r < r1; r += 32) add(mat.b_col[r], VALUES ? sav * b_val[r] : V(0));
        }
        if (__syncthreads_or(by_cta)) {  // (one barrier when no row of B is that long)
            const int nq = s_qn;
            for (int jq = 0; jq < nq; ++jq)
                for (int r = s_q0[jq] + t; r < s_q1[jq]; r += 256)
                    add(mat.b_col[r], VALUES ? s_qa[jq] * b_val[r] : V(0));
            __syncthreads();
            if (t == 0) s_qn = 0;
            __syncthreads();
        }
    }
}

// Reading the rows of a wave back: a CTA per segment of kSgSegCols
// columns of a row (d.segs segments per row; CTA b takes segment b % segs
// of the wave's row b / segs), a thread per kSgWordsPerThread consecutive
// words of bits (read as 16-byte loads), so that no thread has more than
// 32 * kSgWordsPerThread entries to handle however full the row is.
// Symbolic: count the segment's columns into seg_cnt and add them to
// row_nnz.  Numeric: write the columns and their values in order from the
// segment's offset (seg_off, an exclusive prefix sum of the symbolic counts
// over all segments).  Both clear the bits and values they read.
template <typename V, bool VALUES>
__global__ void __launch_bounds__(256)
sg_dense_finish_kernel(SgDense d, int64_t j0, int64_t *__restrict__ row_nnz, const int64_t *__restrict__ c_ptr,
                       int32_t *__restrict__ c_col, V *__restrict__ c_val, int32_t *error) {
    constexpr int WPT = kSgWordsPerThread;
    const int t = threadIdx.x;
    const int64_t slot = blockIdx.x / d.segs, seg = blockIdx.x % d.segs;
    const int64_t j = j0 + slot;
    const int i = d.drows[j];
    unsigned *bits = d.bits + slot * d.words;
    V *dense = VALUES ? static_cast<V *>(d.vals) + slot * d.n : nullptr;
    const int64_t q0 = seg * (kSgSegCols / 32) + (int64_t)t * WPT;  // my first word
    unsigned w[WPT];
    int cnt = 0;
    if (q0 + WPT <= d.words) {  // rows of bits are padded to a multiple of WPT words: 16-byte aligned
#pragma unroll
        for (int u = 0; u < WPT; u += 4) {
            const uint4 v4 = *reinterpret_cast<const uint4 *>(bits + q0 + u);
            w[u] = v4.x;
            w[u + 1] = v4.y;
            w[u + 2] = v4.z;
            w[u + 3] = v4.w;
        }
    } else {
#pragma unroll
        for (int u = 0; u < WPT; ++u) w[u] = q0 + u < d.words ? bits[q0 + u] : 0u;
    }
#pragma unroll
    for (int u = 0; u < WPT; ++u) cnt += __popc(w[u]);
    long long tot;
    const long long before = sg_cta_scan(cnt, &tot);
    const int64_t g = j * d.segs + seg;
    if (!VALUES) {
        if (t == 0) {
            d.seg_cnt[g] = tot;
            if (tot) atomicAdd(reinterpret_cast<unsigned long long *>(row_nnz + i), (unsigned long long)tot);
        }
    } else {
        const int64_t base = c_ptr[i] + (d.seg_off[g] - d.seg_off[j * d.segs]);
        const int64_t end = c_ptr[i + 1];
        int64_t o = base + before;
#pragma unroll
        for (int u = 0; u < WPT; ++u)
            for (unsigned b = w[u]; b;) {
                // up to four set bits at a time: four independent loads in flight
                int64_t cs[4];
                V vs[4];
                int nb = 0;
#pragma unroll
                for (int z = 0; z < 4; ++z)
                    if (b) {
                        cs[z] = (q0 + u) * 32 + __ffs(b) - 1;
                        b &= b - 1;
                        nb = z + 1;
                    }
#pragma unroll
                for (int z = 0; z < 4; ++z)
                    if (z < nb) vs[z] = dense[cs[z]];
#pragma unroll
                for (int z = 0; z < 4; ++z)
                    if (z < nb) {
                        if (o < end) {
                            c_col[o] = (int32_t)cs[z];
                            c_val[o] = vs[z];
                        } else {
                            atomicOr(error, 2);
                        }
                        dense[cs[z]] = V(0);
                        ++o;
                    }
            }
    }
#pragma unroll
    for (int u = 0; u < WPT; ++u)
        if (w[u]) bits[q0 + u] = 0u;
}

__global__ void __launch_bounds__(256)
sg_narrow_kernel(int64_t n, const int64_t *__restrict__ in, int32_t *__restrict__ out) {
    const int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x;
    if (i < n) out[i] = (int32_t)in[i];
}

unsigned sg_blocks(int64_t n) { return (unsigned)((n + 255) / 256); }

template <typename V, int TS, int G, int GROUPS, bool VALUES>
cudaError_t sg_launch_hash(const SgCsr &mat, const void *a_val, const void *b_val, const int32_t *rows, int64_t nrows,
                           int64_t *row_nnz, const int64_t *c_ptr, int32_t *c_col, void *c_val, int32_t *error,
                           cudaStream_t stream) {
    if (nrows <= 0) return cudaSuccess;
    const size_t smem = GROUPS * sg_group_smem<TS, G, VALUES>(sizeof(V));
    auto kern = sg_hash_kernel<V, TS, G, GROUPS, VALUES>;
    // set on every launch: the setting belongs to the current device
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, G * GROUPS, smem);
    if (e != cudaSuccess) return e;
    long long grid = (nrows + GROUPS - 1) / GROUPS;
    const long long cap = (long long)device_sm_count() * (per_sm > 0 ? per_sm : 1);
    if (grid > cap) grid = cap;
    kern<<<(unsigned)grid, G * GROUPS, smem, stream>>>(mat, static_cast<const V *>(a_val),
                                                       static_cast<const V *>(b_val), rows, nrows, row_nnz, c_ptr,
                                                       c_col, static_cast<V *>(c_val), error);
    return cudaGetLastError();
}

// One phase over the bins: the symbolic phase bins rows by products, the
// numeric phase by the entries the symbolic phase found (the dense bin and
// the list bin hold the same rows in both).
template <typename V, bool VALUES>
cudaError_t sg_phase(const SpgemmArgs &a, const void *a_val, const void *b_val, int32_t *c_col, void *c_val,
                     cudaStream_t stream) {
    const SgCsr mat{a.a_ptr, a.a_col, a.b_ptr, a.b_col};
    const int64_t *count = VALUES ? a.num_bin_count : a.bin_count;
    const int32_t *r[kSgBins];
    r[0] = VALUES ? a.num_bin_rows : a.bin_rows;
    for (int b = 1; b < kSgBins; ++b) r[b] = r[b - 1] + count[b - 1];
    cudaError_t e = cudaSuccess;
    if (count[0] > 0) {
        long long grid = (count[0] + 255) / 256;
        const long long cap = (long long)device_sm_count() * 4;
        if (grid > cap) grid = cap;
        sg_list_kernel<V, VALUES><<<(unsigned)grid, 256, 0, stream>>>(
            mat, static_cast<const V *>(a_val), static_cast<const V *>(b_val), r[0], count[0], a.row_nnz,
            a.c_ptr, c_col, static_cast<V *>(c_val), a.error);
        e = cudaGetLastError();
    }
#define SG_HASH(BIN, TS, G, GROUPS)                                                                              \
    if (e == cudaSuccess)                                                                                        \
        e = sg_launch_hash<V, TS, G, GROUPS, VALUES>(mat, a_val, b_val, r[BIN], count[BIN], a.row_nnz,           \
                                                     a.c_ptr, c_col, c_val, a.error, stream);
    SG_HASH(1, 256, 32, 8)
    SG_HASH(2, 1024, 32, 4)
    SG_HASH(3, 2048, 128, 1)
    SG_HASH(4, 4096, 256, 1)
    SG_HASH(5, 8192, 256, 1)
#undef SG_HASH
    const int64_t dense_rows = count[kSgBins - 1];
    if (e == cudaSuccess && dense_rows > 0) {
        const SgDense d{r[kSgBins - 1], a.dense_e_off, a.dense_pp, a.dense_piece_k0, a.dense_piece_e,
                        a.dense_piece_row, a.n, spgemm_bit_words(a.n), a.dense_bits, a.dense_vals,
                        a.dense_segs, a.dense_seg_cnt, a.dense_seg_off};
        for (int64_t w = 0; w < a.dense_waves && e == cudaSuccess; ++w) {
            const int64_t j0 = a.h_wave_row[w], j1 = a.h_wave_row[w + 1];
            const int64_t c0 = a.h_wave_piece[w], c1 = a.h_wave_piece[w + 1];
            sg_dense_accumulate_kernel<V, VALUES><<<(unsigned)(c1 - c0), 256, 0, stream>>>(
                mat, static_cast<const V *>(a_val), static_cast<const V *>(b_val), d, c0, j0);
            e = cudaGetLastError();
            if (e != cudaSuccess) break;
            sg_dense_finish_kernel<V, VALUES><<<(unsigned)((j1 - j0) * a.dense_segs), 256, 0, stream>>>(
                d, j0, a.row_nnz, a.c_ptr, c_col, static_cast<V *>(c_val), a.error);
            e = cudaGetLastError();
        }
    }
    return e;
}

}  // namespace

int64_t spgemm_chunks(int32_t m) {
    const int64_t c = ((int64_t)m + kSgChunk - 1) / kSgChunk;
    return c < 1 ? 1 : c;
}

int64_t spgemm_piece_products() { return kSgPiece; }

int64_t spgemm_segments(int32_t n) { return ((int64_t)n + kSgSegCols - 1) / kSgSegCols; }

int64_t spgemm_bit_words(int32_t n) {
    const int64_t w = ((int64_t)n + 31) / 32;
    return (w + kSgWordsPerThread - 1) / kSgWordsPerThread * kSgWordsPerThread;
}

cudaError_t launch_spgemm_dense_layout(const SpgemmArgs &a, const int32_t *drows, int64_t nrows, int64_t *alen,
                                       int64_t *e_off, int64_t *scan_scratch, cudaStream_t stream) {
    sg_dense_alen_kernel<<<sg_blocks(nrows), 256, 0, stream>>>(nrows, drows, a.a_ptr, alen);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) e = launch_exclusive_scan(alen, nrows, e_off, scan_scratch, stream);
    return e;
}

cudaError_t launch_spgemm_dense_products(const SpgemmArgs &a, const int32_t *drows, int64_t nrows,
                                         const int64_t *e_off, int64_t entries, int64_t *blen, int64_t *pp,
                                         int64_t *rowp, int64_t *scan_scratch, cudaStream_t stream) {
    sg_dense_blen_kernel<<<(unsigned)nrows, 256, 0, stream>>>(drows, e_off, a.a_ptr, a.a_col, a.b_ptr, blen);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) e = launch_exclusive_scan(blen, entries, pp, scan_scratch, stream);
    if (e == cudaSuccess) {
        sg_dense_rowp_kernel<<<sg_blocks(nrows + 1), 256, 0, stream>>>(nrows, e_off, pp, rowp);
        e = cudaGetLastError();
    }
    return e;
}

cudaError_t launch_spgemm_dense_locate(int64_t pieces, const int64_t *piece_k0, const int64_t *pp, int64_t entries,
                                       int64_t *piece_e, cudaStream_t stream) {
    if (pieces <= 0) return cudaSuccess;
    sg_dense_locate_kernel<<<sg_blocks(pieces), 256, 0, stream>>>(pieces, piece_k0, pp, entries, piece_e);
    return cudaGetLastError();
}

// Two-pass binning of rows 0 .. m-1 by key (sg_bin): counts per chunk and
// bin, one exclusive scan over [bin][chunk], then the rows of each bin in
// increasing order.
static cudaError_t sg_binning(int32_t m, const int64_t *key, int64_t *chunk_counts, int64_t *chunk_offsets,
                              int64_t *scan_scratch, int32_t *rows, cudaStream_t stream) {
    const int64_t chunks = spgemm_chunks(m);
    sg_bin_count_kernel<<<(unsigned)chunks, 256, 0, stream>>>(m, key, chunks, chunk_counts);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) e = launch_exclusive_scan(chunk_counts, kSgBins * chunks, chunk_offsets, scan_scratch, stream);
    if (e == cudaSuccess) {
        sg_bin_scatter_kernel<<<(unsigned)chunks, 256, 0, stream>>>(m, key, chunks, chunk_offsets, rows);
        e = cudaGetLastError();
    }
    return e;
}

cudaError_t launch_spgemm_analysis(const SpgemmArgs &a, int64_t *chunk_counts, int64_t *chunk_offsets,
                                   int64_t *scan_scratch, cudaStream_t stream) {
    if (a.m <= 0) return cudaSuccess;
    sg_products_kernel<<<sg_blocks((int64_t)a.m * 32), 256, 0, stream>>>(a.m, a.a_ptr, a.a_col, a.b_ptr, a.products);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) e = sg_binning(a.m, a.products, chunk_counts, chunk_offsets, scan_scratch, a.bin_rows, stream);
    return e;
}

// key of the numeric binning: the products for the list and dense bins,
// else the row's entries (at least 17, so that such rows stay out of the
// list bin)
__global__ void __launch_bounds__(256)
sg_numeric_key_kernel(int32_t m, const int64_t *__restrict__ products, const int64_t *__restrict__ c_ptr,
                      int64_t *__restrict__ key) {
    const int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x;
    if (i >= m) return;
    const int64_t p = products[i];
    const int64_t nnz = c_ptr[i + 1] - c_ptr[i];
    key[i] = (p <= 16 || p > 4096) ? p : (nnz < 17 ? 17 : nnz);
}

cudaError_t launch_spgemm_numeric_bins(const SpgemmArgs &a, int64_t *key, int64_t *chunk_counts,
                                       int64_t *chunk_offsets, int64_t *scan_scratch, int32_t *num_bin_rows,
                                       cudaStream_t stream) {
    if (a.m <= 0) return cudaSuccess;
    sg_numeric_key_kernel<<<sg_blocks(a.m), 256, 0, stream>>>(a.m, a.products, a.c_ptr, key);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) e = sg_binning(a.m, key, chunk_counts, chunk_offsets, scan_scratch, num_bin_rows, stream);
    return e;
}

cudaError_t launch_spgemm_symbolic(spmv_dtype_t dtype, const SpgemmArgs &a, int64_t *scan_scratch,
                                   cudaStream_t stream) {
    if (a.m <= 0) return cudaSuccess;
    cudaError_t e = dtype == SPMV_F64 ? sg_phase<double, false>(a, nullptr, nullptr, nullptr, nullptr, stream)
                                      : sg_phase<float, false>(a, nullptr, nullptr, nullptr, nullptr, stream);
    if (e == cudaSuccess) e = launch_exclusive_scan(a.row_nnz, a.m, a.c_ptr, scan_scratch, stream);
    const int64_t dense_segments = a.bin_count[kSgBins - 1] * a.dense_segs;
    if (e == cudaSuccess && dense_segments > 0)
        e = launch_exclusive_scan(a.dense_seg_cnt, dense_segments, a.dense_seg_off, a.dense_seg_scan, stream);
    return e;
}

cudaError_t launch_spgemm_numeric(spmv_dtype_t dtype, const SpgemmArgs &a, const void *a_val, const void *b_val,
                                  int32_t *c_row_ptr, int32_t *c_col, void *c_val, cudaStream_t stream) {
    if (a.m <= 0) {
        return c_row_ptr ? cudaMemsetAsync(c_row_ptr, 0, sizeof(int32_t), stream) : cudaSuccess;
    }
    cudaError_t e = dtype == SPMV_F64 ? sg_phase<double, true>(a, a_val, b_val, c_col, c_val, stream)
                                      : sg_phase<float, true>(a, a_val, b_val, c_col, c_val, stream);
    if (e == cudaSuccess && c_row_ptr) {
        sg_narrow_kernel<<<sg_blocks((int64_t)a.m + 1), 256, 0, stream>>>((int64_t)a.m + 1, a.c_ptr, c_row_ptr);
        e = cudaGetLastError();
    }
    return e;
}

}  // namespace lbcsr
