// Merge-path CSR SpMV: persistent warps over warp-sized tiles, with a fused
// carry-out fix-up.
//
// Schedule: "A GPU load-balancing programming model" (Osama, Porumbescu,
// Owens), section 5.2.1 -- every row end and every nonzero is one unit of
// work, the m + nnz units are split into equal tiles of T units, and each
// worker finds where its share starts by a search over (row ends, nonzero
// indices).  The plan computes the tile splits once (plan_kernels.cu).
//
// A tile here is T = 32 * IPL units and belongs to one warp.  Each warp owns
// a contiguous run of tiles (all tiles cost the same, so equal runs balance
// the GPU) and never waits for another warp.  Per tile it
//
//  1. has the tile's col_idx, vals and row ends row_ptr[i0+1 .. i1] copied
//     into its own shared-memory stage by the Tensor Memory Accelerator (one
//     bulk copy per array, issued by one lane, completion signalled on an
//     mbarrier) -- the next tile's copy is always in flight while the current
//     one is processed.  When beta != 0 the tile's slice of y comes along.
//     A copy must start and end on 16-byte boundaries: it is rounded out to
//     them wherever that stays inside the array, and only at an array's end
//     do lanes load the last few elements;
//  2. marks in a bitmap, for every row with a nonzero in the tile, the
//     position of its last one;
//  3. splits the tile's nonzeros over the 32 lanes in runs of Q = the odd
//     number nearest above nnz/32 (odd, so the lanes' shared-memory reads hit
//     distinct banks); each lane loads its run's values and gathers its x
//     values into registers through the read-only path -- all at once, and
//     before the bitmap is built, so their latency overlaps that work;
//  4. adds its run up in order (one fused multiply-add per nonzero) and,
//     where the bitmap marks a row's last nonzero, closes the row and keeps
//     its sum in that nonzero's slot (no other lane reads it).  Row ends cost
//     no floating-point work, so every lane of every warp-wide FMA does
//     useful work -- this matters on GB300, whose fp64 unit runs 2 lanes per
//     clock per SM and charges a warp instruction the same for 1 or 32
//     lanes;
//  5. a segmented warp scan adds the sum carried into each lane's first
//     closed row (it stops once every open segment has reached its start);
//     the sum still open at the tile's end is carried to the warp's next
//     tile in a register;
//  6. writes the finished rows to y, coalesced.  A row with no nonzero in
//     the tile contributes 0.
//
// Rows cut by the boundary between two warps' runs ("partial tiles" in the
// section) are finished without a second kernel and without any waiting:
// each warp holding part of such a row stores its partial sum, then counts
// itself in on the row's arrival counter; the warp that arrives last (the
// counter says how many to expect: the warps from the one holding the row's
// first nonzero to the one holding its end) adds the partials in warp order
// with a tree and writes y.  The order of the sum does not depend on which
// warp arrives last, so results are deterministic.  (The CUB implementation
// the paper compares with runs a separate fix-up step for these rows.)
#include <climits>
#include <cstdlib>

#include <atomic>

#include "internal.cuh"
#include "tma.cuh"

namespace lbcsr {

namespace {

using namespace tma;

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
// Copy stages per warp (stages_for below): 2 keeps the next tile's copy in
// flight while a tile is processed; 1 halves the shared memory, and the copy
// of tile t + 1 starts when tile t is done.  Shared memory is taken from the
// SM's L1, where the x gathers in flight live: measured on GB300, the random
// gathers slow down once more than about 96 KB per SM goes to shared memory
// (by 1.3x at 160 KB and 1.7x at 192 KB), so large tiles take one stage.
// LBCSR_MP_STAGES (1 or 2) overrides the choice at build time, for tuning.
template <typename V, int IPL>
__host__ __device__ constexpr int stage_bytes();
template <typename V, int IPL>
__host__ __device__ constexpr int stages_for() {
#ifdef LBCSR_MP_STAGES
    return LBCSR_MP_STAGES;
#else
    // fp32 with 24 items per lane is the banded case (the plan picks it for
    // matrices within n/64 of the diagonal): its gathers hit L1, so the
    // copy in flight pays (27-point stencil 128^3: 89 us with two stages,
    // 117 us with one)
    return (2 * stage_bytes<V, IPL>() <= 7168 || (sizeof(V) == 4 && IPL == 24)) ? 2 : 1;
#endif
}

template <typename V>
struct MPParams {
    int32_t m;
    int32_t n;  // columns (the debug build checks the gathers against it)
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
    long long num_tiles;  // P
    long long num_warps;  // W <= P: warps with a run of tiles
    V *tail_partial;      // per warp
    V *head_partial;      // per warp
    int32_t *arrivals;    // per warp, zero between products
    int32_t *error;       // bit 0 set if a copy never completed (may be null)
};

// One stage of a warp's shared memory, for a tile with n nonzeros and r row
// ends (n + r <= T):
//   col[ns] | val[ns] | row_ends[rs] | y_old[ys] (beta != 0 only) | bitmap
// ns = (sh + n + 4) & ~3 <= n + 7, rs and ys likewise <= r + 7 slots (sh and
// the other shifts < 4 align the 16-byte copies), bitmap (n + 31) / 32 + 2
// words.  With 4 + sizeof(V) bytes per nonzero and at most 4 + sizeof(V) per
// row this is bounded by:
template <typename V, int IPL>
__host__ __device__ constexpr int stage_bytes() {
    constexpr int T = 32 * IPL;
    constexpr int per_unit = sizeof(int) + sizeof(V);
    return ((per_unit * (T + 16) + 4 * (T / 32 + 16)) + 15) & ~15;
}
// A warp's region: two mbarriers (16 bytes), then its stages.
template <typename V, int IPL>
__host__ __device__ constexpr int warp_region_bytes() {
    return 16 + stages_for<V, IPL>() * stage_bytes<V, IPL>();
}

// Where a tile's arrays sit in its stage.
template <typename V>
struct StageView {
    int *col;      // col[k + sh]: the tile's nonzero k
    V *val;        // val[k + sh]
    int *re;       // re[r]: absolute end of row i0 + r
    V *yo;         // yo[r] = y[i0 + r] before the product (beta != 0)
    unsigned *bm;  // bitmap over the tile's nonzeros
};

template <typename V>
__device__ __forceinline__ StageView<V> stage_view(unsigned char *stage, int4 t, bool with_y) {
    const int i0 = t.x, j0 = t.y, i1 = t.z, j1 = t.w;
    const int ns = ((j0 & 3) + (j1 - j0) + 4) & ~3;
    const int rsh = (i0 + 1) & 3;
    const int rs = (rsh + (i1 - i0) + 4) & ~3;
    const int ysh = i0 & 3;
    const int ys = with_y ? (ysh + (i1 - i0) + 4) & ~3 : 0;
    StageView<V> v;
    v.col = reinterpret_cast<int *>(stage);
    v.val = reinterpret_cast<V *>(v.col + ns);
    int *re_raw = reinterpret_cast<int *>(v.val + ns);
    v.re = re_raw + rsh;
    V *y_raw = reinterpret_cast<V *>(re_raw + rs);
    v.yo = y_raw + ysh;
    v.bm = reinterpret_cast<unsigned *>(y_raw + ys);
    return v;
}

// The bulk-copied part of elements [b, e) of an array of n elements, b a
// multiple of 4: rounded up to a 16-byte boundary when that stays inside the
// array, else down (the few elements left are loaded by lanes).
__device__ __forceinline__ int bulk_end(int b, int e, long long n) {
    const int up = (e + 3) & ~3;
    return max(b, (long long)up <= n ? up : (e & ~3));
}

// Lanes tail_lane0.. load the elements [from, e) the bulk copy left out.
template <typename E>
__device__ __forceinline__ void stage_tail(E *dst, const E *src, int b, int from, int e, int lane, int tail_lane0) {
    const int t = lane - tail_lane0;
    if (t >= 0 && from + t < e) dst[from - b + t] = ld_stream(src + from + t);
}

// Start the copies of tile t into a stage.  Lane 0 first fences the generic
// proxy (lanes may have written this stage) against the asynchronous one,
// announces the bytes to the stage's barrier and issues one copy per array.
template <typename V, bool VEC>
__device__ __forceinline__ void issue_tile(const MPParams<V> &p, unsigned char *stage, uint64_t *bar, int4 t,
                                           int lane, uint64_t pol) {
    const bool with_y = p.mode & 2;
    const StageView<V> v = stage_view<V>(stage, t, with_y);
    const int i0 = t.x, j0 = t.y, i1 = t.z, j1 = t.w;
    const int base = j0 & ~3;
    const int rb = (i0 + 1) & ~3;
    const int yb = i0 & ~3;
    int *re_raw = v.re - ((i0 + 1) - rb);
    V *y_raw = v.yo - (i0 - yb);
    if (!VEC) {
        for (int q = base + lane; q < j1; q += 32) {
            v.col[q - base] = ld_stream(p.col_idx + q);
            v.val[q - base] = ld_stream(p.vals + q);
        }
        for (int q = rb + lane; q < i1 + 1; q += 32) re_raw[q - rb] = ld_stream(p.row_ptr + q);
        if (with_y)
            for (int q = yb + lane; q < i1; q += 32) y_raw[q - yb] = p.y[q];
        return;
    }
    const int ne = bulk_end(base, j1, p.nnz);
    const int re_end = bulk_end(rb, i1 + 1, (long long)p.m + 1);
    const int ye = with_y ? bulk_end(yb, i1, p.m) : yb;
    if (lane == 0) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        const uint32_t nb = (uint32_t)(ne - base), rbytes = 4u * (uint32_t)(re_end - rb);
        const uint32_t ybytes = (uint32_t)sizeof(V) * (uint32_t)(ye - yb);
        mbar_expect_tx(bar, nb * (4u + sizeof(V)) + rbytes + ybytes);
        if (nb) {
            bulk_copy(v.col, p.col_idx + base, 4u * nb, bar, pol);
            bulk_copy(v.val, p.vals + base, (uint32_t)sizeof(V) * nb, bar, pol);
        }
        if (rbytes) bulk_copy(re_raw, p.row_ptr + rb, rbytes, bar, pol);
        if (ybytes) bulk_copy(y_raw, p.y + yb, ybytes, bar, pol);
    }
    // elements past the last 16-byte boundary, only at an array's end
    if (ne < j1 || re_end < i1 + 1 || ye < (with_y ? i1 : yb)) {
        stage_tail<int>(v.col, p.col_idx, base, ne, j1, lane, 1);
        stage_tail<V>(v.val, p.vals, base, ne, j1, lane, 4);
        stage_tail<int>(re_raw, p.row_ptr, rb, re_end, i1 + 1, lane, 8);
        if (with_y) stage_tail<V>(y_raw, p.y, yb, ye, i1, lane, 12);
    }
}

__device__ __forceinline__ int4 tile_bounds(const int2 *part, long long t) {
    const int2 a = part[t];
    const int2 b = part[t + 1];
    return make_int4(a.x, a.y, b.x, b.y);
}

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
__device__ __forceinline__ V warp_sum(V v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

__device__ __forceinline__ long long warp_of_tile(long long t, long long P, long long W) {
    return ((t + 1) * W - 1) / P;  // warp w owns tiles [w*P/W, (w+1)*P/W)
}


// The tile's finished rows, written to y coalesced: row q's sum is in the
// slot of its last nonzero in the tile (a row with none there contributes 0,
// or the carried sum when it is the tile's first row).  MODE (bit 0: alpha
// != 1, bit 1: beta != 0) is fixed per launch; taking it as a template
// parameter keeps the alpha and beta arithmetic out of the loop when it is
// not needed.  Returns the first row's sum when that row is cut between
// warps (it is then finished by the cut-row protocol, not written here).
template <typename V, int MODE>
__device__ __forceinline__ V finish_rows(const MPParams<V> &p, const StageView<V> &sv, int i0, int j0, int nrows,
                                         int sh, V carry_row0, bool cut_head, int lane, uint64_t pol) {
    V head_val = V(0);
    for (int q = lane; q < nrows; q += 32) {
        const int e = sv.re[q] - j0;
        const int ep = q == 0 ? 0 : sv.re[q - 1] - j0;
        const V sum = e > ep ? sv.val[e - 1 + sh] : (q == 0 ? carry_row0 : V(0));
        if (q == 0 && cut_head) {
            head_val = sum;
        } else {
            V res = sum;
            if (MODE & 1) res = p.alpha * res;
            if (MODE & 2) res = fma(p.beta, sv.yo[q], res);
            store_stream(p.y + i0 + q, res, pol);
        }
    }
    return head_val;
}

// The tail partials of warps first .. last-1, summed in a fixed order whose
// depth grows with the logarithm of their number: chunks of 32 warps by a
// shuffle tree, the chunk sums pairwise by a binary counter (level k holds
// the sum of 2^k chunks).  A row cut across W warps then goes through at
// most 5 + 2 log2(W / 32) + 1 additions here (W < 2^17 for every size the
// interface accepts).
template <typename V>
__device__ __forceinline__ V sum_partials(const V *tail, long long first, long long last, int lane) {
    constexpr int kLevels = 16;  // up to 2^16 chunks of 32 warps
    V level[kLevels];
    unsigned occupied = 0;
    for (long long c = first; c < last; c += 32) {
        V s = c + lane < last ? __ldcg(tail + c + lane) : V(0);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
#pragma unroll
        for (int k = 0; k < kLevels; ++k) {
            if (occupied & (1u << k)) {
                s = level[k] + s;
                occupied &= ~(1u << k);
            } else {
                level[k] = s;
                occupied |= 1u << k;
                break;
            }
        }
    }
    V total = V(0);
#pragma unroll
    for (int k = 0; k < kLevels; ++k)
        if (occupied & (1u << k)) total = level[k] + total;
    return total;
}

// Cut rows: store this warp's partial, count in; the last to arrive adds all
// partials (warps first..last-1 as tails, warp last as head) and writes y.
// Called by the whole warp; `lane_with_value` holds the partial.
template <typename V>
__device__ void cut_row(const MPParams<V> &p, int lane, int lane_with_value, V partial, bool as_head, long long me,
                        int row, long long first, long long last) {
    int finisher = 0;
    if (lane == lane_with_value) {
        if (as_head) p.head_partial[me] = partial;
        else p.tail_partial[me] = partial;
        __threadfence();
        const int before = atomicAdd(p.arrivals + last, 1);
        finisher = before == (int)(last - first);
        if (finisher) __threadfence();
    }
    if (!__shfl_sync(0xffffffffu, finisher, lane_with_value)) return;
    V s = sum_partials(p.tail_partial, first, last, lane);
    if (lane == 0) {
        s += __ldcg(p.head_partial + last);
        p.y[row] = finish_row(s, p.alpha, p.beta, p.mode, p.y, row);
        p.arrivals[last] = 0;  // ready for the next product
    }
}

// Resident CTAs the register allocation must allow (0: the compiler's
// choice).  LBCSR_MP_FP64_MIN_CTAS and LBCSR_MP_FP32_MIN_CTAS set it for
// tiles of at most 12 items per lane, for tuning.
#ifndef LBCSR_MP_FP64_MIN_CTAS
#define LBCSR_MP_FP64_MIN_CTAS 0
#endif
#ifndef LBCSR_MP_FP32_MIN_CTAS
#define LBCSR_MP_FP32_MIN_CTAS 0
#endif
template <typename V, int IPL>
constexpr int min_ctas() {
    return IPL > 12 ? 0 : sizeof(V) == 8 ? LBCSR_MP_FP64_MIN_CTAS : LBCSR_MP_FP32_MIN_CTAS;
}

template <typename V, int IPL, bool VEC>
__global__ void __launch_bounds__(kThreads, min_ctas<V, IPL>())
merge_path_spmv_kernel(const MPParams<V> p) {
    constexpr int T = 32 * IPL;
    constexpr int kStages = stages_for<V, IPL>();
    static_assert(kStages == 1 || kStages == 2, "one or two stages");
    extern __shared__ __align__(16) unsigned char dsm[];

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const long long me = (long long)blockIdx.x * kWarps + warp;
    if (me >= p.num_warps) return;  // warps never wait for each other
    const long long P = p.num_tiles;
    const long long W = p.num_warps;
    const long long t_begin = me * P / W;
    const long long t_end = (me + 1) * P / W;  // non-empty: W <= P
    unsigned char *region = dsm + (size_t)warp * warp_region_bytes<V, IPL>();
    uint64_t *bars = reinterpret_cast<uint64_t *>(region);
    unsigned char *stages = region + 16;
    const uint64_t stream_pol = l2_policy_evict_first();
    const uint64_t x_pol = l2_policy_evict_last();
    if (VEC) {
        if (lane == 0) {
            mbar_init(bars);
            mbar_init(bars + 1);
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        }
        __syncwarp();
    }

    // the warp's run starts inside a row whose beginning belongs to an earlier warp
    const int4 first_tile = tile_bounds(p.part, t_begin);
    bool head_pending = first_tile.x < p.m && p.row_ptr[first_tile.x] < first_tile.y;

    int4 cur = first_tile;
    int4 nxt = make_int4(0, 0, 0, 0);
    issue_tile<V, VEC>(p, stages, bars, cur, lane, stream_pol);
    if (kStages == 2 && t_begin + 1 < t_end) {
        nxt = tile_bounds(p.part, t_begin + 1);
        issue_tile<V, VEC>(p, stages + stage_bytes<V, IPL>(), bars + 1, nxt, lane, stream_pol);
    }

    const bool with_y = p.mode & 2;
    V carry = V(0);  // sum of the row open at the previous tile's end
    // tiles that lie inside one row (no row end) leave their sums in the
    // lanes, one per lane, and skip the scan
    V lane_part = V(0);
    bool parts_pending = false;
    for (long long t = t_begin; t < t_end; ++t) {
        const int s = kStages == 2 ? (int)((t - t_begin) & 1) : 0;
        unsigned char *stage = stages + s * stage_bytes<V, IPL>();
        const int i0 = cur.x, j0 = cur.y, i1 = cur.z, j1 = cur.w;
        const int nrows = i1 - i0;
        const int nnzt = j1 - j0;
        const int sh = j0 & 3;
        const StageView<V> sv = stage_view<V>(stage, cur, with_y);
        const int nwords = (nnzt + 31) >> 5;
        // bounds of the tile that goes into this stage next (load early)
        const int4 after = t + kStages < t_end ? tile_bounds(p.part, t + kStages) : cur;

        if (VEC) {  // this tile's copies are done (the next tile's may not be)
            const uint32_t parity = (uint32_t)(((t - t_begin) / kStages) & 1);
            const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(bars + s, parity));
            if (!ok) {  // a copy never completed: report it and stop this warp
                if (lane == 0 && p.error) atomicOr(p.error, 1);
                mbar_wait_bounded(bars + s, parity);
                if (kStages == 2 && t + 1 < t_end)
                    mbar_wait_bounded(bars + (s ^ 1), (uint32_t)(((t + 1 - t_begin) >> 1) & 1));
                return;
            }
        }
        __syncwarp();  // the lanes' tail loads are visible too

        // ---- values and x into registers.  A tile with row ends splits its
        // nonzeros into lane runs [k0, k0 + run) of Q consecutive ones (Q
        // odd, so the lanes' shared-memory reads hit distinct banks).  A tile
        // that lies inside one row may split them any way: it takes them
        // interleaved (nonzero lane + 32 i), so that the gathers of a row
        // with dense columns share cache lines.
        const bool inside = nrows == 0;
        const int Q = ((nnzt + 31) >> 5) | 1;
        const int k0 = min(lane * Q, nnzt);
        const int run = min(Q, nnzt - k0);
        const int steps = inside ? (nnzt + 31) >> 5 : Q;  // the same for all lanes
        V xr[IPL + 1], vr[IPL + 1];
        if (inside) {
            const int *c = sv.col + sh + lane;
            const V *w = sv.val + sh + lane;
#pragma unroll
            for (int i = 0; i <= IPL; ++i) {
                if (sizeof(V) == 8 && i >= steps) break;
                const bool in = i * 32 + lane < nnzt;
                xr[i] = in ? gather_keep(p.x + debug_col(c[i * 32], p.n, p.error), x_pol) : V(0);
                vr[i] = in ? w[i * 32] : V(0);
            }
        } else {
            const int *c = sv.col + sh + k0;
            const V *w = sv.val + sh + k0;
#pragma unroll
            for (int i = 0; i <= IPL; ++i) {
                if (sizeof(V) == 8 && i >= Q) break;
                xr[i] = i < run ? gather_keep(p.x + debug_col(c[i], p.n, p.error), x_pol) : V(0);
                vr[i] = i < run ? w[i] : V(0);
            }
        }
        if (inside) {
            // the lanes keep their shares; they join the carry once, when a
            // row end or the end of the run comes
            V acc = V(0);
#pragma unroll
            for (int i = 0; i <= IPL; ++i) {
                if (sizeof(V) == 8 && i >= steps) break;
                acc = fma(vr[i], xr[i], acc);
            }
            lane_part += acc;
            parts_pending = true;
        } else {
        // lanes past the tile's last nonzero take no part (lane 0 always
        // does: it brings the carried sum)
        const unsigned holding = __ballot_sync(0xffffffffu, run > 0);
        const int last_lane = holding ? 31 - __clz(holding) : 0;
        if (parts_pending) {
            carry += warp_sum(lane_part);
            lane_part = V(0);
            parts_pending = false;
        }
        // ---- mark each row's last nonzero in the tile (while the gathers fly)
        for (int w = lane; w < nwords + 2; w += 32) sv.bm[w] = 0u;
        __syncwarp();
        // The carried sum belongs to row i0.  If that row ends before the
        // tile's first nonzero, it takes the carry and nothing flows on.
        const bool row0_ends_first = sv.re[0] == j0;
        const V carry_row0 = row0_ends_first ? carry : V(0);
        if (row0_ends_first) carry = V(0);
        for (int r = lane; r < nrows; r += 32) {
            const int e = sv.re[r] - j0;
            const int ep = r == 0 ? 0 : sv.re[r - 1] - j0;
            if (e > ep) atomicOr(sv.bm + ((e - 1) >> 5), 1u << ((e - 1) & 31));
        }
        __syncwarp();
        // bit i of `bits`: nonzero k0 + i is the last of a row in this tile
        // (Q <= 33 and only the run's bits are kept)
        const unsigned long long two = ((unsigned long long)sv.bm[(k0 >> 5) + 1] << 32) | sv.bm[k0 >> 5];
        const unsigned long long shifted = two >> (k0 & 31);
        const unsigned long long run_mask = run >= 64 ? ~0ull : ((1ull << run) - 1);
        const unsigned long long bits = shifted & run_mask;

        // ---- add the run up.  Lane 0 starts from the carried sum.  A closed
        // row's sum goes to the slot of its last nonzero, which no other lane
        // touches.  fp64 keeps a lane's first closed row in a register
        // instead (it still lacks the sum carried in from earlier lanes), so
        // that the carry is added once, in registers; fp32, whose walk runs
        // fully predicated, keeps the walk short and adds the carry to the
        // slot afterwards.
        V acc = lane == 0 ? carry : V(0);
        V first_sum = V(0);
        bool closed = false;
#pragma unroll
        for (int i = 0; i <= IPL; ++i) {
            // fp64: every warp-wide FMA costs the fp64 unit the same, so stop
            // at Q (the same for all lanes); fp32 runs fully predicated
            if (sizeof(V) == 8 && i >= Q) break;
            acc = fma(vr[i], xr[i], acc);  // vr[i] = 0 past the run
            if ((bits >> i) & 1ull) {
                if (sizeof(V) == 4 || closed) sv.val[k0 + i + sh] = acc;
                else first_sum = acc;
                closed = true;
                acc = V(0);
            }
        }
        const int first_pos = bits ? k0 + (__ffsll((long long)bits) - 1) : -1;
        if (sizeof(V) == 4 && first_pos >= 0) first_sum = sv.val[first_pos + sh];

        // ---- segmented inclusive scan of (row closed, running sum) over the
        // lanes that hold nonzeros; lane last_lane ends with the open sum
        V v = lane <= last_lane ? acc : V(0);
        int f = first_pos >= 0 || lane > last_lane;
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
        const V carry_in = __shfl_up_sync(0xffffffffu, v, 1);
        if (first_pos >= 0) sv.val[first_pos + sh] = lane == 0 ? first_sum : carry_in + first_sum;
        carry = __shfl_sync(0xffffffffu, v, last_lane);
        __syncwarp();

        // ---- finished rows; the warp's first row end may be a cut row
        const bool cut_head = head_pending;
        V head_val = V(0);
        switch (p.mode) {
        case 0: head_val = finish_rows<V, 0>(p, sv, i0, j0, nrows, sh, carry_row0, cut_head, lane, stream_pol); break;
        case 1: head_val = finish_rows<V, 1>(p, sv, i0, j0, nrows, sh, carry_row0, cut_head, lane, stream_pol); break;
        case 2: head_val = finish_rows<V, 2>(p, sv, i0, j0, nrows, sh, carry_row0, cut_head, lane, stream_pol); break;
        default: head_val = finish_rows<V, 3>(p, sv, i0, j0, nrows, sh, carry_row0, cut_head, lane, stream_pol);
        }
        if (cut_head) {
            head_pending = false;
            const long long first = warp_of_tile(((long long)p.row_ptr[i0] + i0) / T, P, W);
            cut_row<V>(p, lane, 0, head_val, true, me, i0, first, me);
        }
        }  // nrows > 0
        __syncwarp();  // this stage may now be refilled

        // ---- tile t + kStages goes into this stage
        if (kStages == 2) {
            cur = nxt;
            if (t + 2 < t_end) {
                nxt = after;
                issue_tile<V, VEC>(p, stage, bars + s, nxt, lane, stream_pol);
            }
        } else {
            cur = after;
            if (t + 1 < t_end) issue_tile<V, VEC>(p, stage, bars + s, cur, lane, stream_pol);
        }
    }

    if (parts_pending) carry += warp_sum(lane_part);
    // ---- the row open at the end of the warp's run, if it has nonzeros here
    const int4 last_tile = tile_bounds(p.part, t_end - 1);
    const int ie = last_tile.z, je = last_tile.w;
    if (ie < p.m) {
        const int32_t rp_ie = p.row_ptr[ie];
        if (je > max(rp_ie, first_tile.y)) {
            const long long first = warp_of_tile(((long long)rp_ie + ie) / T, P, W);
            const long long last = warp_of_tile(((long long)p.row_ptr[ie + 1] + ie) / T, P, W);
            cut_row<V>(p, lane, 0, carry, false, me, ie, first, last);
        }
    }
}

// occupancy per (type, IPL, VEC, device); 0 until first computed.  Host
// threads may fill an entry at the same time: they compute the same value.
std::atomic<int> g_ctas_per_sm[2][33][2][64];

// Tuning override of the CTAs per SM (SPMV_MP_CTAS_PER_SM, 0 = as many as
// fit), read once.
int ctas_per_sm_override() {
    static const int v = [] {
        const char *s = getenv("SPMV_MP_CTAS_PER_SM");
        return s ? atoi(s) : 0;
    }();
    return v;
}

// CTAs of the kernel per SM (cached per device), with its attributes set:
// as many as fit, and the rest of the SM's storage left to L1.
template <typename V, int IPL, bool VEC>
cudaError_t ctas_per_sm(int &out) {
    constexpr size_t smem = (size_t)kWarps * warp_region_bytes<V, IPL>();
    int dev = 0;
    cudaGetDevice(&dev);
    std::atomic<int> &cached = g_ctas_per_sm[sizeof(V) == 8][IPL][VEC][dev & 63];
    int per_sm = cached.load(std::memory_order_acquire);
    if (per_sm == 0) {
        cudaError_t e = cudaFuncSetAttribute(merge_path_spmv_kernel<V, IPL, VEC>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        int nb = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, merge_path_spmv_kernel<V, IPL, VEC>, kThreads, smem);
        if (e != cudaSuccess) return e;
        int want = nb > 0 ? nb : 1;
        if (ctas_per_sm_override() > 0 && ctas_per_sm_override() < want) want = ctas_per_sm_override();
        // leave the rest of the SM's storage to L1, where the x gathers in
        // flight live
        const int pct = carveout_percent(want, smem);
        if (pct >= 0) {
            e = cudaFuncSetAttribute(merge_path_spmv_kernel<V, IPL, VEC>,
                                     cudaFuncAttributePreferredSharedMemoryCarveout, pct);
            if (e != cudaSuccess) return e;
        }
        per_sm = want;
        cached.store(want, std::memory_order_release);
    }
    out = per_sm;
    return cudaSuccess;
}

// Warps with a run of tiles: one per tile, as many as the GPU holds at once,
// and more (queued behind the first wave; warps never wait for each other)
// when a run would otherwise exceed max_run(IPL) tiles -- so that the sum of
// a long row stays shallow at every size the interface accepts.  A term of
// a row's sum passes, at most, through: the FMA chain of its lane (Q <= IPL
// + 1), one addition per later tile of the run (K), the warp's tree (5), the
// carry into the next tile's lane 0 and that lane's chain (1 + Q), the scan
// (5), the pairwise sum over the warps the row spans (5 + 2 * 12 + 1), and
// alpha and beta (2): 2 Q + K + 43 roundings.  With K <= 120 - 2 (IPL + 1)
// that is at most 163, and 163 * 2^-24 < 1e-5, the fp32 accuracy bound (for
// fp64, 163 * 2^-53 is far below 1e-13).  At most cap warps when cap > 0.
long long max_run(int ipl) { return 120 - 2 * (ipl + 1); }
long long warps_for(long long num_tiles, int per_sm, int ipl, int64_t cap) {
    const long long max_warps = (long long)per_sm * device_sm_count() * kWarps;
    long long w = num_tiles < max_warps ? num_tiles : max_warps;
    const long long run = max_run(ipl);
    if (num_tiles > w * run) w = (num_tiles + run - 1) / run;
    if (cap > 0 && w > cap) w = cap;
    return w;
}

template <typename V, int IPL, bool VEC>
cudaError_t launch_typed(const MergePathArgs &a, cudaStream_t stream) {
    if (a.num_tiles <= 0) return cudaSuccess;
    constexpr size_t smem = (size_t)kWarps * warp_region_bytes<V, IPL>();
    int per_sm = 0;
    cudaError_t e = ctas_per_sm<V, IPL, VEC>(per_sm);
    if (e != cudaSuccess) return e;
    MPParams<V> p;
    p.m = a.m;
    p.n = a.n;
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
    p.num_tiles = a.num_tiles;
    p.num_warps = warps_for(a.num_tiles, per_sm, IPL, a.max_warps);
    p.tail_partial = static_cast<V *>(a.tail_partial);
    p.head_partial = static_cast<V *>(a.head_partial);
    p.arrivals = a.arrivals;
    p.error = a.error;
    const unsigned grid = (unsigned)((p.num_warps + kWarps - 1) / kWarps);
    merge_path_spmv_kernel<V, IPL, VEC><<<grid, kThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

template <typename V, bool VEC>
cudaError_t launch_ipl(int ipl, const MergePathArgs &a, cudaStream_t stream) {
    switch (ipl) {
    case 8: return launch_typed<V, 8, VEC>(a, stream);
    case 12: return launch_typed<V, 12, VEC>(a, stream);
    case 16: return launch_typed<V, 16, VEC>(a, stream);
    case 24: return launch_typed<V, 24, VEC>(a, stream);
    case 32: return launch_typed<V, 32, VEC>(a, stream);
    default: return cudaErrorInvalidValue;
    }
}

template <typename V, bool VEC>
cudaError_t ctas_ipl(int ipl, int &out) {
    switch (ipl) {
    case 8: return ctas_per_sm<V, 8, VEC>(out);
    case 12: return ctas_per_sm<V, 12, VEC>(out);
    case 16: return ctas_per_sm<V, 16, VEC>(out);
    case 24: return ctas_per_sm<V, 24, VEC>(out);
    case 32: return ctas_per_sm<V, 32, VEC>(out);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

int64_t merge_path_num_warps(spmv_dtype_t dtype, int ipl, bool aligned, int64_t num_tiles) {
    if (num_tiles <= 0) return 0;
    int per_sm = 0;
    cudaError_t e = dtype == SPMV_F64 ? (aligned ? ctas_ipl<double, true>(ipl, per_sm) : ctas_ipl<double, false>(ipl, per_sm))
                                      : (aligned ? ctas_ipl<float, true>(ipl, per_sm) : ctas_ipl<float, false>(ipl, per_sm));
    if (e != cudaSuccess) return -1;
    return warps_for(num_tiles, per_sm, ipl, 0);
}

bool merge_path_supported(int ipl) { return ipl == 8 || ipl == 12 || ipl == 16 || ipl == 24 || ipl == 32; }

int merge_path_threads() { return 32; }

int merge_path_min_items() { return 8; }

// Tile size from the row statistics.  Measured on GB300: matrices whose
// nonzeros stay near the diagonal (the gathers of a tile hit few cache lines)
// run best with large tiles, which spread the per-tile work over more
// nonzeros; scattered columns run best with smaller ones, which keep the
// shared memory per SM small and so leave L1 room for the gathers in flight.
// fp32: 24 items per lane when the bandwidth is below n/64, else 16 (power
// law: 266-268 us at 16 against 269-274 us at 12 and 286 us at 8).
// fp64: 16 when the bandwidth is below 4096, else 12 (short rows in a band
// of +-1024: 216 us at 16 against 236 us at 12 with two stages; skew: 242 us
// at 12 against 262 us at 16 and 287 us at 8).
int merge_path_choose_items(spmv_dtype_t dtype, int32_t n, const spmv_row_stats_t &s) {
    if (dtype == SPMV_F64) return s.bandwidth <= 4096 ? 16 : 12;
    return (int64_t)s.bandwidth * 64 <= (int64_t)n ? 24 : 16;
}

cudaError_t launch_merge_path_spmv(spmv_dtype_t dtype, int ipl, const MergePathArgs &a, cudaStream_t stream) {
    // bulk copies need row_ptr, col_idx, vals and (when it is read) y 16-byte
    // aligned
    const bool reads_y = dtype == SPMV_F64 ? a.beta != 0.0 : (float)a.beta != 0.0f;
    const bool vec = (reinterpret_cast<uintptr_t>(a.row_ptr) % 16 == 0) &&
                     (reinterpret_cast<uintptr_t>(a.col_idx) % 16 == 0) &&
                     (reinterpret_cast<uintptr_t>(a.vals) % 16 == 0) &&
                     (!reads_y || reinterpret_cast<uintptr_t>(a.y) % 16 == 0);
    if (dtype == SPMV_F64)
        return vec ? launch_ipl<double, true>(ipl, a, stream) : launch_ipl<double, false>(ipl, a, stream);
    return vec ? launch_ipl<float, true>(ipl, a, stream) : launch_ipl<float, false>(ipl, a, stream);
}

}  // namespace lbcsr
