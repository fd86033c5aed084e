// Ceilings of the x gather: how fast a column pattern can be gathered from x
// by each load path the GPU offers, with no matrix values and no arithmetic
// beyond an integer checksum.
//
// The Row-grouped CSR page (sections 3 and 4) found the x gather to decide
// SpMV speed once the matrix stream is coalesced: binding x to the texture
// cache gave 1.3-1.8x.  On GB300 a random gather that misses in L1 costs the
// L1 one tag lookup per distinct cache line, about one per SM clock, whatever
// the hit rate in L2 -- so a matrix whose columns are scattered (a power-law
// graph) is bound by that rate, not by HBM.  The paths measured here:
//
//   STREAM   col_idx only (no gather): the floor set by the column stream
//   L1       ld.global.nc (the read-only path the SpMV kernels use)
//   L2       ld.global.cg (cached in L2 only)
//   BULK16   per lane, a 16-byte cp.async.bulk of the aligned block holding
//            x[c] into shared memory (the Tensor Memory Accelerator)
//   TMA4     cp.async.bulk.tensor tile::gather4 over x viewed as rows of 32
//            bytes: one instruction fetches the rows of 4 gathers
//   L1_TMA4  half the gathers by L1, half by TMA4, to see whether the two
//            paths add up
//   L1_TMA4_QUARTER  three quarters by L1, one quarter by TMA4
//   TMA4_16  TMA4 over rows of 16 bytes (the narrowest row a tensor copy
//            takes)
//
// and, to see what bringing in the matrix stream costs the gathers, three
// paths that also read the values (L1 gathers in all three):
//
//   STREAM_LDG      columns and values by coalesced loads into registers
//   STREAM_BULK     columns and values by one bulk copy each per chunk into
//                   shared memory (two stages per warp)
//   STREAM_CPASYNC  columns and values by 16-byte cp.async per lane into
//                   shared memory (two stages per warp)
//   STREAM_LDG_OCC  as STREAM_LDG, with the shared memory of the staged
//                   paths reserved (the same warps per SM)
//   STREAM_LDG_STS  coalesced loads into registers, stored to shared memory
//                   and read back by the lanes (staging done by the lanes)
//   STREAM_LDG_FEW  as STREAM_LDG, with no shared memory but only as many
//                   CTAs per SM as the staged paths fit
//   STREAM_LDG_RES_k (k = 1..6)  as STREAM_LDG with 4 CTAs per SM and
//                   32 * k KB of shared memory reserved per SM, unused: how
//                   the gathers depend on the L1 left to them
//
// Each warp takes chunks of 32 * U consecutive nonzeros (grid-stride), loads
// their columns with coalesced loads and adds the bit patterns of the
// gathered x values into a 64-bit checksum, identical for every path.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.cuh"
#include "tma.cuh"

namespace lbcsr {
namespace {

using namespace tma;

constexpr int kGThreads = 256;
constexpr int kGWarps = kGThreads / 32;

__device__ __forceinline__ unsigned long long bits_of(float v) { return __float_as_uint(v); }
__device__ __forceinline__ unsigned long long bits_of(double v) {
    return (unsigned long long)__double_as_longlong(v);
}

__device__ __forceinline__ float ld_l2(const float *p) { return __ldcg(p); }
__device__ __forceinline__ double ld_l2(const double *p) { return __ldcg(p); }

// tile::gather4: rows r0..r3 of the 2-D view of x (all columns of each row's
// box) into 4 consecutive boxes at dst (128-byte aligned).
__device__ __forceinline__ void tma_gather4(void *dst, const CUtensorMap *map, int r0, int r1, int r2, int r3,
                                            uint64_t *bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7], %8;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(smem_u32(bar)),
        "l"(pol)
        : "memory");
}

template <typename V>
struct GatherParams {
    long long nnz;
    int32_t n;
    const int32_t *col;
    const V *x;
    const V *vals;       // STREAM_* paths
    int32_t rows;        // TMA4: rows in the 2-D view of x
    unsigned long long *checksum;
    int32_t *error;
};

constexpr int kBoxBytes = 128;  // 4 rows, one gather4 destination (128-byte aligned)

// TMA4 row: 32 bytes (one L2 sector), or 16 for TMA4_16
__host__ __device__ constexpr int g_row_bytes(int path) { return path == 7 ? 16 : 32; }
// gathers by TMA4 among a lane's U: all (4, 7), even u (5), u % 4 == 0 (6)
__host__ __device__ constexpr bool g_by_tma(int path, int u) {
    return path == 4 || path == 7 || (path == 5 && (u & 1) == 0) || (path == 6 && (u & 3) == 0);
}
// slot of gather u among the TMA4 gathers of a lane
__host__ __device__ constexpr int g_slot(int path, int u) { return path == 5 ? u / 2 : path == 6 ? u / 4 : u; }

// Bytes a stage's copies deliver: 16 per BULK16 gather, 4 rows per gather4.
template <int PATH, int U>
__host__ __device__ constexpr int g_tx_bytes() {
    return PATH == 3 ? U * 32 * 16
                     : PATH == 4 || PATH == 7 ? U * 8 * 4 * g_row_bytes(PATH)
                     : PATH == 5 ? (U / 2) * 8 * 4 * g_row_bytes(PATH)
                     : PATH == 6 ? (U / 4) * 8 * 4 * g_row_bytes(PATH) : 0;
}
// Shared memory per warp and stage for U gathers per lane.
template <int PATH, int U>
__host__ __device__ constexpr int g_stage_bytes() {
    return PATH == 3 ? U * 32 * 16
                     : PATH == 4 || PATH == 7 ? U * 8 * kBoxBytes
                     : PATH == 5 ? (U / 2) * 8 * kBoxBytes
                     : PATH == 6 ? (U / 4) * 8 * kBoxBytes : 0;
}

template <typename V, int PATH, int U>
__global__ void __launch_bounds__(kGThreads) gather_ceiling_kernel(const GatherParams<V> p,
                                                                   const __grid_constant__ CUtensorMap map) {
    constexpr int SB = g_stage_bytes<PATH, U>();
    constexpr bool ASYNC = SB > 0;
    constexpr int CH = 32 * U;
    constexpr int kRowBytes = g_row_bytes(PATH);
    constexpr int EPR = kRowBytes / (int)sizeof(V);  // x elements per TMA4 row
    constexpr int E16 = 16 / (int)sizeof(V);         // x elements per 16 bytes
    extern __shared__ __align__(16) unsigned char dsm[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // 128-byte aligned per-warp region: two barriers, then two stages
    const uint32_t base_u32 = smem_u32(dsm);
    unsigned char *aligned = dsm + (((base_u32 + 127u) & ~127u) - base_u32);
    unsigned char *region = aligned + (size_t)warp * (128 + 2 * SB);
    uint64_t *bars = reinterpret_cast<uint64_t *>(region);
    unsigned char *stages = region + 128;
    const uint64_t pol = l2_policy_evict_last();

    const long long chunks = (p.nnz + CH - 1) / CH;
    const long long gw = (long long)blockIdx.x * kGWarps + warp;
    const long long step = (long long)gridDim.x * kGWarps;
    unsigned long long sum = 0;

    if (!ASYNC) {
        for (long long c = gw; c < chunks; c += step) {
            int cc[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const long long k = c * CH + u * 32 + lane;
                cc[u] = k < p.nnz ? ld_stream(p.col + k) : -1;
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (cc[u] < 0) continue;
                if (PATH == 0) sum += (unsigned)cc[u];
                else if (PATH == 1) sum += bits_of(gather_keep(p.x + cc[u], pol));
                else sum += bits_of(ld_l2(p.x + cc[u]));
            }
        }
    } else {
        if (lane == 0) {
            mbar_init(bars);
            mbar_init(bars + 1);
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        }
        __syncwarp();
        // issue the copies of chunk c into stage s; returns the columns
        auto issue = [&](long long c, int s, int (&cc)[U]) {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const long long k = c * CH + u * 32 + lane;
                cc[u] = k < p.nnz ? ld_stream(p.col + k) : -1;
            }
            unsigned char *st = stages + s * SB;
            if (lane == 0) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                mbar_expect_tx(bars + s, (uint32_t)g_tx_bytes<PATH, U>());
            }
            __syncwarp();
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c0 = cc[u] < 0 ? 0 : cc[u];
                if (PATH == 3) {
                    // the 16-byte block holding x[c0], if it lies inside x;
                    // else block 0 (the lane then loads its value directly)
                    const long long blk = (long long)(c0 / E16) * E16;
                    const long long src = blk + E16 <= p.n ? blk : 0;
                    bulk_copy(st + (u * 32 + lane) * 16, p.x + src, 16u, bars + s, pol);
                } else {
                    if (!g_by_tma(PATH, u)) continue;
                    const int slot = g_slot(PATH, u);
                    int row = c0 / EPR;
                    if (row >= p.rows) row = 0;  // past the view: loaded directly
                    const int r0 = __shfl_sync(0xffffffffu, row, lane & ~3);
                    const int r1 = __shfl_sync(0xffffffffu, row, (lane & ~3) + 1);
                    const int r2 = __shfl_sync(0xffffffffu, row, (lane & ~3) + 2);
                    const int r3 = __shfl_sync(0xffffffffu, row, (lane & ~3) + 3);
                    if ((lane & 3) == 0)
                        tma_gather4(st + (slot * 8 + (lane >> 2)) * kBoxBytes, &map, r0, r1, r2, r3, bars + s, pol);
                }
            }
        };
        auto consume = [&](int s, const int (&cc)[U]) {
            const unsigned char *st = stages + s * SB;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (cc[u] < 0) continue;
                const int c = cc[u];
                V v;
                if (PATH == 3) {
                    const long long blk = (long long)(c / E16) * E16;
                    v = blk + E16 <= p.n
                            ? reinterpret_cast<const V *>(st + (u * 32 + lane) * 16)[c - blk]
                            : gather_keep(p.x + c, pol);
                } else if (!g_by_tma(PATH, u)) {
                    v = gather_keep(p.x + c, pol);
                } else {
                    const int slot = g_slot(PATH, u);
                    v = c / EPR < p.rows
                            ? reinterpret_cast<const V *>(st + (slot * 8 + (lane >> 2)) * kBoxBytes +
                                                          (lane & 3) * kRowBytes)[c % EPR]
                            : gather_keep(p.x + c, pol);
                }
                sum += bits_of(v);
            }
        };
        int cur[U], nxt[U];
        long long c = gw;
        uint32_t uses = 0u;  // bit s: parity of stage s's next completion
        if (c < chunks) issue(c, 0, cur);
        int s = 0;
        for (; c < chunks; c += step) {
            const long long cn = c + step;
            if (cn < chunks) issue(cn, s ^ 1, nxt);
            const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(bars + s, (uses >> s) & 1u));
            if (!ok) {
                if (lane == 0) atomicOr(p.error, 1);
                if (cn < chunks) mbar_wait_bounded(bars + (s ^ 1), (uses >> (s ^ 1)) & 1u);
                return;
            }
            uses ^= 1u << s;
            consume(s, cur);
            __syncwarp();  // the stage is read before it is refilled
#pragma unroll
            for (int u = 0; u < U; ++u) cur[u] = nxt[u];
            s ^= 1;
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    if (lane == 0 && sum) atomicAdd(p.checksum, sum);
}


// Path 20: x read by element fetches from a linear texture object over x
// (the Row-grouped CSR page reads x through the texture cache).  fp64 is
// fetched as int2, its two 32-bit halves.
__device__ __forceinline__ unsigned long long tex_bits(cudaTextureObject_t t, int c, float *) {
    return __float_as_uint(tex1Dfetch<float>(t, c));
}
__device__ __forceinline__ unsigned long long tex_bits(cudaTextureObject_t t, int c, double *) {
    const int2 v = tex1Dfetch<int2>(t, c);
    return ((unsigned long long)(unsigned)v.y << 32) | (unsigned)v.x;
}

template <typename V>
__global__ void __launch_bounds__(kGThreads) tex_gather_kernel(const GatherParams<V> p, cudaTextureObject_t tex) {
    constexpr int U = 8, CH = 32 * U;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const long long chunks = (p.nnz + CH - 1) / CH;
    const long long gw = (long long)blockIdx.x * kGWarps + warp;
    const long long step = (long long)gridDim.x * kGWarps;
    unsigned long long sum = 0;
    for (long long c = gw; c < chunks; c += step) {
        int cc[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const long long k = c * CH + u * 32 + lane;
            cc[u] = k < p.nnz ? ld_stream(p.col + k) : -1;
        }
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (cc[u] >= 0) sum += tex_bits(tex, cc[u], static_cast<V *>(nullptr));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    if (lane == 0 && sum) atomicAdd(p.checksum, sum);
}

template <typename V>
cudaError_t launch_tex_gather(const GatherParams<V> &p, cudaStream_t stream) {
    int max_width = 0, dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&max_width, cudaDevAttrMaxTexture1DLinearWidth, dev);
    if (e != cudaSuccess) return e;
    if ((long long)p.n > max_width) return cudaErrorInvalidValue;
    cudaResourceDesc res;
    memset(&res, 0, sizeof(res));
    res.resType = cudaResourceTypeLinear;
    res.res.linear.devPtr = const_cast<V *>(p.x);
    res.res.linear.desc = sizeof(V) == 8 ? cudaCreateChannelDesc<int2>() : cudaCreateChannelDesc<float>();
    res.res.linear.sizeInBytes = (size_t)p.n * sizeof(V);
    cudaTextureDesc td;
    memset(&td, 0, sizeof(td));
    td.readMode = cudaReadModeElementType;
    td.filterMode = cudaFilterModePoint;
    td.addressMode[0] = cudaAddressModeClamp;
    cudaTextureObject_t tex = 0;
    e = cudaCreateTextureObject(&tex, &res, &td, nullptr);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, tex_gather_kernel<V>, kGThreads, 0);
    if (e == cudaSuccess) {
        const long long chunks = (p.nnz + 255) / 256;
        long long grid = (long long)(per_sm > 0 ? per_sm : 1) * device_sm_count();
        const long long need = (chunks + kGWarps - 1) / kGWarps;
        if (grid > need) grid = need;
        if (grid < 1) grid = 1;
        tex_gather_kernel<V><<<(unsigned)grid, kGThreads, 0, stream>>>(p, tex);
        e = cudaGetLastError();
    }
    // the object must outlive the launch that uses it
    const cudaError_t es = cudaStreamSynchronize(stream);
    cudaDestroyTextureObject(tex);
    return e != cudaSuccess ? e : es;
}

// Paths 8-10: the gather with the matrix stream (columns and values).  Each
// warp takes chunks of 256 nonzeros; the checksum adds the gathered x and
// the values' bit patterns.  Full chunks go through the path's staging; the
// last, partial chunk is loaded directly.
constexpr int kSChunk = 256;

template <typename V>
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}

template <typename V, int PATH>
__global__ void __launch_bounds__(kGThreads) stream_gather_kernel(const GatherParams<V> p) {
    constexpr int U = kSChunk / 32;
    constexpr int SB = kSChunk * (4 + (int)sizeof(V));  // columns, then values
    extern __shared__ __align__(16) unsigned char dsm[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t base_u32 = smem_u32(dsm);
    unsigned char *aligned = dsm + (((base_u32 + 127u) & ~127u) - base_u32);
    unsigned char *region = aligned + (size_t)warp * (128 + 2 * SB);
    uint64_t *bars = reinterpret_cast<uint64_t *>(region);
    unsigned char *stages = region + 128;
    const uint64_t pol = l2_policy_evict_last();
    const uint64_t spol = l2_policy_evict_first();
    const long long chunks = (p.nnz + kSChunk - 1) / kSChunk;
    const long long full = p.nnz / kSChunk;
    const long long gw = (long long)blockIdx.x * kGWarps + warp;
    const long long step = (long long)gridDim.x * kGWarps;
    unsigned long long sum = 0;

    auto direct = [&](long long c) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const long long k = c * kSChunk + u * 32 + lane;
            if (k < p.nnz) sum += bits_of(gather_keep(p.x + ld_stream(p.col + k), pol)) + bits_of(ld_stream(p.vals + k));
        }
    };
    if (PATH == 8 || PATH == 11 || PATH >= 13) {
        for (long long c = gw; c < chunks; c += step) direct(c);
    } else if (PATH == 12) {
        int *sc = reinterpret_cast<int *>(stages);
        V *sv = reinterpret_cast<V *>(stages + kSChunk * 4);
        for (long long c = gw; c < full; c += step) {
            int cr[U];
            V vr[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                cr[u] = ld_stream(p.col + c * kSChunk + u * 32 + lane);
                vr[u] = ld_stream(p.vals + c * kSChunk + u * 32 + lane);
            }
            __syncwarp();  // the previous chunk is read
#pragma unroll
            for (int u = 0; u < U; ++u) {
                sc[u * 32 + lane] = cr[u];
                sv[u * 32 + lane] = vr[u];
            }
            __syncwarp();
#pragma unroll
            for (int u = 0; u < U; ++u)  // read back in another lane order
                sum += bits_of(gather_keep(p.x + sc[u * 32 + (lane ^ 1)], pol)) + bits_of(sv[u * 32 + (lane ^ 1)]);
        }
        for (long long t = full + ((gw - full) % step + step) % step; t < chunks; t += step) direct(t);
    } else {
        if (PATH == 9 && lane == 0) {
            mbar_init(bars);
            mbar_init(bars + 1);
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        }
        __syncwarp();
        auto issue = [&](long long c, int s) {
            unsigned char *st = stages + s * SB;
            if (PATH == 9) {
                if (lane == 0) {
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    mbar_expect_tx(bars + s, (uint32_t)SB);
                    bulk_copy(st, p.col + c * kSChunk, kSChunk * 4u, bars + s, spol);
                    bulk_copy(st + kSChunk * 4, p.vals + c * kSChunk, kSChunk * (uint32_t)sizeof(V), bars + s, spol);
                }
            } else {
                const unsigned char *gc = reinterpret_cast<const unsigned char *>(p.col + c * kSChunk);
                const unsigned char *gv = reinterpret_cast<const unsigned char *>(p.vals + c * kSChunk);
                for (int q = lane; q < kSChunk * 4 / 16; q += 32) cp_async16<V>(st + q * 16, gc + q * 16);
                for (int q = lane; q < kSChunk * (int)sizeof(V) / 16; q += 32)
                    cp_async16<V>(st + kSChunk * 4 + q * 16, gv + q * 16);
                asm volatile("cp.async.commit_group;" ::: "memory");
            }
        };
        uint32_t uses = 0u;
        long long c = gw;
        if (c < full) issue(c, 0);
        int s = 0;
        for (; c < full; c += step) {
            const long long cn = c + step;
            const bool more = cn < full;
            if (more) issue(cn, s ^ 1);
            if (PATH == 9) {
                const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(bars + s, (uses >> s) & 1u));
                if (!ok) {
                    if (lane == 0) atomicOr(p.error, 1);
                    if (more) mbar_wait_bounded(bars + (s ^ 1), (uses >> (s ^ 1)) & 1u);
                    return;
                }
                uses ^= 1u << s;
            } else {
                if (more) asm volatile("cp.async.wait_group 1;" ::: "memory");
                else asm volatile("cp.async.wait_group 0;" ::: "memory");
                __syncwarp();
            }
            const unsigned char *st = stages + s * SB;
            const int *sc = reinterpret_cast<const int *>(st);
            const V *sv = reinterpret_cast<const V *>(st + kSChunk * 4);
#pragma unroll
            for (int u = 0; u < U; ++u)
                sum += bits_of(gather_keep(p.x + sc[u * 32 + lane], pol)) + bits_of(sv[u * 32 + lane]);
            __syncwarp();  // the stage is read before it is refilled
            s ^= 1;
        }
        for (long long t = full + ((gw - full) % step + step) % step; t < chunks; t += step) direct(t);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    if (lane == 0 && sum) atomicAdd(p.checksum, sum);
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

template <typename V, int PATH, int U>
cudaError_t launch_gather(const GatherParams<V> &p, const CUtensorMap &map, cudaStream_t stream) {
    constexpr int SB = g_stage_bytes<PATH, U>();
    const size_t smem = SB ? 128 + (size_t)kGWarps * (128 + 2 * SB) : 0;
    auto kern = gather_ceiling_kernel<V, PATH, U>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kGThreads, smem);
    if (e != cudaSuccess) return e;
    const int pct = carveout_percent(per_sm > 0 ? per_sm : 1, smem);
    if (pct >= 0 && (e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, pct)) != cudaSuccess)
        return e;
    const long long chunks = (p.nnz + 32 * U - 1) / (32 * U);
    long long grid = (long long)(per_sm > 0 ? per_sm : 1) * device_sm_count();
    const long long need = (chunks + kGWarps - 1) / kGWarps;
    if (grid > need) grid = need;
    if (grid < 1) grid = 1;
    kern<<<(unsigned)grid, kGThreads, smem, stream>>>(p, map);
    return cudaGetLastError();
}


template <typename V, int PATH>
cudaError_t launch_stream_gather(const GatherParams<V> &p, cudaStream_t stream) {
    const size_t staged = 128 + (size_t)kGWarps * (128 + 2 * kSChunk * (4 + sizeof(V)));
    // PATH 11 reserves the staged paths' shared memory without using it;
    // PATH 13 uses none but launches as few CTAs as they fit
    const size_t smem = PATH == 8 || PATH == 13 ? 0 : PATH >= 14 ? (size_t)(PATH - 13) * 8192 - 1024 : staged;
    auto kern = stream_gather_kernel<V, PATH>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(staged > smem ? staged : smem));
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kGThreads, PATH == 13 ? staged : smem);
    if (e != cudaSuccess) return e;
    // STREAM_LDG_OCC keeps the runtime's own choice (it shows what reserved
    // shared memory costs); the others leave the rest of the SM to L1
    if (PATH >= 14) per_sm = per_sm < 4 ? per_sm : 4;
    const int pct = PATH == 11 || PATH == 13 ? -1 : carveout_percent(per_sm > 0 ? per_sm : 1, smem);
    if (pct >= 0 && (e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, pct)) != cudaSuccess)
        return e;
    const long long chunks = (p.nnz + kSChunk - 1) / kSChunk;
    long long grid = (long long)(per_sm > 0 ? per_sm : 1) * device_sm_count();
    const long long need = (chunks + kGWarps - 1) / kGWarps;
    if (grid > need) grid = need;
    if (grid < 1) grid = 1;
    kern<<<(unsigned)grid, kGThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

template <typename V>
spmv_status_t gather_typed(int path, int32_t nnz, const int32_t *col, int32_t n, const void *x, const void *vals,
                           unsigned long long *checksum, int32_t *error, cudaStream_t stream) {
    GatherParams<V> p;
    p.nnz = nnz;
    p.n = n;
    p.col = col;
    p.x = static_cast<const V *>(x);
    p.vals = static_cast<const V *>(vals);
    const int row_bytes = g_row_bytes(path);
    p.rows = (int32_t)(((long long)n * (long long)sizeof(V)) / row_bytes);
    p.checksum = checksum;
    p.error = error;
    CUtensorMap map;
    memset(&map, 0, sizeof(map));
    if (path == 3 && reinterpret_cast<uintptr_t>(x) % 16 != 0) return SPMV_ERR_UNSUPPORTED;
    if (path == 9 || path == 10) {
        if (reinterpret_cast<uintptr_t>(col) % 16 != 0 || reinterpret_cast<uintptr_t>(vals) % 16 != 0)
            return SPMV_ERR_UNSUPPORTED;
    }
    if (path >= 4 && path <= 7) {
        if (reinterpret_cast<uintptr_t>(x) % 16 != 0 || p.rows < 1) return SPMV_ERR_UNSUPPORTED;
        PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
        if (!enc) return SPMV_ERR_UNSUPPORTED;
        const cuuint64_t dims[2] = {(cuuint64_t)(row_bytes / sizeof(V)), (cuuint64_t)p.rows};
        const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
        const cuuint32_t box[2] = {(cuuint32_t)(row_bytes / sizeof(V)), 1u};
        const cuuint32_t estr[2] = {1u, 1u};
        const CUresult r = enc(&map, sizeof(V) == 8 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT64 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                               2, const_cast<void *>(x), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                               CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return SPMV_ERR_UNSUPPORTED;
    }
    cudaError_t e;
    switch (path) {
    case 0: e = launch_gather<V, 0, 8>(p, map, stream); break;
    case 1: e = launch_gather<V, 1, 8>(p, map, stream); break;
    case 2: e = launch_gather<V, 2, 8>(p, map, stream); break;
    case 3: e = launch_gather<V, 3, 4>(p, map, stream); break;
    case 4: e = launch_gather<V, 4, 4>(p, map, stream); break;
    case 5: e = launch_gather<V, 5, 4>(p, map, stream); break;
    case 6: e = launch_gather<V, 6, 4>(p, map, stream); break;
    case 7: e = launch_gather<V, 7, 4>(p, map, stream); break;
    case 8: e = launch_stream_gather<V, 8>(p, stream); break;
    case 9: e = launch_stream_gather<V, 9>(p, stream); break;
    case 10: e = launch_stream_gather<V, 10>(p, stream); break;
    case 11: e = launch_stream_gather<V, 11>(p, stream); break;
    case 12: e = launch_stream_gather<V, 12>(p, stream); break;
    case 13: e = launch_stream_gather<V, 13>(p, stream); break;
    case 14: e = launch_stream_gather<V, 14>(p, stream); break;
    case 15: e = launch_stream_gather<V, 15>(p, stream); break;
    case 16: e = launch_stream_gather<V, 16>(p, stream); break;
    case 17: e = launch_stream_gather<V, 17>(p, stream); break;
    case 18: e = launch_stream_gather<V, 18>(p, stream); break;
    case 19: e = launch_stream_gather<V, 19>(p, stream); break;
    case 20: e = launch_tex_gather<V>(p, stream); break;
    default: return SPMV_ERR_INVALID_ARG;
    }
    return e == cudaSuccess ? SPMV_OK : SPMV_ERR_CUDA;
}

}  // namespace
}  // namespace lbcsr

using namespace lbcsr;

extern "C" spmv_status_t spmv_gather_ceiling(int32_t path, int32_t nnz, const int32_t *col_idx, int32_t n,
                                             const void *x, const void *vals, spmv_dtype_t dtype,
                                             uint64_t *checksum, int32_t *error, spmv_stream_t stream) {
    if (path < 0 || path > 20 || nnz < 0 || n < 0) return SPMV_ERR_INVALID_ARG;
    if (dtype != SPMV_F32 && dtype != SPMV_F64) return SPMV_ERR_INVALID_ARG;
    if (nnz == 0) return SPMV_OK;
    if (!col_idx || !checksum || !error || (path > 0 && (!x || n < 1)) || (path >= 8 && !vals))
        return SPMV_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    unsigned long long *cs = reinterpret_cast<unsigned long long *>(checksum);
    return dtype == SPMV_F64 ? gather_typed<double>(path, nnz, col_idx, n, x, vals, cs, error, s)
                             : gather_typed<float>(path, nnz, col_idx, n, x, vals, cs, error, s);
}
