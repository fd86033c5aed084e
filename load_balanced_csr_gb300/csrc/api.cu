// C ABI of the load-balanced CSR SpMV library: plan creation (analysis,
// kernel choice, schedule), execution, inspection.  Declarations and the
// contract of every entry point are in include/spmv.h.
//
// Memory: a plan makes its device allocations once, at creation, in one
// arena (OpSparse, section 5.1: all metadata sized up front and allocated
// with one cudaMalloc, since allocation is far slower than use), plus a
// second allocation only for kernels that keep a reordered copy of A.
// spmv_execute allocates and frees nothing and never waits for the device.
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <string>

#include "internal.cuh"

using namespace lbcsr;

struct spmv_plan_s {
    int32_t m = 0, n = 0, nnz = 0;
    spmv_dtype_t dtype = SPMV_F32;
    const int32_t *row_ptr = nullptr;
    const int32_t *col_idx = nullptr;
    const void *vals = nullptr;

    spmv_kernel_t kernel = SPMV_KERNEL_MERGE_PATH;
    int ipt = 7;
    int64_t tile = 0;        // T
    int64_t num_tiles = 0;   // P
    int rgcsr_group = 0;
    int32_t num_long_rows = 0;

    void *arena = nullptr;
    size_t arena_bytes = 0;
    int2 *part = nullptr;
    void *tail_partial = nullptr;
    void *head_partial = nullptr;
    int32_t *arrivals = nullptr;
    int32_t *device_error = nullptr;  // set by kernels whose copies time out

    // Row-grouped CSR and long-row kernels (a second allocation, `aux`, and
    // the interleaved copy of A, `rg`)
    void *aux = nullptr;
    size_t aux_bytes = 0;
    int32_t long_min = 0;            // rows this long go to the long-row kernel (0: none)
    int32_t *long_rows = nullptr;    // [num_long_rows]
    int64_t *seg_begin = nullptr;    // [num_long_rows + 1]
    int64_t num_segs = 0;
    void *seg_partial = nullptr;     // [num_segs]
    int32_t *long_arrivals = nullptr;  // [num_long_rows]
    int g_log2 = 0;
    int64_t ngroups = 0;
    int64_t rg_slots = 0;
    int64_t *group_ptr = nullptr;    // [ngroups + 1]
    int32_t *row_len = nullptr;      // [m] by position
    int32_t *perm = nullptr;         // [m] row at each position (window-sorted copy only)
    void *rg = nullptr;
    size_t rg_bytes = 0;

    // A^T in CSR form (spmv_execute_transposed) and its own plan
    void *tr = nullptr;
    size_t tr_bytes = 0;
    int32_t *t_ptr = nullptr, *t_idx = nullptr, *t_src = nullptr;
    void *t_vals = nullptr;
    spmv_plan_s *tplan = nullptr;

    // SpMM (spmv_execute_multi): warps and their scratch
    bool with_spmm = false;
    bool has_partition = false;
    int64_t spmm_warps = 0;
    void *spmm = nullptr;
    size_t spmm_bytes = 0;
    void *spmm_tail = nullptr, *spmm_head = nullptr;
    int32_t *spmm_arrivals = nullptr;
    int32_t *rg_col = nullptr;       // [rg_slots]
    void *rg_val = nullptr;          // [rg_slots]

    spmv_row_stats_t stats{};
};

namespace {

thread_local std::string g_last_error;

spmv_status_t fail(spmv_status_t s, const std::string &msg) {
    g_last_error = msg;
    return s;
}

spmv_status_t cuda_fail(cudaError_t e, const char *what) {
    return fail(SPMV_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

size_t value_size(spmv_dtype_t d) { return d == SPMV_F64 ? 8 : 4; }

int env_int(const char *name, int fallback) {
    const char *v = std::getenv(name);
    if (!v || !*v) return fallback;
    return std::atoi(v);
}

spmv_kernel_t env_kernel() {
    const char *v = std::getenv("SPMV_FORCE_KERNEL");
    if (!v || !*v) return SPMV_KERNEL_AUTO;
    if (!std::strcmp(v, "merge_path")) return SPMV_KERNEL_MERGE_PATH;
    if (!std::strcmp(v, "thread_row")) return SPMV_KERNEL_THREAD_ROW;
    if (!std::strcmp(v, "rgcsr")) return SPMV_KERNEL_RGCSR;
    if (!std::strcmp(v, "long_rows")) return SPMV_KERNEL_LONG_ROWS;
    if (!std::strcmp(v, "rgcsr_sorted")) return SPMV_KERNEL_RGCSR_SORTED;
    if (!std::strcmp(v, "group_mapped")) return SPMV_KERNEL_GROUP_MAPPED;
    return SPMV_KERNEL_AUTO;
}

// Kernel choice from the measured row-length statistics.
//  * n == 1 with short rows: thread per row, CUB's special case for a
//    single-column matrix named in "A GPU load-balancing programming model"
//    (section 6.1): perfectly balanced work needs no balancing.
//  * small matrices: the same paper's rule (section 6.2) -- merge path unless
//    (rows < 500 or columns < 500) and nnz < 10000 -- with rows capped at 256
//    nonzeros so the per-row sum stays accurate; and on GB300 any matrix of
//    at most 65,536 rows (one wave of thread-per-row CTAs) whose rows hold
//    at most 64 nonzeros: such products are latency-bound, and one thread
//    per row has the shortest chain (5-point Laplacian 64x64: 6.1 us, against
//    8.1 us Row-grouped and 12.2 us merge path);
//  * rows so even that a Row-grouped CSR copy with groups of 32 rows pads at
//    most 10 % (the Row-grouped CSR page, section 4, names padding as the
//    format's weakness): the Row-grouped kernel, which measured faster than
//    merge path on such matrices (27-point stencil 128^3: 82.6 us against
//    90.0 us; 5-point Laplacian 64x64: 8.2 us against 12.6 us) and 2-8x
//    slower on irregular ones;
//  * everything else: merge path.
spmv_kernel_t choose_kernel(const spmv_plan_s &p) {
    const spmv_row_stats_t &s = p.stats;
    if (p.n == 1 && s.max_len <= 32) return SPMV_KERNEL_THREAD_ROW;
    if ((p.m < 500 || p.n < 500) && p.nnz < 10000 && s.max_len <= 256) return SPMV_KERNEL_THREAD_ROW;
    if (p.m <= 65536 && s.max_len <= 64) return SPMV_KERNEL_THREAD_ROW;
    if (p.nnz > 0 && (double)s.rg_slots[0] <= 1.1 * (double)p.nnz) return SPMV_KERNEL_RGCSR;
    return SPMV_KERNEL_MERGE_PATH;
}

// Row-grouped CSR group size: 32.  The Row-grouped CSR page needs G >= 32
// for coalesced loads and found 128 best on its hardware (section 4), where
// a warp read each level straight from global memory.  Here the copy is
// staged by bulk copies and G = 32 makes a group one warp's rows, so warps
// never synchronise; it also pads least (a group's padding is set by its
// longest row, and smaller groups have shorter longest rows).
int choose_rgcsr_group(const spmv_row_stats_t &, int64_t) { return 32; }

// Rows in length classes that can hold a row of at least `len` nonzeros:
// an upper bound on the number of long rows.
int64_t rows_at_least(const spmv_row_stats_t &s, int32_t len) {
    int c = 0;
    while (c < 31 && (len >> c) != 0) ++c;  // class of len
    int64_t r = 0;
    for (int k = c; k < 32; ++k) r += s.hist[k];
    return r;
}

void destroy_plan(spmv_plan_s *p) {
    if (!p) return;
    if (p->tplan) destroy_plan(p->tplan);
    if (p->tr) cudaFree(p->tr);
    if (p->rg) cudaFree(p->rg);
    if (p->aux) cudaFree(p->aux);
    if (p->spmm) cudaFree(p->spmm);
    if (p->arena) cudaFree(p->arena);
    delete p;
}

constexpr int32_t kDefaultLongRowMin = 512;

// The long-row list and, for the Row-grouped kernel, its layout and copy of
// A.  Two passes over row_ptr per structure, sized on the host from the
// statistics where they bound it, read back where they do not.
bool is_rgcsr(spmv_kernel_t k) { return k == SPMV_KERNEL_RGCSR || k == SPMV_KERNEL_RGCSR_SORTED; }

spmv_status_t build_row_layouts(spmv_plan_s *p, const spmv_options_t &opt, cudaStream_t stream) {
    const int32_t m = p->m;
    const bool rgcsr = is_rgcsr(p->kernel);
    const bool sorted = p->kernel == SPMV_KERNEL_RGCSR_SORTED;
    p->long_min = opt.long_row_min ? opt.long_row_min : kDefaultLongRowMin;
    const bool has_long = m > 0 && p->stats.max_len >= p->long_min;
    const size_t vs = value_size(p->dtype);

    const int nc = long_rows_num_chunks(m);
    const int64_t long_ub = has_long ? rows_at_least(p->stats, p->long_min) : 0;
    const int64_t segs_ub = has_long ? (int64_t)p->nnz / kLongSegmentNnz + long_ub : 0;
    if (rgcsr) {
        const int G = sorted ? 32 : opt.rgcsr_group ? opt.rgcsr_group : choose_rgcsr_group(p->stats, p->nnz);
        p->rgcsr_group = G;
        p->g_log2 = 0;
        while ((1 << p->g_log2) < G) ++p->g_log2;
        p->ngroups = ((int64_t)m + G - 1) / G;
    }
    const int64_t scan_n = rgcsr && p->ngroups > nc ? p->ngroups : nc;

    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = align_up(off + bytes, 256);
        return o;
    };
    const size_t o_long = take(sizeof(int32_t) * long_ub);
    const size_t o_segb = take(sizeof(int64_t) * (long_ub + 1));
    const size_t o_segp = take(vs * segs_ub);
    const size_t o_larr = take(sizeof(int32_t) * long_ub);
    const size_t o_crow = take(sizeof(int64_t) * nc);
    const size_t o_cseg = take(sizeof(int64_t) * nc);
    const size_t o_crow_off = take(sizeof(int64_t) * (nc + 1));
    const size_t o_cseg_off = take(sizeof(int64_t) * (nc + 1));
    const size_t o_rlen = take(rgcsr ? sizeof(int32_t) * m : 0);
    const size_t o_perm = take(sorted ? sizeof(int32_t) * m : 0);
    const size_t o_gsize = take(rgcsr ? sizeof(int64_t) * p->ngroups : 0);
    const size_t o_gp = take(rgcsr ? sizeof(int64_t) * (p->ngroups + 1) : 0);
    const size_t o_scr = take(sizeof(int64_t) * scan_scratch_elems(scan_n));
    p->aux_bytes = off;
    cudaError_t e = cudaMalloc(&p->aux, p->aux_bytes);
    if (e != cudaSuccess) {
        p->aux = nullptr;
        return fail(SPMV_ERR_ALLOC, std::string("cudaMalloc of the row-kernel workspace: ") + cudaGetErrorString(e));
    }
    char *base = static_cast<char *>(p->aux);
    p->long_rows = reinterpret_cast<int32_t *>(base + o_long);
    p->seg_begin = reinterpret_cast<int64_t *>(base + o_segb);
    p->seg_partial = base + o_segp;
    p->long_arrivals = reinterpret_cast<int32_t *>(base + o_larr);
    int64_t *chunk_rows = reinterpret_cast<int64_t *>(base + o_crow);
    int64_t *chunk_segs = reinterpret_cast<int64_t *>(base + o_cseg);
    int64_t *chunk_row_off = reinterpret_cast<int64_t *>(base + o_crow_off);
    int64_t *chunk_seg_off = reinterpret_cast<int64_t *>(base + o_cseg_off);
    int64_t *gsize = reinterpret_cast<int64_t *>(base + o_gsize);
    int64_t *scratch = reinterpret_cast<int64_t *>(base + o_scr);
    if (rgcsr) {
        p->row_len = reinterpret_cast<int32_t *>(base + o_rlen);
        p->group_ptr = reinterpret_cast<int64_t *>(base + o_gp);
    }
    if (sorted) p->perm = reinterpret_cast<int32_t *>(base + o_perm);

    // sizes read back: long rows, segments, Row-grouped slots
    int64_t sizes[3] = {0, 0, 0};
    if (long_ub > 0) e = cudaMemsetAsync(p->long_arrivals, 0, sizeof(int32_t) * long_ub, stream);
    if (e == cudaSuccess && has_long) {
        e = launch_long_rows_count(m, p->row_ptr, p->long_min, chunk_rows, chunk_segs, stream);
        if (e == cudaSuccess) e = launch_exclusive_scan(chunk_rows, nc, chunk_row_off, scratch, stream);
        if (e == cudaSuccess) e = launch_exclusive_scan(chunk_segs, nc, chunk_seg_off, scratch, stream);
        if (e == cudaSuccess)
            e = launch_long_rows_scatter(m, p->row_ptr, p->long_min, chunk_row_off, chunk_seg_off, p->long_rows,
                                         p->seg_begin, stream);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(&sizes[0], chunk_row_off + nc, sizeof(int64_t), cudaMemcpyDeviceToHost, stream);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(&sizes[1], chunk_seg_off + nc, sizeof(int64_t), cudaMemcpyDeviceToHost, stream);
    }
    if (e == cudaSuccess && rgcsr && m > 0) {
        if (sorted)
            e = launch_window_sort(m, p->row_ptr, has_long ? p->long_min : 0, p->perm, p->row_len, gsize, stream);
        else
            e = launch_rgcsr_lengths(m, p->row_ptr, p->g_log2, has_long ? p->long_min : 0, p->row_len, gsize,
                                     stream);
        if (e == cudaSuccess) e = launch_exclusive_scan(gsize, p->ngroups, p->group_ptr, scratch, stream);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(&sizes[2], p->group_ptr + p->ngroups, sizeof(int64_t), cudaMemcpyDeviceToHost,
                                stream);
    } else if (e == cudaSuccess && rgcsr) {
        e = cudaMemsetAsync(p->group_ptr, 0, sizeof(int64_t), stream);
    }
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, "row-kernel layout");
    p->num_long_rows = (int32_t)sizes[0];
    p->num_segs = sizes[1];
    p->rg_slots = sizes[2];
    if (p->num_long_rows > long_ub || p->num_segs > segs_ub)
        return fail(SPMV_ERR_CUDA, "long-row count exceeds its bound");

    if (rgcsr && p->rg_slots > 0) {
        const size_t col_bytes = align_up(sizeof(int32_t) * (size_t)p->rg_slots, 256);
        p->rg_bytes = col_bytes + vs * (size_t)p->rg_slots;
        e = cudaMalloc(&p->rg, p->rg_bytes);
        if (e != cudaSuccess) {
            p->rg = nullptr;
            return fail(SPMV_ERR_ALLOC, std::string("cudaMalloc of the Row-grouped copy: ") + cudaGetErrorString(e));
        }
        p->rg_col = static_cast<int32_t *>(p->rg);
        p->rg_val = static_cast<char *>(p->rg) + col_bytes;
        e = cudaMemsetAsync(p->rg, 0, p->rg_bytes, stream);  // pads: column 0, value 0
        if (e == cudaSuccess)
            e = launch_rgcsr_pack(p->dtype, m, p->row_ptr, p->col_idx, p->vals, p->g_log2, p->group_ptr, p->row_len,
                                  p->perm, p->rg_col, p->rg_val, true, stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
        if (e != cudaSuccess) return cuda_fail(e, "Row-grouped copy");
    }
    return SPMV_OK;
}

// A^T in CSR form (one allocation the plan keeps), built with a temporary
// scratch, and a plan of its own for it.
spmv_status_t build_transpose(spmv_plan_s *p, cudaStream_t stream) {
    const size_t vs = value_size(p->dtype);
    const size_t o_ptr = 0;
    const size_t o_idx = align_up(o_ptr + sizeof(int32_t) * ((size_t)p->n + 1), 256);
    const size_t o_src = align_up(o_idx + sizeof(int32_t) * (size_t)p->nnz, 256);
    const size_t o_val = align_up(o_src + sizeof(int32_t) * (size_t)p->nnz, 256);
    p->tr_bytes = align_up(o_val + vs * (size_t)p->nnz, 256);
    cudaError_t e = cudaMalloc(&p->tr, p->tr_bytes);
    if (e != cudaSuccess) {
        p->tr = nullptr;
        return fail(SPMV_ERR_ALLOC, std::string("cudaMalloc of the transpose: ") + cudaGetErrorString(e));
    }
    char *b = static_cast<char *>(p->tr);
    p->t_ptr = reinterpret_cast<int32_t *>(b + o_ptr);
    p->t_idx = reinterpret_cast<int32_t *>(b + o_idx);
    p->t_src = reinterpret_cast<int32_t *>(b + o_src);
    p->t_vals = b + o_val;
    void *scratch = nullptr;
    e = cudaMalloc(&scratch, (size_t)transpose_scratch_bytes(p->n, p->nnz));
    if (e != cudaSuccess) return fail(SPMV_ERR_ALLOC, std::string("cudaMalloc of the transpose scratch: ") + cudaGetErrorString(e));
    e = launch_transpose(p->dtype, p->m, p->n, p->nnz, p->row_ptr, p->col_idx, p->vals, scratch, p->t_ptr, p->t_idx,
                         p->t_vals, p->t_src, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    cudaFree(scratch);
    if (e != cudaSuccess) return cuda_fail(e, "transpose");
    spmv_plan_t t = nullptr;
    const spmv_status_t st = spmv_plan_create_ex(&t, p->n, p->m, p->nnz, p->t_ptr, p->t_idx, p->t_vals, p->dtype,
                                                 nullptr, reinterpret_cast<spmv_stream_t>(stream));
    if (st != SPMV_OK) return st;
    p->tplan = t;
    return SPMV_OK;
}

cudaError_t launch_long_part(const spmv_plan_s *p, const void *x, void *y, double alpha, double beta,
                             cudaStream_t stream) {
    LongRowsArgs a;
    a.row_ptr = p->row_ptr;
    a.col_idx = p->col_idx;
    a.vals = p->vals;
    a.x = x;
    a.y = y;
    a.alpha = alpha;
    a.beta = beta;
    a.long_rows = p->long_rows;
    a.seg_begin = p->seg_begin;
    a.num_long = p->num_long_rows;
    a.num_segs = p->num_segs;
    a.seg_partial = p->seg_partial;
    a.arrivals = p->long_arrivals;
    return launch_long_rows_spmv(p->dtype, a, stream);
}

}  // namespace

extern "C" {

const char *spmv_status_string(spmv_status_t s) {
    switch (s) {
    case SPMV_OK: return "ok";
    case SPMV_ERR_INVALID_ARG: return "invalid argument";
    case SPMV_ERR_INVALID_CSR: return "invalid CSR matrix";
    case SPMV_ERR_ALLOC: return "allocation failed";
    case SPMV_ERR_CUDA: return "CUDA error";
    case SPMV_ERR_UNSUPPORTED: return "unsupported";
    }
    return "unknown status";
}

const char *spmv_last_error(void) { return g_last_error.c_str(); }

spmv_status_t spmv_plan_create(spmv_plan_t *out, int32_t m, int32_t n, int32_t nnz, const int32_t *row_ptr,
                               const int32_t *col_idx, const void *vals, spmv_dtype_t dtype,
                               spmv_stream_t stream) {
    return spmv_plan_create_ex(out, m, n, nnz, row_ptr, col_idx, vals, dtype, nullptr, stream);
}

spmv_status_t spmv_plan_create_ex(spmv_plan_t *out, int32_t m, int32_t n, int32_t nnz,
                                  const int32_t *row_ptr, const int32_t *col_idx, const void *vals,
                                  spmv_dtype_t dtype, const spmv_options_t *options,
                                  spmv_stream_t stream_handle) {
    g_last_error.clear();
    if (!out) return fail(SPMV_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    if (m < 0 || n < 0 || nnz < 0) return fail(SPMV_ERR_INVALID_ARG, "negative size");
    if ((int64_t)m + (int64_t)nnz >= (1LL << 31)) return fail(SPMV_ERR_INVALID_ARG, "m + nnz must be < 2^31");
    if (dtype != SPMV_F32 && dtype != SPMV_F64) return fail(SPMV_ERR_INVALID_ARG, "unknown dtype");
    if (!row_ptr) return fail(SPMV_ERR_INVALID_ARG, "row_ptr is NULL");
    if (nnz > 0 && (!col_idx || !vals)) return fail(SPMV_ERR_INVALID_ARG, "col_idx or vals is NULL");

    spmv_options_t opt{};
    if (options) opt = *options;
    spmv_kernel_t forced = (spmv_kernel_t)opt.kernel;
    if (forced == SPMV_KERNEL_AUTO) forced = env_kernel();
    if (forced < SPMV_KERNEL_AUTO || forced > SPMV_KERNEL_GROUP_MAPPED)
        return fail(SPMV_ERR_INVALID_ARG, "unknown kernel option");
    if (opt.rgcsr_group && opt.rgcsr_group != 32 && opt.rgcsr_group != 64 && opt.rgcsr_group != 128 &&
        opt.rgcsr_group != 256)
        return fail(SPMV_ERR_INVALID_ARG, "rgcsr_group must be 32, 64, 128 or 256");
    if (opt.long_row_min != 0 && opt.long_row_min < 32)
        return fail(SPMV_ERR_INVALID_ARG, "long_row_min must be 0 or at least 32");
    const int ipt_forced = opt.items_per_thread ? opt.items_per_thread : env_int("SPMV_ITEMS_PER_THREAD", 0);
    if (ipt_forced && !merge_path_supported(ipt_forced))
        return fail(SPMV_ERR_INVALID_ARG, "items_per_thread must be 8, 12, 16, 24 or 32");

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10 || minor != 3)
        return fail(SPMV_ERR_UNSUPPORTED, "this library is built for sm_103 (GB300) only");

    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_handle);
    spmv_plan_s *p = new (std::nothrow) spmv_plan_s();
    if (!p) return fail(SPMV_ERR_ALLOC, "host allocation failed");
    p->m = m;
    p->n = n;
    p->nnz = nnz;
    p->dtype = dtype;
    p->row_ptr = row_ptr;
    p->col_idx = col_idx;
    p->vals = vals;
    // the tile size is chosen after the analysis: size the arena for the
    // smallest one
    const int64_t total = (int64_t)m + nnz;
    const int64_t min_tile = (int64_t)merge_path_threads() * (ipt_forced ? ipt_forced : merge_path_min_items());
    const int64_t max_tiles = total > 0 ? (total + min_tile - 1) / min_tile : 1;

    // ---- one arena: analysis scratch + merge-path schedule and carry state
    const int stats_ctas = stats_num_ctas(m, nnz);
    const size_t vs = value_size(dtype);
    const size_t P = (size_t)max_tiles;
    size_t off = 0;
    const size_t off_partials = off;
    off = align_up(off + sizeof(StatsPartial) * stats_ctas, 256);
    const size_t off_stats = off;
    off = align_up(off + sizeof(spmv_row_stats_t), 256);
    const size_t off_part = off;
    off = align_up(off + sizeof(int2) * (P + 1), 256);
    const size_t off_tail = off;
    off = align_up(off + vs * P, 256);
    const size_t off_head = off;
    off = align_up(off + vs * P, 256);
    const size_t off_arr = off;
    off = align_up(off + sizeof(int32_t) * P, 256);
    const size_t off_err = off;
    off = align_up(off + sizeof(int32_t), 256);
    p->arena_bytes = off;
    e = cudaMalloc(&p->arena, p->arena_bytes);
    if (e != cudaSuccess) {
        p->arena = nullptr;
        destroy_plan(p);
        return fail(SPMV_ERR_ALLOC, std::string("cudaMalloc of the plan workspace: ") + cudaGetErrorString(e));
    }
    char *base = static_cast<char *>(p->arena);
    StatsPartial *partials = reinterpret_cast<StatsPartial *>(base + off_partials);
    spmv_row_stats_t *d_stats = reinterpret_cast<spmv_row_stats_t *>(base + off_stats);
    p->part = reinterpret_cast<int2 *>(base + off_part);
    p->tail_partial = base + off_tail;
    p->head_partial = base + off_head;
    p->arrivals = reinterpret_cast<int32_t *>(base + off_arr);
    p->device_error = reinterpret_cast<int32_t *>(base + off_err);

    // ---- analysis: statistics + validity, read back once
    e = cudaMemsetAsync(p->arrivals, 0, off_err + sizeof(int32_t) - off_arr, stream);
    if (e == cudaSuccess) e = launch_row_stats(m, n, nnz, row_ptr, col_idx, partials, stats_ctas, d_stats, stream);
    if (e == cudaSuccess) e = cudaMemcpyAsync(&p->stats, d_stats, sizeof(spmv_row_stats_t), cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) {
        destroy_plan(p);
        return cuda_fail(e, "plan analysis");
    }
    if (p->stats.flags) {
        const int f = p->stats.flags;
        destroy_plan(p);
        char msg[160];
        std::snprintf(msg, sizeof msg, "invalid CSR:%s%s%s%s", (f & 1) ? " row_ptr[0] != 0;" : "",
                      (f & 2) ? " row_ptr decreases;" : "", (f & 4) ? " row_ptr[m] != nnz;" : "",
                      (f & 8) ? " column index outside [0, n);" : "");
        return fail(SPMV_ERR_INVALID_CSR, msg);
    }

    // ---- kernel choice and schedule
    p->kernel = forced != SPMV_KERNEL_AUTO ? forced : choose_kernel(*p);
    p->ipt = ipt_forced ? ipt_forced : merge_path_choose_items(dtype, n, p->stats);
    p->tile = (int64_t)merge_path_threads() * p->ipt;
    p->num_tiles = total > 0 ? (total + p->tile - 1) / p->tile : 1;
    p->with_spmm = opt.with_spmm != 0;
    if ((p->kernel == SPMV_KERNEL_MERGE_PATH || p->with_spmm) && m > 0) {
        e = launch_merge_path_partition(m, nnz, row_ptr, p->tile, p->num_tiles, p->part, stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
        if (e != cudaSuccess) {
            destroy_plan(p);
            return cuda_fail(e, "merge-path partition");
        }
        p->has_partition = true;
    }
    if (p->with_spmm && m > 0) {
        p->spmm_warps = spmm_warps(p->num_tiles);
        const size_t part_bytes = align_up(vs * kSpmmBlocks * 32 * (size_t)p->spmm_warps, 256);
        p->spmm_bytes = 2 * part_bytes + align_up(sizeof(int32_t) * (size_t)p->spmm_warps, 256);
        e = cudaMalloc(&p->spmm, p->spmm_bytes);
        if (e != cudaSuccess) {
            p->spmm = nullptr;
            destroy_plan(p);
            return fail(SPMV_ERR_ALLOC, std::string("cudaMalloc of the SpMM scratch: ") + cudaGetErrorString(e));
        }
        p->spmm_tail = p->spmm;
        p->spmm_head = static_cast<char *>(p->spmm) + part_bytes;
        p->spmm_arrivals = reinterpret_cast<int32_t *>(static_cast<char *>(p->spmm) + 2 * part_bytes);
        e = cudaMemsetAsync(p->spmm_arrivals, 0, sizeof(int32_t) * (size_t)p->spmm_warps, stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
        if (e != cudaSuccess) {
            destroy_plan(p);
            return cuda_fail(e, "SpMM scratch");
        }
    }
    if (opt.with_transpose) {
        const spmv_status_t st = build_transpose(p, stream);
        if (st != SPMV_OK) {
            destroy_plan(p);
            return st;
        }
    }
    if (is_rgcsr(p->kernel) || p->kernel == SPMV_KERNEL_LONG_ROWS) {
        const spmv_status_t st = build_row_layouts(p, opt, stream);
        if (st != SPMV_OK) {
            destroy_plan(p);
            return st;
        }
    }
    *out = p;
    return SPMV_OK;
}

spmv_status_t spmv_execute(spmv_plan_t p, double alpha, const void *x, double beta, void *y,
                           spmv_stream_t stream_handle) {
    if (!p) return fail(SPMV_ERR_INVALID_ARG, "plan is NULL");
    if (p->m == 0) return SPMV_OK;
    if (!y) return fail(SPMV_ERR_INVALID_ARG, "y is NULL");
    if (!x && p->nnz > 0) return fail(SPMV_ERR_INVALID_ARG, "x is NULL");
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_handle);
    cudaError_t e = cudaSuccess;
    switch (p->kernel) {
    case SPMV_KERNEL_THREAD_ROW:
        e = launch_thread_per_row(p->dtype, p->m, p->row_ptr, p->col_idx, p->vals, x, y, alpha, beta, 0, stream);
        break;
    case SPMV_KERNEL_GROUP_MAPPED:
        e = launch_group_mapped(p->dtype, p->m, p->row_ptr, p->col_idx, p->vals, x, y, alpha, beta, stream);
        break;
    case SPMV_KERNEL_LONG_ROWS:
        // long rows first (they take longest), then the others
        if (p->num_long_rows > 0) e = launch_long_part(p, x, y, alpha, beta, stream);
        if (e == cudaSuccess)
            e = launch_thread_per_row(p->dtype, p->m, p->row_ptr, p->col_idx, p->vals, x, y, alpha, beta,
                                      p->num_long_rows > 0 ? p->long_min : 0, stream);
        break;
    case SPMV_KERNEL_RGCSR:
    case SPMV_KERNEL_RGCSR_SORTED:
        if (p->num_long_rows > 0) e = launch_long_part(p, x, y, alpha, beta, stream);
        if (e == cudaSuccess)
            e = launch_rgcsr_spmv(p->dtype, p->m, p->g_log2, p->group_ptr, p->row_len, p->perm, p->rg_col, p->rg_val,
                                  x, y, alpha, beta, p->device_error, stream);
        break;
    case SPMV_KERNEL_MERGE_PATH:
    default: {
        MergePathArgs a;
        a.m = p->m;
        a.nnz = p->nnz;
        a.row_ptr = p->row_ptr;
        a.col_idx = p->col_idx;
        a.vals = p->vals;
        a.x = x;
        a.y = y;
        a.alpha = alpha;
        a.beta = beta;
        a.part = p->part;
        a.num_tiles = p->num_tiles;
        a.tail_partial = p->tail_partial;
        a.head_partial = p->head_partial;
        a.arrivals = p->arrivals;
        a.error = p->device_error;
        e = launch_merge_path_spmv(p->dtype, p->ipt, a, stream);
        break;
    }
    }
    if (e != cudaSuccess) return cuda_fail(e, "spmv_execute launch");
    return SPMV_OK;
}

spmv_status_t spmv_execute_multi(spmv_plan_t p, int32_t k, double alpha, const void *X, int64_t ldx, double beta,
                                 void *Y, int64_t ldy, spmv_stream_t stream_handle) {
    if (!p) return fail(SPMV_ERR_INVALID_ARG, "plan is NULL");
    if (k < 0) return fail(SPMV_ERR_INVALID_ARG, "k < 0");
    if (!p->with_spmm) return fail(SPMV_ERR_INVALID_ARG, "plan was created without with_spmm");
    if (p->m == 0 || k == 0) return SPMV_OK;
    if (!Y || (!X && p->nnz > 0)) return fail(SPMV_ERR_INVALID_ARG, "X or Y is NULL");
    if (ldx < k || ldy < k) return fail(SPMV_ERR_INVALID_ARG, "leading dimension smaller than k");
    const int32_t rg_kmax = p->dtype == SPMV_F64 ? 16 : 32;  // one slice of columns: the matrix read once
    if (is_rgcsr(p->kernel) && p->g_log2 == 5 && p->num_long_rows == 0 && (p->rg_slots > 0 || p->nnz == 0) &&
        k <= rg_kmax) {
        // the Row-grouped copy serves SpMM too: one thread per row (27-point
        // stencil 128^3, k = 8: 174 us against 612 us on the merge path;
        // wider X is sliced and re-reads the matrix, where merge path wins)
        RgSpmmArgs r;
        r.m = p->m;
        r.k = k;
        r.group_ptr = p->group_ptr;
        r.row_len = p->row_len;
        r.perm = p->perm;
        r.rg_col = p->rg_col;
        r.rg_val = p->rg_val;
        r.X = X;
        r.ldx = ldx;
        r.Y = Y;
        r.ldy = ldy;
        r.alpha = alpha;
        r.beta = beta;
        const cudaError_t e = launch_rg_spmm(p->dtype, r, reinterpret_cast<cudaStream_t>(stream_handle));
        if (e != cudaSuccess) return cuda_fail(e, "spmv_execute_multi launch");
        return SPMV_OK;
    }
    SpmmArgs a;
    a.m = p->m;
    a.nnz = p->nnz;
    a.k = k;
    a.row_ptr = p->row_ptr;
    a.col_idx = p->col_idx;
    a.vals = p->vals;
    a.X = X;
    a.ldx = ldx;
    a.Y = Y;
    a.ldy = ldy;
    a.alpha = alpha;
    a.beta = beta;
    a.part = p->part;
    a.num_tiles = p->num_tiles;
    a.tile = p->tile;
    a.num_warps = p->spmm_warps;
    a.tail = p->spmm_tail;
    a.head = p->spmm_head;
    a.arrivals = p->spmm_arrivals;
    const cudaError_t e = launch_spmm(p->dtype, a, reinterpret_cast<cudaStream_t>(stream_handle));
    if (e != cudaSuccess) return cuda_fail(e, "spmv_execute_multi launch");
    return SPMV_OK;
}

spmv_status_t spmv_execute_transposed(spmv_plan_t p, double alpha, const void *x, double beta, void *y,
                                      spmv_stream_t stream) {
    if (!p) return fail(SPMV_ERR_INVALID_ARG, "plan is NULL");
    if (!p->tplan) return fail(SPMV_ERR_INVALID_ARG, "plan was created without with_transpose");
    return spmv_execute(p->tplan, alpha, x, beta, y, stream);
}

spmv_status_t spmv_plan_update_values(spmv_plan_t p, const void *vals, spmv_stream_t stream_handle) {
    if (!p) return fail(SPMV_ERR_INVALID_ARG, "plan is NULL");
    if (!vals && p->nnz > 0) return fail(SPMV_ERR_INVALID_ARG, "vals is NULL");
    p->vals = vals;
    if (p->tplan) {  // A^T's values in their new order, then its plan's own copy
        const cudaError_t e = launch_transpose_values(p->dtype, p->nnz, p->t_src, nullptr, vals, nullptr, p->t_vals,
                                                      reinterpret_cast<cudaStream_t>(stream_handle));
        if (e != cudaSuccess) return cuda_fail(e, "spmv_plan_update_values");
        const spmv_status_t st = spmv_plan_update_values(p->tplan, p->t_vals, stream_handle);
        if (st != SPMV_OK) return st;
    }
    if (is_rgcsr(p->kernel) && p->rg_slots > 0) {
        // the pattern is unchanged: only the values move into the copy
        const cudaError_t e = launch_rgcsr_pack(p->dtype, p->m, p->row_ptr, p->col_idx, vals, p->g_log2, p->group_ptr,
                                                p->row_len, p->perm, p->rg_col, p->rg_val, false,
                                                reinterpret_cast<cudaStream_t>(stream_handle));
        if (e != cudaSuccess) return cuda_fail(e, "spmv_plan_update_values");
    }
    return SPMV_OK;
}

spmv_status_t spmv_plan_destroy(spmv_plan_t p) {
    if (!p) return SPMV_OK;
    destroy_plan(p);
    return SPMV_OK;
}

spmv_status_t spmv_plan_info(spmv_plan_t p, spmv_plan_info_t *info) {
    if (!p || !info) return fail(SPMV_ERR_INVALID_ARG, "plan or info is NULL");
    std::memset(info, 0, sizeof *info);
    info->m = p->m;
    info->n = p->n;
    info->nnz = p->nnz;
    info->dtype = p->dtype;
    info->kernel = p->kernel;
    info->threads_per_tile = merge_path_threads();
    info->items_per_thread = p->ipt;
    info->rgcsr_group = p->rgcsr_group;
    info->items_per_tile = p->tile;
    info->num_tiles = p->num_tiles;
    info->num_long_rows = p->num_long_rows;
    info->launches_per_execute = p->m > 0 ? 1 + (p->num_long_rows > 0 ? 1 : 0) : 0;
    info->workspace_bytes = (int64_t)(p->arena_bytes + p->aux_bytes + p->rg_bytes + p->spmm_bytes + p->tr_bytes);
    info->transposed_kernel = p->tplan ? p->tplan->kernel : -1;
    if (p->tplan) {
        spmv_plan_info_t ti;
        spmv_plan_info(p->tplan, &ti);
        info->transposed_launches = ti.launches_per_execute;
    }
    info->stats = p->stats;
    info->long_row_min = p->num_long_rows > 0 ? p->long_min : 0;
    info->long_segment_nnz = kLongSegmentNnz;
    info->num_long_segments = p->num_segs;
    info->rgcsr_slots = p->rg_slots;
    return SPMV_OK;
}

spmv_status_t spmv_plan_device_status(spmv_plan_t p, int32_t *flags) {
    if (!p || !flags) return fail(SPMV_ERR_INVALID_ARG, "plan or flags is NULL");
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(flags, p->device_error, sizeof(int32_t), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "spmv_plan_device_status");
    return SPMV_OK;
}

spmv_status_t spmv_plan_export(spmv_plan_t p, spmv_export_t what, void *dst, size_t bytes, size_t *needed) {
    if (!p) return fail(SPMV_ERR_INVALID_ARG, "plan is NULL");
    const void *src = nullptr;
    size_t size = 0;
    switch (what) {
    case SPMV_EXPORT_PARTITION:
        if (!p->has_partition) return fail(SPMV_ERR_INVALID_ARG, "plan has no merge-path partition");
        src = p->part;
        size = sizeof(int2) * (size_t)(p->num_tiles + 1);
        break;
    case SPMV_EXPORT_RG_GROUP_PTR:
    case SPMV_EXPORT_RG_ROW_LEN:
    case SPMV_EXPORT_RG_COL:
    case SPMV_EXPORT_RG_VAL:
        if (!is_rgcsr(p->kernel)) return fail(SPMV_ERR_INVALID_ARG, "plan has no Row-grouped copy");
        if (what == SPMV_EXPORT_RG_GROUP_PTR) {
            src = p->group_ptr;
            size = sizeof(int64_t) * (size_t)(p->ngroups + 1);
        } else if (what == SPMV_EXPORT_RG_ROW_LEN) {
            src = p->row_len;
            size = sizeof(int32_t) * (size_t)p->m;
        } else if (what == SPMV_EXPORT_RG_COL) {
            src = p->rg_col;
            size = sizeof(int32_t) * (size_t)p->rg_slots;
        } else {
            src = p->rg_val;
            size = value_size(p->dtype) * (size_t)p->rg_slots;
        }
        break;
    case SPMV_EXPORT_LONG_ROWS:
    case SPMV_EXPORT_LONG_SEG_BEGIN:
        if (!is_rgcsr(p->kernel) && p->kernel != SPMV_KERNEL_LONG_ROWS)
            return fail(SPMV_ERR_INVALID_ARG, "plan has no long-row list");
        if (what == SPMV_EXPORT_LONG_ROWS) {
            src = p->long_rows;
            size = sizeof(int32_t) * (size_t)p->num_long_rows;
        } else {
            src = p->seg_begin;
            size = p->num_long_rows > 0 ? sizeof(int64_t) * (size_t)(p->num_long_rows + 1) : 0;
        }
        break;
    case SPMV_EXPORT_T_PTR:
    case SPMV_EXPORT_T_IDX:
    case SPMV_EXPORT_T_VALS:
    case SPMV_EXPORT_T_SRC:
        if (!p->tr) return fail(SPMV_ERR_INVALID_ARG, "plan has no transpose");
        if (what == SPMV_EXPORT_T_PTR) {
            src = p->t_ptr;
            size = sizeof(int32_t) * ((size_t)p->n + 1);
        } else if (what == SPMV_EXPORT_T_IDX) {
            src = p->t_idx;
            size = sizeof(int32_t) * (size_t)p->nnz;
        } else if (what == SPMV_EXPORT_T_SRC) {
            src = p->t_src;
            size = sizeof(int32_t) * (size_t)p->nnz;
        } else {
            src = p->t_vals;
            size = value_size(p->dtype) * (size_t)p->nnz;
        }
        break;
    case SPMV_EXPORT_RG_PERM:
        if (p->kernel != SPMV_KERNEL_RGCSR_SORTED) return fail(SPMV_ERR_INVALID_ARG, "plan has no row order");
        src = p->perm;
        size = sizeof(int32_t) * (size_t)p->m;
        break;
    default: return fail(SPMV_ERR_INVALID_ARG, "plan does not hold this array");
    }
    if (needed) *needed = size;
    if (!dst) return SPMV_OK;
    if (bytes < size) return fail(SPMV_ERR_INVALID_ARG, "destination too small");
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess && size) e = cudaMemcpy(dst, src, size, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "spmv_plan_export");
    return SPMV_OK;
}

}  // extern "C"
