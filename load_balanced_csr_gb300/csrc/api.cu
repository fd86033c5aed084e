// C ABI of the load-balanced CSR SpMV library: plan creation (analysis,
// kernel choice, schedule), execution, inspection.  Declarations and the
// contract of every entry point are in include/spmv.h.
//
// Memory: a plan makes its device allocations once, at creation, in one
// arena (OpSparse, section 5.1: all metadata sized up front and allocated
// with one cudaMalloc, since allocation is far slower than use), plus a
// second allocation only for kernels that keep a reordered copy of A.
// spmv_execute allocates and frees nothing and never waits for the device.
#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "row_spmm.cuh"
#include "spgemm.cuh"

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
    // SpMM over long rows (rows longer than kRowSpmmMaxLen): their list,
    // segments, partials and arrival counters, one allocation
    void *spmm_long = nullptr;
    size_t spmm_long_bytes = 0;
    int32_t spmm_num_long = 0;
    int64_t spmm_num_segs = 0;
    int32_t *spmm_long_rows = nullptr;
    int64_t *spmm_seg_begin = nullptr;
    void *spmm_seg_partial = nullptr;
    int32_t *spmm_long_arrivals = nullptr;
    // SpMM over the long rows a Row-grouped plan leaves out: k-wide segment
    // partials (32 values per segment) and arrival counters
    void *spmm_rg_long = nullptr;
    int32_t *spmm_rg_arrivals = nullptr;
    int32_t *rg_col = nullptr;       // [rg_slots]
    void *rg_val = nullptr;          // [rg_slots]

    spmv_row_stats_t stats{};
};

// SpGEMM handle: the borrowed patterns, the binning and the symbolic
// result, and the dense-bin scratch.
struct spmv_spgemm_s {
    int32_t m = 0, k = 0, n = 0, a_nnz = 0, b_nnz = 0;
    spmv_dtype_t dtype = SPMV_F32;
    int64_t c_nnz = 0, products = 0;
    void *arena = nullptr;
    size_t arena_bytes = 0;
    void *dense = nullptr;     // the slots of a wave of dense rows
    size_t dense_bytes = 0;
    void *layout = nullptr;    // dense bin: entry space, pieces, segments
    void *pieces = nullptr;    // the pieces when they outgrow their place in `layout`
    size_t layout_bytes = 0;
    int64_t dense_pieces = 0;
    std::vector<int64_t> wave_row, wave_piece;  // HOST, [waves + 1]
    SpgemmArgs args{};
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


// ---------------------------------------------------------------- fault injection
// Host-side failures injected into plan and SpGEMM-handle creation, so that
// tests can walk every clean-up path without faulting a GPU.  With
// SPMV_FAULT=alloc:N the N-th device allocation of a creation call fails as
// if the device were out of memory; with SPMV_FAULT=launch:N its N-th launch
// step reports a launch failure without launching anything.  The variable
// is read at the start of each creation call and counts on the calling
// thread; unset (the normal case) it costs one getenv per creation.
struct FaultPlan {
    int kind = 0;  // 1: allocation, 2: launch step
    long long at = 0;
    long long allocs = 0, launches = 0;
};
thread_local FaultPlan g_fault;

void fault_arm() {
    g_fault = FaultPlan{};
    const char *v = getenv("SPMV_FAULT");
    if (!v) return;
    if (!strncmp(v, "alloc:", 6)) g_fault.kind = 1, g_fault.at = atoll(v + 6);
    else if (!strncmp(v, "launch:", 7)) g_fault.kind = 2, g_fault.at = atoll(v + 7);
}

template <typename T>
cudaError_t dev_malloc(T **ptr, size_t bytes) {
    if (g_fault.kind == 1 && ++g_fault.allocs == g_fault.at) {
        *ptr = nullptr;
        return cudaErrorMemoryAllocation;
    }
    return cudaMalloc(reinterpret_cast<void **>(ptr), bytes);
}

bool launch_fault() { return g_fault.kind == 2 && ++g_fault.launches == g_fault.at; }

// Arms the injection for one creation call and disarms it on return (a
// plan's creation of the plan for its transpose counts as part of it).
thread_local int g_fault_depth = 0;
struct FaultScope {
    FaultScope() {
        if (g_fault_depth++ == 0) fault_arm();
    }
    ~FaultScope() {
        if (--g_fault_depth == 0) g_fault = FaultPlan{};
    }
};

}  // namespace

// A launch step of a creation call (the injected failure skips the launch).
#define LAUNCH(call) (launch_fault() ? cudaErrorLaunchFailure : (call))

namespace {

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
// `why`, when given, receives the rule that decided.
spmv_kernel_t choose_kernel(const spmv_plan_s &p, const char **why = nullptr) {
    const spmv_row_stats_t &s = p.stats;
    const char *unused = nullptr;
    const char *&rule = why ? *why : unused;
    if (p.n == 1 && s.max_len <= 32) {
        rule = "one column, rows of at most 32";
        return SPMV_KERNEL_THREAD_ROW;
    }
    if ((p.m < 500 || p.n < 500) && p.nnz < 10000 && s.max_len <= 256) {
        rule = "small matrix (rows or columns < 500, nnz < 10000)";
        return SPMV_KERNEL_THREAD_ROW;
    }
    if (p.m <= 65536 && s.max_len <= 64) {
        rule = "at most 65536 rows of at most 64";
        return SPMV_KERNEL_THREAD_ROW;
    }
    if (p.nnz > 0 && (double)s.rg_slots[0] <= 1.1 * (double)p.nnz) {
        rule = "Row-grouped copy pads at most 10 %";
        return SPMV_KERNEL_RGCSR;
    }
    rule = "default";
    return SPMV_KERNEL_MERGE_PATH;
}

const char *kernel_name(spmv_kernel_t k) {
    switch (k) {
    case SPMV_KERNEL_MERGE_PATH: return "merge_path";
    case SPMV_KERNEL_THREAD_ROW: return "thread_row";
    case SPMV_KERNEL_RGCSR: return "rgcsr";
    case SPMV_KERNEL_LONG_ROWS: return "long_rows";
    case SPMV_KERNEL_RGCSR_SORTED: return "rgcsr_sorted";
    case SPMV_KERNEL_GROUP_MAPPED: return "group_mapped";
    default: return "?";
    }
}

// SPMV_LOG=1: one line per plan on stderr with its statistics and the
// kernel choice (read at each creation; unset, it costs one getenv).
void log_plan(const spmv_plan_s &p, const char *why) {
    if (env_int("SPMV_LOG", 0) == 0) return;
    const spmv_row_stats_t &s = p.stats;
    const double fill = p.nnz > 0 ? (double)s.rg_slots[0] / (double)p.nnz - 1.0 : 0.0;
    std::fprintf(stderr,
                 "spmv plan: m=%d n=%d nnz=%d %s rows[min=%d max=%d mean=%.2f empty=%d] bandwidth=%d "
                 "rgcsr32_fill=%.3f -> kernel=%s (%s) items_per_thread=%d tiles=%lld long_rows=%d\n",
                 p.m, p.n, p.nnz, p.dtype == SPMV_F64 ? "f64" : "f32", s.min_len, s.max_len,
                 p.m > 0 ? (double)s.sum_len / p.m : 0.0, s.n_empty, s.bandwidth, fill, kernel_name(p.kernel), why,
                 p.ipt, (long long)p.num_tiles, p.num_long_rows);
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
    if (p->spmm_long) cudaFree(p->spmm_long);
    if (p->spmm_rg_long) cudaFree(p->spmm_rg_long);
    if (p->arena) cudaFree(p->arena);
    delete p;
}

constexpr int32_t kDefaultLongRowMin = 512;

// A creation call that fails after launching work waits for that work
// before it frees the memory the work writes.
void abandon_plan(spmv_plan_s *p, cudaStream_t stream) {
    cudaStreamSynchronize(stream);
    destroy_plan(p);
}

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
    cudaError_t e = dev_malloc(&p->aux, p->aux_bytes);
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
        e = LAUNCH(launch_long_rows_count(m, p->row_ptr, p->long_min, chunk_rows, chunk_segs, stream));
        if (e == cudaSuccess) e = LAUNCH(launch_exclusive_scan(chunk_rows, nc, chunk_row_off, scratch, stream));
        if (e == cudaSuccess) e = LAUNCH(launch_exclusive_scan(chunk_segs, nc, chunk_seg_off, scratch, stream));
        if (e == cudaSuccess)
            e = LAUNCH(launch_long_rows_scatter(m, p->row_ptr, p->long_min, chunk_row_off, chunk_seg_off, p->long_rows,
                                         p->seg_begin, stream));
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(&sizes[0], chunk_row_off + nc, sizeof(int64_t), cudaMemcpyDeviceToHost, stream);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(&sizes[1], chunk_seg_off + nc, sizeof(int64_t), cudaMemcpyDeviceToHost, stream);
    }
    if (e == cudaSuccess && rgcsr && m > 0) {
        if (sorted)
            e = LAUNCH(launch_window_sort(m, p->row_ptr, has_long ? p->long_min : 0, p->perm, p->row_len, gsize, stream));
        else
            e = LAUNCH(launch_rgcsr_lengths(m, p->row_ptr, p->g_log2, has_long ? p->long_min : 0, p->row_len, gsize,
                                     stream));
        if (e == cudaSuccess) e = LAUNCH(launch_exclusive_scan(gsize, p->ngroups, p->group_ptr, scratch, stream));
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
        e = dev_malloc(&p->rg, p->rg_bytes);
        if (e != cudaSuccess) {
            p->rg = nullptr;
            return fail(SPMV_ERR_ALLOC, std::string("cudaMalloc of the Row-grouped copy: ") + cudaGetErrorString(e));
        }
        p->rg_col = static_cast<int32_t *>(p->rg);
        p->rg_val = static_cast<char *>(p->rg) + col_bytes;
        e = cudaMemsetAsync(p->rg, 0, p->rg_bytes, stream);  // pads: column 0, value 0
        if (e == cudaSuccess)
            e = LAUNCH(launch_rgcsr_pack(p->dtype, m, p->row_ptr, p->col_idx, p->vals, p->g_log2, p->group_ptr, p->row_len,
                                  p->perm, p->rg_col, p->rg_val, true, stream));
        if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
        if (e != cudaSuccess) return cuda_fail(e, "Row-grouped copy");
    }
    return SPMV_OK;
}

// A^T in CSR form (one allocation the plan keeps), built with a temporary
// scratch, and a plan of its own for it.
// The long rows of SpMM: rows of at least kSpmmLongMin nonzeros, listed
// with the same two passes as the long rows of SpMV, with segment partials
// of 32 values (one slice of columns).
spmv_status_t build_spmm_long_rows(spmv_plan_s *p, cudaStream_t stream) {
    const int32_t m = p->m;
    const size_t vs = value_size(p->dtype);
    const int nc = long_rows_num_chunks(m);
    const int64_t long_ub = rows_at_least(p->stats, kSpmmLongMin);
    const int64_t segs_ub = (int64_t)p->nnz / kLongSegmentNnz + long_ub;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = align_up(off + bytes, 256);
        return o;
    };
    const size_t o_long = take(sizeof(int32_t) * long_ub);
    const size_t o_segb = take(sizeof(int64_t) * (long_ub + 1));
    const size_t o_segp = take(vs * 32 * segs_ub);
    const size_t o_larr = take(sizeof(int32_t) * long_ub);
    const size_t o_crow = take(sizeof(int64_t) * nc);
    const size_t o_cseg = take(sizeof(int64_t) * nc);
    const size_t o_crow_off = take(sizeof(int64_t) * (nc + 1));
    const size_t o_cseg_off = take(sizeof(int64_t) * (nc + 1));
    const size_t o_scr = take(sizeof(int64_t) * scan_scratch_elems(nc));
    p->spmm_long_bytes = off;
    cudaError_t e = dev_malloc(&p->spmm_long, p->spmm_long_bytes);
    if (e != cudaSuccess) {
        p->spmm_long = nullptr;
        return fail(SPMV_ERR_ALLOC, std::string("cudaMalloc of the SpMM long-row workspace: ") + cudaGetErrorString(e));
    }
    char *base = static_cast<char *>(p->spmm_long);
    p->spmm_long_rows = reinterpret_cast<int32_t *>(base + o_long);
    p->spmm_seg_begin = reinterpret_cast<int64_t *>(base + o_segb);
    p->spmm_seg_partial = base + o_segp;
    p->spmm_long_arrivals = reinterpret_cast<int32_t *>(base + o_larr);
    int64_t *chunk_rows = reinterpret_cast<int64_t *>(base + o_crow);
    int64_t *chunk_segs = reinterpret_cast<int64_t *>(base + o_cseg);
    int64_t *chunk_row_off = reinterpret_cast<int64_t *>(base + o_crow_off);
    int64_t *chunk_seg_off = reinterpret_cast<int64_t *>(base + o_cseg_off);
    int64_t *scratch = reinterpret_cast<int64_t *>(base + o_scr);
    int64_t sizes[2] = {0, 0};
    e = cudaMemsetAsync(p->spmm_long_arrivals, 0, sizeof(int32_t) * long_ub, stream);
    if (e == cudaSuccess) e = LAUNCH(launch_long_rows_count(m, p->row_ptr, kSpmmLongMin, chunk_rows, chunk_segs, stream));
    if (e == cudaSuccess) e = LAUNCH(launch_exclusive_scan(chunk_rows, nc, chunk_row_off, scratch, stream));
    if (e == cudaSuccess) e = LAUNCH(launch_exclusive_scan(chunk_segs, nc, chunk_seg_off, scratch, stream));
    if (e == cudaSuccess)
        e = LAUNCH(launch_long_rows_scatter(m, p->row_ptr, kSpmmLongMin, chunk_row_off, chunk_seg_off, p->spmm_long_rows,
                                     p->spmm_seg_begin, stream));
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(&sizes[0], chunk_row_off + nc, sizeof(int64_t), cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(&sizes[1], chunk_seg_off + nc, sizeof(int64_t), cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, "SpMM long rows");
    if (sizes[0] > long_ub || sizes[1] > segs_ub) return fail(SPMV_ERR_CUDA, "SpMM long-row count exceeds its bound");
    p->spmm_num_long = (int32_t)sizes[0];
    p->spmm_num_segs = sizes[1];
    return SPMV_OK;
}

spmv_status_t build_transpose(spmv_plan_s *p, cudaStream_t stream) {
    const size_t vs = value_size(p->dtype);
    const size_t o_ptr = 0;
    const size_t o_idx = align_up(o_ptr + sizeof(int32_t) * ((size_t)p->n + 1), 256);
    const size_t o_src = align_up(o_idx + sizeof(int32_t) * (size_t)p->nnz, 256);
    const size_t o_val = align_up(o_src + sizeof(int32_t) * (size_t)p->nnz, 256);
    p->tr_bytes = align_up(o_val + vs * (size_t)p->nnz, 256);
    cudaError_t e = dev_malloc(&p->tr, p->tr_bytes);
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
    e = dev_malloc(&scratch, (size_t)transpose_scratch_bytes(p->n, p->nnz));
    if (e != cudaSuccess) return fail(SPMV_ERR_ALLOC, std::string("cudaMalloc of the transpose scratch: ") + cudaGetErrorString(e));
    e = LAUNCH(launch_transpose(p->dtype, p->m, p->n, p->nnz, p->row_ptr, p->col_idx, p->vals, scratch, p->t_ptr, p->t_idx,
                         p->t_vals, p->t_src, stream));
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
    a.n = p->n;
    a.error = p->device_error;
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
    FaultScope fault_scope;
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
    e = dev_malloc(&p->arena, p->arena_bytes);
    if (e != cudaSuccess) {
        p->arena = nullptr;
        abandon_plan(p, stream);
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
    if (e == cudaSuccess) e = LAUNCH(launch_row_stats(m, n, nnz, row_ptr, col_idx, partials, stats_ctas, d_stats, stream));
    if (e == cudaSuccess) e = cudaMemcpyAsync(&p->stats, d_stats, sizeof(spmv_row_stats_t), cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) {
        abandon_plan(p, stream);
        return cuda_fail(e, "plan analysis");
    }
    if (p->stats.flags) {
        const int f = p->stats.flags;
        abandon_plan(p, stream);
        char msg[160];
        std::snprintf(msg, sizeof msg, "invalid CSR:%s%s%s%s", (f & 1) ? " row_ptr[0] != 0;" : "",
                      (f & 2) ? " row_ptr decreases;" : "", (f & 4) ? " row_ptr[m] != nnz;" : "",
                      (f & 8) ? " column index outside [0, n);" : "");
        return fail(SPMV_ERR_INVALID_CSR, msg);
    }

    // ---- kernel choice and schedule
    const char *why = "forced";
    p->kernel = forced != SPMV_KERNEL_AUTO ? forced : choose_kernel(*p, &why);
    p->ipt = ipt_forced ? ipt_forced : merge_path_choose_items(dtype, n, p->stats);
    p->tile = (int64_t)merge_path_threads() * p->ipt;
    p->num_tiles = total > 0 ? (total + p->tile - 1) / p->tile : 1;
    p->with_spmm = opt.with_spmm != 0;
    if ((p->kernel == SPMV_KERNEL_MERGE_PATH || p->with_spmm) && m > 0) {
        e = LAUNCH(launch_merge_path_partition(m, nnz, row_ptr, p->tile, p->num_tiles, p->part, stream));
        if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
        if (e != cudaSuccess) {
            abandon_plan(p, stream);
            return cuda_fail(e, "merge-path partition");
        }
        p->has_partition = true;
    }
    if (p->with_spmm && m > 0) {
        p->spmm_warps = spmm_warps(p->num_tiles);
        const size_t part_bytes = align_up(vs * kSpmmBlocks * 32 * (size_t)p->spmm_warps, 256);
        p->spmm_bytes = 2 * part_bytes + align_up(sizeof(int32_t) * (size_t)p->spmm_warps, 256);
        e = dev_malloc(&p->spmm, p->spmm_bytes);
        if (e != cudaSuccess) {
            p->spmm = nullptr;
            abandon_plan(p, stream);
            return fail(SPMV_ERR_ALLOC, std::string("cudaMalloc of the SpMM scratch: ") + cudaGetErrorString(e));
        }
        p->spmm_tail = p->spmm;
        p->spmm_head = static_cast<char *>(p->spmm) + part_bytes;
        p->spmm_arrivals = reinterpret_cast<int32_t *>(static_cast<char *>(p->spmm) + 2 * part_bytes);
        e = cudaMemsetAsync(p->spmm_arrivals, 0, sizeof(int32_t) * (size_t)p->spmm_warps, stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
        if (e != cudaSuccess) {
            abandon_plan(p, stream);
            return cuda_fail(e, "SpMM scratch");
        }
    }
    if (p->with_spmm && m > 0 && p->stats.max_len > kRowSpmmMaxLen) {
        const spmv_status_t st = build_spmm_long_rows(p, stream);
        if (st != SPMV_OK) {
            abandon_plan(p, stream);
            return st;
        }
    }
    if (opt.with_transpose) {
        const spmv_status_t st = build_transpose(p, stream);
        if (st != SPMV_OK) {
            abandon_plan(p, stream);
            return st;
        }
    }
    if (is_rgcsr(p->kernel) || p->kernel == SPMV_KERNEL_LONG_ROWS) {
        const spmv_status_t st = build_row_layouts(p, opt, stream);
        if (st != SPMV_OK) {
            abandon_plan(p, stream);
            return st;
        }
    }
    if (p->with_spmm && is_rgcsr(p->kernel) && p->num_long_rows > 0) {
        // SpMM partials for the long rows the Row-grouped copy leaves out
        const size_t part = align_up(value_size(dtype) * 32 * (size_t)p->num_segs, 256);
        e = dev_malloc(&p->spmm_rg_long, part + sizeof(int32_t) * (size_t)p->num_long_rows);
        if (e != cudaSuccess) {
            p->spmm_rg_long = nullptr;
            abandon_plan(p, stream);
            return fail(SPMV_ERR_ALLOC, std::string("cudaMalloc of the SpMM long-row partials: ") + cudaGetErrorString(e));
        }
        p->spmm_rg_arrivals = reinterpret_cast<int32_t *>(static_cast<char *>(p->spmm_rg_long) + part);
        e = cudaMemsetAsync(p->spmm_rg_arrivals, 0, sizeof(int32_t) * (size_t)p->num_long_rows, stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
        if (e != cudaSuccess) {
            abandon_plan(p, stream);
            return cuda_fail(e, "SpMM long-row partials");
        }
    }
    log_plan(*p, why);
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
        e = LAUNCH(launch_thread_per_row(p->dtype, p->m, p->n, p->row_ptr, p->col_idx, p->vals, x, y, alpha, beta, 0,
                                         p->device_error, stream));
        break;
    case SPMV_KERNEL_GROUP_MAPPED:
        e = LAUNCH(launch_group_mapped(p->dtype, p->m, p->n, p->row_ptr, p->col_idx, p->vals, x, y, alpha, beta,
                                       p->device_error, stream));
        break;
    case SPMV_KERNEL_LONG_ROWS:
        // long rows first (they take longest), then the others
        if (p->num_long_rows > 0) e = LAUNCH(launch_long_part(p, x, y, alpha, beta, stream));
        if (e == cudaSuccess)
            e = LAUNCH(launch_thread_per_row(p->dtype, p->m, p->n, p->row_ptr, p->col_idx, p->vals, x, y, alpha, beta,
                                             p->num_long_rows > 0 ? p->long_min : 0, p->device_error, stream));
        break;
    case SPMV_KERNEL_RGCSR:
    case SPMV_KERNEL_RGCSR_SORTED:
        if (p->num_long_rows > 0) e = LAUNCH(launch_long_part(p, x, y, alpha, beta, stream));
        if (e == cudaSuccess)
            e = LAUNCH(launch_rgcsr_spmv(p->dtype, p->m, p->n, p->g_log2, p->group_ptr, p->row_len, p->perm, p->rg_col, p->rg_val,
                                  x, y, alpha, beta, p->device_error, stream));
        break;
    case SPMV_KERNEL_MERGE_PATH:
    default: {
        MergePathArgs a;
        a.m = p->m;
        a.n = p->n;
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
        e = LAUNCH(launch_merge_path_spmv(p->dtype, p->ipt, a, stream));
        break;
    }
    }
    if (e != cudaSuccess) return cuda_fail(e, "spmv_execute launch");
    return SPMV_OK;
}

spmv_status_t spmv_execute_host(spmv_plan_t p, double alpha, const void *x_host, double beta, void *y_host,
                                void *x_dev, void *y_dev, spmv_stream_t stream_handle) {
    if (!p) return fail(SPMV_ERR_INVALID_ARG, "plan is NULL");
    if (p->m == 0) return SPMV_OK;
    if (!y_host || !y_dev) return fail(SPMV_ERR_INVALID_ARG, "y_host or y_dev is NULL");
    if (p->nnz > 0 && (!x_host || !x_dev)) return fail(SPMV_ERR_INVALID_ARG, "x_host or x_dev is NULL");
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_handle);
    const size_t vs = value_size(p->dtype);
    cudaError_t e = cudaSuccess;
    if (p->nnz > 0) e = cudaMemcpyAsync(x_dev, x_host, vs * (size_t)p->n, cudaMemcpyHostToDevice, stream);
    // y is read when beta, rounded to the value type, is not zero
    const bool reads_y = p->dtype == SPMV_F64 ? beta != 0.0 : (float)beta != 0.0f;
    if (e == cudaSuccess && reads_y)
        e = cudaMemcpyAsync(y_dev, y_host, vs * (size_t)p->m, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return cuda_fail(e, "spmv_execute_host copy to the device");
    const spmv_status_t st = spmv_execute(p, alpha, p->nnz > 0 ? x_dev : nullptr, beta, y_dev, stream_handle);
    if (st != SPMV_OK) return st;
    e = cudaMemcpyAsync(y_host, y_dev, vs * (size_t)p->m, cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return cuda_fail(e, "spmv_execute_host copy to the host");
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
    // Row-grouped plans: long rows, if any, must be rare (as for the CSR path:
    // a power-law matrix forced onto the window-sorted copy took 5.3 ms at
    // k = 32 against 3.1 ms on the merge path)
    const bool rg_long_ok = p->num_long_rows == 0 ||
                            (p->spmm_rg_long && (int64_t)p->num_long_rows * kSpmmRowsPerLongRow <= p->m);
    if (is_rgcsr(p->kernel) && p->g_log2 == 5 && rg_long_ok && (p->rg_slots > 0 || p->nnz == 0)) {
        // the Row-grouped copy serves SpMM too, in slices of 32 (fp32) or 16
        // (fp64) columns, each slice reading the matrix again (27-point
        // stencil 128^3: k = 8 in 174 us against 612 us on the merge path)
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
        cudaError_t e = cudaSuccess;
        if (p->num_long_rows > 0) {  // the rows the copy leaves out
            LongSpmmArgs l;
            l.k = k;
            l.row_ptr = p->row_ptr;
            l.col_idx = p->col_idx;
            l.vals = p->vals;
            l.X = X;
            l.ldx = ldx;
            l.Y = Y;
            l.ldy = ldy;
            l.alpha = alpha;
            l.beta = beta;
            l.num_long = p->num_long_rows;
            l.num_segs = p->num_segs;
            l.long_rows = p->long_rows;
            l.seg_begin = p->seg_begin;
            l.seg_partial = p->spmm_rg_long;
            l.arrivals = p->spmm_rg_arrivals;
            e = LAUNCH(launch_long_spmm(p->dtype, l, reinterpret_cast<cudaStream_t>(stream_handle)));
        }
        if (e == cudaSuccess) e = LAUNCH(launch_rg_spmm(p->dtype, r, reinterpret_cast<cudaStream_t>(stream_handle)));
        if (e != cudaSuccess) return cuda_fail(e, "spmv_execute_multi launch");
        return SPMV_OK;
    }
    // with long rows, at most two slices of columns (each slice reads the
    // matrix again; skew, fp64, k = 128 in 8 slices: 24.4 ms against 23.3 ms
    // on the merge path)
    const bool rare_long = p->spmm_num_long > 0 && (int64_t)p->spmm_num_long * kSpmmRowsPerLongRow <= p->m &&
                           k <= (p->dtype == SPMV_F64 ? 32 : 64);
#ifndef LBCSR_SPMM_CSR_PATH
#define LBCSR_SPMM_CSR_PATH 1  // 0: the merge-path SpMM takes these matrices too (tuning)
#endif
    if (LBCSR_SPMM_CSR_PATH && (p->stats.max_len <= kRowSpmmMaxLen || rare_long) &&
        row_spmm_supported(p->dtype, k, X, ldx, Y, ldy)) {
        // a warp per 32 rows straight from CSR, lanes sharing X rows; rows
        // longer than kRowSpmmMaxLen, if any, by a warp per 4096-nonzero segment
        RowSpmmArgs r;
        r.m = p->m;
        r.k = k;
        r.row_ptr = p->row_ptr;
        r.col_idx = p->col_idx;
        r.vals = p->vals;
        r.X = X;
        r.ldx = ldx;
        r.Y = Y;
        r.ldy = ldy;
        r.alpha = alpha;
        r.beta = beta;
        r.long_min = kSpmmLongMin;
        r.num_long = p->spmm_num_long;
        r.num_segs = p->spmm_num_segs;
        r.long_rows = p->spmm_long_rows;
        r.seg_begin = p->spmm_seg_begin;
        r.seg_partial = p->spmm_seg_partial;
        r.arrivals = p->spmm_long_arrivals;
        const cudaError_t e = LAUNCH(launch_row_spmm(p->dtype, r, reinterpret_cast<cudaStream_t>(stream_handle)));
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
    const cudaError_t e = LAUNCH(launch_spmm(p->dtype, a, reinterpret_cast<cudaStream_t>(stream_handle)));
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
        const cudaError_t e = LAUNCH(launch_transpose_values(p->dtype, p->nnz, p->t_src, nullptr, vals, nullptr, p->t_vals,
                                                      reinterpret_cast<cudaStream_t>(stream_handle)));
        if (e != cudaSuccess) return cuda_fail(e, "spmv_plan_update_values");
        const spmv_status_t st = spmv_plan_update_values(p->tplan, p->t_vals, stream_handle);
        if (st != SPMV_OK) return st;
    }
    if (is_rgcsr(p->kernel) && p->rg_slots > 0) {
        // the pattern is unchanged: only the values move into the copy
        const cudaError_t e = LAUNCH(launch_rgcsr_pack(p->dtype, p->m, p->row_ptr, p->col_idx, vals, p->g_log2, p->group_ptr,
                                                p->row_len, p->perm, p->rg_col, p->rg_val, false,
                                                reinterpret_cast<cudaStream_t>(stream_handle)));
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
    info->workspace_bytes =
        (int64_t)(p->arena_bytes + p->aux_bytes + p->rg_bytes + p->spmm_bytes + p->spmm_long_bytes + p->tr_bytes);
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
    if (p->kernel == SPMV_KERNEL_MERGE_PATH && p->m > 0) {
        const bool aligned = reinterpret_cast<uintptr_t>(p->row_ptr) % 16 == 0 &&
                             reinterpret_cast<uintptr_t>(p->col_idx) % 16 == 0 &&
                             reinterpret_cast<uintptr_t>(p->vals) % 16 == 0;
        info->merge_path_warps = merge_path_num_warps(p->dtype, p->ipt, aligned, p->num_tiles);
    }
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

// ---------------------------------------------------------------- SpGEMM

static void destroy_spgemm(spmv_spgemm_s *h) {
    if (!h) return;
    cudaDeviceSynchronize();
    if (h->arena) cudaFree(h->arena);
    if (h->dense) cudaFree(h->dense);
    if (h->layout) cudaFree(h->layout);
    if (h->pieces) cudaFree(h->pieces);
    delete h;
}

// The dense bin's layout (see spgemm.cu): entry offsets of the dense rows,
// products before each entry, pieces and their first entries, waves, and
// the slots of one wave.  Synchronises the stream.
static spmv_status_t spgemm_dense_plan(spmv_spgemm_s *h, cudaStream_t stream) {
    SpgemmArgs &a = h->args;
    const int64_t D = a.bin_count[kSpgemmBins - 1];
    int64_t before = 0;
    for (int b = 0; b < kSpgemmBins - 1; ++b) before += a.bin_count[b];
    const int32_t *drows = a.bin_rows + before;
    const size_t vs = value_size(h->dtype);

    // entries of A of the dense rows: e_off, then their products: pp
    int64_t *tmp = nullptr;
    const int64_t scan_d = scan_scratch_elems(D);
    cudaError_t e = dev_malloc(&tmp, sizeof(int64_t) * (size_t)(2 * (D + 1) + scan_d));
    if (e != cudaSuccess) return fail(SPMV_ERR_ALLOC, std::string("cudaMalloc of the SpGEMM dense layout: ") + cudaGetErrorString(e));
    int64_t *alen = tmp, *e_off_tmp = tmp + (D + 1), *scan_tmp = tmp + 2 * (D + 1);
    int64_t entries = 0;
    e = LAUNCH(launch_spgemm_dense_layout(a, drows, D, alen, e_off_tmp, scan_tmp, stream));
    if (e == cudaSuccess) e = cudaMemcpyAsync(&entries, e_off_tmp + D, sizeof(int64_t), cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) {
        cudaFree(tmp);
        return cuda_fail(e, "SpGEMM dense layout");
    }
    // pieces: each dense row's products cut evenly into ceil(products / piece) parts.
    // The layout arena is sized for the most pieces the rows can need (known after
    // rowp), so rowp is computed in a first arena and the pieces in a second.
    const int64_t scan_e = scan_scratch_elems(std::max<int64_t>(entries, 1));
    size_t off = 0;
    const size_t o_eoff = off;
    off = align_up(off + sizeof(int64_t) * (size_t)(D + 1), 256);
    const size_t o_pp = off;
    off = align_up(off + sizeof(int64_t) * (size_t)(entries + 1), 256);
    const size_t o_rowp = off;
    off = align_up(off + sizeof(int64_t) * (size_t)(D + 1), 256);
    const size_t o_blen = off;  // scratch: B lengths, then the pieces
    off = align_up(off + sizeof(int64_t) * (size_t)std::max<int64_t>(entries, 1), 256);
    const size_t o_scan = off;
    off = align_up(off + sizeof(int64_t) * (size_t)scan_e, 256);
    const int64_t segs = spgemm_segments(h->n), nseg = D * segs;
    const size_t o_segcnt = off;
    off = align_up(off + sizeof(int64_t) * (size_t)nseg, 256);
    const size_t o_segoff = off;
    off = align_up(off + sizeof(int64_t) * (size_t)(nseg + 1), 256);
    const size_t o_segscan = off;
    off = align_up(off + sizeof(int64_t) * (size_t)scan_scratch_elems(nseg), 256);
    const size_t first_bytes = off;
    void *first = nullptr;
    e = dev_malloc(&first, first_bytes);
    if (e != cudaSuccess) {
        cudaFree(tmp);
        return fail(SPMV_ERR_ALLOC, std::string("cudaMalloc of the SpGEMM dense layout: ") + cudaGetErrorString(e));
    }
    char *fb = static_cast<char *>(first);
    int64_t *e_off = reinterpret_cast<int64_t *>(fb + o_eoff);
    int64_t *pp = reinterpret_cast<int64_t *>(fb + o_pp);
    int64_t *rowp = reinterpret_cast<int64_t *>(fb + o_rowp);
    std::vector<int64_t> h_rowp((size_t)D + 1);
    e = cudaMemcpyAsync(e_off, e_off_tmp, sizeof(int64_t) * (size_t)(D + 1), cudaMemcpyDeviceToDevice, stream);
    if (e == cudaSuccess)
        e = LAUNCH(launch_spgemm_dense_products(a, drows, D, e_off, entries, reinterpret_cast<int64_t *>(fb + o_blen), pp,
                                         rowp, reinterpret_cast<int64_t *>(fb + o_scan), stream));
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(h_rowp.data(), rowp, sizeof(int64_t) * (size_t)(D + 1), cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    cudaFree(tmp);
    h->layout = first;
    h->layout_bytes = first_bytes;
    if (e != cudaSuccess) return cuda_fail(e, "SpGEMM dense products");

    // pieces (HOST), then their first entries (device)
    const int64_t piece = spgemm_piece_products();
    std::vector<int32_t> piece_row;
    std::vector<int64_t> piece_k0, row_piece((size_t)D + 1);
    for (int64_t j = 0; j < D; ++j) {
        row_piece[(size_t)j] = (int64_t)piece_row.size();
        const int64_t k0 = h_rowp[(size_t)j], len = h_rowp[(size_t)j + 1] - k0;
        const int64_t np = std::max<int64_t>(1, (len + piece - 1) / piece);
        for (int64_t c = 0; c < np; ++c) {
            piece_row.push_back((int32_t)j);
            piece_k0.push_back(k0 + len * c / np);
        }
    }
    row_piece[(size_t)D] = (int64_t)piece_row.size();
    piece_k0.push_back(h_rowp[(size_t)D]);
    const int64_t P = (int64_t)piece_row.size();
    h->dense_pieces = P;
    // the pieces live in the blen + scan scratch of the first arena when they fit
    const size_t need = align_up(sizeof(int64_t) * (size_t)(P + 1), 256) + align_up(sizeof(int64_t) * (size_t)P, 256) +
                        align_up(sizeof(int32_t) * (size_t)P, 256);
    if (need > o_segcnt - o_blen) {
        // a separate allocation for the pieces
        void *more = nullptr;
        e = dev_malloc(&more, need);
        if (e != cudaSuccess) return fail(SPMV_ERR_ALLOC, std::string("cudaMalloc of the SpGEMM pieces: ") + cudaGetErrorString(e));
        h->pieces = more;
        h->layout_bytes += need;
    }
    char *pb = h->pieces ? static_cast<char *>(h->pieces) : fb + o_blen;
    int64_t *d_k0 = reinterpret_cast<int64_t *>(pb);
    int64_t *d_pe = reinterpret_cast<int64_t *>(pb + align_up(sizeof(int64_t) * (size_t)(P + 1), 256));
    int32_t *d_prow = reinterpret_cast<int32_t *>(reinterpret_cast<char *>(d_pe) + align_up(sizeof(int64_t) * (size_t)P, 256));
    e = cudaMemcpyAsync(d_k0, piece_k0.data(), sizeof(int64_t) * (size_t)(P + 1), cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(d_prow, piece_row.data(), sizeof(int32_t) * (size_t)P, cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess) e = LAUNCH(launch_spgemm_dense_locate(P, d_k0, pp, entries, d_pe, stream));
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, "SpGEMM pieces");
    a.dense_e_off = e_off;
    a.dense_pp = pp;
    a.dense_piece_k0 = d_k0;
    a.dense_piece_e = d_pe;
    a.dense_piece_row = d_prow;
    a.dense_segs = segs;
    a.dense_seg_cnt = reinterpret_cast<int64_t *>(fb + o_segcnt);
    a.dense_seg_off = reinterpret_cast<int64_t *>(fb + o_segoff);
    a.dense_seg_scan = reinterpret_cast<int64_t *>(fb + o_segscan);
    e = cudaMemsetAsync(a.dense_seg_cnt, 0, sizeof(int64_t) * (size_t)nseg, stream);
    if (e != cudaSuccess) return cuda_fail(e, "SpGEMM segments");

    // slots and waves
    const int32_t n = h->n;
    const size_t words = (size_t)spgemm_bit_words(n);
    const size_t per_slot = (size_t)n * vs + words * sizeof(unsigned);
    int64_t S = std::min<int64_t>(D, 1024);
    S = std::max<int64_t>(1, std::min<int64_t>(S, (int64_t)((size_t(8) << 30) / std::max<size_t>(per_slot, 1))));
    const size_t vals_bytes = align_up((size_t)n * vs * (size_t)S, 256);
    h->dense_bytes = vals_bytes + align_up(words * sizeof(unsigned) * (size_t)S, 256);
    e = dev_malloc(&h->dense, h->dense_bytes);
    if (e != cudaSuccess) {
        h->dense = nullptr;
        return fail(SPMV_ERR_ALLOC, std::string("cudaMalloc of the SpGEMM dense rows: ") + cudaGetErrorString(e));
    }
    e = cudaMemsetAsync(h->dense, 0, h->dense_bytes, stream);
    if (e != cudaSuccess) return cuda_fail(e, "SpGEMM dense rows");
    a.dense_slots = S;
    a.dense_vals = h->dense;
    a.dense_bits = reinterpret_cast<unsigned *>(static_cast<char *>(h->dense) + vals_bytes);
    h->wave_row.clear();
    h->wave_piece.clear();
    for (int64_t j = 0; j < D; j += S) {
        h->wave_row.push_back(j);
        h->wave_piece.push_back(row_piece[(size_t)j]);
    }
    h->wave_row.push_back(D);
    h->wave_piece.push_back(P);
    a.dense_waves = (int64_t)h->wave_row.size() - 1;
    a.h_wave_row = h->wave_row.data();
    a.h_wave_piece = h->wave_piece.data();
    return SPMV_OK;
}

spmv_status_t spmv_spgemm_create(spmv_spgemm_t *out, int32_t m, int32_t k, int32_t n, int32_t a_nnz,
                                 const int32_t *a_row_ptr, const int32_t *a_col_idx, int32_t b_nnz,
                                 const int32_t *b_row_ptr, const int32_t *b_col_idx, spmv_dtype_t dtype,
                                 int64_t *c_nnz, spmv_stream_t stream_handle) {
    g_last_error.clear();
    FaultScope fault_scope;
    if (!out) return fail(SPMV_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    if (!c_nnz) return fail(SPMV_ERR_INVALID_ARG, "c_nnz is NULL");
    if (m < 0 || k < 0 || n < 0 || a_nnz < 0 || b_nnz < 0) return fail(SPMV_ERR_INVALID_ARG, "negative size");
    if ((int64_t)m + a_nnz >= (1LL << 31) || (int64_t)k + b_nnz >= (1LL << 31))
        return fail(SPMV_ERR_INVALID_ARG, "m + a_nnz and k + b_nnz must be < 2^31");
    if (dtype != SPMV_F32 && dtype != SPMV_F64) return fail(SPMV_ERR_INVALID_ARG, "unknown dtype");
    if (!a_row_ptr || !b_row_ptr) return fail(SPMV_ERR_INVALID_ARG, "a_row_ptr or b_row_ptr is NULL");
    if ((a_nnz > 0 && !a_col_idx) || (b_nnz > 0 && !b_col_idx))
        return fail(SPMV_ERR_INVALID_ARG, "a_col_idx or b_col_idx is NULL");
    int dev = 0, major = 0, minor = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10 || minor != 3) return fail(SPMV_ERR_UNSUPPORTED, "this library is built for sm_103 (GB300) only");
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_handle);

    spmv_spgemm_s *h = new (std::nothrow) spmv_spgemm_s();
    if (!h) return fail(SPMV_ERR_ALLOC, "host allocation failed");
    h->m = m;
    h->k = k;
    h->n = n;
    h->a_nnz = a_nnz;
    h->b_nnz = b_nnz;
    h->dtype = dtype;

    // ---- one arena: checks of A and B, row products, bins, row sizes of C
    const int ctas_a = stats_num_ctas(m, a_nnz), ctas_b = stats_num_ctas(k, b_nnz);
    const int64_t chunks = spgemm_chunks(m);
    const int64_t scan_elems = std::max(scan_scratch_elems(kSpgemmBins * chunks), scan_scratch_elems(std::max<int64_t>(m, 1)));
    const size_t M = (size_t)std::max<int32_t>(m, 1);
    size_t off = 0;
    const size_t off_pa = off;
    off = align_up(off + sizeof(StatsPartial) * ctas_a, 256);
    const size_t off_pb = off;
    off = align_up(off + sizeof(StatsPartial) * ctas_b, 256);
    const size_t off_stats = off;
    off = align_up(off + 2 * sizeof(spmv_row_stats_t), 256);
    const size_t off_products = off;
    off = align_up(off + sizeof(int64_t) * M, 256);
    const size_t off_rows = off;
    off = align_up(off + sizeof(int32_t) * M, 256);
    const size_t off_num_rows = off;
    off = align_up(off + sizeof(int32_t) * M, 256);
    const size_t off_nnz = off;
    off = align_up(off + sizeof(int64_t) * (M + 1), 256);
    const size_t off_cptr = off;
    off = align_up(off + sizeof(int64_t) * (M + 1), 256);
    const size_t off_counts = off;
    off = align_up(off + sizeof(int64_t) * kSpgemmBins * chunks, 256);
    const size_t off_offsets = off;
    off = align_up(off + sizeof(int64_t) * (kSpgemmBins * chunks + 1), 256);
    const size_t off_scan = off;
    off = align_up(off + sizeof(int64_t) * scan_elems, 256);
    const size_t off_err = off;
    off = align_up(off + sizeof(int32_t), 256);
    h->arena_bytes = off;
    e = dev_malloc(&h->arena, h->arena_bytes);
    if (e != cudaSuccess) {
        h->arena = nullptr;
        cudaStreamSynchronize(stream);
        destroy_spgemm(h);
        return fail(SPMV_ERR_ALLOC, std::string("cudaMalloc of the SpGEMM workspace: ") + cudaGetErrorString(e));
    }
    char *base = static_cast<char *>(h->arena);
    spmv_row_stats_t *d_stats = reinterpret_cast<spmv_row_stats_t *>(base + off_stats);
    SpgemmArgs &a = h->args;
    a.m = m;
    a.n = n;
    a.a_ptr = a_row_ptr;
    a.a_col = a_col_idx;
    a.b_ptr = b_row_ptr;
    a.b_col = b_col_idx;
    a.products = reinterpret_cast<int64_t *>(base + off_products);
    a.bin_rows = reinterpret_cast<int32_t *>(base + off_rows);
    int32_t *num_rows = reinterpret_cast<int32_t *>(base + off_num_rows);
    a.num_bin_rows = num_rows;
    a.row_nnz = reinterpret_cast<int64_t *>(base + off_nnz);
    a.c_ptr = reinterpret_cast<int64_t *>(base + off_cptr);
    a.error = reinterpret_cast<int32_t *>(base + off_err);
    int64_t *counts = reinterpret_cast<int64_t *>(base + off_counts);
    int64_t *offsets = reinterpret_cast<int64_t *>(base + off_offsets);
    int64_t *scan = reinterpret_cast<int64_t *>(base + off_scan);

    // ---- checks of both patterns, read back once
    spmv_row_stats_t st[2];
    e = cudaMemsetAsync(base, 0, h->arena_bytes, stream);
    if (e == cudaSuccess)
        e = LAUNCH(launch_row_stats(m, k, a_nnz, a_row_ptr, a_col_idx, reinterpret_cast<StatsPartial *>(base + off_pa),
                             ctas_a, d_stats, stream));
    if (e == cudaSuccess)
        e = LAUNCH(launch_row_stats(k, n, b_nnz, b_row_ptr, b_col_idx, reinterpret_cast<StatsPartial *>(base + off_pb),
                             ctas_b, d_stats + 1, stream));
    if (e == cudaSuccess) e = cudaMemcpyAsync(st, d_stats, sizeof st, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) {
        cudaStreamSynchronize(stream);
        destroy_spgemm(h);
        return cuda_fail(e, "SpGEMM analysis");
    }
    for (int w = 0; w < 2; ++w)
        if (st[w].flags) {
            const int f = st[w].flags;
            cudaStreamSynchronize(stream);
        destroy_spgemm(h);
            char msg[160];
            std::snprintf(msg, sizeof msg, "invalid CSR (%s):%s%s%s%s", w ? "B" : "A", (f & 1) ? " row_ptr[0] != 0;" : "",
                          (f & 2) ? " row_ptr decreases;" : "", (f & 4) ? " row_ptr[m] != nnz;" : "",
                          (f & 8) ? " column index outside its range;" : "");
            return fail(SPMV_ERR_INVALID_CSR, msg);
        }

    // ---- products per row and bins
    e = LAUNCH(launch_spgemm_analysis(a, counts, offsets, scan, stream));
    int64_t host_off[kSpgemmBins + 1] = {};
    if (e == cudaSuccess && m > 0)
        for (int b = 0; b <= kSpgemmBins && e == cudaSuccess; ++b)
            e = cudaMemcpyAsync(host_off + b, offsets + b * chunks, sizeof(int64_t), cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) {
        cudaStreamSynchronize(stream);
        destroy_spgemm(h);
        return cuda_fail(e, "SpGEMM binning");
    }
    for (int b = 0; b < kSpgemmBins; ++b) a.bin_count[b] = host_off[b + 1] - host_off[b];

    // ---- the dense bin: entry space, pieces of at most spgemm_piece_products()
    //      products, waves of rows that fit the slots (at most 8 GiB of them)
    const int64_t dense_rows = a.bin_count[kSpgemmBins - 1];
    if (dense_rows > 0) {
        const spmv_status_t st = spgemm_dense_plan(h, stream);
        if (st != SPMV_OK) {
            cudaStreamSynchronize(stream);
        destroy_spgemm(h);
            return st;
        }
    }

    // ---- symbolic phase: the size of every row of C
    e = LAUNCH(launch_spgemm_symbolic(dtype, a, scan, stream));
    int64_t tot[2] = {0, 0};
    if (e == cudaSuccess && m > 0) e = cudaMemcpyAsync(tot, a.c_ptr + m, sizeof(int64_t), cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess && m > 0) {
        // the total of the products (for the info), summed into row_nnz,
        // which the numeric phase does not use
        e = LAUNCH(launch_exclusive_scan(a.products, m, a.row_nnz, scan, stream));
        if (e == cudaSuccess) e = cudaMemcpyAsync(tot + 1, a.row_nnz + m, sizeof(int64_t), cudaMemcpyDeviceToHost, stream);
    }
    // ---- the numeric phase's bins, by the entries of each row of C (row_nnz as the key)
    int64_t num_off[kSpgemmBins + 1] = {};
    if (e == cudaSuccess && m > 0) {
        e = LAUNCH(launch_spgemm_numeric_bins(a, a.row_nnz, counts, offsets, scan, num_rows, stream));
        for (int b = 0; b <= kSpgemmBins && e == cudaSuccess; ++b)
            e = cudaMemcpyAsync(num_off + b, offsets + b * chunks, sizeof(int64_t), cudaMemcpyDeviceToHost, stream);
    }
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) {
        cudaStreamSynchronize(stream);
        destroy_spgemm(h);
        return cuda_fail(e, "SpGEMM symbolic phase");
    }
    for (int b = 0; b < kSpgemmBins; ++b) a.num_bin_count[b] = num_off[b + 1] - num_off[b];
    h->c_nnz = tot[0];
    h->products = tot[1];
    *c_nnz = h->c_nnz;
    if (h->c_nnz >= (1LL << 31)) {
        cudaStreamSynchronize(stream);
        destroy_spgemm(h);
        return fail(SPMV_ERR_INVALID_ARG, "C has 2^31 entries or more (int32 indices)");
    }
    *out = h;
    return SPMV_OK;
}

spmv_status_t spmv_spgemm_compute(spmv_spgemm_t h, const void *a_vals, const void *b_vals, int32_t *c_row_ptr,
                                  int32_t *c_col_idx, void *c_vals, spmv_stream_t stream_handle) {
    if (!h) return fail(SPMV_ERR_INVALID_ARG, "handle is NULL");
    if (!c_row_ptr) return fail(SPMV_ERR_INVALID_ARG, "c_row_ptr is NULL");
    if ((h->a_nnz > 0 && !a_vals) || (h->b_nnz > 0 && !b_vals)) return fail(SPMV_ERR_INVALID_ARG, "a_vals or b_vals is NULL");
    if (h->c_nnz > 0 && (!c_col_idx || !c_vals)) return fail(SPMV_ERR_INVALID_ARG, "c_col_idx or c_vals is NULL");
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_handle);
    const cudaError_t e = LAUNCH(launch_spgemm_numeric(h->dtype, h->args, a_vals, b_vals, c_row_ptr, c_col_idx, c_vals, stream));
    if (e != cudaSuccess) return cuda_fail(e, "spmv_spgemm_compute launch");
    return SPMV_OK;
}

spmv_status_t spmv_spgemm_info(spmv_spgemm_t h, spmv_spgemm_info_t *info) {
    if (!h || !info) return fail(SPMV_ERR_INVALID_ARG, "handle or info is NULL");
    std::memset(info, 0, sizeof *info);
    info->m = h->m;
    info->k = h->k;
    info->n = h->n;
    info->dtype = h->dtype;
    info->a_nnz = h->a_nnz;
    info->b_nnz = h->b_nnz;
    info->c_nnz = h->c_nnz;
    info->products = h->products;
    int launches = h->m > 0 ? 1 : 0;  // the int32 row pointers (m == 0: a memset)
    for (int b = 0; b < kSpgemmBins; ++b) {
        info->bin_rows[b] = h->args.bin_count[b];
        info->numeric_bin_rows[b] = h->args.num_bin_count[b];
        if (b < kSpgemmBins - 1) launches += h->args.num_bin_count[b] > 0;
    }
    launches += 2 * (int)h->args.dense_waves;  // accumulate + finish per wave
    info->dense_slots = (int32_t)h->args.dense_slots;
    info->dense_pieces = h->dense_pieces;
    info->dense_waves = h->args.dense_waves;
    info->launches_per_compute = launches;
    info->workspace_bytes = (int64_t)(h->arena_bytes + h->dense_bytes + h->layout_bytes);
    return SPMV_OK;
}

spmv_status_t spmv_spgemm_device_status(spmv_spgemm_t h, int32_t *flags) {
    if (!h || !flags) return fail(SPMV_ERR_INVALID_ARG, "handle or flags is NULL");
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(flags, h->args.error, sizeof(int32_t), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "spmv_spgemm_device_status");
    return SPMV_OK;
}

spmv_status_t spmv_spgemm_destroy(spmv_spgemm_t h) {
    destroy_spgemm(h);
    return SPMV_OK;
}

}  // extern "C"
