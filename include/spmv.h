/*
 * Load-balanced CSR sparse matrix-vector product for one GB300 (sm_103a).
 *
 *     y = alpha * A * x + beta * y
 *
 * A is an m-by-n matrix in CSR form with int32 indices and fp32 or fp64
 * values.  CSR as defined on the Row-grouped CSR page ("New Row-grouped CSR
 * format for storing the sparse matrices on GPU with implementation in CUDA",
 * section 3, Figure 1): the nonzeros are stored row by row in `vals` with
 * their column indices in `col_idx`; `row_ptr` has m+1 entries, row i owns
 * positions row_ptr[i] .. row_ptr[i+1]-1, and row_ptr[m] = nnz.  The same
 * three arrays are the SpMV kernel's inputs in the load-balancing paper
 * (Osama, Porumbescu, Owens, "A GPU load-balancing programming model",
 * section 4.3, Listing 3), which computes each y entry as the row's sum of
 * values[nz] * x[indices[nz]].
 *
 * The library works in two steps.  spmv_plan_create analyses the row
 * lengths on the GPU (statistics by length class, after OpSparse's row
 * binning, section 5.1), chooses a kernel, and precomputes its schedule --
 * for the default merge-path kernel, the exact split of the m + nnz units
 * of work (every row end and every nonzero, "A GPU load-balancing
 * programming model", section 5.2.1) into equal tiles.  spmv_execute then
 * runs the product on a stream with no allocation and no synchronisation.
 *
 * All array arguments are DEVICE pointers (for example from torch CUDA
 * tensors) on the current CUDA device, except where a function says HOST.
 * Streams are cudaStream_t handles; NULL is the legacy default stream.
 * Every function returns an spmv_status_t; spmv_last_error() gives a
 * one-line description of the last failure on the calling thread.
 */
#ifndef LBCSR_SPMV_H
#define LBCSR_SPMV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
/* a cudaStream_t */
typedef struct CUstream_st *spmv_stream_t;

typedef struct spmv_plan_s *spmv_plan_t;

typedef enum { SPMV_F32 = 0, SPMV_F64 = 1 } spmv_dtype_t;

typedef enum {
    SPMV_OK = 0,
    SPMV_ERR_INVALID_ARG = 1, /* null pointer, negative size, size limits, bad option */
    SPMV_ERR_INVALID_CSR = 2, /* row_ptr[0] != 0, row_ptr decreasing, row_ptr[m] != nnz,
                                 or a column index outside [0, n) */
    SPMV_ERR_ALLOC = 3,       /* device or host allocation failed in plan creation */
    SPMV_ERR_CUDA = 4,        /* a CUDA call or kernel launch failed */
    SPMV_ERR_UNSUPPORTED = 5  /* device is not sm_103 / option not available */
} spmv_status_t;

/* Kernels a plan can run. */
typedef enum {
    SPMV_KERNEL_AUTO = 0,       /* let the plan choose from the row-length statistics */
    SPMV_KERNEL_MERGE_PATH = 1, /* equal shares of rows + nonzeros per warp tile, fused carry-out fix-up */
    SPMV_KERNEL_THREAD_ROW = 2, /* one thread per row */
    SPMV_KERNEL_RGCSR = 3,      /* Row-grouped CSR (interleaved copy of A built by the plan);
                                   long rows, if any, by the long-row kernel */
    SPMV_KERNEL_LONG_ROWS = 4,  /* long rows by the long-row kernel (one warp per segment of
                                   4096 nonzeros), the other rows one thread per row */
    SPMV_KERNEL_RGCSR_SORTED = 5,/* Row-grouped CSR (groups of 32) over the rows listed, in
                                   each window of 1024 rows, by decreasing length, which
                                   cuts the padding; long rows by the long-row kernel */
    SPMV_KERNEL_GROUP_MAPPED = 6 /* group-level schedule ("A GPU load-balancing programming
                                   model", section 5.2.3): a CTA per 256 rows, their
                                   nonzeros shared by the CTA's threads */
} spmv_kernel_t;

/* Options for spmv_plan_create_ex; zero-initialise and set what you need. */
typedef struct {
    int32_t kernel;           /* spmv_kernel_t; SPMV_KERNEL_AUTO (0) = choose */
    int32_t items_per_thread; /* merge-path work items (rows + nonzeros) per
                                 thread; a tile is one warp, T = 32 * items.
                                 0 = chosen from the statistics (8-24).
                                 Allowed: 8, 12, 16, 24, 32 */
    int32_t rgcsr_group;      /* Row-grouped CSR group size G; 0 = chosen from
                                 the statistics (the largest G whose padding
                                 is at most 10 %, else the least padded).
                                 Allowed: 32, 64, 128, 256 */
    int32_t long_row_min;     /* Row-grouped CSR and long-row kernels: rows with
                                 at least this many nonzeros count as long and
                                 go to the long-row kernel; 0 = default (512).
                                 Allowed: 0 or >= 32 */
    int32_t with_spmm;        /* nonzero: also prepare spmv_execute_multi (the
                                 merge-path partition and its scratch, about
                                 1 KB per warp slot for fp32, 2 KB for fp64) */
    int32_t with_transpose;   /* nonzero: also prepare spmv_execute_transposed
                                 (the plan builds A^T in CSR form, 12-16 bytes
                                 per nonzero, and a plan for it) */
} spmv_options_t;

/*
 * Row-length statistics measured by the plan.  hist[k] counts rows whose
 * length falls in class k: class 0 = empty rows, class k >= 1 = lengths in
 * [2^(k-1), 2^k).  rg_slots[g] = storage (slots) a Row-grouped CSR layout
 * with group size 32 << g would need (each group padded to its longest
 * row).  bandwidth: the largest |column - row| over every row's first and
 * last stored nonzero.  flags: bit0 row_ptr[0] != 0, bit1 row_ptr
 * decreases, bit2 row_ptr[m] != nnz, bit3 a column index outside [0, n).
 */
typedef struct {
    int64_t hist[32];
    int64_t sum_len;
    int64_t rg_slots[4];
    int32_t min_len;
    int32_t max_len;
    int32_t n_empty;
    int32_t flags;
    int32_t bandwidth;
    int32_t reserved;
} spmv_row_stats_t;

typedef struct {
    int32_t m, n, nnz;
    int32_t dtype;                /* spmv_dtype_t */
    int32_t kernel;               /* spmv_kernel_t actually used */
    int32_t threads_per_tile;     /* merge-path kernel: one warp per tile */
    int32_t items_per_thread;     /* merge-path kernel */
    int32_t rgcsr_group;          /* Row-grouped CSR kernel */
    int64_t items_per_tile;       /* merge-path tile T = threads * items (rows + nonzeros) */
    int64_t num_tiles;            /* merge-path tiles P = ceil((m + nnz) / T), at least 1 */
    int32_t num_long_rows;        /* rows handled by the long-row kernels */
    int32_t launches_per_execute; /* kernel launches one spmv_execute issues */
    int64_t workspace_bytes;      /* device memory the plan owns */
    spmv_row_stats_t stats;
    int32_t long_row_min;         /* threshold of the long-row kernel (0 if unused) */
    int32_t long_segment_nnz;     /* nonzeros per long-row segment (one warp each) */
    int64_t num_long_segments;    /* segments over all long rows */
    int64_t rgcsr_slots;          /* slots of the Row-grouped copy (group_ptr[last]) */
    int32_t transposed_kernel;    /* spmv_kernel_t of the plan for A^T (-1: none) */
    int32_t transposed_launches;  /* kernel launches one spmv_execute_transposed issues */
    int64_t merge_path_warps;     /* merge-path kernel: warps W, each owning a contiguous run of
                                     about num_tiles / W tiles (for 16-byte aligned arrays; 0 when
                                     the plan runs another kernel) */
} spmv_plan_info_t;

/* What spmv_plan_export copies out. */
typedef enum {
    SPMV_EXPORT_PARTITION = 0,   /* int32 pairs (row, nonzero), num_tiles + 1 of them */
    SPMV_EXPORT_RG_GROUP_PTR = 1,/* int64[ceil(m/G) + 1] */
    SPMV_EXPORT_RG_ROW_LEN = 2,  /* int32[m] by position: row length, -1 for a row left to the
                                    long-row kernel */
    SPMV_EXPORT_RG_COL = 3,      /* int32[group_ptr[last]] */
    SPMV_EXPORT_RG_VAL = 4,      /* value type [group_ptr[last]] */
    SPMV_EXPORT_LONG_ROWS = 5,   /* int32[num_long_rows], ascending */
    SPMV_EXPORT_LONG_SEG_BEGIN = 6,/* int64[num_long_rows + 1]: first segment of each long row */
    SPMV_EXPORT_RG_PERM = 7,     /* int32[m]: the row at each position of the window-sorted copy */
    SPMV_EXPORT_T_PTR = 8,       /* int32[n + 1]: A^T in CSR form, row pointers */
    SPMV_EXPORT_T_IDX = 9,       /* int32[nnz]: its column indices (rows of A) */
    SPMV_EXPORT_T_VALS = 10,     /* value type [nnz] */
    SPMV_EXPORT_T_SRC = 11       /* int32[nnz]: each entry's position in A */
} spmv_export_t;

/*
 * Build a plan for A (device arrays row_ptr[m+1], col_idx[nnz], vals[nnz]).
 *
 * Limits: m >= 0, n >= 0, 0 <= nnz, m + nnz < 2^31.  When nnz > 0 the
 * pointers must be non-null; row_ptr must be non-null when m >= 0.
 * Ownership: the plan BORROWS row_ptr, col_idx and vals; they must stay
 * allocated and unchanged until spmv_plan_destroy (values may change if
 * spmv_plan_update_values is called afterwards).  The plan OWNS one device
 * workspace, allocated here and freed by spmv_plan_destroy.
 * Synchronisation: runs its analysis kernels on `stream` and waits for that
 * stream once (to read the ~0.4 KB statistics back) -- three times for the
 * Row-grouped CSR and long-row kernels, whose layouts are sized on the
 * device (long-row count, segment count, Row-grouped slots) before their
 * last allocation.  Results are synchronous.
 * Errors: INVALID_ARG for bad sizes/pointers; INVALID_CSR when the analysis
 * finds a malformed row_ptr or a column index outside [0, n); ALLOC; CUDA;
 * UNSUPPORTED when the current device is not compute capability 10.3.
 * On error *out is set to NULL and nothing is leaked.
 * Environment, read at each creation: SPMV_LOG=1 prints one line per plan
 * on stderr (the row statistics, the kernel and the rule that chose it);
 * SPMV_FORCE_KERNEL (a kernel name) and SPMV_ITEMS_PER_THREAD override the
 * choice when the options leave it open; SPMV_FAULT=alloc:N|launch:N makes
 * the N-th device allocation or launch step of the call fail, for testing
 * the clean-up paths.
 */
spmv_status_t spmv_plan_create(spmv_plan_t *out, int32_t m, int32_t n, int32_t nnz,
                               const int32_t *row_ptr, const int32_t *col_idx, const void *vals,
                               spmv_dtype_t dtype, spmv_stream_t stream);

/* As spmv_plan_create, with options (NULL = defaults). */
spmv_status_t spmv_plan_create_ex(spmv_plan_t *out, int32_t m, int32_t n, int32_t nnz,
                                  const int32_t *row_ptr, const int32_t *col_idx, const void *vals,
                                  spmv_dtype_t dtype, const spmv_options_t *options,
                                  spmv_stream_t stream);

/*
 * y = alpha * A * x + beta * y on `stream` (device x[n], y[m] of the plan's
 * value type).  alpha and beta are rounded to the value type.  If beta == 0
 * y is write-only: its old contents (NaN included) are not read.  x and y
 * must not overlap.  Asynchronous: returns after queueing the kernels; no
 * allocation, no host synchronisation.  A plan must not run on two streams
 * at once (its workspace holds per-execution carry state).
 * Errors: INVALID_ARG (null plan, or null x/y when the sizes need them),
 * CUDA (launch failure).
 */
spmv_status_t spmv_execute(spmv_plan_t plan, double alpha, const void *x, double beta, void *y,
                           spmv_stream_t stream);

/*
 * The same product with x and y in HOST memory (x_host[n], y_host[m] of
 * the plan's value type): on `stream`, copy x_host into the caller's
 * device buffer x_dev[n] (and y_host into y_dev[m] when beta != 0), run
 * spmv_execute(plan, alpha, x_dev, beta, y_dev, stream), and copy y_dev
 * back into y_host -- one cudaMemcpyAsync per copy.  Asynchronous like
 * spmv_execute: y_host holds the result once the stream has passed the
 * last copy (synchronise the stream before reading it).  For copies that
 * overlap other work the host buffers should be page-locked
 * (cudaHostAlloc, or pinned torch tensors); pageable memory also works.
 * x_dev and y_dev must not overlap each other or the plan's arrays.
 * Allocates nothing.  This is the call an application with its vectors on
 * the host makes; the product itself is the one above.
 * Errors: as spmv_execute, INVALID_ARG also for a null host or device
 * buffer the sizes need, CUDA when a copy cannot be queued.
 */
spmv_status_t spmv_execute_host(spmv_plan_t plan, double alpha, const void *x_host, double beta, void *y_host,
                                void *x_dev, void *y_dev, spmv_stream_t stream);

/*
 * Y = alpha * A * X + beta * Y for k right-hand sides ("A GPU
 * load-balancing programming model", section 4.3, Listing 4: the row loop
 * of SpMV with an inner loop over the columns of a dense matrix).  X is
 * n-by-k and Y m-by-k, device, row-major with leading dimensions ldx >= k
 * and ldy >= k (element (c, t) of X at X[c*ldx + t]); value type of the
 * plan.  alpha and beta as for spmv_execute (beta == 0: Y is write-only).
 * X and Y must not overlap.  The plan must have been created with
 * options.with_spmm != 0 (it then holds the merge-path partition, and the
 * long-row lists the paths below need).
 *
 * The call takes the first path that applies: (1) over the plan's
 * Row-grouped copy (groups of 32; long rows the copy leaves out, if at
 * most one per 4096 rows, by a warp per 4096-nonzero segment), in slices
 * of 32 (fp32) or 16 (fp64) columns; (2) for matrices whose rows have at
 * most 64 nonzeros, or with rows of 65 or more at most one per 4096 rows
 * and k <= 64 (fp32) / 32 (fp64): a warp per 32 rows straight from CSR,
 * long rows by a warp per segment -- both need k a multiple of 16 bytes'
 * worth of values and X, Y 16-byte aligned row by row; (3) otherwise the
 * merge-path partition, 128 columns per launch.  Every path gives the
 * same sums up to rounding order; none allocates; asynchronous.  A plan
 * must not run two products at once.
 * Errors: INVALID_ARG (null plan or pointers, k < 0, ld < k, plan without
 * with_spmm), CUDA (launch failure).  k == 0 or m == 0 is a no-op.
 */
spmv_status_t spmv_execute_multi(spmv_plan_t plan, int32_t k, double alpha, const void *X, int64_t ldx,
                                 double beta, void *Y, int64_t ldy, spmv_stream_t stream);

/*
 * y = alpha * A^T * x + beta * y: x has m entries, y has n (device, plan's
 * value type).  The plan must have been created with
 * options.with_transpose != 0: it then holds A^T in compressed-row form
 * (A in compressed-column form, the CSC of "A GPU load-balancing
 * programming model", section 4.1), each column's entries in increasing
 * row order, built by a stable radix sort on the GPU, and a plan of its own
 * for it (statistics, kernel choice, schedule), whose product this runs.
 * Semantics, synchronisation and errors as for spmv_execute.
 */
spmv_status_t spmv_execute_transposed(spmv_plan_t plan, double alpha, const void *x, double beta, void *y,
                                      spmv_stream_t stream);

/*
 * Point the plan at new values with the same sparsity pattern (vals[nnz],
 * device).  Plans that keep a reordered copy of the values (the
 * Row-grouped CSR kernel, A^T) repack it on `stream`; the others only
 * record the pointer.  Same ownership rule as at creation.
 */
spmv_status_t spmv_plan_update_values(spmv_plan_t plan, const void *vals, spmv_stream_t stream);

/* Free the plan's workspace (waits for the device to finish using it). NULL is a no-op. */
spmv_status_t spmv_plan_destroy(spmv_plan_t plan);

/* Fill *info (HOST) with the plan's sizes, chosen kernel and statistics. */
spmv_status_t spmv_plan_info(spmv_plan_t plan, spmv_plan_info_t *info);

/*
 * Copy one of the plan's internal arrays into HOST memory dst of `bytes`
 * bytes (for tests and inspection; synchronous).  INVALID_ARG if the plan
 * does not hold that array or bytes is smaller than its size; the size is
 * written to *needed when needed != NULL.
 */
spmv_status_t spmv_plan_export(spmv_plan_t plan, spmv_export_t what, void *dst, size_t bytes,
                               size_t *needed);

/*
 * One product y = alpha * A * x + beta * y that allocates nothing: no plan,
 * no cudaMalloc/cudaFree, no allocating library call.  The pages have no
 * counterpart; this entry point exists for callers that cannot allocate
 * device memory when they need a product -- for example a service that
 * hands the whole device to its own memory pool at start-up (a cudaMalloc
 * would fail or fragment the pool), or a latency-critical loop where a
 * cudaMalloc would synchronise the device and stall work queued on other
 * streams.
 *
 * Arguments as spmv_plan_create plus spmv_execute (device arrays, the
 * caller's stream).  It runs the merge-path kernel (tiles of 384 rows plus
 * nonzeros) with its scratch in one fixed-size array (about 6 MB) inside the
 * library's device image, which every GPU that loads the library holds
 * until the process exits.  Limit: m + nnz <= 2^28 = 268,435,456; larger
 * sizes return SPMV_ERR_INVALID_ARG.  The matrix is NOT checked (use
 * spmv_plan_create once to validate it); invalid indices give undefined
 * results.  All calls share the scratch array and each call clears what must
 * start at zero, so calls that overlap on the GPU (two streams, two host
 * threads) race.  Every call looks up the array's device address (a host
 * table lookup once the library's module is loaded on the device); the first
 * call on a device loads that module, so make it before any stream capture.
 * Asynchronous otherwise.  A tile copy that does not complete within about a
 * second stops that part of the product and sets a flag that
 * spmv_noalloc_device_status reports.  Returns SPMV_OK, SPMV_ERR_INVALID_ARG
 * or SPMV_ERR_CUDA (no message is set for spmv_last_error).
 */
spmv_status_t spmv_execute_noalloc(int32_t m, int32_t n, int32_t nnz, const int32_t *row_ptr,
                                   const int32_t *col_idx, const void *vals, spmv_dtype_t dtype,
                                   double alpha, const void *x, double beta, void *y,
                                   spmv_stream_t stream);

/*
 * Kernel-side failure flags of the last spmv_execute_noalloc on the current
 * device (HOST *flags; waits for the whole device, so not during a stream
 * capture; allocates nothing).  0 = no failure; bit 0: a tile copy did not
 * complete within about a second, and that product's y is incomplete.  The
 * pages have no counterpart.  Returns SPMV_OK, SPMV_ERR_INVALID_ARG or
 * SPMV_ERR_CUDA.
 */
spmv_status_t spmv_noalloc_device_status(int32_t *flags);

/*
 * Kernel-side failure flags of a plan (HOST *flags; waits for the device).
 * 0 = no failure.  Bit 0: a kernel's wait for its tile copies ran past its
 * time limit (about a second); the kernel then stopped that part of the work
 * instead of waiting forever, so the y of that product is incomplete.
 * Bit 2 (value 4), debug build only (libspmv_debug.so, compiled with
 * -DSPMV_DEBUG): an SpMV kernel met a column index outside [0, n) -- an
 * array changed after the plan was created, which the plan borrows
 * unmodified -- and gathered x[0] in its place; that y is wrong.  The
 * release build does not check (creation validates every index once).
 */
spmv_status_t spmv_plan_device_status(spmv_plan_t plan, int32_t *flags);

/*
 * Diagnostic: the ceiling of the x gather for a column pattern, by load
 * path.  The Row-grouped CSR page (sections 3 and 4) names the gather of x
 * as what limits SpMV once the matrix stream is coalesced (x through the
 * texture cache gave 1.3-1.8x); this call measures how fast each of the
 * GPU's load paths can gather x[col_idx[k]] for k = 0 .. nnz-1, with no
 * matrix values and no floating-point work, so that a kernel's time can be
 * set against the best one.
 *
 * path (spmv_gather_path_t): STREAM reads col_idx only; L1 gathers through
 * the read-only path (ld.global.nc); L2 through L2 only (ld.global.cg);
 * BULK16 by one 16-byte Tensor Memory Accelerator copy per gather into
 * shared memory; TMA4 by tile::gather4 tensor copies (x viewed as rows of
 * 32 bytes, four rows per instruction); L1_TMA4 half by L1, half by TMA4;
 * L1_TMA4_QUARTER three quarters by L1, one by TMA4; TMA4_16 as TMA4 over
 * rows of 16 bytes.  Three paths also stream the values vals[nnz] (device,
 * dtype) beside the L1 gathers, to measure what bringing in the matrix
 * costs the gathers: STREAM_LDG by coalesced loads, STREAM_BULK by one bulk
 * copy per 256 nonzeros and array into shared memory, STREAM_CPASYNC by
 * 16-byte cp.async (both need col_idx and vals 16-byte aligned),
 * STREAM_LDG_OCC as STREAM_LDG with the staged paths' shared memory reserved
 * (as many warps per SM), STREAM_LDG_STS by coalesced loads that the lanes
 * store to shared memory and read back, STREAM_LDG_FEW as STREAM_LDG with no
 * shared memory but only as many CTAs per SM as the staged paths fit,
 * STREAM_LDG_RES_1 .. _6 as STREAM_LDG with 4 CTAs per SM and 32, 64, ...,
 * 192 KB of shared memory reserved per SM (the L1 left to the gathers);
 * their checksum adds the values' bit patterns too.
 * col_idx[nnz] (device, int32, each in [0, n)), x[n] (device, dtype; 16-byte
 * aligned for the copy paths, BULK16 to TMA4_16, which also need
 * n * sizeof(value) >= 32).  *checksum (device uint64, zeroed by the caller) receives the sum,
 * modulo 2^64, of the bit patterns of the gathered values (the same for
 * every path except STREAM, which sums the columns instead).  *error
 * (device int32, zeroed by the caller): bit 0 is set if a copy did not
 * complete within about a second.  Asynchronous on `stream`; allocates
 * nothing.  Errors: INVALID_ARG; UNSUPPORTED when x is misaligned for the
 * path or the tensor-map encoder is unavailable; CUDA on launch failure.
 */
typedef enum {
    SPMV_GATHER_STREAM = 0,
    SPMV_GATHER_L1 = 1,
    SPMV_GATHER_L2 = 2,
    SPMV_GATHER_BULK16 = 3,
    SPMV_GATHER_TMA4 = 4,
    SPMV_GATHER_L1_TMA4 = 5,
    SPMV_GATHER_L1_TMA4_QUARTER = 6,
    SPMV_GATHER_TMA4_16 = 7,
    SPMV_GATHER_STREAM_LDG = 8,
    SPMV_GATHER_STREAM_BULK = 9,
    SPMV_GATHER_STREAM_CPASYNC = 10,
    SPMV_GATHER_STREAM_LDG_OCC = 11,
    SPMV_GATHER_STREAM_LDG_STS = 12,
    SPMV_GATHER_STREAM_LDG_FEW = 13,
    SPMV_GATHER_STREAM_LDG_RES_1 = 14, /* .. _RES_6 = 19 */
    SPMV_GATHER_STREAM_LDG_RES_6 = 19,
    SPMV_GATHER_TEX = 20               /* element fetches from a linear texture object over x (the call
                                          synchronises the stream: the object must outlive the launch) */
} spmv_gather_path_t;

spmv_status_t spmv_gather_ceiling(int32_t path, int32_t nnz, const int32_t *col_idx, int32_t n, const void *x,
                                  const void *vals, spmv_dtype_t dtype, uint64_t *checksum, int32_t *error,
                                  spmv_stream_t stream);

/*
 * Sparse times sparse, C = A * B, after OpSparse ("OpSparse: a highly
 * optimized framework for sparse general matrix multiplication on GPUs",
 * sections 3 and 5): Gustavson's row-by-row product (row i of C sums, over
 * the entries a_ip of row i of A, a_ip times row p of B), in two phases.
 *
 * spmv_spgemm_create takes the PATTERNS of A (m-by-k: a_row_ptr[m+1],
 * a_col_idx[a_nnz]) and B (k-by-n: b_row_ptr[k+1], b_col_idx[b_nnz]), device
 * int32 CSR arrays that the handle borrows until it is destroyed (their
 * contents must not change meanwhile).  It checks both as
 * spmv_plan_create does, counts the products of each row of C, bins the
 * rows by that count, sizes every row of C (the symbolic phase: sorted
 * lists for rows of at most 16 products, hash sets in shared memory up to
 * 4096; above, a dense row of C per row in global memory, the row's
 * products cut into equal pieces of at most 32768, a CTA each, with up to
 * 8 GiB of such rows at once),
 * and writes the number of entries of C to *c_nnz (HOST).  An entry of C
 * exists where at least one product lands, even if the products sum to
 * zero.  Synchronous (it waits for `stream` several times).
 * Limits: m, k, n >= 0; m + a_nnz and k + b_nnz < 2^31; C must have fewer
 * than 2^31 entries (else INVALID_ARG, with *c_nnz still set).
 * Errors: INVALID_ARG, INVALID_CSR, ALLOC, CUDA, UNSUPPORTED.  On error
 * *out is NULL.
 *
 * spmv_spgemm_compute is the numeric phase: with the values a_vals[a_nnz]
 * and b_vals[b_nnz] (device, the handle's value type) it writes C in CSR
 * form into caller-allocated device arrays c_row_ptr[m+1] (int32),
 * c_col_idx[c_nnz] (int32, increasing within each row) and c_vals[c_nnz].
 * It may be called again with new values of the same patterns.
 * Asynchronous on `stream`; allocates nothing.  Outside the rows of at
 * most 16 products (summed in the order of the row's products), the
 * products of an entry are added in an order that may change from call to
 * call (atomics), so its last bits may too; the pattern is always the same.
 * Errors: INVALID_ARG (null handle or pointers), CUDA.
 */
typedef struct spmv_spgemm_s *spmv_spgemm_t;

typedef struct {
    int32_t m, k, n;
    int32_t dtype;               /* spmv_dtype_t */
    int64_t a_nnz, b_nnz, c_nnz;
    int64_t products;            /* sum over the rows of C of their products */
    int64_t bin_rows[8];         /* rows of C by products: <= 16, <= 128, <= 512, <= 1024,
                                    <= 2048, <= 4096, more (the dense bin); [7] unused */
    int32_t dense_slots;         /* dense-bin rows of C held at once (one wave) */
    int32_t launches_per_compute;/* kernel launches one spmv_spgemm_compute issues */
    int64_t workspace_bytes;     /* device memory the handle owns */
    int64_t dense_pieces;        /* dense-bin pieces of at most 32768 products, a CTA each */
    int64_t dense_waves;         /* waves of dense-bin rows (two launches each) */
    int64_t numeric_bin_rows[8]; /* the numeric phase's bins: rows of at most 16 products,
                                    then by entries of C (<= 128, <= 512, <= 1024, <= 2048,
                                    <= 4096; tables of twice that), the dense bin as above */
} spmv_spgemm_info_t;

spmv_status_t spmv_spgemm_create(spmv_spgemm_t *out, int32_t m, int32_t k, int32_t n, int32_t a_nnz,
                                 const int32_t *a_row_ptr, const int32_t *a_col_idx, int32_t b_nnz,
                                 const int32_t *b_row_ptr, const int32_t *b_col_idx, spmv_dtype_t dtype,
                                 int64_t *c_nnz, spmv_stream_t stream);

spmv_status_t spmv_spgemm_compute(spmv_spgemm_t handle, const void *a_vals, const void *b_vals,
                                  int32_t *c_row_ptr, int32_t *c_col_idx, void *c_vals, spmv_stream_t stream);

/* Fill *info (HOST). */
spmv_status_t spmv_spgemm_info(spmv_spgemm_t handle, spmv_spgemm_info_t *info);

/* Kernel-side failure flags (HOST *flags; waits for the device).  Bit 1: a
 * row of C outgrew the size the symbolic phase found (the patterns changed
 * after creation); that row is incomplete. */
spmv_status_t spmv_spgemm_device_status(spmv_spgemm_t handle, int32_t *flags);

/* Free the handle's workspace (waits for the device).  NULL is a no-op. */
spmv_status_t spmv_spgemm_destroy(spmv_spgemm_t handle);

/* Static text for a status code. */
const char *spmv_status_string(spmv_status_t status);

/* Description of the last error on the calling thread ("" if none). */
const char *spmv_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* LBCSR_SPMV_H */
