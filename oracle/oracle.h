/*
 * CPU oracle for the load-balanced CSR SpMV library.
 *
 * TEST INFRASTRUCTURE ONLY.  Plain, single-threaded, obviously-correct C that
 * the tests, the smoke check and the benchmark's CPU-baseline leg use to
 * check the CUDA path.  The product library never includes, links or calls
 * anything here, and nothing here includes or calls the product library.
 *
 * Sources (web pages on load-balanced CSR SpMV):
 *   [RgCSR]  "New Row-grouped CSR format for storing the sparse matrices on
 *            GPU with implementation in CUDA" (arXiv 1012.2270): CSR
 *            definition (section 3, Figure 1), Row-grouped CSR layout
 *            (section 3, Figure 5), bytes-per-nonzero peak model (section 3).
 *   [LBPM]   Osama, Porumbescu, Owens, "A GPU load-balancing programming
 *            model" (PPoPP'23): CSR as atoms/tiles (section 4.1, Listing 1),
 *            SpMV as a row loop (section 4.3, Listing 3), merge-path
 *            schedule (section 5.2.1).
 *   [OpSparse] "OpSparse: a highly optimized framework for sparse general
 *            matrix multiplication on GPUs" (arXiv 2206.07244): row binning
 *            by length class (section 5.1, Algorithms 1-3).
 */
#ifndef SPMV_ORACLE_H
#define SPMV_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/*
 * y = alpha*A*x + beta*y_old, accumulated in long double.  [LBPM] section
 * 4.3 (Listing 3: for every row, sum values[nz]*x[indices[nz]] over the row's
 * nonzeros, then store the sum); [RgCSR] section 3 (CSR definition).
 * alpha and beta are first rounded to the value type (they reach the library
 * as double).  If beta == 0, y_old is not read.  If rows != NULL only the
 * listed rows are computed and y_out[t], mag_out[t] refer to rows[t];
 * otherwise all m rows.  mag_out (may be NULL) receives
 *   |alpha| * sum_k |val[k] * x[col[k]]| + |beta * y_old[i]|,
 * the scale of the accuracy tolerance.  Returns 0, or 1 on bad arguments.
 */
int oracle_spmv_f64(int32_t m, int32_t n, const int32_t *row_ptr, const int32_t *col_idx,
                    const double *vals, const double *x, double alpha, double beta,
                    const double *y_old, const int32_t *rows, int64_t nrows, double *y_out,
                    double *mag_out);
int oracle_spmv_f32(int32_t m, int32_t n, const int32_t *row_ptr, const int32_t *col_idx,
                    const float *vals, const float *x, double alpha, double beta,
                    const float *y_old, const int32_t *rows, int64_t nrows, float *y_out,
                    double *mag_out);

/*
 * Merge-path partition.  [LBPM] section 5.2.1: every nonzero and every row
 * end is one unit of work; the m + nnz units are split evenly; a worker's
 * start is the (row, nonzero) pair where its share begins.  Units are taken
 * in merge order: in state (i, j) the next unit is the end of row i when
 * row_ptr[i+1] <= j, otherwise nonzero j.  After d units the state is
 *   i(d) = #{ r in [0, m) : row_ptr[r+1] + r < d },  j(d) = d - i(d).
 * For p = 0..P the split of diagonal d_p = min(p*T, m+nnz) is written to
 * part[2p] = i(d_p), part[2p+1] = j(d_p).  Returns 0, or 1 on bad arguments.
 */
int oracle_merge_path_partition(int32_t m, int32_t nnz, const int32_t *row_ptr, int64_t T,
                                int64_t P, int32_t *part);

/*
 * Row-length statistics.  Length classes after [OpSparse] section 5.1
 * (rows binned by size): class 0 holds empty rows, class k >= 1 holds lengths
 * in [2^(k-1), 2^k).  rg_slots[g] is the storage a Row-grouped CSR layout
 * with group size 32 << g needs ([RgCSR] section 3: each group of G rows is
 * padded to its longest row): sum over groups of G * max length, the last
 * partial group padded with empty rows.
 * bandwidth = the largest |column - row| over every row's first and last
 * stored nonzero (the distance of a sorted row's outermost entries from the
 * diagonal; 0 for a matrix without nonzeros).
 * Flags: bit0 row_ptr[0] != 0, bit1 row_ptr decreases somewhere,
 * bit2 row_ptr[m] != nnz, bit3 a column index outside [0, n).
 * Statistics are computed only if no row_ptr flag (bits 0-2) is set.
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
} oracle_stats_t;

int oracle_row_stats(int32_t m, int32_t n, int32_t nnz, const int32_t *row_ptr,
                     const int32_t *col_idx, oracle_stats_t *out);

/*
 * Row-grouped CSR layout, [RgCSR] section 3 and Figure 5: rows are taken in
 * groups of G; within a group the k-th nonzeros of all rows are stored
 * together, padded to the group's longest row.  group_ptr[g] (ngroups + 1
 * entries, ngroups = ceil(m / G)) is the offset of group g; element k of row
 * i lives at group_ptr[i / G] + k*G + (i mod G).  Padding slots get column 0
 * and value 0.  row_len[i] = row_ptr[i+1] - row_ptr[i].
 * oracle_rgcsr_layout fills group_ptr and row_len; the pack functions also
 * fill the interleaved column and value arrays (group_ptr[ngroups] slots).
 */
int oracle_rgcsr_layout(int32_t m, const int32_t *row_ptr, int32_t G, int64_t *group_ptr,
                        int32_t *row_len);
int oracle_rgcsr_pack_f64(int32_t m, const int32_t *row_ptr, const int32_t *col_idx,
                          const double *vals, int32_t G, const int64_t *group_ptr,
                          int32_t *rg_col, double *rg_val);
int oracle_rgcsr_pack_f32(int32_t m, const int32_t *row_ptr, const int32_t *col_idx,
                          const float *vals, int32_t G, const int64_t *group_ptr,
                          int32_t *rg_col, float *rg_val);

/*
 * Long rows: the bin of rows with at least min_len nonzeros ([OpSparse]
 * section 5.1 bins rows by length; the order inside a bin and the segment
 * size are this library's choice, as the pages fix neither).  ids[] gets the
 * long rows in ascending order; seg_begin[t] (count + 1 entries) is the
 * number of seg_nnz-nonzero segments of the long rows before ids[t]:
 * seg_begin[0] = 0, seg_begin[t+1] = seg_begin[t] + ceil(len(ids[t]) / seg_nnz).
 * *count gets the number of long rows; ids and seg_begin may be NULL to
 * count only.  Returns 0, or 1 on bad arguments (min_len < 1, seg_nnz < 1).
 */
int oracle_long_rows(int32_t m, const int32_t *row_ptr, int32_t min_len, int32_t seg_nnz, int32_t *ids,
                     int64_t *seg_begin, int64_t *count);

/*
 * Y = alpha*A*X + beta*Y_old for k right-hand sides ([LBPM] section 4.3,
 * Listing 4: the SpMV row loop with an inner loop over the columns of a
 * dense matrix).  X is n-by-k and Y m-by-k, both row-major with leading
 * dimensions ldx, ldy >= k: X[c][t] = X[c*ldx + t].  Sums in long double;
 * mag_out[i*k + t] (may be NULL) = |alpha|*sum_j |a_ij X[j][t]| +
 * |beta*Y_old[i][t]|.  If beta == 0, Y_old is not read.  Y_out is m-by-k
 * with leading dimension k.  Returns 0, or 1 on bad arguments.
 */
int oracle_spmm_f64(int32_t m, int32_t n, int32_t k, const int32_t *row_ptr, const int32_t *col_idx,
                    const double *vals, const double *X, int64_t ldx, double alpha, double beta,
                    const double *Y_old, int64_t ldy, double *Y_out, double *mag_out);
int oracle_spmm_f32(int32_t m, int32_t n, int32_t k, const int32_t *row_ptr, const int32_t *col_idx,
                    const float *vals, const float *X, int64_t ldx, double alpha, double beta,
                    const float *Y_old, int64_t ldy, float *Y_out, double *mag_out);

/*
 * The transpose of A in CSR form (= A in compressed-column form, the
 * "CSC" the load-balancing paper lists among the formats its CSR
 * abstraction carries, section 4.1): t_ptr[n+1], t_idx[nnz] (row indices)
 * and t_vals[nnz], each column's entries in increasing row order, and
 * t_src[nnz] (may be NULL) the position in A of each entry.  Returns 0, or
 * 1 on bad arguments.
 */
int oracle_transpose_f64(int32_t m, int32_t n, const int32_t *row_ptr, const int32_t *col_idx, const double *vals,
                         int32_t *t_ptr, int32_t *t_idx, double *t_vals, int32_t *t_src);
int oracle_transpose_f32(int32_t m, int32_t n, const int32_t *row_ptr, const int32_t *col_idx, const float *vals,
                         int32_t *t_ptr, int32_t *t_idx, float *t_vals, int32_t *t_src);

/*
 * y = alpha * A^T * x + beta * y_old (x has m entries, y n): y_j = alpha *
 * sum_i a_ij x_i + beta * y_old_j, summed over A's rows in increasing i,
 * in long double.  mag_out as for oracle_spmv.  Returns 0, or 1 on bad
 * arguments.
 */
int oracle_spmv_transposed_f64(int32_t m, int32_t n, const int32_t *row_ptr, const int32_t *col_idx,
                               const double *vals, const double *x, double alpha, double beta, const double *y_old,
                               double *y_out, double *mag_out);
int oracle_spmv_transposed_f32(int32_t m, int32_t n, const int32_t *row_ptr, const int32_t *col_idx,
                               const float *vals, const float *x, double alpha, double beta, const float *y_old,
                               float *y_out, double *mag_out);

/*
 * C = A * B for A m-by-k and B k-by-n in CSR form ([OpSparse], the
 * Gustavson row-by-row product its sections 4-5 build on: row i of C is
 * the sum over A's entries a_iq of a_iq times row q of B).  Accumulated in
 * long double in a dense row; C's entries are the columns any product
 * reaches (an exact zero sum stays an entry), listed in increasing column
 * order.  Call with c_col == NULL to get c_row_ptr (m + 1 entries) only;
 * then again with c_col and c_val of c_row_ptr[m] entries.  Returns 0, or
 * 1 on bad arguments.
 */
int oracle_spgemm_f64(int32_t m, int32_t k, int32_t n, const int32_t *a_ptr, const int32_t *a_col,
                      const double *a_val, const int32_t *b_ptr, const int32_t *b_col, const double *b_val,
                      int64_t *c_row_ptr, int32_t *c_col, double *c_val);
int oracle_spgemm_f32(int32_t m, int32_t k, int32_t n, const int32_t *a_ptr, const int32_t *a_col,
                      const float *a_val, const int32_t *b_ptr, const int32_t *b_col, const float *b_val,
                      int64_t *c_row_ptr, int32_t *c_col, float *c_val);

/*
 * Row order of the window-sorted Row-grouped layout (an extension of
 * [RgCSR] section 3, whose weakness is the padding of a group to its
 * longest row, section 4): inside each window of `window` consecutive rows
 * (the last window may be shorter), rows are listed by decreasing length,
 * equal lengths by increasing row index; rows of length >= long_min (when
 * long_min > 0) count as length -1, i.e. they come last.  perm[p] (m
 * entries) is the row at position p; eff_len[p] (may be NULL) its length,
 * or -1 for a long row.  Returns 0, or 1 on bad arguments (window < 1).
 */
int oracle_window_sort(int32_t m, const int32_t *row_ptr, int32_t window, int32_t long_min, int32_t *perm,
                       int32_t *eff_len);

#ifdef __cplusplus
}
#endif

#endif
