/*
 * CPU oracle for the load-balanced CSR SpMV library (see oracle.h).
 *
 * TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check and the
 * benchmark's CPU-baseline leg; never by the product library.
 *
 * Everything is a direct restatement of a definition on the pages, in the
 * plainest loop that states it.  Sums are carried in long double.
 * Build with -ffp-contract=off so the compiler does not fuse operations.
 */
#include "oracle.h"

#include <stddef.h>
#include <stdlib.h>

static int check_row_ptr_basic(int32_t m, const int32_t *row_ptr) {
    return m >= 0 && row_ptr != NULL;
}

/* [LBPM] section 4.3 / [RgCSR] section 3: y_i = alpha * sum_k a_ik x_k + beta * y_i */
int oracle_spmv_f64(int32_t m, int32_t n, const int32_t *row_ptr, const int32_t *col_idx,
                    const double *vals, const double *x, double alpha, double beta,
                    const double *y_old, const int32_t *rows, int64_t nrows, double *y_out,
                    double *mag_out) {
    if (!check_row_ptr_basic(m, row_ptr) || n < 0 || y_out == NULL) return 1;
    if (beta != 0.0 && y_old == NULL) return 1;
    const long double a = (long double)(double)alpha;
    const long double b = (long double)(double)beta;
    int64_t count = rows ? nrows : m;
    for (int64_t t = 0; t < count; ++t) {
        int32_t i = rows ? rows[t] : (int32_t)t;
        if (i < 0 || i >= m) return 1;
        long double acc = 0.0L, mag = 0.0L;
        for (int32_t k = row_ptr[i]; k < row_ptr[i + 1]; ++k) {
            long double prod = (long double)vals[k] * (long double)x[col_idx[k]];
            acc += prod;
            mag += prod < 0 ? -prod : prod;
        }
        long double y = a * acc;
        long double by = 0.0L;
        if (beta != 0.0) {
            by = b * (long double)y_old[i];
            y += by;
        }
        y_out[t] = (double)y;
        if (mag_out) {
            long double aa = a < 0 ? -a : a;
            mag_out[t] = (double)(aa * mag + (by < 0 ? -by : by));
        }
    }
    return 0;
}

int oracle_spmv_f32(int32_t m, int32_t n, const int32_t *row_ptr, const int32_t *col_idx,
                    const float *vals, const float *x, double alpha, double beta,
                    const float *y_old, const int32_t *rows, int64_t nrows, float *y_out,
                    double *mag_out) {
    if (!check_row_ptr_basic(m, row_ptr) || n < 0 || y_out == NULL) return 1;
    if (beta != 0.0 && y_old == NULL) return 1;
    const long double a = (long double)(float)alpha;
    const long double b = (long double)(float)beta;
    int64_t count = rows ? nrows : m;
    for (int64_t t = 0; t < count; ++t) {
        int32_t i = rows ? rows[t] : (int32_t)t;
        if (i < 0 || i >= m) return 1;
        long double acc = 0.0L, mag = 0.0L;
        for (int32_t k = row_ptr[i]; k < row_ptr[i + 1]; ++k) {
            long double prod = (long double)vals[k] * (long double)x[col_idx[k]];
            acc += prod;
            mag += prod < 0 ? -prod : prod;
        }
        long double y = a * acc;
        long double by = 0.0L;
        if (beta != 0.0) {
            by = b * (long double)y_old[i];
            y += by;
        }
        y_out[t] = (float)y;
        if (mag_out) {
            long double aa = a < 0 ? -a : a;
            mag_out[t] = (double)(aa * mag + (by < 0 ? -by : by));
        }
    }
    return 0;
}

/*
 * [LBPM] section 5.2.1.  The row end r is the unit at merge position
 * row_ptr[r+1] + r (all of row r's nonzeros and the r earlier row ends come
 * before it).  So after d units, the row ends taken are those with
 * row_ptr[r+1] + r < d.  The diagonals d_p rise with p and so does
 * row_ptr[r+1] + r with r, so one forward sweep over the rows counts them
 * for every p in turn.
 */
int oracle_merge_path_partition(int32_t m, int32_t nnz, const int32_t *row_ptr, int64_t T,
                                int64_t P, int32_t *part) {
    if (!check_row_ptr_basic(m, row_ptr) || nnz < 0 || T <= 0 || P < 1 || part == NULL) return 1;
    const int64_t total = (int64_t)m + (int64_t)nnz;
    int64_t i = 0;
    for (int64_t p = 0; p <= P; ++p) {
        int64_t d = p * T < total ? p * T : total;
        while (i < m && (int64_t)row_ptr[i + 1] + i < d) ++i;
        part[2 * p] = (int32_t)i;
        part[2 * p + 1] = (int32_t)(d - i);
    }
    return 0;
}

static int length_class(int32_t len) {
    int k = 0;
    while (k < 31 && (len >> k) != 0) ++k;
    return k; /* 0 for len == 0, else 1 + floor(log2(len)) */
}

int oracle_row_stats(int32_t m, int32_t n, int32_t nnz, const int32_t *row_ptr,
                     const int32_t *col_idx, oracle_stats_t *out) {
    if (!check_row_ptr_basic(m, row_ptr) || out == NULL || nnz < 0 || n < 0) return 1;
    for (int b = 0; b < 32; ++b) out->hist[b] = 0;
    for (int g = 0; g < 4; ++g) out->rg_slots[g] = 0;
    out->sum_len = 0;
    out->min_len = 0;
    out->max_len = 0;
    out->n_empty = 0;
    out->flags = 0;
    out->bandwidth = 0;
    out->reserved = 0;

    if (row_ptr[0] != 0) out->flags |= 1;
    for (int32_t i = 0; i < m; ++i)
        if (row_ptr[i + 1] < row_ptr[i]) out->flags |= 2;
    if (row_ptr[m] != nnz) out->flags |= 4;
    if (out->flags) return 0;

    for (int32_t k = 0; k < nnz; ++k)
        if (col_idx[k] < 0 || col_idx[k] >= n) out->flags |= 8;

    for (int32_t i = 0; i < m; ++i) {
        int32_t len = row_ptr[i + 1] - row_ptr[i];
        out->hist[length_class(len)] += 1;
        out->sum_len += len;
        if (i == 0 || len < out->min_len) out->min_len = len;
        if (i == 0 || len > out->max_len) out->max_len = len;
        if (len == 0) out->n_empty += 1;
        if (len > 0) {
            int64_t d_first = (int64_t)col_idx[row_ptr[i]] - i;
            int64_t d_last = (int64_t)col_idx[row_ptr[i + 1] - 1] - i;
            if (d_first < 0) d_first = -d_first;
            if (d_last < 0) d_last = -d_last;
            if (d_first > out->bandwidth) out->bandwidth = (int32_t)d_first;
            if (d_last > out->bandwidth) out->bandwidth = (int32_t)d_last;
        }
    }
    for (int g = 0; g < 4; ++g) {
        int32_t G = 32 << g;
        for (int32_t start = 0; start < m; start += G) {
            int32_t longest = 0;
            for (int32_t i = start; i < start + G && i < m; ++i) {
                int32_t len = row_ptr[i + 1] - row_ptr[i];
                if (len > longest) longest = len;
            }
            out->rg_slots[g] += (int64_t)G * longest;
        }
    }
    return 0;
}

/* [RgCSR] section 3, Figure 5 */
int oracle_rgcsr_layout(int32_t m, const int32_t *row_ptr, int32_t G, int64_t *group_ptr,
                        int32_t *row_len) {
    if (!check_row_ptr_basic(m, row_ptr) || G <= 0 || group_ptr == NULL) return 1;
    int32_t ngroups = (m + G - 1) / G;
    group_ptr[0] = 0;
    for (int32_t g = 0; g < ngroups; ++g) {
        int32_t longest = 0;
        for (int32_t i = g * G; i < (g + 1) * G && i < m; ++i) {
            int32_t len = row_ptr[i + 1] - row_ptr[i];
            if (len > longest) longest = len;
        }
        group_ptr[g + 1] = group_ptr[g] + (int64_t)G * longest;
    }
    if (row_len)
        for (int32_t i = 0; i < m; ++i) row_len[i] = row_ptr[i + 1] - row_ptr[i];
    return 0;
}

int oracle_rgcsr_pack_f64(int32_t m, const int32_t *row_ptr, const int32_t *col_idx,
                          const double *vals, int32_t G, const int64_t *group_ptr,
                          int32_t *rg_col, double *rg_val) {
    if (!check_row_ptr_basic(m, row_ptr) || G <= 0 || !group_ptr || !rg_col || !rg_val) return 1;
    int32_t ngroups = (m + G - 1) / G;
    for (int64_t s = 0; s < group_ptr[ngroups]; ++s) {
        rg_col[s] = 0;
        rg_val[s] = 0.0;
    }
    for (int32_t i = 0; i < m; ++i) {
        int64_t base = group_ptr[i / G] + (i % G);
        for (int32_t k = 0; k < row_ptr[i + 1] - row_ptr[i]; ++k) {
            rg_col[base + (int64_t)k * G] = col_idx[row_ptr[i] + k];
            rg_val[base + (int64_t)k * G] = vals[row_ptr[i] + k];
        }
    }
    return 0;
}

int oracle_rgcsr_pack_f32(int32_t m, const int32_t *row_ptr, const int32_t *col_idx,
                          const float *vals, int32_t G, const int64_t *group_ptr,
                          int32_t *rg_col, float *rg_val) {
    if (!check_row_ptr_basic(m, row_ptr) || G <= 0 || !group_ptr || !rg_col || !rg_val) return 1;
    int32_t ngroups = (m + G - 1) / G;
    for (int64_t s = 0; s < group_ptr[ngroups]; ++s) {
        rg_col[s] = 0;
        rg_val[s] = 0.0f;
    }
    for (int32_t i = 0; i < m; ++i) {
        int64_t base = group_ptr[i / G] + (i % G);
        for (int32_t k = 0; k < row_ptr[i + 1] - row_ptr[i]; ++k) {
            rg_col[base + (int64_t)k * G] = col_idx[row_ptr[i] + k];
            rg_val[base + (int64_t)k * G] = vals[row_ptr[i] + k];
        }
    }
    return 0;
}

/* [OpSparse] section 5.1: a row belongs to the bin when its length reaches
 * the bin's lower bound; the rows are listed in the order they are met. */
int oracle_long_rows(int32_t m, const int32_t *row_ptr, int32_t min_len, int32_t seg_nnz, int32_t *ids,
                     int64_t *seg_begin, int64_t *count) {
    if (!check_row_ptr_basic(m, row_ptr) || min_len < 1 || seg_nnz < 1 || count == NULL) return 1;
    int64_t t = 0, segs = 0;
    if (seg_begin) seg_begin[0] = 0;
    for (int32_t i = 0; i < m; ++i) {
        int32_t len = row_ptr[i + 1] - row_ptr[i];
        if (len < min_len) continue;
        segs += ((int64_t)len + seg_nnz - 1) / seg_nnz;
        if (ids) ids[t] = i;
        if (seg_begin) seg_begin[t + 1] = segs;
        ++t;
    }
    *count = t;
    return 0;
}

/* Selection of the next row by (length descending, index ascending), one
 * window at a time: the plainest statement of the order, quadratic in the
 * window size. */
int oracle_window_sort(int32_t m, const int32_t *row_ptr, int32_t window, int32_t long_min, int32_t *perm,
                       int32_t *eff_len) {
    if (!check_row_ptr_basic(m, row_ptr) || window < 1 || perm == NULL) return 1;
    char *taken = (char *)malloc((size_t)window);
    if (!taken) return 1;
    for (int32_t w0 = 0; w0 < m; w0 += window) {
        int32_t w1 = w0 + window < m ? w0 + window : m;
        for (int32_t i = w0; i < w1; ++i) taken[i - w0] = 0;
        for (int32_t p = w0; p < w1; ++p) {
            int32_t best = -1, best_len = 0;
            for (int32_t i = w0; i < w1; ++i) {
                if (taken[i - w0]) continue;
                int32_t len = row_ptr[i + 1] - row_ptr[i];
                if (long_min > 0 && len >= long_min) len = -1;
                if (best < 0 || len > best_len) {
                    best = i;
                    best_len = len;
                }
            }
            perm[p] = best;
            taken[best - w0] = 1;
            if (eff_len) eff_len[p] = best_len;
        }
    }
    free(taken);
    return 0;
}

/* [LBPM] section 4.3, Listing 4: for every row, for every column t of X,
 * sum vals[nz] * X[indices[nz]][t] over the row's nonzeros. */
#define ORACLE_SPMM(NAME, T)                                                                               \
    int NAME(int32_t m, int32_t n, int32_t k, const int32_t *row_ptr, const int32_t *col_idx,            \
             const T *vals, const T *X, int64_t ldx, double alpha, double beta, const T *Y_old,          \
             int64_t ldy, T *Y_out, double *mag_out) {                                                    \
        if (!check_row_ptr_basic(m, row_ptr) || n < 0 || k < 0 || Y_out == NULL || ldx < k) return 1;    \
        if (beta != 0.0 && (Y_old == NULL || ldy < k)) return 1;                                          \
        const long double a = (long double)(T)alpha;                                                      \
        const long double b = (long double)(T)beta;                                                       \
        for (int32_t i = 0; i < m; ++i) {                                                                 \
            for (int32_t t = 0; t < k; ++t) {                                                             \
                long double acc = 0.0L, mag = 0.0L;                                                       \
                for (int32_t q = row_ptr[i]; q < row_ptr[i + 1]; ++q) {                                   \
                    long double prod = (long double)vals[q] * (long double)X[(int64_t)col_idx[q] * ldx + t]; \
                    acc += prod;                                                                          \
                    mag += prod < 0 ? -prod : prod;                                                       \
                }                                                                                         \
                long double y = a * acc, by = 0.0L;                                                       \
                if (beta != 0.0) {                                                                        \
                    by = b * (long double)Y_old[(int64_t)i * ldy + t];                                    \
                    y += by;                                                                              \
                }                                                                                         \
                Y_out[(int64_t)i * k + t] = (T)y;                                                         \
                if (mag_out) {                                                                            \
                    long double aa = a < 0 ? -a : a;                                                      \
                    mag_out[(int64_t)i * k + t] = (double)(aa * mag + (by < 0 ? -by : by));               \
                }                                                                                         \
            }                                                                                             \
        }                                                                                                 \
        return 0;                                                                                         \
    }
ORACLE_SPMM(oracle_spmm_f64, double)
ORACLE_SPMM(oracle_spmm_f32, float)

/* Counting: column sizes, their prefix sums, then every entry of A in row
 * order appended to its column -- which lists each column's rows in
 * increasing order. */
#define ORACLE_TRANSPOSE(NAME, T)                                                                         \
    int NAME(int32_t m, int32_t n, const int32_t *row_ptr, const int32_t *col_idx, const T *vals,        \
             int32_t *t_ptr, int32_t *t_idx, T *t_vals, int32_t *t_src) {                                 \
        if (!check_row_ptr_basic(m, row_ptr) || n < 0 || !t_ptr || !t_idx || !t_vals) return 1;         \
        int32_t nnz = row_ptr[m];                                                                         \
        for (int32_t j = 0; j <= n; ++j) t_ptr[j] = 0;                                                    \
        for (int32_t q = 0; q < nnz; ++q) {                                                               \
            if (col_idx[q] < 0 || col_idx[q] >= n) return 1;                                              \
            t_ptr[col_idx[q] + 1] += 1;                                                                   \
        }                                                                                                 \
        for (int32_t j = 0; j < n; ++j) t_ptr[j + 1] += t_ptr[j];                                         \
        int32_t *next = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n > 0 ? n : 1));                     \
        if (!next) return 1;                                                                              \
        for (int32_t j = 0; j < n; ++j) next[j] = t_ptr[j];                                               \
        for (int32_t i = 0; i < m; ++i)                                                                   \
            for (int32_t q = row_ptr[i]; q < row_ptr[i + 1]; ++q) {                                       \
                int32_t pos = next[col_idx[q]]++;                                                         \
                t_idx[pos] = i;                                                                           \
                t_vals[pos] = vals[q];                                                                    \
                if (t_src) t_src[pos] = q;                                                                \
            }                                                                                             \
        free(next);                                                                                       \
        return 0;                                                                                         \
    }
ORACLE_TRANSPOSE(oracle_transpose_f64, double)
ORACLE_TRANSPOSE(oracle_transpose_f32, float)

/* y_j = alpha * sum_i a_ij x_i + beta * y_old_j, rows of A in order. */
#define ORACLE_SPMV_T(NAME, T)                                                                            \
    int NAME(int32_t m, int32_t n, const int32_t *row_ptr, const int32_t *col_idx, const T *vals,        \
             const T *x, double alpha, double beta, const T *y_old, T *y_out, double *mag_out) {          \
        if (!check_row_ptr_basic(m, row_ptr) || n < 0 || y_out == NULL) return 1;                        \
        if (beta != 0.0 && y_old == NULL) return 1;                                                       \
        const long double a = (long double)(T)alpha;                                                      \
        const long double b = (long double)(T)beta;                                                       \
        long double *acc = (long double *)calloc((size_t)(n > 0 ? n : 1), sizeof(long double));           \
        long double *mag = (long double *)calloc((size_t)(n > 0 ? n : 1), sizeof(long double));           \
        if (!acc || !mag) {                                                                               \
            free(acc);                                                                                    \
            free(mag);                                                                                    \
            return 1;                                                                                     \
        }                                                                                                 \
        for (int32_t i = 0; i < m; ++i)                                                                   \
            for (int32_t q = row_ptr[i]; q < row_ptr[i + 1]; ++q) {                                       \
                long double prod = (long double)vals[q] * (long double)x[i];                              \
                acc[col_idx[q]] += prod;                                                                  \
                mag[col_idx[q]] += prod < 0 ? -prod : prod;                                               \
            }                                                                                             \
        for (int32_t j = 0; j < n; ++j) {                                                                 \
            long double y = a * acc[j], by = 0.0L;                                                        \
            if (beta != 0.0) {                                                                            \
                by = b * (long double)y_old[j];                                                           \
                y += by;                                                                                  \
            }                                                                                             \
            y_out[j] = (T)y;                                                                              \
            if (mag_out) {                                                                                \
                long double aa = a < 0 ? -a : a;                                                          \
                mag_out[j] = (double)(aa * mag[j] + (by < 0 ? -by : by));                                 \
            }                                                                                             \
        }                                                                                                 \
        free(acc);                                                                                        \
        free(mag);                                                                                        \
        return 0;                                                                                         \
    }
ORACLE_SPMV_T(oracle_spmv_transposed_f64, double)
ORACLE_SPMV_T(oracle_spmv_transposed_f32, float)

/* Row by row: scatter every product of row i into a dense long double row
 * with a mark per column, listing each column the first time a product
 * lands on it; then sort that list and gather the row's entries in column
 * order.  (Only the listed columns are visited, so a row costs its products
 * plus the sort of its entries, not a pass over all n columns.) */
static int cmp_i32(const void *a, const void *b) {
    const int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}
#define ORACLE_SPGEMM(NAME, T)                                                                            \
    int NAME(int32_t m, int32_t k, int32_t n, const int32_t *a_ptr, const int32_t *a_col, const T *a_val, \
             const int32_t *b_ptr, const int32_t *b_col, const T *b_val, int64_t *c_row_ptr,              \
             int32_t *c_col, T *c_val) {                                                                  \
        if (!check_row_ptr_basic(m, a_ptr) || !check_row_ptr_basic(k, b_ptr) || n < 0 || !c_row_ptr)     \
            return 1;                                                                                     \
        long double *acc = (long double *)calloc((size_t)(n > 0 ? n : 1), sizeof(long double));           \
        char *mark = (char *)calloc((size_t)(n > 0 ? n : 1), 1);                                          \
        int32_t *touched = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n > 0 ? n : 1));                  \
        if (!acc || !mark || !touched) {                                                                  \
            free(acc);                                                                                    \
            free(mark);                                                                                   \
            free(touched);                                                                                \
            return 1;                                                                                     \
        }                                                                                                 \
        c_row_ptr[0] = 0;                                                                                 \
        for (int32_t i = 0; i < m; ++i) {                                                                 \
            int64_t nt = 0;                                                                               \
            for (int32_t p = a_ptr[i]; p < a_ptr[i + 1]; ++p) {                                           \
                int32_t q = a_col[p];                                                                     \
                if (q < 0 || q >= k) {                                                                    \
                    free(acc);                                                                            \
                    free(mark);                                                                           \
                    free(touched);                                                                        \
                    return 1;                                                                             \
                }                                                                                         \
                for (int32_t r = b_ptr[q]; r < b_ptr[q + 1]; ++r) {                                       \
                    const int32_t j = b_col[r];                                                           \
                    acc[j] += (long double)a_val[p] * (long double)b_val[r];                              \
                    if (!mark[j]) {                                                                       \
                        mark[j] = 1;                                                                      \
                        touched[nt++] = j;                                                                \
                    }                                                                                     \
                }                                                                                         \
            }                                                                                             \
            qsort(touched, (size_t)nt, sizeof(int32_t), cmp_i32);                                         \
            int64_t cnt = 0, out = c_row_ptr[i];                                                          \
            for (int64_t t = 0; t < nt; ++t) {                                                            \
                const int32_t j = touched[t];                                                             \
                if (mark[j]) {                                                                            \
                    if (c_col) {                                                                          \
                        c_col[out + cnt] = j;                                                             \
                        c_val[out + cnt] = (T)acc[j];                                                     \
                    }                                                                                     \
                    ++cnt;                                                                                \
                    mark[j] = 0;                                                                          \
                    acc[j] = 0.0L;                                                                        \
                }                                                                                         \
            }                                                                                             \
            c_row_ptr[i + 1] = c_row_ptr[i] + cnt;                                                        \
        }                                                                                                 \
        free(acc);                                                                                        \
        free(mark);                                                                                       \
        free(touched);                                                                                    \
        return 0;                                                                                         \
    }
ORACLE_SPGEMM(oracle_spgemm_f64, double)
ORACLE_SPGEMM(oracle_spgemm_f32, float)
