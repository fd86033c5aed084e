/*
 * Seeded synthetic inputs for the CSR SpMV library: sparse matrices in CSR
 * form (row lengths, sorted distinct column sets, values) and dense vectors.
 *
 * This file is shared by the tests, the benchmark and the oracle checks.  It
 * holds none of the SpMV arithmetic: it only draws numbers.  Row pointers are
 * formed by the caller (a running sum of the lengths drawn here).
 *
 * Random numbers: every array is drawn from its own named stream so that the
 * arrays do not depend on the order in which they are generated, and every
 * row (or every chunk of 65536 vector entries) seeds its own generator, so
 * rows can be filled in parallel and the result does not depend on the
 * thread count.
 *   - seeding: SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom
 *     number generators", OOPSLA 2014);
 *   - draws: xoshiro256** (Blackman, Vigna, "Scrambled linear pseudorandom
 *     number generators", 2018).
 * Uniform doubles take the top 53 bits; normals use Marsaglia's polar method;
 * bounded integers use the high half of a 64x64-bit product (Lemire 2019;
 * the bias is below 2^-40 for the ranges used here).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct { uint64_t s[4]; } rng_t;

static uint64_t sm64(uint64_t *state) {
    uint64_t z = (*state += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static void rng_init(rng_t *r, uint64_t seed, uint64_t stream, uint64_t index) {
    uint64_t k = seed;
    uint64_t a = sm64(&k);
    k = a ^ (stream * 0xD6E8FEB86659FD93ull);
    uint64_t b = sm64(&k);
    k = b ^ (index * 0xA0761D6478BD642Full);
    for (int i = 0; i < 4; ++i) r->s[i] = sm64(&k);
    if ((r->s[0] | r->s[1] | r->s[2] | r->s[3]) == 0) r->s[0] = 1;
}

static inline uint64_t rotl64(uint64_t v, int k) { return (v << k) | (v >> (64 - k)); }

static inline uint64_t rng_next(rng_t *r) {
    uint64_t *s = r->s;
    uint64_t out = rotl64(s[1] * 5, 7) * 9;
    uint64_t t = s[1] << 17;
    s[2] ^= s[0];
    s[3] ^= s[1];
    s[1] ^= s[2];
    s[0] ^= s[3];
    s[2] ^= t;
    s[3] = rotl64(s[3], 45);
    return out;
}

/* uniform in [0, 1) */
static inline double rng_u01(rng_t *r) { return (double)(rng_next(r) >> 11) * 0x1.0p-53; }

/* uniform integer in [0, k) */
static inline uint64_t rng_below(rng_t *r, uint64_t k) {
    return (uint64_t)(((unsigned __int128)rng_next(r) * (unsigned __int128)k) >> 64);
}

static inline double rng_normal(rng_t *r) {
    for (;;) {
        double u = 2.0 * rng_u01(r) - 1.0;
        double v = 2.0 * rng_u01(r) - 1.0;
        double q = u * u + v * v;
        if (q > 0.0 && q < 1.0) return u * sqrt(-2.0 * log(q) / q);
    }
}

/* stream identifiers */
enum { ST_LEN = 1, ST_COL = 2, ST_VAL = 3, ST_PLACE = 4, ST_VEC = 16 };

/* value distributions */
enum { DIST_UNIFORM_PM1 = 0, DIST_NORMAL = 1, DIST_SMALL_INT = 2 };

static inline double draw_value(rng_t *r, int dist) {
    switch (dist) {
    case DIST_NORMAL: return rng_normal(r);
    case DIST_SMALL_INT: return (double)((int64_t)rng_below(r, 7) - 3); /* -3..3, exact */
    default: return 2.0 * rng_u01(r) - 1.0;
    }
}

/* ------------------------------------------------------------------ */
/* dense vectors                                                        */

#define VEC_CHUNK 65536

/* out[i] for i in [0, n): dist as above; f64 != 0 selects double output. */
int synth_vector(int64_t n, int dist, uint64_t seed, uint64_t stream, int f64, void *out) {
    if (n < 0 || (n > 0 && !out)) return 1;
    int64_t nchunks = (n + VEC_CHUNK - 1) / VEC_CHUNK;
#pragma omp parallel for schedule(static)
    for (int64_t c = 0; c < nchunks; ++c) {
        rng_t r;
        rng_init(&r, seed, ST_VEC + stream, (uint64_t)c);
        int64_t lo = c * VEC_CHUNK, hi = lo + VEC_CHUNK < n ? lo + VEC_CHUNK : n;
        for (int64_t i = lo; i < hi; ++i) {
            double v = draw_value(&r, dist);
            if (f64) ((double *)out)[i] = v;
            else ((float *)out)[i] = (float)v;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* row lengths                                                          */

/* Uniform integer lengths in [lo, hi] per row. */
int synth_lengths_uniform(int32_t m, int32_t lo, int32_t hi, uint64_t seed, int32_t *len) {
    if (m < 0 || lo < 0 || hi < lo) return 1;
#pragma omp parallel for schedule(static)
    for (int32_t i = 0; i < m; ++i) {
        rng_t r;
        rng_init(&r, seed, ST_LEN, (uint64_t)i);
        len[i] = lo + (int32_t)rng_below(&r, (uint64_t)(hi - lo + 1));
    }
    return 0;
}

/*
 * Power-law lengths: X = (1-u)^(-1/(a-1)) (Pareto with x_min = 1, so the
 * density falls as X^-a), then L = clip(round(s*X), 1, cap) with the scale s
 * found by bisection so that the mean of L is target_mean +- tol.  X is
 * scaled before rounding: scaling an already-floored X makes the mean jump
 * by about 0.5 whenever the half of the rows with floor(X) = 1 change their
 * rounded length together, and the target could not be met.
 * Returns 0 on success, 2 if the target mean could not be reached.
 */
int synth_lengths_powerlaw(int32_t m, double exponent, int32_t cap, double target_mean,
                           double tol, uint64_t seed, int32_t *len, double *scale_out) {
    if (m <= 0 || exponent <= 1.0 || cap < 1) return 1;
    double *base = (double *)malloc(sizeof(double) * (size_t)m);
    if (!base) return 3;
    double inv = -1.0 / (exponent - 1.0);
#pragma omp parallel for schedule(static)
    for (int32_t i = 0; i < m; ++i) {
        rng_t r;
        rng_init(&r, seed, ST_LEN, (uint64_t)i);
        double u = rng_u01(&r);
        base[i] = pow(1.0 - u, inv);
    }
    double lo = 1e-3, hi = 1e3, s = 1.0;
    int ok = 0;
    for (int it = 0; it < 200; ++it) {
        s = 0.5 * (lo + hi);
        int64_t total = 0;
#pragma omp parallel for reduction(+ : total) schedule(static)
        for (int32_t i = 0; i < m; ++i) {
            double v = round(s * base[i]);
            int64_t l = v < 1.0 ? 1 : (v > (double)cap ? cap : (int64_t)v);
            total += l;
        }
        double mean = (double)total / (double)m;
        if (fabs(mean - target_mean) <= tol) { ok = 1; break; }
        if (mean < target_mean) lo = s; else hi = s;
    }
#pragma omp parallel for schedule(static)
    for (int32_t i = 0; i < m; ++i) {
        double v = round(s * base[i]);
        len[i] = v < 1.0 ? 1 : (v > (double)cap ? cap : (int32_t)v);
    }
    free(base);
    if (scale_out) *scale_out = s;
    return ok ? 0 : 2;
}

/*
 * Extreme skew: lengths uniform in [lo, hi] everywhere, then the rows picked
 * (distinct, uniform over [0, m), from the placement stream) get the given
 * heavy lengths, in order: heavy_len[0] goes to the first pick, and so on.
 * The picked row indices are written to rows_out (nheavy entries).
 */
int synth_lengths_skew(int32_t m, int32_t lo, int32_t hi, int32_t nheavy, const int32_t *heavy_len,
                       uint64_t seed, int32_t *len, int32_t *rows_out) {
    if (nheavy < 0 || nheavy > m) return 1;
    int rc = synth_lengths_uniform(m, lo, hi, seed, len);
    if (rc) return rc;
    rng_t r;
    rng_init(&r, seed, ST_PLACE, 0);
    for (int32_t h = 0; h < nheavy; ++h) {
        for (;;) {
            int32_t cand = (int32_t)rng_below(&r, (uint64_t)m);
            int dup = 0;
            for (int32_t q = 0; q < h; ++q) dup |= rows_out[q] == cand;
            if (!dup) { rows_out[h] = cand; break; }
        }
        len[rows_out[h]] = heavy_len[h];
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* column sets                                                          */

static int cmp_i32(const void *a, const void *b) {
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

static void sort_i32(int32_t *v, int64_t n) {
    if (n <= 32) {
        for (int64_t i = 1; i < n; ++i) {
            int32_t t = v[i];
            int64_t j = i - 1;
            while (j >= 0 && v[j] > t) { v[j + 1] = v[j]; --j; }
            v[j + 1] = t;
        }
    } else {
        qsort(v, (size_t)n, sizeof(int32_t), cmp_i32);
    }
}

static int64_t unique_sorted(int32_t *v, int64_t n) {
    if (n == 0) return 0;
    int64_t w = 1;
    for (int64_t i = 1; i < n; ++i)
        if (v[i] != v[w - 1]) v[w++] = v[i];
    return w;
}

/*
 * Draw L distinct columns from [lo, lo+R), sorted ascending, into out.
 * Dense requests use selection sampling (Knuth, TAOCP vol. 2, Algorithm S);
 * sparse ones draw, sort, drop duplicates and top up.  tmp holds >= L ints.
 */
static void draw_columns(rng_t *r, int32_t lo, int64_t R, int64_t L, int32_t *out, int32_t *tmp) {
    if (L <= 0) return;
    if (L * 8 >= R) {
        int64_t need = L, left = R, w = 0;
        for (int64_t c = 0; c < R && need > 0; ++c, --left) {
            if ((int64_t)rng_below(r, (uint64_t)left) < need) { out[w++] = lo + (int32_t)c; --need; }
        }
        return;
    }
    int64_t have = 0;
    while (have < L) {
        int64_t want = L - have;
        for (int64_t k = 0; k < want; ++k) tmp[k] = lo + (int32_t)rng_below(r, (uint64_t)R);
        memcpy(out + have, tmp, sizeof(int32_t) * (size_t)want);
        have += want;
        sort_i32(out, have);
        have = unique_sorted(out, have);
    }
}

/*
 * Fill the columns and values of a CSR matrix whose row pointers are given.
 * Row i draws its columns uniformly without repetition from
 *   [max(0, i-band), min(n-1, i+band)]  if band >= 0,
 *   [0, n)                              if band < 0,
 * sorted ascending, and its values from dist.  f64 selects the value type.
 * Returns 1 on bad arguments, 2 if a row is longer than its column range.
 */
int synth_fill_random(int32_t m, int32_t n, const int32_t *rp, int32_t band, int dist,
                      uint64_t seed, int f64, int32_t *col, void *val) {
    if (m < 0 || n < 0 || !rp) return 1;
    int32_t maxlen = 0;
    for (int32_t i = 0; i < m; ++i) {
        int32_t l = rp[i + 1] - rp[i];
        if (l < 0) return 1;
        if (l > maxlen) maxlen = l;
        int64_t lo = band < 0 ? 0 : (i - (int64_t)band < 0 ? 0 : i - (int64_t)band);
        int64_t hi = band < 0 ? n - 1 : (i + (int64_t)band > n - 1 ? n - 1 : i + (int64_t)band);
        if (l > 0 && (hi < lo || l > hi - lo + 1)) return 2;
    }
    int err = 0;
#pragma omp parallel
    {
        int32_t *tmp = (int32_t *)malloc(sizeof(int32_t) * ((size_t)maxlen + 1));
        if (!tmp) err = 3;
#pragma omp for schedule(dynamic, 4096)
        for (int32_t i = 0; i < m; ++i) {
            if (!tmp) continue;
            int64_t l = rp[i + 1] - rp[i];
            if (l == 0) continue;
            int64_t lo = band < 0 ? 0 : (i - (int64_t)band < 0 ? 0 : i - (int64_t)band);
            int64_t hi = band < 0 ? n - 1 : (i + (int64_t)band > n - 1 ? n - 1 : i + (int64_t)band);
            rng_t rc, rv;
            rng_init(&rc, seed, ST_COL, (uint64_t)i);
            rng_init(&rv, seed, ST_VAL, (uint64_t)i);
            draw_columns(&rc, (int32_t)lo, hi - lo + 1, l, col + rp[i], tmp);
            for (int64_t k = 0; k < l; ++k) {
                double v = draw_value(&rv, dist);
                if (f64) ((double *)val)[rp[i] + k] = v;
                else ((float *)val)[rp[i] + k] = (float)v;
            }
        }
        free(tmp);
    }
    return err;
}

/* ------------------------------------------------------------------ */
/* structured matrices                                                  */

/* 2-D 5-point Laplacian on an nx-by-ny grid, Dirichlet boundary:
 * row lengths (pass 1) */
int synth_laplace2d_lengths(int32_t nx, int32_t ny, int32_t *len) {
    if (nx <= 0 || ny <= 0) return 1;
    for (int32_t r = 0; r < ny; ++r)
        for (int32_t c = 0; c < nx; ++c)
            len[(int64_t)r * nx + c] = 1 + (r > 0) + (r < ny - 1) + (c > 0) + (c < nx - 1);
    return 0;
}

/* pass 2: columns ascending; 4 on the diagonal, -1 off it */
int synth_laplace2d_fill(int32_t nx, int32_t ny, const int32_t *rp, int f64, int32_t *col, void *val) {
    if (nx <= 0 || ny <= 0) return 1;
    for (int32_t r = 0; r < ny; ++r)
        for (int32_t c = 0; c < nx; ++c) {
            int64_t i = (int64_t)r * nx + c;
            int64_t k = rp[i];
            int64_t cols[5];
            double vals[5];
            int q = 0;
            if (r > 0) { cols[q] = i - nx; vals[q++] = -1.0; }
            if (c > 0) { cols[q] = i - 1; vals[q++] = -1.0; }
            cols[q] = i; vals[q++] = 4.0;
            if (c < nx - 1) { cols[q] = i + 1; vals[q++] = -1.0; }
            if (r < ny - 1) { cols[q] = i + nx; vals[q++] = -1.0; }
            for (int t = 0; t < q; ++t) {
                col[k + t] = (int32_t)cols[t];
                if (f64) ((double *)val)[k + t] = vals[t];
                else ((float *)val)[k + t] = (float)vals[t];
            }
        }
    return 0;
}

/* 3-D 27-point stencil on a g^3 grid, Dirichlet boundary: row lengths */
int synth_stencil27_lengths(int32_t g, int32_t *len) {
    if (g <= 0) return 1;
    int64_t gg = (int64_t)g * g;
#pragma omp parallel for schedule(static)
    for (int32_t z = 0; z < g; ++z)
        for (int32_t y = 0; y < g; ++y)
            for (int32_t x = 0; x < g; ++x) {
                int a = 1 + (x > 0) + (x < g - 1);
                int b = 1 + (y > 0) + (y < g - 1);
                int c = 1 + (z > 0) + (z < g - 1);
                len[z * gg + (int64_t)y * g + x] = a * b * c;
            }
    return 0;
}

/* pass 2: columns ascending; off-diagonal values from dist, diagonal = diag */
int synth_stencil27_fill(int32_t g, const int32_t *rp, int dist, double diag, uint64_t seed, int f64,
                         int32_t *col, void *val) {
    if (g <= 0) return 1;
    int64_t gg = (int64_t)g * g;
#pragma omp parallel for schedule(static)
    for (int32_t z = 0; z < g; ++z)
        for (int32_t y = 0; y < g; ++y)
            for (int32_t x = 0; x < g; ++x) {
                int64_t i = z * gg + (int64_t)y * g + x;
                int64_t k = rp[i];
                rng_t rv;
                rng_init(&rv, seed, ST_VAL, (uint64_t)i);
                for (int dz = -1; dz <= 1; ++dz) {
                    if (z + dz < 0 || z + dz >= g) continue;
                    for (int dy = -1; dy <= 1; ++dy) {
                        if (y + dy < 0 || y + dy >= g) continue;
                        for (int dx = -1; dx <= 1; ++dx) {
                            if (x + dx < 0 || x + dx >= g) continue;
                            int64_t j = (z + dz) * gg + (int64_t)(y + dy) * g + (x + dx);
                            double v = (j == i) ? diag : draw_value(&rv, dist);
                            col[k] = (int32_t)j;
                            if (f64) ((double *)val)[k] = v;
                            else ((float *)val)[k] = (float)v;
                            ++k;
                        }
                    }
                }
            }
    return 0;
}
