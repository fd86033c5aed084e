"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each check is chosen so that a plausible slip in the oracle (a dropped term,
a wrong sign, a swapped index, a transposed operand, an off-by-one in the
merge order or the length classes) fails at least one of them:

* SpMV: a dense product on exactly representable inputs (exact equality),
  the 5-point Laplacian times the all-ones vector (closed form), A e_j equals
  column j, 1^T (A x) = (A^T 1)^T x, linearity in alpha and beta, empty rows.
* merge-path partition: a literal step-by-step merge walk on every small
  row-pointer array, the interval characterisation of the split on larger
  ones, monotonicity and the end points.
* row statistics: counting by other means.
* Row-grouped CSR: the worked example of the Row-grouped CSR page
  (tests/golden/rgcsr_figure5.json) and a decode round trip.
"""
import itertools
import json
import os

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def dense(A: synth.CSR) -> np.ndarray:
    D = np.zeros((A.m, A.n), dtype=np.float64)
    for i in range(A.m):
        for k in range(A.row_ptr[i], A.row_ptr[i + 1]):
            D[i, A.col_idx[k]] += float(A.vals[k])
    return D


# ---------------------------------------------------------------- SpMV


@pytest.mark.parametrize("dtype", ["f64", "f32"])
@pytest.mark.parametrize("shape", [(1, 1), (7, 3), (3, 7), (33, 64), (64, 64), (64, 17)])
def test_spmv_equals_dense_product_exactly(dtype, shape):
    """Small integers make every product and partial sum exact, so the
    oracle must equal the dense product bit for bit (non-square shapes catch
    a transposed operand)."""
    m, n = shape
    for seed in range(3):
        A = synth.random_csr(m, n, max_len=max(1, n // 2), empty_frac=0.2,
                             dist=synth.DIST_SMALL_INT, seed=seed, dtype=dtype)
        x = synth.vector(n, synth.DIST_SMALL_INT, seed, synth.STREAM_X, dtype)
        y0 = synth.vector(m, synth.DIST_SMALL_INT, seed, synth.STREAM_Y, dtype)
        D = dense(A)
        for alpha, beta in [(1.0, 0.0), (2.0, -3.0), (-1.0, 1.0), (0.0, 1.0), (0.5, 0.25)]:
            y, mag = oracle.spmv(A.row_ptr, A.col_idx, A.vals, x, alpha, beta, y0)
            want = alpha * (D @ x.astype(np.float64)) + beta * y0.astype(np.float64)
            np.testing.assert_array_equal(y.astype(np.float64), want)
            want_mag = abs(alpha) * (np.abs(D) @ np.abs(x.astype(np.float64))) + np.abs(beta * y0.astype(np.float64))
            np.testing.assert_array_equal(mag, want_mag)


def test_spmv_random_reals_against_dense():
    for seed in range(4):
        A = synth.random_csr(50, 40, max_len=30, empty_frac=0.1, dist=synth.DIST_NORMAL, seed=seed)
        x = synth.vector(40, synth.DIST_NORMAL, seed, synth.STREAM_X, "f64")
        y0 = synth.vector(50, synth.DIST_NORMAL, seed, synth.STREAM_Y, "f64")
        y, mag = oracle.spmv(A.row_ptr, A.col_idx, A.vals, x, 1.5, -0.5, y0)
        want = 1.5 * (dense(A) @ x) - 0.5 * y0
        assert np.all(np.abs(y - want) <= 1e-14 * mag + 1e-300)


@pytest.mark.parametrize("nx,ny", [(64, 64), (5, 9), (1, 6), (2, 2)])
def test_laplacian_times_ones_closed_form(nx, ny):
    """5-point Laplacian (4 on the diagonal, -1 per grid neighbour): A*1 is 0
    on interior rows and the number of missing neighbours on boundary rows."""
    A = synth.laplace2d(nx, ny, "f64")
    ones = np.ones(A.n)
    y, _ = oracle.spmv(A.row_ptr, A.col_idx, A.vals, ones)
    for r in range(ny):
        for c in range(nx):
            missing = (r == 0) + (r == ny - 1) + (c == 0) + (c == nx - 1)
            assert y[r * nx + c] == float(missing)


def test_spmv_unit_vectors_give_columns():
    A = synth.random_csr(40, 25, max_len=10, empty_frac=0.25, dist=synth.DIST_NORMAL, seed=5)
    for j in range(A.n):
        e = np.zeros(A.n)
        e[j] = 1.0
        y, _ = oracle.spmv(A.row_ptr, A.col_idx, A.vals, e)
        col = np.zeros(A.m)
        for i in range(A.m):
            seg = slice(A.row_ptr[i], A.row_ptr[i + 1])
            hit = A.col_idx[seg] == j
            col[i] = A.vals[seg][hit].sum()
        np.testing.assert_array_equal(y, col)


def test_spmv_transpose_identity():
    """1^T (A x) = (A^T 1)^T x, with A^T 1 the column sums taken by bincount."""
    for seed in range(3):
        A = synth.random_csr(300, 200, max_len=40, empty_frac=0.1, dist=synth.DIST_NORMAL, seed=seed)
        x = synth.vector(200, synth.DIST_NORMAL, seed, synth.STREAM_X, "f64")
        y, mag = oracle.spmv(A.row_ptr, A.col_idx, A.vals, x)
        colsum = np.bincount(A.col_idx, weights=A.vals, minlength=A.n)
        lhs = np.sum(y.astype(np.longdouble))
        rhs = np.sum(colsum.astype(np.longdouble) * x.astype(np.longdouble))
        assert abs(float(lhs - rhs)) <= 1e-12 * mag.sum()


def test_spmv_linearity_in_alpha_beta():
    A = synth.random_csr(100, 90, max_len=20, empty_frac=0.2, dist=synth.DIST_NORMAL, seed=11)
    x = synth.vector(90, synth.DIST_NORMAL, 11, synth.STREAM_X, "f64")
    y0 = synth.vector(100, synth.DIST_NORMAL, 11, synth.STREAM_Y, "f64")
    ax, mag = oracle.spmv(A.row_ptr, A.col_idx, A.vals, x)
    for alpha, beta in [(2.0, 0.0), (-1.25, 0.5), (0.0, -2.0), (3.0, 1.0)]:
        y, _ = oracle.spmv(A.row_ptr, A.col_idx, A.vals, x, alpha, beta, y0)
        want = alpha * ax + beta * y0
        assert np.all(np.abs(y - want) <= 1e-15 * (abs(alpha) * mag + np.abs(beta * y0)) + 1e-300)


def test_spmv_beta_zero_ignores_y_and_empty_rows():
    A = synth.random_csr(64, 64, max_len=6, empty_frac=0.5, dist=synth.DIST_NORMAL, seed=2)
    x = synth.vector(64, synth.DIST_NORMAL, 2, synth.STREAM_X, "f64")
    nan_y = np.full(64, np.nan)
    y, _ = oracle.spmv(A.row_ptr, A.col_idx, A.vals, x, 1.0, 0.0, nan_y)
    assert np.all(np.isfinite(y))
    empty = np.diff(A.row_ptr) == 0
    assert empty.any()
    assert np.all(y[empty] == 0.0)
    y0 = synth.vector(64, synth.DIST_NORMAL, 2, synth.STREAM_Y, "f64")
    y2, _ = oracle.spmv(A.row_ptr, A.col_idx, A.vals, x, 1.0, 0.75, y0)
    np.testing.assert_array_equal(y2[empty], 0.75 * y0[empty])


def test_spmv_rows_subset_matches_full():
    A = synth.random_csr(80, 80, max_len=12, empty_frac=0.1, dist=synth.DIST_NORMAL, seed=4, dtype="f32")
    x = synth.vector(80, synth.DIST_NORMAL, 4, synth.STREAM_X, "f32")
    y0 = synth.vector(80, synth.DIST_NORMAL, 4, synth.STREAM_Y, "f32")
    full, fmag = oracle.spmv(A.row_ptr, A.col_idx, A.vals, x, 1.5, 0.5, y0)
    rows = np.array([79, 0, 13, 13, 40], dtype=np.int32)
    sub, smag = oracle.spmv(A.row_ptr, A.col_idx, A.vals, x, 1.5, 0.5, y0, rows=rows)
    np.testing.assert_array_equal(sub, full[rows])
    np.testing.assert_array_equal(smag, fmag[rows])


def test_spmv_f32_products_are_exact_in_long_double():
    """fp32 x fp32 products are exact in long double, so a row with one
    nonzero returns the correctly rounded fp32 product."""
    rp = np.arange(5, dtype=np.int32)
    col = np.array([0, 1, 2, 3], dtype=np.int32)
    vals = np.array([1.1, -3.7, 1e-20, 7e30], dtype=np.float32)
    x = np.array([0.3, 2.9, 5e-20, -1e-3], dtype=np.float32)
    y, _ = oracle.spmv(rp, col, vals, x)
    np.testing.assert_array_equal(y, vals * x)


# ---------------------------------------------------------------- merge path


def merge_walk(row_ptr):
    """Literal merge of the row-end list with the nonzero indices: returns the
    (i, j) state after every number of steps d = 0 .. m + nnz."""
    m = len(row_ptr) - 1
    nnz = row_ptr[-1]
    i = j = 0
    states = [(0, 0)]
    while i < m or j < nnz:
        if i < m and row_ptr[i + 1] <= j:
            i += 1  # end of row i is next (ties go to the row end)
        else:
            j += 1  # nonzero j is next
        states.append((i, j))
    return states


def all_row_ptrs(m, nnz):
    for cuts in itertools.combinations_with_replacement(range(nnz + 1), m - 1):
        yield [0, *cuts, nnz]


def test_partition_matches_literal_merge_walk_exhaustively():
    count = 0
    for m in range(1, 6):
        for nnz in range(0, 9):
            for rp in all_row_ptrs(m, nnz):
                states = merge_walk(rp)
                total = m + nnz
                for T in (1, 2, 3, 5, total + 3):
                    P = max(1, -(-total // T))
                    part = oracle.merge_path_partition(np.array(rp), T, P)
                    for p in range(P + 1):
                        d = min(p * T, total)
                        assert tuple(part[p]) == states[d], (rp, T, p)
                count += 1
    assert count > 2000


def test_partition_empty_matrix_shapes():
    part = oracle.merge_path_partition(np.array([0], dtype=np.int32), 4, 1)
    assert part.tolist() == [[0, 0], [0, 0]]
    part = oracle.merge_path_partition(np.zeros(4, dtype=np.int32), 2, 2)
    assert part.tolist() == [[0, 0], [2, 0], [3, 0]]


@pytest.mark.parametrize("kind", ["random", "one_huge_row", "leading_trailing_empty", "all_empty"])
def test_partition_interval_property(kind):
    rng = np.random.default_rng(7)
    m = 3000
    if kind == "random":
        lens = rng.integers(0, 12, size=m)
    elif kind == "one_huge_row":
        lens = rng.integers(0, 3, size=m)
        lens[1234] = 50000
    elif kind == "leading_trailing_empty":
        lens = rng.integers(1, 9, size=m)
        lens[:400] = 0
        lens[-500:] = 0
    else:
        lens = np.zeros(m, dtype=np.int64)
    rp = synth.row_ptr_from_lengths(lens.astype(np.int32))
    nnz = int(rp[-1])
    total = m + nnz
    for T in (1, 7, 256, 2048):
        part = oracle.merge_path_partition(rp, T).astype(np.int64)
        d = np.minimum(np.arange(len(part), dtype=np.int64) * T, total)
        i, j = part[:, 0], part[:, 1]
        assert np.all(i + j == d)
        assert i[0] == 0 and j[0] == 0 and i[-1] == m and j[-1] == nnz
        assert np.all(np.diff(i) >= 0) and np.all(np.diff(j) >= 0)
        # state (i, j) after d units: row_ptr[i] + i <= d <= row_ptr[i+1] + i
        rpl = rp.astype(np.int64)
        upper = np.where(i < m, rpl[np.minimum(i + 1, m)] + i, np.iinfo(np.int64).max)
        assert np.all(rpl[i] + i <= d) and np.all(d <= upper)
        if T == 1:
            assert np.all(np.diff(i) <= 1)


# ---------------------------------------------------------------- row statistics


def brute_stats(rp, col, n):
    lens = np.diff(np.asarray(rp, dtype=np.int64))
    cls = np.array([int(v).bit_length() for v in lens], dtype=np.int64)
    hist = np.bincount(cls, minlength=32)[:32]
    slots = []
    m = len(lens)
    for g in range(4):
        G = 32 << g
        padded = np.zeros(-(-m // G) * G, dtype=np.int64)
        padded[:m] = lens
        slots.append(int(G * padded.reshape(-1, G).max(axis=1).sum()) if m else 0)
    bw = 0
    for i in range(m):
        seg = np.asarray(col[rp[i]:rp[i + 1]], dtype=np.int64)
        if len(seg):
            bw = max(bw, int(abs(seg[0] - i)), int(abs(seg[-1] - i)))
    return {"hist": hist.tolist(), "sum_len": int(lens.sum()), "rg_slots": slots,
            "min_len": int(lens.min()) if m else 0, "max_len": int(lens.max()) if m else 0,
            "n_empty": int((lens == 0).sum()), "flags": int(bool(np.any((col < 0) | (col >= n)))) * 8,
            "bandwidth": bw}


@pytest.mark.parametrize("seed", range(4))
def test_row_stats_brute_force(seed):
    rng = np.random.default_rng(seed)
    m = int(rng.integers(1, 3000))
    lens = (rng.pareto(1.2, size=m) * 3).astype(np.int64)
    lens[rng.random(m) < 0.1] = 0
    lens = np.minimum(lens, 5000)
    A = synth.fill_random(lens.astype(np.int32), 6000, seed=seed)
    s = oracle.row_stats(A.row_ptr, A.col_idx, A.n)
    assert s == brute_stats(A.row_ptr, A.col_idx, A.n)
    assert sum(s["hist"]) == m and s["sum_len"] == A.nnz


def test_row_stats_flags():
    rp = np.array([0, 2, 1, 3], dtype=np.int32)
    assert oracle.row_stats(rp, np.zeros(3, np.int32), 4)["flags"] & 2
    rp = np.array([1, 2, 3], dtype=np.int32)
    assert oracle.row_stats(rp, np.zeros(3, np.int32), 4, nnz=3)["flags"] & 1
    rp = np.array([0, 2, 3], dtype=np.int32)
    assert oracle.row_stats(rp, np.zeros(4, np.int32), 4, nnz=4)["flags"] & 4
    rp = np.array([0, 2, 3], dtype=np.int32)
    assert oracle.row_stats(rp, np.array([0, 4, 1], np.int32), 4)["flags"] == 8
    assert oracle.row_stats(rp, np.array([0, -1, 1], np.int32), 4)["flags"] == 8
    assert oracle.row_stats(rp, np.array([0, 3, 1], np.int32), 4)["flags"] == 0


def test_bandwidth_of_known_matrices():
    """5-point Laplacian on an nx-wide grid: outermost entries at +-nx; a
    band-limited random matrix stays within its band; the identity has 0."""
    A = synth.laplace2d(16, 9, "f64")
    assert oracle.row_stats(A.row_ptr, A.col_idx, A.n)["bandwidth"] == 16
    B = synth.fill_random(synth.lengths_uniform(5000, 1, 6, 3), 5000, band=37, seed=3)
    bw = oracle.row_stats(B.row_ptr, B.col_idx, B.n)["bandwidth"]
    assert 30 <= bw <= 37
    rp = np.arange(11, dtype=np.int32)
    assert oracle.row_stats(rp, np.arange(10, dtype=np.int32), 10)["bandwidth"] == 0
    assert oracle.row_stats(rp, np.arange(10, dtype=np.int32)[::-1].copy(), 10)["bandwidth"] == 9


def test_length_class_boundaries():
    lens = np.array([0, 1, 2, 3, 4, 7, 8, 1023, 1024, 2**20], dtype=np.int32)
    A = synth.fill_random(lens, 2**21, seed=1)
    s = oracle.row_stats(A.row_ptr, A.col_idx, A.n)
    want = np.zeros(32, dtype=np.int64)
    for v, k in [(0, 0), (1, 1), (2, 2), (3, 2), (4, 3), (7, 3), (8, 4), (1023, 10), (1024, 11), (2**20, 21)]:
        want[k] += 1
    assert s["hist"] == want.tolist()


# ---------------------------------------------------------------- Row-grouped CSR


def test_rgcsr_worked_example_from_the_page():
    g = json.load(open(os.path.join(GOLDEN, "rgcsr_figure5.json")))
    rp = np.array(g["row_ptr"], dtype=np.int32)
    assert np.diff(rp).tolist() == g["row_len"]
    assert rp[:-1].tolist() == [0, 2, 3, 4, 5, 6, 8, 11] and rp[-1] == 13
    gp, rl = oracle.rgcsr_layout(rp, g["rgcsr_group_size"])
    assert gp.tolist() == g["rgcsr_group_ptr"]
    assert rl.tolist() == g["row_len"]
    assert gp[-1] - rp[-1] == g["rgcsr_padding"]
    # ELLPACK is the one-group case: width = longest row, padding 11
    gp_ell, _ = oracle.rgcsr_layout(rp, g["m"])
    assert gp_ell[-1] == g["m"] * g["ellpack_width"]
    assert gp_ell[-1] - rp[-1] == g["ellpack_padding"]
    assert g["block_csr_stored"] - rp[-1] == g["block_csr_padding"]


@pytest.mark.parametrize("G", [1, 4, 32, 128])
def test_rgcsr_pack_decodes_back_to_csr(G):
    A = synth.random_csr(301, 77, max_len=9, empty_frac=0.2, dist=synth.DIST_NORMAL, seed=G)
    gp, rl, rg_col, rg_val = oracle.rgcsr_pack(A.row_ptr, A.col_idx, A.vals, G)
    used = np.zeros(len(rg_col), dtype=bool)
    for i in range(A.m):
        for k in range(rl[i]):
            s = gp[i // G] + k * G + i % G
            assert rg_col[s] == A.col_idx[A.row_ptr[i] + k]
            assert rg_val[s] == A.vals[A.row_ptr[i] + k]
            used[s] = True
    assert used.sum() == A.nnz
    assert np.all(rg_col[~used] == 0) and np.all(rg_val[~used] == 0.0)
    s = oracle.row_stats(A.row_ptr, A.col_idx, A.n)
    if G in (32, 128):
        assert gp[-1] == s["rg_slots"][{32: 0, 128: 2}[G]]


# ---------------------------------------------------------------- long rows


def test_long_rows_worked_example():
    """Lengths 0, 5, 40, 4096, 4097, 12000, 31, 32 with the bin starting at 32
    and segments of 4096: rows 2, 3, 4, 5, 7 are long, with 1, 1, 2, 3, 1
    segments (counted by hand)."""
    lens = np.array([0, 5, 40, 4096, 4097, 12000, 31, 32], dtype=np.int64)
    rp = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    ids, seg_begin = oracle.long_rows(rp, 32, 4096)
    assert ids.tolist() == [2, 3, 4, 5, 7]
    assert seg_begin.tolist() == [0, 1, 2, 4, 7, 8]
    ids, seg_begin = oracle.long_rows(rp, 4097, 1000)
    assert ids.tolist() == [4, 5] and seg_begin.tolist() == [0, 5, 17]
    ids, seg_begin = oracle.long_rows(rp, 20000, 4096)
    assert ids.size == 0 and seg_begin.tolist() == [0]


@pytest.mark.parametrize("seed", range(3))
def test_long_rows_cover_every_long_row_once(seed):
    """Invariants: ascending, exactly the rows reaching the bound, and each
    row's segments hold its nonzeros with the last one non-empty."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(0, 300, size=500)
    lens[rng.integers(0, 500, size=20)] = rng.integers(300, 5000, size=20)
    rp = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    S, L = 97, 150
    ids, seg_begin = oracle.long_rows(rp, L, S)
    assert np.all(np.diff(ids) > 0)
    members = set(ids.tolist())
    for i in range(500):
        assert (i in members) == (lens[i] >= L)
    counts = np.diff(seg_begin)
    assert seg_begin[0] == 0
    for t, i in enumerate(ids):
        assert counts[t] * S >= lens[i] > (counts[t] - 1) * S


# ---------------------------------------------------------------- window-sorted rows


def test_window_sort_worked_example():
    """Lengths 2, 5, 0, 5, 1 | 3, 9, 3 in windows of 5, long rows from 9 on:
    window 1 lists rows 1, 3 (length 5, by index), 0, 4, 2; window 2 lists
    5, 7 (length 3) and then the long row 6 (sorted by hand)."""
    lens = np.array([2, 5, 0, 5, 1, 3, 9, 3])
    rp = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    perm, eff = oracle.window_sort(rp, 5, 9)
    assert perm.tolist() == [1, 3, 0, 4, 2, 5, 7, 6]
    assert eff.tolist() == [5, 5, 2, 1, 0, 3, 3, -1]
    perm, eff = oracle.window_sort(rp, 5, 0)  # no long rows
    assert perm.tolist() == [1, 3, 0, 4, 2, 6, 5, 7]
    perm, _ = oracle.window_sort(rp, 1, 0)  # windows of one row: identity
    assert perm.tolist() == list(range(8))


@pytest.mark.parametrize("window", [1, 32, 96, 1000])
def test_window_sort_invariants(window):
    """A permutation that never leaves its window, lengths non-increasing
    inside a window, ties in index order."""
    A = synth.random_csr(777, 300, max_len=9, empty_frac=0.2, seed=window)
    perm, eff = oracle.window_sort(A.row_ptr, window, 7)
    lens = np.diff(A.row_ptr)
    assert sorted(perm.tolist()) == list(range(A.m))
    for p in range(A.m):
        assert p // window == perm[p] // window
        want = -1 if lens[perm[p]] >= 7 else lens[perm[p]]
        assert eff[p] == want
        if p + 1 < A.m and (p + 1) // window == p // window:
            assert eff[p] > eff[p + 1] or (eff[p] == eff[p + 1] and perm[p] < perm[p + 1])


# ---------------------------------------------------------------- SpMM


@pytest.mark.parametrize("k", [1, 3, 8])
def test_spmm_equals_dense_product_exactly(k):
    """Small integers: every product and sum is exact, so Y must equal the
    dense integer product alpha*A@X + beta*Y_old exactly."""
    rng = np.random.default_rng(k)
    m, n = 37, 23
    A = synth.random_csr(m, n, max_len=9, empty_frac=0.2, dist=synth.DIST_SMALL_INT, seed=k, dtype="f64")
    dense = np.zeros((m, n), dtype=np.int64)
    for i in range(m):
        for q in range(A.row_ptr[i], A.row_ptr[i + 1]):
            dense[i, A.col_idx[q]] = int(A.vals[q])
    X = rng.integers(-3, 4, size=(n, k)).astype(np.float64)
    Y0 = rng.integers(-5, 6, size=(m, k)).astype(np.float64)
    for alpha, beta in [(1, 0), (2, -3), (0, 1), (-1, 0.5)]:
        Y, _ = oracle.spmm(A.row_ptr, A.col_idx, A.vals, X, alpha, beta, Y0)
        want = alpha * (dense @ X.astype(np.int64)) + beta * Y0
        np.testing.assert_array_equal(Y, want)


def test_spmm_identity_right_hand_sides_give_columns():
    """X = I (n columns): column t of Y is column t of A, exactly."""
    A = synth.random_csr(40, 12, max_len=6, empty_frac=0.1, dist=synth.DIST_NORMAL, seed=5, dtype="f64")
    Y, _ = oracle.spmm(A.row_ptr, A.col_idx, A.vals, np.eye(12))
    want = np.zeros((40, 12))
    for i in range(40):
        for q in range(A.row_ptr[i], A.row_ptr[i + 1]):
            want[i, A.col_idx[q]] = A.vals[q]
    np.testing.assert_array_equal(Y, want)


def test_spmm_columns_are_independent():
    """Scaling one column of X scales the same column of Y only (powers of
    two keep it exact)."""
    A = synth.random_csr(50, 30, max_len=8, empty_frac=0.2, dist=synth.DIST_NORMAL, seed=6, dtype="f64")
    X = synth.vector(30 * 4, synth.DIST_NORMAL, 6, synth.STREAM_X, "f64").reshape(30, 4)
    Y, _ = oracle.spmm(A.row_ptr, A.col_idx, A.vals, X)
    X2 = X.copy()
    X2[:, 2] *= 4.0
    Y2, _ = oracle.spmm(A.row_ptr, A.col_idx, A.vals, X2)
    np.testing.assert_array_equal(Y2[:, [0, 1, 3]], Y[:, [0, 1, 3]])
    np.testing.assert_array_equal(Y2[:, 2], 4.0 * Y[:, 2])


# ---------------------------------------------------------------- transpose


def test_transpose_worked_example():
    """A = [[1, 0, 2], [0, 3, 0], [4, 5, 6], [0, 0, 7]] (4 x 3), transposed by
    hand: columns [1, 4], [3, 5], [2, 6, 7] at rows [0, 2], [1, 2], [0, 2, 3]."""
    rp = np.array([0, 2, 3, 6, 7], dtype=np.int32)
    ci = np.array([0, 2, 1, 0, 1, 2, 2], dtype=np.int32)
    v = np.array([1, 2, 3, 4, 5, 6, 7], dtype=np.float64)
    tp, ti, tv, ts = oracle.transpose(rp, ci, v, 3)
    assert tp.tolist() == [0, 2, 4, 7]
    assert ti.tolist() == [0, 2, 1, 2, 0, 2, 3]
    assert tv.tolist() == [1, 4, 3, 5, 2, 6, 7]
    assert ts.tolist() == [0, 3, 2, 4, 1, 5, 6]


@pytest.mark.parametrize("seed", range(3))
def test_transpose_twice_is_identity(seed):
    A = synth.random_csr(300, 200, max_len=12, empty_frac=0.2, dist=synth.DIST_NORMAL, seed=seed, dtype="f64")
    tp, ti, tv, _ = oracle.transpose(A.row_ptr, A.col_idx, A.vals, A.n)
    rp2, ci2, v2, _ = oracle.transpose(tp, ti, tv, A.m)
    np.testing.assert_array_equal(rp2, A.row_ptr)
    np.testing.assert_array_equal(ci2, A.col_idx)  # random_csr sorts each row's columns
    np.testing.assert_array_equal(v2, A.vals)


def test_spmv_transposed_equals_dense_product_exactly():
    A = synth.random_csr(41, 29, max_len=9, empty_frac=0.2, dist=synth.DIST_SMALL_INT, seed=3, dtype="f64")
    dense = np.zeros((41, 29), dtype=np.int64)
    for i in range(41):
        for q in range(A.row_ptr[i], A.row_ptr[i + 1]):
            dense[i, A.col_idx[q]] = int(A.vals[q])
    rng = np.random.default_rng(3)
    x = rng.integers(-4, 5, size=41).astype(np.float64)
    y0 = rng.integers(-4, 5, size=29).astype(np.float64)
    for alpha, beta in [(1, 0), (-2, 3), (0, 1)]:
        y, _ = oracle.spmv_transposed(A.row_ptr, A.col_idx, A.vals, x, 29, alpha, beta, y0)
        np.testing.assert_array_equal(y, alpha * (dense.T @ x.astype(np.int64)) + beta * y0)


# ---------------------------------------------------------------- SpGEMM


def _dense(A, n):
    D = np.zeros((A.m, n), dtype=np.int64)
    for i in range(A.m):
        for q in range(A.row_ptr[i], A.row_ptr[i + 1]):
            D[i, A.col_idx[q]] = int(A.vals[q])
    return D


def test_spgemm_equals_dense_product_exactly():
    """Small integers: values exact; the pattern is the set of (i, j) some
    product reaches (a zero sum stays an entry), columns in order."""
    A = synth.random_csr(23, 17, max_len=6, empty_frac=0.2, dist=synth.DIST_SMALL_INT, seed=1, dtype="f64")
    B = synth.random_csr(17, 29, max_len=7, empty_frac=0.2, dist=synth.DIST_SMALL_INT, seed=2, dtype="f64")
    rp, col, val = oracle.spgemm(A.row_ptr, A.col_idx, A.vals, B.row_ptr, B.col_idx, B.vals, 29)
    DA, DB = _dense(A, 17), _dense(B, 29)
    SA, SB = np.zeros((23, 17), np.int64), np.zeros((17, 29), np.int64)  # stored entries, zeros included
    for i in range(23):
        SA[i, A.col_idx[A.row_ptr[i]:A.row_ptr[i + 1]]] = 1
    for i in range(17):
        SB[i, B.col_idx[B.row_ptr[i]:B.row_ptr[i + 1]]] = 1
    reach = (SA @ SB) > 0
    C = DA @ DB
    for i in range(23):
        cols = col[rp[i]:rp[i + 1]]
        assert cols.tolist() == np.flatnonzero(reach[i]).tolist()
        np.testing.assert_array_equal(val[rp[i]:rp[i + 1]], C[i, cols])


def test_spgemm_with_identity_and_permutation():
    A = synth.random_csr(40, 30, max_len=8, empty_frac=0.1, dist=synth.DIST_NORMAL, seed=4, dtype="f64")
    eye_p = np.arange(31, dtype=np.int32)
    rp, col, val = oracle.spgemm(A.row_ptr, A.col_idx, A.vals, eye_p, np.arange(30, dtype=np.int32),
                                 np.ones(30), 30)
    np.testing.assert_array_equal(rp, A.row_ptr)
    np.testing.assert_array_equal(col, A.col_idx)
    np.testing.assert_array_equal(val, A.vals)
    perm = np.random.default_rng(4).permutation(30).astype(np.int32)  # B maps column q to perm[q]
    rp, col, val = oracle.spgemm(A.row_ptr, A.col_idx, A.vals, eye_p, perm, np.ones(30), 30)
    for i in range(40):
        cols = A.col_idx[A.row_ptr[i]:A.row_ptr[i + 1]]
        order = np.argsort(perm[cols])
        assert col[rp[i]:rp[i + 1]].tolist() == perm[cols][order].tolist()
        np.testing.assert_array_equal(val[rp[i]:rp[i + 1]], A.vals[A.row_ptr[i]:A.row_ptr[i + 1]][order])
