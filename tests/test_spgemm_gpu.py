"""SpGEMM C = A*B on the GPU against the CPU oracle: the pattern of C
(row pointers and the columns of every row, in increasing order) bit for
bit, and every value within the bound of a sum of products taken in any
order,

    |c_ij - c_ref_ij| <= (n_ij + 2) * u * sum_p |a_ip b_pj|,

n_ij the number of products that land on the entry (the oracle's product of
the two patterns with all values 1), u the unit roundoff of the value type
(one rounding per product and per addition, plus the rounding of the
oracle's long double result).  Rows cover every bin of the row binning
(products <= 16, <= 128, <= 512, <= 1024,
<= 2048, <= 4096, more), empty rows and columns, both value
types, degenerate shapes, invalid input, repeated numeric phases, and A*A of
the full-size workloads on sampled rows."""
import numpy as np
import pytest

import oracle
import synth
from helpers import to_gpu

pytestmark = pytest.mark.gpu

U = {"f32": 2.0 ** -24, "f64": 2.0 ** -53}


def _dtype_name(vals):
    return "f64" if vals.dtype == np.float64 else "f32"


def reference(A, B, rows=None):
    """(row_ptr, col, val, count, mag) of rows `rows` of A*B by the oracle."""
    if rows is not None:
        A = submatrix_rows(A, rows)
    rp, col, val = oracle.spgemm(A.row_ptr, A.col_idx, A.vals, B.row_ptr, B.col_idx, B.vals, B.n)
    ones = lambda v: np.ones(len(v), dtype=np.float64)
    _, _, cnt = oracle.spgemm(A.row_ptr, A.col_idx, ones(A.vals), B.row_ptr, B.col_idx, ones(B.vals), B.n,
                              c_row_ptr=rp)
    _, _, mag = oracle.spgemm(A.row_ptr, A.col_idx, np.abs(A.vals).astype(np.float64), B.row_ptr, B.col_idx,
                              np.abs(B.vals).astype(np.float64), B.n, c_row_ptr=rp)
    return rp, col, val, cnt, mag


def submatrix_rows(A, rows):
    rows = np.asarray(rows)
    lens = (A.row_ptr[rows + 1] - A.row_ptr[rows]).astype(np.int64)
    rp = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    idx = np.concatenate([np.arange(A.row_ptr[r], A.row_ptr[r + 1]) for r in rows]) if lens.sum() else \
        np.zeros(0, np.int64)
    return synth.CSR(len(rows), A.n, rp, A.col_idx[idx].astype(np.int32), A.vals[idx])


def check_values(got, ref, cnt, mag, dt, label):
    err = np.abs(got.astype(np.float64) - ref.astype(np.float64))
    bound = (cnt + 2.0) * U[dt] * mag * 1.0001 + 1e-300
    bad = ~(err <= bound)
    if bad.any():
        i = np.flatnonzero(bad)[0]
        raise AssertionError(f"{label}: {bad.sum()} values out of bound, e.g. #{i}: got {got[i]} want {ref[i]} "
                             f"bound {bound[i]} ({cnt[i]:.0f} products)")


def run_gpu(A, B):
    import torch
    import load_balanced_csr_gb300 as lb
    arp, acol, aval = to_gpu(A)
    brp, bcol, bval = to_gpu(B)
    with lb.SpGEMM(arp, acol, brp, bcol, B.n, aval.dtype) as h:
        rp, col, val = h.compute(aval, bval)
        torch.cuda.synchronize()
        assert h.device_status() == 0
        info = h.info()
    return rp.cpu().numpy(), col.cpu().numpy(), val.cpu().numpy(), info


def check_all(A, B, label):
    rp, col, val, info = run_gpu(A, B)
    r_rp, r_col, r_val, cnt, mag = reference(A, B)
    np.testing.assert_array_equal(rp.astype(np.int64), r_rp, err_msg=f"{label}: row pointers")
    np.testing.assert_array_equal(col, r_col, err_msg=f"{label}: columns")
    check_values(val, r_val, cnt, mag, _dtype_name(A.vals), label)
    assert info["c_nnz"] == len(r_col)
    return info


def mixed_pair(dtype, seed):
    """A (3000 x 2500) and B (2500 x 4000) whose rows of C fall into all
    seven bins: B has a few long rows (1500 entries), some of 200 and many
    short ones, A rows of 0..12 entries plus rows that pick the longer rows
    of B."""
    rng = np.random.default_rng(seed)
    k, n = 2500, 4000
    b_lens = rng.integers(0, 12, size=k).astype(np.int32)
    long_b = rng.choice(k, 40, replace=False)
    b_lens[long_b] = 1500
    mid_b = rng.choice(np.setdiff1d(np.arange(k), long_b), 40, replace=False)
    b_lens[mid_b] = 200
    b_lens[rng.choice(np.setdiff1d(np.arange(k), np.concatenate([long_b, mid_b])), 200, replace=False)] = 0
    B = synth.fill_random(b_lens, n, dist=synth.DIST_NORMAL, seed=seed + 1, dtype=dtype)
    m = 3000
    a_lens = rng.integers(0, 13, size=m).astype(np.int32)
    a_lens[rng.random(m) < 0.1] = 0
    A0 = synth.fill_random(a_lens, k, dist=synth.DIST_NORMAL, seed=seed + 2, dtype=dtype)
    # rows 0..59 pick 1, 2 or 5 long rows of B (products <= 2048, <= 4096 and more), rows 60..119
    # one or two rows of 200 (<= 512), rows 120..179 three or four (<= 1024); row 180 picks all 40
    # long rows and 900 others
    rows = []
    for i in range(m):
        c = A0.col_idx[A0.row_ptr[i]:A0.row_ptr[i + 1]]
        v = A0.vals[A0.row_ptr[i]:A0.row_ptr[i + 1]]
        if i < 60:
            extra = rng.choice(long_b, [1, 2, 5][i % 3], replace=False)
            c = np.unique(np.concatenate([c, extra]))
            v = rng.standard_normal(len(c)).astype(A0.vals.dtype)
        elif i < 120:
            c = np.unique(np.concatenate([c, rng.choice(mid_b, 1 + i % 2, replace=False)]))
            v = rng.standard_normal(len(c)).astype(A0.vals.dtype)
        elif i < 180:
            c = np.unique(np.concatenate([c, rng.choice(mid_b, 3 + i % 2, replace=False)]))
            v = rng.standard_normal(len(c)).astype(A0.vals.dtype)
        elif i == 180:
            c = np.unique(np.concatenate([long_b, rng.choice(k, 900, replace=False)]))
            v = rng.standard_normal(len(c)).astype(A0.vals.dtype)
        rows.append((c.astype(np.int32), v))
    lens = np.array([len(c) for c, _ in rows])
    rp = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    A = synth.CSR(m, k, rp, np.concatenate([c for c, _ in rows]).astype(np.int32),
                  np.concatenate([v for _, v in rows]).astype(A0.vals.dtype))
    return A, B


@pytest.mark.parametrize("dtype", ["f32", "f64"])
def test_spgemm_every_bin(dtype):
    A, B = mixed_pair(dtype, 7)
    info = check_all(A, B, f"spgemm bins {dtype}")
    assert all(c > 0 for c in info["bin_rows"]), info["bin_rows"]
    assert sum(info["bin_rows"]) == A.m and sum(info["numeric_bin_rows"]) == A.m
    assert info["numeric_bin_rows"][0] == info["bin_rows"][0]
    assert info["numeric_bin_rows"][6] == info["bin_rows"][6]


@pytest.mark.parametrize("dtype", ["f32", "f64"])
def test_spgemm_square_stencil_identity_permutation(dtype):
    A = synth.stencil27(10, dist=synth.DIST_UNIFORM_PM1, diag=27.0, seed=3, dtype=dtype)
    check_all(A, A, f"stencil A*A {dtype}")
    t = A.vals.dtype
    eye = synth.CSR(A.n, A.n, np.arange(A.n + 1, dtype=np.int32), np.arange(A.n, dtype=np.int32),
                    np.ones(A.n, t))
    rp, col, val, _ = run_gpu(A, eye)
    np.testing.assert_array_equal(rp, A.row_ptr)
    np.testing.assert_array_equal(col, A.col_idx)
    np.testing.assert_array_equal(val, A.vals)  # one product per entry, times 1: exact
    perm = np.random.default_rng(1).permutation(A.n).astype(np.int32)
    P = synth.CSR(A.n, A.n, np.arange(A.n + 1, dtype=np.int32), perm, np.ones(A.n, t))
    rp, col, val, _ = run_gpu(P, A)  # rows of A in permuted order
    want_rp = np.concatenate([[0], np.cumsum(np.diff(A.row_ptr)[perm])])
    np.testing.assert_array_equal(rp, want_rp)
    for i in range(0, A.n, 97):
        r = perm[i]
        np.testing.assert_array_equal(col[rp[i]:rp[i + 1]], A.col_idx[A.row_ptr[r]:A.row_ptr[r + 1]])
        np.testing.assert_array_equal(val[rp[i]:rp[i + 1]], A.vals[A.row_ptr[r]:A.row_ptr[r + 1]])


@pytest.mark.parametrize("dtype", ["f32", "f64"])
def test_spgemm_many_products_few_columns(dtype):
    """Rows whose products pile onto few columns: B's rows all live in
    columns 0..39, so a row of C has at most 40 entries however many
    products it takes (up to about 3000 here).  The numeric phase sizes its
    tables by those entries, not by the products."""
    import torch
    import load_balanced_csr_gb300 as lb
    rng = np.random.default_rng(21)
    k, n = 600, 5000
    b_lens = rng.integers(1, 40, size=k).astype(np.int32)
    B0 = synth.fill_random(b_lens, 40, dist=synth.DIST_NORMAL, seed=22, dtype=dtype)
    B = synth.CSR(k, n, B0.row_ptr, B0.col_idx, B0.vals)
    a_lens = rng.integers(0, 150, size=800).astype(np.int32)
    A = synth.fill_random(a_lens, k, dist=synth.DIST_NORMAL, seed=23, dtype=dtype)
    info = check_all(A, B, f"few columns {dtype}")
    assert sum(info["numeric_bin_rows"]) == A.m
    # rows with more than 128 products but at most 40 entries move to the smallest table
    assert info["numeric_bin_rows"][1] > info["bin_rows"][1]


def test_spgemm_degenerate_shapes():
    z = np.zeros(0, np.int32)
    cases = [
        (synth.CSR(0, 5, np.zeros(1, np.int32), z, np.zeros(0)), synth.random_csr(5, 7, max_len=3, seed=1)),
        (synth.CSR(4, 0, np.zeros(5, np.int32), z, np.zeros(0)), synth.CSR(0, 6, np.zeros(1, np.int32), z,
                                                                           np.zeros(0))),
        (synth.random_csr(50, 40, max_len=6, seed=2), synth.CSR(40, 0, np.zeros(41, np.int32), z, np.zeros(0))),
        (synth.CSR(30, 20, np.zeros(31, np.int32), z, np.zeros(0)), synth.random_csr(20, 25, max_len=6, seed=3)),
        (synth.random_csr(30, 20, max_len=6, seed=4), synth.CSR(20, 25, np.zeros(21, np.int32), z, np.zeros(0))),
        (synth.random_csr(1, 300, max_len=300, seed=5), synth.random_csr(300, 1, max_len=1, seed=6)),
    ]
    for j, (A, B) in enumerate(cases):
        A = synth.CSR(A.m, A.n, A.row_ptr, A.col_idx, A.vals.astype(np.float64))
        B = synth.CSR(B.m, B.n, B.row_ptr, B.col_idx, B.vals.astype(np.float64))
        check_all(A, B, f"degenerate case {j}")


def test_spgemm_invalid_input():
    import torch
    import load_balanced_csr_gb300 as lb
    A = synth.random_csr(40, 30, max_len=5, seed=8)
    B = synth.random_csr(30, 20, max_len=5, seed=9)
    arp, acol, _ = to_gpu(A)
    brp, bcol, _ = to_gpu(B)
    bad = bcol.clone()
    bad[3] = 20  # outside [0, n)
    with pytest.raises(lb.SpmvError) as e:
        lb.SpGEMM(arp, acol, brp, bad, 20, torch.float64)
    assert e.value.status == 2 and "(B)" in str(e.value)
    bad = acol.clone()
    bad[0] = -1
    with pytest.raises(lb.SpmvError) as e:
        lb.SpGEMM(arp, bad, brp, bcol, 20, torch.float64)
    assert e.value.status == 2 and "(A)" in str(e.value)
    with pytest.raises(ValueError):
        with lb.SpGEMM(arp, acol, brp, bcol, 20, torch.float64) as h:
            h.compute(torch.zeros(3, dtype=torch.float64, device="cuda"), torch.zeros(B.nnz, dtype=torch.float64,
                                                                                        device="cuda"))


@pytest.mark.parametrize("dtype", ["f32", "f64"])
def test_spgemm_numeric_phase_again(dtype):
    """New values through the same handle, into caller-supplied arrays: the
    same pattern, values within the bound for each set of values."""
    import torch
    import load_balanced_csr_gb300 as lb
    A, B = mixed_pair(dtype, 11)
    arp, acol, aval = to_gpu(A)
    brp, bcol, bval = to_gpu(B)
    r_rp, r_col, r_val, cnt, mag = reference(A, B)
    with lb.SpGEMM(arp, acol, brp, bcol, B.n, aval.dtype) as h:
        out = (torch.empty(A.m + 1, dtype=torch.int32, device="cuda"),
               torch.empty(h.c_nnz, dtype=torch.int32, device="cuda"),
               torch.empty(h.c_nnz, dtype=aval.dtype, device="cuda"))
        h.compute(aval, bval, out=out)
        check_values(out[2].cpu().numpy(), r_val, cnt, mag, dtype, "first values")
        A2 = synth.CSR(A.m, A.n, A.row_ptr, A.col_idx,
                       synth.vector(A.nnz, synth.DIST_UNIFORM_PM1, 5, synth.STREAM_X, dtype))
        B2 = synth.CSR(B.m, B.n, B.row_ptr, B.col_idx,
                       synth.vector(B.nnz, synth.DIST_UNIFORM_PM1, 6, synth.STREAM_Y, dtype))
        h.compute(torch.from_numpy(A2.vals).cuda(), torch.from_numpy(B2.vals).cuda(), out=out)
        torch.cuda.synchronize()
        _, _, r_val2, cnt2, mag2 = reference(A2, B2)
        np.testing.assert_array_equal(out[0].cpu().numpy().astype(np.int64), r_rp)
        np.testing.assert_array_equal(out[1].cpu().numpy(), r_col)
        check_values(out[2].cpu().numpy(), r_val2, cnt2, mag2, dtype, "second values")
        assert h.device_status() == 0


@pytest.mark.parametrize("name", ["stencil27_128", "powerlaw_4M", "skew_8M"])
def test_spgemm_full_size_square(name):
    """C = A*A of a full-size workload, every row of C against the oracle:
    row sizes and columns exactly, values within the summation bound.  The
    oracle runs on blocks of rows in threads (plain C through ctypes, which
    releases the interpreter lock; its arithmetic is unchanged), and each
    block is compared as it comes so that host memory stays bounded."""
    import concurrent.futures as cf
    import os
    import torch
    import load_balanced_csr_gb300 as lb
    A = synth.workload(name).A
    arp, acol, aval = to_gpu(A)
    with lb.SpGEMM(arp, acol, arp, acol, A.n, aval.dtype) as h:
        rp, col, val = h.compute(aval, aval)
        torch.cuda.synchronize()
        assert h.device_status() == 0
        info = h.info()
    assert rp[0].item() == 0 and rp[-1].item() == h.c_nnz
    bl = np.diff(A.row_ptr).astype(np.int64)
    prod = np.add.reduceat(np.concatenate([bl[A.col_idx], [0]]), A.row_ptr[:-1])
    prod = np.where(np.diff(A.row_ptr) > 0, prod, 0)
    assert info["products"] == int(prod.sum())
    rp_h = rp.cpu().numpy().astype(np.int64)
    nb = 2 * (os.cpu_count() or 4)  # few blocks: each oracle call allocates an n-long accumulator
    edges = np.linspace(0, A.m, nb + 1).astype(np.int64)
    blocks = [(int(edges[i]), int(edges[i + 1])) for i in range(nb) if edges[i + 1] > edges[i]]

    def block_reference(b):  # rows [r0, r1) of A as a CSR matrix of their own (views, no copies)
        r0, r1 = b
        lo, hi = int(A.row_ptr[r0]), int(A.row_ptr[r1])
        sub = synth.CSR(r1 - r0, A.n, (A.row_ptr[r0:r1 + 1] - lo).astype(np.int32), A.col_idx[lo:hi],
                        A.vals[lo:hi])
        return reference(sub, A)

    checked = 0
    with cf.ThreadPoolExecutor(max_workers=os.cpu_count() or 4) as ex:
        for (r0, r1), (r_rp, r_col, r_val, cnt, mag) in zip(blocks, ex.map(block_reference, blocks)):
            np.testing.assert_array_equal(np.diff(rp_h[r0:r1 + 1]), np.diff(r_rp), err_msg=f"{name}: row sizes")
            lo, hi = int(rp_h[r0]), int(rp_h[r1])
            np.testing.assert_array_equal(col[lo:hi].cpu().numpy(), r_col, err_msg=f"{name}: columns")
            check_values(val[lo:hi].cpu().numpy(), r_val, cnt, mag, A.dtype, f"{name} A*A rows {r0}..{r1}")
            checked += r1 - r0
    assert checked == A.m
