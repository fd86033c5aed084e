"""Shared test helpers: move seeded CSR inputs to the GPU and compare the
CUDA path with the oracle under the accuracy bound

    |y_i - y_ref_i| <= tau * (|alpha| sum_j |a_ij x_j| + |beta y_old_i|) + 1e-30,

tau = 1e-5 for fp32 and 1e-13 for fp64."""
import numpy as np

import oracle

TAU = {"f32": 1e-5, "f64": 1e-13}


def to_gpu(A):
    import torch
    return (torch.from_numpy(A.row_ptr).cuda(), torch.from_numpy(A.col_idx).cuda(),
            torch.from_numpy(A.vals).cuda())


def assert_close_to_oracle(A, x, y_gpu, alpha, beta, y_old, rows=None, label=""):
    """y_gpu: numpy result (all rows, or the rows listed)."""
    ref, mag = oracle.spmv(A.row_ptr, A.col_idx, A.vals, x, alpha, beta, y_old, rows=rows)
    got = y_gpu if rows is None else y_gpu[rows]
    err = np.abs(got.astype(np.float64) - ref.astype(np.float64))
    bound = TAU[A.dtype] * mag + 1e-30
    bad = ~(err <= bound)
    if bad.any():
        idx = np.flatnonzero(bad)[:5]
        rr = idx if rows is None else np.asarray(rows)[idx]
        raise AssertionError(f"{label}: {bad.sum()} rows out of tolerance, e.g. rows {rr.tolist()}: "
                             f"got {got[idx].tolist()} want {ref[idx].tolist()} bound {bound[idx].tolist()}")
    # empty rows: exactly beta*y_old in the value type (0 when beta == 0)
    lens = np.diff(A.row_ptr)
    sel = np.arange(A.m) if rows is None else np.asarray(rows)
    empty = lens[sel] == 0
    if empty.any():
        t = np.float64 if A.dtype == "f64" else np.float32
        want = (t(beta) * y_old[sel][empty]).astype(t) if beta != 0 else np.zeros(empty.sum(), t)
        np.testing.assert_array_equal(got[empty], want, err_msg=f"{label}: empty rows")
        # and the sign of a zero (alpha * +0 is -0 for alpha < 0), as the oracle has it
        np.testing.assert_array_equal(np.signbit(got[empty]), np.signbit(ref[empty]),
                                      err_msg=f"{label}: sign of empty rows")


def _blocks(m, parts):
    edges = np.linspace(0, m, parts + 1).astype(np.int64)
    return [np.arange(edges[i], edges[i + 1], dtype=np.int32) for i in range(parts) if edges[i + 1] > edges[i]]


def oracle_spmv_all(A, x, alpha, beta, y_old):
    """The oracle's (y, mag) for every row, computed on blocks of rows in
    threads (the oracle is plain C called through ctypes, which releases the
    interpreter lock; its arithmetic is unchanged)."""
    import concurrent.futures as cf
    import os
    if A.m == 0:
        return oracle.spmv(A.row_ptr, A.col_idx, A.vals, x, alpha, beta, y_old)
    blocks = _blocks(A.m, min(64, max(1, A.m // 1024)))
    with cf.ThreadPoolExecutor(max_workers=os.cpu_count() or 4) as ex:
        parts = list(ex.map(lambda r: oracle.spmv(A.row_ptr, A.col_idx, A.vals, x, alpha, beta, y_old, rows=r),
                            blocks))
    return np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts])


def assert_all_rows_close(A, x, y_gpu, alpha, beta, y_old, ref=None, label=""):
    """Every row of y_gpu against the oracle (ref = (y, mag) if already
    computed), with the exact checks of assert_close_to_oracle on empty rows."""
    y_ref, mag = ref if ref is not None else oracle_spmv_all(A, x, alpha, beta, y_old)
    err = np.abs(y_gpu.astype(np.float64) - y_ref.astype(np.float64))
    bound = TAU[A.dtype] * mag + 1e-30
    bad = ~(err <= bound)
    if bad.any():
        idx = np.flatnonzero(bad)[:5]
        raise AssertionError(f"{label}: {bad.sum()} of {A.m} rows out of tolerance, e.g. rows {idx.tolist()}: "
                             f"got {y_gpu[idx].tolist()} want {y_ref[idx].tolist()} bound {bound[idx].tolist()}")
    empty = np.diff(A.row_ptr) == 0
    if empty.any():
        t = np.float64 if A.dtype == "f64" else np.float32
        want = (t(beta) * y_old[empty]).astype(t) if beta != 0 else np.zeros(empty.sum(), t)
        np.testing.assert_array_equal(y_gpu[empty], want, err_msg=f"{label}: empty rows")
        np.testing.assert_array_equal(np.signbit(y_gpu[empty]), np.signbit(y_ref[empty]),
                                      err_msg=f"{label}: sign of empty rows")
