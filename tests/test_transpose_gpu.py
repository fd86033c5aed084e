"""The transposed product y = alpha*A^T*x + beta*y: A^T built on the GPU in
CSR form (a stable radix sort by column) compared array by array with the
oracle's transpose -- bit for bit, for column counts needing one, two and
three 8-bit passes -- and the product compared with the oracle's
transposed product, for both value types, several alpha/beta, a value
update, degenerate shapes, and the full-size skewed and power-law
matrices."""
import numpy as np
import pytest

import oracle
import synth
from helpers import TAU, to_gpu

pytestmark = pytest.mark.gpu


def make(A, **kw):
    import load_balanced_csr_gb300 as lb
    rp, col, val = to_gpu(A)
    return lb.Plan(rp, col, val, A.n, with_transpose=True, **kw), (rp, col, val)


def check_layout(plan, A):
    tp, ti, tv, ts = oracle.transpose(A.row_ptr, A.col_idx, A.vals, A.n)
    np.testing.assert_array_equal(plan.export("t_ptr"), tp)
    np.testing.assert_array_equal(plan.export("t_idx"), ti)
    np.testing.assert_array_equal(plan.export("t_src"), ts)
    np.testing.assert_array_equal(plan.export("t_vals"), tv)


def run_t(plan, A, x, y0, alpha, beta):
    import torch
    xd = torch.from_numpy(x).cuda()
    yd = torch.from_numpy(y0.copy()).cuda() if beta != 0 else torch.full((A.n,), float("nan"), dtype=xd.dtype,
                                                                            device="cuda")
    plan.execute_transposed(xd, yd, alpha, beta)
    torch.cuda.synchronize()
    return yd.cpu().numpy()


def check_product(A, x, y0, got, alpha, beta, label, cols=None):
    ref, mag = oracle.spmv_transposed(A.row_ptr, A.col_idx, A.vals, x, A.n, alpha, beta, y0)
    sel = slice(None) if cols is None else cols
    err = np.abs(got[sel].astype(np.float64) - ref[sel].astype(np.float64))
    bad = ~(err <= TAU[A.dtype] * mag[sel] + 1e-30)
    assert not bad.any(), f"{label}: {bad.sum()} entries out of tolerance"


@pytest.mark.parametrize("dtype", ["f32", "f64"])
@pytest.mark.parametrize("m,n", [(3000, 200), (5000, 40000), (2000, 300000)])
def test_transpose_layout_and_product(dtype, m, n):
    """n = 200, 40,000, 300,000: one, two and three radix passes."""
    A = synth.random_csr(m, n, max_len=30, empty_frac=0.2, dist=synth.DIST_NORMAL, seed=n, dtype=dtype)
    x = synth.vector(A.m, synth.DIST_NORMAL, 1, synth.STREAM_X, dtype)
    y0 = synth.vector(A.n, synth.DIST_NORMAL, 1, synth.STREAM_Y, dtype)
    plan, _ = make(A)
    check_layout(plan, A)
    assert plan.info()["transposed_kernel"] > 0
    for alpha, beta in [(1.0, 0.0), (1.5, -0.5), (0.0, 2.0)]:
        got = run_t(plan, A, x, y0, alpha, beta)
        check_product(A, x, y0, got, alpha, beta, f"A^T x {dtype} m={m} n={n}")
    assert plan.device_status() == 0
    plan.close()


@pytest.mark.parametrize("dtype", ["f32", "f64"])
def test_transpose_skewed_columns_and_update(dtype):
    """A dense column (every row holds column 7), long rows (dense rows of
    A^T's short columns), empty rows and empty columns; then new values."""
    import torch
    rng = np.random.default_rng(5)
    m, n = 6000, 9000
    lens = rng.integers(0, 6, size=m).astype(np.int32)
    lens[100] = 8000
    A0 = synth.fill_random(lens, n, dist=synth.DIST_NORMAL, seed=5, dtype=dtype)
    # add column 7 to every row (kept sorted and distinct)
    rows = []
    for i in range(m):
        c = A0.col_idx[A0.row_ptr[i]:A0.row_ptr[i + 1]]
        v = A0.vals[A0.row_ptr[i]:A0.row_ptr[i + 1]]
        if 7 not in c:
            c = np.append(c, 7)
            v = np.append(v, v.dtype.type(0.25))
        o = np.argsort(c, kind="stable")
        rows.append((c[o], v[o]))
    lens = np.array([len(c) for c, _ in rows])
    rp = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    A = synth.CSR(m, n, rp, np.concatenate([c for c, _ in rows]).astype(np.int32),
                  np.concatenate([v for _, v in rows]).astype(A0.vals.dtype))
    x = synth.vector(m, synth.DIST_NORMAL, 2, synth.STREAM_X, dtype)
    y0 = synth.vector(n, synth.DIST_NORMAL, 2, synth.STREAM_Y, dtype)
    plan, _ = make(A)
    check_layout(plan, A)
    got = run_t(plan, A, x, y0, 0.5, 1.0)
    check_product(A, x, y0, got, 0.5, 1.0, f"A^T x skewed {dtype}")
    new_vals = synth.vector(A.nnz, synth.DIST_UNIFORM_PM1, 9, synth.STREAM_X, dtype)
    plan.update_values(torch.from_numpy(new_vals).cuda())
    A2 = synth.CSR(m, n, A.row_ptr, A.col_idx, new_vals)
    check_layout(plan, A2)
    got = run_t(plan, A2, x, y0, 1.0, 0.0)
    check_product(A2, x, y0, got, 1.0, 0.0, f"A^T x after update {dtype}")
    plan.close()


def test_transpose_degenerate_and_checks():
    import torch
    import load_balanced_csr_gb300 as lb
    for lens, n in [(np.zeros(500, np.int32), 300), (np.array([50], np.int32), 60), (np.ones(700, np.int32), 1)]:
        A = synth.fill_random(lens, n, dist=synth.DIST_NORMAL, seed=3, dtype="f64")
        x = synth.vector(A.m, synth.DIST_NORMAL, 3, synth.STREAM_X, "f64")
        y0 = synth.vector(A.n, synth.DIST_NORMAL, 3, synth.STREAM_Y, "f64")
        plan, _ = make(A)
        check_layout(plan, A)
        got = run_t(plan, A, x, y0, 2.0, 0.5)
        check_product(A, x, y0, got, 2.0, 0.5, f"A^T x degenerate n={n}")
        plan.close()
    A = synth.random_csr(100, 100, max_len=5, seed=0, dtype="f32")
    rp, col, val = to_gpu(A)
    with lb.Plan(rp, col, val, A.n) as plan:
        with pytest.raises(lb.SpmvError):
            plan.execute_transposed(torch.zeros(100, device="cuda"), torch.zeros(100, device="cuda"))


@pytest.mark.parametrize("name", ["skew_8M", "powerlaw_4M"])
def test_transpose_full_size(name):
    """Full-size matrices: the whole transpose bit for bit, and the product
    in every column against the oracle."""
    import torch
    W = synth.workload(name)
    A = W.A
    plan, _ = make(A)
    tp, ti, tv, ts = oracle.transpose(A.row_ptr, A.col_idx, A.vals, A.n)
    np.testing.assert_array_equal(plan.export("t_ptr"), tp)
    np.testing.assert_array_equal(plan.export("t_src"), ts)
    x = synth.vector(A.m, synth.DIST_NORMAL, 0, synth.STREAM_X, A.dtype)
    xd = torch.from_numpy(x).cuda()
    yd = torch.full((A.n,), float("nan"), dtype=xd.dtype, device="cuda")
    plan.execute_transposed(xd, yd)
    torch.cuda.synchronize()
    got = yd.cpu().numpy()
    assert np.all(np.isfinite(got))
    check_product(A, x, None, got, 1.0, 0.0, f"A^T x {name}")
    plan.close()
