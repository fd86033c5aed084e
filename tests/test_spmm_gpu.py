"""SpMM Y = alpha*A*X + beta*Y (row-major X, k right-hand sides) on the
merge-path partition, against the CPU oracle element by element: column
counts around the 32-lane and 128-column slices, padded rows of X and Y,
rows cut between many warps, empty rows, both value types, several
alpha/beta; plus its argument checks and determinism."""
import numpy as np
import pytest

import oracle
import synth
from helpers import TAU, to_gpu

pytestmark = pytest.mark.gpu


def dense_inputs(A, k, seed, ld_pad=0):
    t = np.float64 if A.dtype == "f64" else np.float32
    X = synth.vector(A.n * k, synth.DIST_NORMAL, seed, synth.STREAM_X, A.dtype).reshape(A.n, k)
    Y0 = synth.vector(A.m * k, synth.DIST_NORMAL, seed, synth.STREAM_Y, A.dtype).reshape(A.m, k)
    return X.astype(t), Y0.astype(t)


def on_gpu(M, pad):
    """M on the GPU as a row-major view with `pad` extra columns per row."""
    import torch
    buf = torch.zeros((M.shape[0], M.shape[1] + pad), dtype=torch.float64 if M.dtype == np.float64 else torch.float32,
                      device="cuda")
    buf[:, :M.shape[1]] = torch.from_numpy(M).cuda()
    return buf[:, :M.shape[1]]


def check(A, X, Y0, Yg, alpha, beta, label):
    ref, mag = oracle.spmm(A.row_ptr, A.col_idx, A.vals, X, alpha, beta, Y0)
    got = Yg.cpu().numpy()
    err = np.abs(got.astype(np.float64) - ref.astype(np.float64))
    bad = ~(err <= TAU[A.dtype] * mag + 1e-30)
    if bad.any():
        i, t = np.argwhere(bad)[0]
        raise AssertionError(f"{label}: {bad.sum()} entries out of tolerance, e.g. ({i}, {t}): got {got[i, t]} "
                             f"want {ref[i, t]}")


def run_spmm(A, k, alpha, beta, kernel="merge_path", pad=0, seed=0):
    import torch
    import load_balanced_csr_gb300 as lb
    X, Y0 = dense_inputs(A, k, seed)
    rp, col, val = to_gpu(A)
    with lb.Plan(rp, col, val, A.n, kernel=kernel, with_spmm=True) as plan:
        Xg = on_gpu(X, pad)
        Yg = on_gpu(Y0, pad) if beta != 0 else on_gpu(np.full_like(Y0, np.nan), pad)
        plan.execute_multi(Xg, Yg, alpha, beta)
        torch.cuda.synchronize()
        assert plan.device_status() == 0
    return X, Y0, Yg


@pytest.mark.parametrize("dtype", ["f32", "f64"])
@pytest.mark.parametrize("k", [1, 2, 3, 8, 16, 17, 32, 33, 64, 100, 130])
def test_spmm_random(dtype, k):
    A = synth.random_csr(2500, 1800, max_len=14, empty_frac=0.2, dist=synth.DIST_NORMAL, seed=k, dtype=dtype)
    for alpha, beta in [(1.0, 0.0), (1.5, -0.5)]:
        X, Y0, Yg = run_spmm(A, k, alpha, beta, pad=3 if k % 2 else 0, seed=k)
        check(A, X, Y0, Yg, alpha, beta, f"spmm {dtype} k={k} alpha={alpha}")


@pytest.mark.parametrize("dtype", ["f32", "f64"])
def test_spmm_wide_lanes_and_fallbacks(dtype):
    """16-byte lanes where X's layout allows them and one value per lane
    where it does not: X aligned with k and ldx multiples of the values per
    16 bytes; X starting one value past an aligned address; a row stride
    that is not such a multiple; k with idle lanes in a row's lane group.
    Rows of up to 300 nonzeros, so that the whole-warp walk runs too."""
    import torch
    import load_balanced_csr_gb300 as lb
    rng = np.random.default_rng(21)
    lens = rng.integers(0, 12, size=6000).astype(np.int32)
    lens[rng.choice(6000, 40, replace=False)] = rng.integers(65, 300, size=40)
    A = synth.fill_random(lens, 5000, dist=synth.DIST_NORMAL, seed=21, dtype=dtype)
    t = torch.float64 if dtype == "f64" else torch.float32
    rp, col, val = to_gpu(A)
    with lb.Plan(rp, col, val, A.n, kernel="merge_path", with_spmm=True) as plan:
        for k, offset, ld in [(8, 0, 8), (8, 1, 12), (8, 0, 10), (12, 0, 12), (24, 0, 28), (128, 0, 128)]:
            X, Y0 = dense_inputs(A, k, k + offset)
            flat = torch.zeros(A.n * ld + offset, dtype=t, device="cuda")
            Xg = flat[offset:].view(A.n, ld)[:, :k]
            Xg.copy_(torch.from_numpy(X).cuda())
            assert Xg.stride(0) == ld and (Xg.data_ptr() % 16 != 0) == (offset != 0)
            Yg = torch.from_numpy(Y0).cuda()
            plan.execute_multi(Xg, Yg, 1.25, 0.5)
            torch.cuda.synchronize()
            assert plan.device_status() == 0
            check(A, X, Y0, Yg, 1.25, 0.5, f"spmm {dtype} k={k} offset={offset} ldx={ld}")


@pytest.mark.parametrize("dtype", ["f32", "f64"])
def test_spmm_rare_long_rows(dtype):
    """A few long rows among many short ones (at most one per 4096 rows):
    with k a multiple of the values per 16 bytes, the short rows go to the
    CSR warp kernel and rows of at least 65 nonzeros to the warp-per-segment
    kernel; rows of 64, 65, 4096 and 4097 nonzeros sit on its boundaries,
    and a row of 60,000 spans 15 segments added by the last to arrive."""
    rng = np.random.default_rng(12)
    lens = rng.integers(0, 9, size=70000).astype(np.int32)
    lens[[5, 700, 33000, 45000, 69999]] = [64, 65, 4096, 4097, 60000]
    A = synth.fill_random(lens, 80000, dist=synth.DIST_NORMAL, seed=12, dtype=dtype)
    for k, alpha, beta in [(8, 0.5, 2.0), (16, 1.0, 0.0), (40, -1.5, 0.25), (4, 1.0, 1.0)]:
        X, Y0, Yg = run_spmm(A, k, alpha, beta, kernel="auto", seed=k)
        check(A, X, Y0, Yg, alpha, beta, f"spmm rare long rows {dtype} k={k}")


@pytest.mark.parametrize("dtype", ["f32", "f64"])
def test_spmm_rows_cut_between_many_warps(dtype):
    """Many long rows among few short ones: the merge-path SpMM, rows cut
    between warps' runs (rows of 64, 65, 4096 and 4097 nonzeros too)."""
    lens = np.full(3000, 2, dtype=np.int32)
    lens[10] = 60000       # spans many warps' runs
    lens[1500:1510] = 5000
    lens[-1] = 20000       # open at the end of the last run
    lens[200:260] = 0
    lens[300], lens[301], lens[302], lens[303] = 64, 65, 4096, 4097
    A = synth.fill_random(lens, 70000, dist=synth.DIST_NORMAL, seed=4, dtype=dtype)
    for k, kernel in [(8, "merge_path"), (40, "auto"), (4, "auto"), (64, "auto"), (7, "merge_path"),
                      (33, "auto")]:
        X, Y0, Yg = run_spmm(A, k, 0.5, 2.0, kernel=kernel, seed=4)
        check(A, X, Y0, Yg, 0.5, 2.0, f"spmm cut rows {dtype} k={k}")


@pytest.mark.parametrize("dtype", ["f32", "f64"])
def test_spmm_on_every_plan_kernel(dtype):
    """The SpMM path uses the merge-path partition whatever kernel the plan
    chose for SpMV."""
    A = synth.stencil27(12, dist=synth.DIST_UNIFORM_PM1, diag=27.0, seed=2, dtype=dtype)
    for kernel in ["auto", "rgcsr", "thread_row", "long_rows"]:
        X, Y0, Yg = run_spmm(A, 16, 1.0, 0.0, kernel=kernel, seed=2)
        check(A, X, Y0, Yg, 1.0, 0.0, f"spmm stencil plan={kernel}")


def test_spmm_deterministic_and_checks():
    import torch
    import load_balanced_csr_gb300 as lb
    lens = np.full(4000, 3, dtype=np.int32)
    lens[7] = 50000
    A = synth.fill_random(lens, 60000, dist=synth.DIST_NORMAL, seed=8, dtype="f32")
    X, _ = dense_inputs(A, 20, 8)
    rp, col, val = to_gpu(A)
    with lb.Plan(rp, col, val, A.n, with_spmm=True) as plan:
        Xg = torch.from_numpy(X).cuda()
        outs = []
        for _ in range(3):
            Yg = torch.zeros((A.m, 20), dtype=torch.float32, device="cuda")
            plan.execute_multi(Xg, Yg)
            outs.append(Yg.cpu().numpy())
        for o in outs[1:]:
            np.testing.assert_array_equal(o.view(np.uint32), outs[0].view(np.uint32))
        with pytest.raises(ValueError):
            plan.execute_multi(Xg, torch.zeros((A.m, 19), dtype=torch.float32, device="cuda"))
        # k = 0 is a no-op
        plan.execute_multi(torch.zeros((A.n, 0), dtype=torch.float32, device="cuda"),
                           torch.zeros((A.m, 0), dtype=torch.float32, device="cuda"))
    with lb.Plan(rp, col, val, A.n) as plan:  # no SpMM scratch
        with pytest.raises(lb.SpmvError):
            plan.execute_multi(Xg, torch.zeros((A.m, 20), dtype=torch.float32, device="cuda"))


@pytest.mark.parametrize("dtype", ["f32", "f64"])
@pytest.mark.parametrize("kernel", ["rgcsr", "rgcsr_sorted"])
def test_spmm_over_the_row_grouped_copy(dtype, kernel):
    """Plans holding a Row-grouped copy (groups of 32, no long rows) run SpMM
    one thread per row over it when one slice of columns (32 fp32, 16 fp64)
    covers k: 16-byte X loads when aligned, scalar loads for a padded X;
    wider X goes to the merge-path SpMM."""
    A = synth.random_csr(3000, 2500, max_len=24, empty_frac=0.2, dist=synth.DIST_NORMAL, seed=11, dtype=dtype)
    for k, pad in [(1, 0), (3, 1), (8, 0), (16, 0), (17, 0), (32, 0), (40, 2), (64, 0)]:
        for alpha, beta in [(1.0, 0.0), (-0.5, 1.5)]:
            X, Y0, Yg = run_spmm(A, k, alpha, beta, kernel=kernel, pad=pad, seed=k)
            check(A, X, Y0, Yg, alpha, beta, f"spmm {kernel} {dtype} k={k} pad={pad}")


@pytest.mark.parametrize("dtype", ["f32", "f64"])
@pytest.mark.parametrize("kernel", ["rgcsr", "rgcsr_sorted"])
def test_spmm_row_grouped_with_long_rows(dtype, kernel):
    """Row-grouped plans whose copy leaves a few long rows out (512 nonzeros
    or more, at most one per 4096 rows): those rows by the long-row SpMM kernel (a warp per 4096-nonzero
    segment, slices of 32 columns), the others over the copy.  Rows of 511,
    512, 4096, 4097 and 30,000 nonzeros; k narrow, wide and odd; X padded."""
    rng = np.random.default_rng(31)
    lens = rng.integers(0, 40, size=20000).astype(np.int32)  # rare long rows: at most one per 4096
    lens[[3, 900, 9000, 13100, 19999]] = [511, 512, 4096, 4097, 30000]
    A = synth.fill_random(lens, 40000, dist=synth.DIST_NORMAL, seed=31, dtype=dtype)
    for k, pad, alpha, beta in [(1, 0, 1.0, 0.0), (8, 0, 0.5, 2.0), (32, 0, 1.0, 0.0), (33, 1, -1.0, 0.5),
                                (70, 0, 1.0, 1.0)]:
        X, Y0, Yg = run_spmm(A, k, alpha, beta, kernel=kernel, pad=pad, seed=k)
        check(A, X, Y0, Yg, alpha, beta, f"spmm {kernel} long rows {dtype} k={k}")
