"""Parity of the CUDA path (called through the C ABI) with the CPU oracle on
seeded inputs at sizes the oracle finishes in seconds: several merge-path
tiles plus a ragged tail, every kernel, both value types, alpha/beta
combinations, and the degenerate cases (empty matrix, empty rows, one row,
one column, one row spanning many tiles, NaN in y with beta = 0)."""
import numpy as np
import pytest

import oracle
import synth
from helpers import TAU, assert_close_to_oracle, to_gpu

pytestmark = pytest.mark.gpu

ALPHA_BETA = [(1.0, 0.0), (1.5, 0.5), (0.0, 1.0), (-2.0, 0.0)]


def run(A, x, y0, alpha, beta, kernel="auto", ipt=0, fill_nan=False):
    import torch
    import load_balanced_csr_gb300 as lb
    rp, col, val = to_gpu(A)
    plan = lb.Plan(rp, col, val, A.n, kernel=kernel, items_per_thread=ipt)
    xd = torch.from_numpy(x).cuda()
    if beta != 0.0:
        yd = torch.from_numpy(y0.copy()).cuda()
    else:
        yd = torch.full((A.m,), float("nan") if fill_nan else 7.0, dtype=val.dtype, device="cuda")
    plan(xd, yd, alpha, beta)
    torch.cuda.synchronize()
    info = plan.info()
    assert plan.device_status() == 0
    plan.close()
    return yd.cpu().numpy(), info


def inputs(m, n, max_len, seed, dtype, empty_frac=0.2, dist=synth.DIST_NORMAL):
    A = synth.random_csr(m, n, max_len=max_len, empty_frac=empty_frac, dist=dist, seed=seed, dtype=dtype)
    x = synth.vector(n, dist, seed, synth.STREAM_X, dtype)
    y0 = synth.vector(m, dist, seed, synth.STREAM_Y, dtype)
    return A, x, y0


@pytest.mark.parametrize("dtype", ["f32", "f64"])
@pytest.mark.parametrize("alpha,beta", ALPHA_BETA)
@pytest.mark.parametrize("kernel", ["merge_path", "thread_row", "group_mapped"])
def test_random_matrices(dtype, alpha, beta, kernel):
    for seed, (m, n, L) in enumerate([(5000, 3000, 20), (20011, 20011, 6), (1, 4000, 4000), (9333, 1, 1)]):
        if kernel == "thread_row" and L > 256:
            continue  # sequential per-row sums: the plan uses this kernel for short rows only
        A, x, y0 = inputs(m, n, L, seed, dtype)
        y, info = run(A, x, y0, alpha, beta, kernel=kernel, fill_nan=True)
        assert info["kernel_name"] == kernel
        if kernel == "merge_path" and m > 100:
            assert info["num_tiles"] >= 3
        assert_close_to_oracle(A, x, y, alpha, beta, y0, label=f"{kernel} {dtype} m={m}")


@pytest.mark.parametrize("ipt", [8, 12, 16, 24, 32])
@pytest.mark.parametrize("dtype", ["f32", "f64"])
def test_items_per_thread_variants(ipt, dtype):
    A, x, y0 = inputs(30000, 25000, 15, ipt, dtype)
    y, info = run(A, x, y0, 1.5, 0.5, kernel="merge_path", ipt=ipt)
    assert info["items_per_thread"] == ipt
    assert info["items_per_tile"] == info["threads_per_tile"] * ipt
    assert_close_to_oracle(A, x, y, 1.5, 0.5, y0, label=f"ipt={ipt}")


@pytest.mark.parametrize("dtype", ["f32", "f64"])
def test_long_rows_spanning_many_tiles(dtype):
    """Rows far longer than a tile: the cut-row fix-up sums partials from
    hundreds of tiles (tree order keeps fp32 within tolerance)."""
    lens = np.full(20000, 3, dtype=np.int32)
    lens[7] = 400000
    lens[5000:5004] = 30000
    lens[-1] = 50000
    lens[100:200] = 0
    A = synth.fill_random(lens, 500000, dist=synth.DIST_NORMAL, seed=3, dtype=dtype)
    x = synth.vector(A.n, synth.DIST_NORMAL, 3, synth.STREAM_X, dtype)
    y0 = synth.vector(A.m, synth.DIST_NORMAL, 3, synth.STREAM_Y, dtype)
    for alpha, beta in [(1.0, 0.0), (0.5, -1.5)]:
        y, info = run(A, x, y0, alpha, beta, kernel="merge_path")
        assert info["num_tiles"] > 200
        assert_close_to_oracle(A, x, y, alpha, beta, y0, label="long rows")


@pytest.mark.parametrize("dtype", ["f32", "f64"])
def test_degenerate_shapes(dtype):
    import torch
    import load_balanced_csr_gb300 as lb
    t = torch.float64 if dtype == "f64" else torch.float32
    # m = 0
    rp = torch.zeros(1, dtype=torch.int32, device="cuda")
    plan = lb.Plan(rp, torch.zeros(0, dtype=torch.int32, device="cuda"), torch.zeros(0, dtype=t, device="cuda"), 5)
    plan(torch.zeros(5, dtype=t, device="cuda"), torch.zeros(0, dtype=t, device="cuda"))
    plan.close()
    # nnz = 0 with rows; all empty -> y = beta*y_old
    for kernel in ("merge_path", "thread_row", "group_mapped"):
        A = synth.fill_random(np.zeros(3000, np.int32), 10, seed=1, dtype=dtype)
        x = synth.vector(10, synth.DIST_NORMAL, 1, synth.STREAM_X, dtype)
        y0 = synth.vector(3000, synth.DIST_NORMAL, 1, synth.STREAM_Y, dtype)
        for alpha, beta in [(1.0, 0.0), (2.0, 0.25)]:
            y, _ = run(A, x, y0, alpha, beta, kernel=kernel, fill_nan=True)
            assert_close_to_oracle(A, x, y, alpha, beta, y0, label=f"all empty {kernel}")
    # n = 0 with m > 0 (every row empty)
    A = synth.fill_random(np.zeros(17, np.int32), 0, seed=1, dtype=dtype)
    y, _ = run(A, np.zeros(0, dtype=A.vals.dtype), None, 1.0, 0.0, fill_nan=True)
    assert np.all(y == 0)
    # single row, single column, single nonzero
    A = synth.fill_random(np.ones(1, np.int32), 1, seed=2, dtype=dtype)
    x = synth.vector(1, synth.DIST_NORMAL, 2, synth.STREAM_X, dtype)
    for kernel in ("auto", "merge_path", "thread_row", "group_mapped"):
        y, _ = run(A, x, None, 1.0, 0.0, kernel=kernel)
        assert_close_to_oracle(A, x, y, 1.0, 0.0, None, label=f"1x1 {kernel}")


@pytest.mark.parametrize("pattern", ["leading_trailing_empty", "tile_aligned_rows", "alternating",
                                     "empty_block"])
def test_adversarial_row_patterns(pattern):
    T = 32 * 8  # fp64 default tile
    if pattern == "leading_trailing_empty":
        lens = np.full(30000, 4, np.int32)
        lens[:5000] = 0
        lens[-7000:] = 0
    elif pattern == "tile_aligned_rows":
        lens = np.full(60, T - 1, np.int32)  # each row plus its end fills a tile exactly
    elif pattern == "alternating":
        lens = np.tile(np.array([0, 2 * T + 5, 0, 1], np.int32), 50)
    else:  # a block of empty rows longer than several tiles, between two rows
        lens = np.zeros(20000, np.int32)
        lens[0] = 7
        lens[3] = 2 * T
        lens[19000] = 5
        lens[-1] = 3
    A = synth.fill_random(lens, 100000, dist=synth.DIST_NORMAL, seed=9, dtype="f64")
    x = synth.vector(A.n, synth.DIST_NORMAL, 9, synth.STREAM_X, "f64")
    y0 = synth.vector(A.m, synth.DIST_NORMAL, 9, synth.STREAM_Y, "f64")
    for alpha, beta in [(1.0, 0.0), (-1.0, 2.0)]:
        y, _ = run(A, x, y0, alpha, beta, kernel="merge_path", fill_nan=True)
        assert_close_to_oracle(A, x, y, alpha, beta, y0, label=pattern)


def test_integer_inputs_are_exact():
    """Small-integer values make every sum exact in fp64: the GPU must then
    equal the oracle bit for bit, whatever the summation order."""
    A, x, y0 = inputs(40000, 30000, 40, 12, "f64", dist=synth.DIST_SMALL_INT)
    for kernel in ("merge_path", "thread_row", "group_mapped"):
        y, _ = run(A, x, y0, 2.0, -1.0, kernel=kernel)
        ref, _ = oracle.spmv(A.row_ptr, A.col_idx, A.vals, x, 2.0, -1.0, y0)
        np.testing.assert_array_equal(y, ref)


def test_deterministic_and_reusable_plan():
    import torch
    import load_balanced_csr_gb300 as lb
    A, x, y0 = inputs(50000, 50000, 30, 21, "f32")
    rp, col, val = to_gpu(A)
    xd = torch.from_numpy(x).cuda()
    with lb.Plan(rp, col, val, A.n, kernel="merge_path") as plan:
        outs = []
        for _ in range(3):
            y = torch.empty(A.m, dtype=torch.float32, device="cuda")
            plan(xd, y)
            outs.append(y.cpu().numpy())
        assert all(np.array_equal(outs[0], o) for o in outs[1:])
        # new values, same pattern
        val2 = val * 2
        plan.update_values(val2)
        y = torch.empty(A.m, dtype=torch.float32, device="cuda")
        plan(xd, y)
        np.testing.assert_array_equal(y.cpu().numpy(), outs[0] * 2)


@pytest.mark.parametrize("T_ipt", [8, 16, 32])
def test_partition_bit_exact(T_ipt):
    import load_balanced_csr_gb300 as lb
    for seed, lens in enumerate([
        synth.lengths_uniform(70000, 0, 9, 1),
        np.zeros(5000, np.int32),
        np.array([0] * 100 + [100000] + [1] * 300 + [0] * 50, np.int32),
    ]):
        A = synth.fill_random(lens, 200000, seed=seed, dtype="f32")
        rp, col, val = to_gpu(A)
        with lb.Plan(rp, col, val, A.n, kernel="merge_path", items_per_thread=T_ipt) as plan:
            info = plan.info()
            part = plan.export("partition")
        want = oracle.merge_path_partition(A.row_ptr, info["items_per_tile"], info["num_tiles"])
        np.testing.assert_array_equal(part, want)


def test_row_stats_exact():
    import load_balanced_csr_gb300 as lb
    rng = np.random.default_rng(5)
    lens = (rng.pareto(1.1, size=100000) * 2).astype(np.int64)
    lens[rng.random(100000) < 0.15] = 0
    lens = np.minimum(lens, 90000).astype(np.int32)
    A = synth.fill_random(lens, 100000, seed=5, dtype="f64")
    rp, col, val = to_gpu(A)
    with lb.Plan(rp, col, val, A.n) as plan:
        got = plan.info()["stats"]
    want = oracle.row_stats(A.row_ptr, A.col_idx, A.n)
    assert got == want


@pytest.mark.parametrize("case", ["row_ptr0", "decreasing", "last", "col_high", "col_negative"])
def test_invalid_csr_is_rejected(case):
    import torch
    import load_balanced_csr_gb300 as lb
    rp = np.array([0, 2, 4, 6], np.int32)
    col = np.array([0, 1, 1, 2, 0, 2], np.int32)
    nnz = 6
    if case == "row_ptr0":
        rp = np.array([1, 2, 4, 6], np.int32)
    elif case == "decreasing":
        rp = np.array([0, 4, 2, 6], np.int32)
    elif case == "last":
        rp = np.array([0, 2, 4, 5], np.int32)
    elif case == "col_high":
        col[3] = 3
    else:
        col[0] = -1
    with pytest.raises(lb.SpmvError) as ei:
        lb.Plan(torch.from_numpy(rp).cuda(), torch.from_numpy(col).cuda(),
                torch.ones(nnz, dtype=torch.float32, device="cuda"), 3)
    assert ei.value.status == 2


@pytest.mark.parametrize("dtype", ["f32", "f64"])
@pytest.mark.parametrize("offset_what", ["matrix", "y", "x", "all"])
def test_unaligned_pointers(dtype, offset_what):
    """Arrays that start one element past a 16-byte boundary (slices of a
    larger buffer): bulk copies need 16-byte aligned sources, so such
    matrices (and y when beta != 0) take the plain-load staging path."""
    import torch
    import load_balanced_csr_gb300 as lb

    def shifted(a, shift):
        t = torch.from_numpy(a).cuda()
        if not shift:
            return t
        buf = torch.empty(a.size + 1, dtype=t.dtype, device="cuda")
        buf[1:] = t
        return buf[1:]

    A, x, y0 = inputs(12000, 9000, 24, 11, dtype)
    sm, sy, sx = (offset_what in ("matrix", "all"), offset_what in ("y", "all"), offset_what in ("x", "all"))
    rp, col, val = shifted(A.row_ptr, sm), shifted(A.col_idx, sm), shifted(A.vals, sm)
    assert (rp.data_ptr() % 16 != 0) == sm
    for alpha, beta in [(1.0, 0.0), (1.5, 0.5)]:
        for ipt in [8, 24]:
            plan = lb.Plan(rp, col, val, A.n, kernel="merge_path", items_per_thread=ipt)
            xd = shifted(x, sx)
            yd = shifted(y0.copy(), sy)
            plan(xd, yd, alpha, beta)
            torch.cuda.synchronize()
            assert plan.device_status() == 0
            plan.close()
            assert_close_to_oracle(A, x, yd.cpu().numpy(), alpha, beta, y0,
                                   label=f"{offset_what} {dtype} ipt={ipt} beta={beta}")
