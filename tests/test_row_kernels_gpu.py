"""Parity of the row-mapped kernels with the CPU oracle: the Row-grouped CSR
kernel (its interleaved copy of A compared slot by slot with the oracle's
layout, its products with the oracle's), the long-row kernel with the
long-row list compared with the oracle's bin, and both combined (long rows
split off a Row-grouped or thread-per-row plan), for both value types and
several alpha/beta, group sizes and thresholds."""
import numpy as np
import pytest

import oracle
import synth
from helpers import assert_close_to_oracle, to_gpu

pytestmark = pytest.mark.gpu

SEG = 4096


def make_plan(A, **kw):
    import load_balanced_csr_gb300 as lb
    rp, col, val = to_gpu(A)
    return lb.Plan(rp, col, val, A.n, **kw), (rp, col, val)


def run_plan(plan, A, x, y0, alpha, beta, fill_nan=True):
    import torch
    xd = torch.from_numpy(x).cuda()
    if beta != 0.0:
        yd = torch.from_numpy(y0.copy()).cuda()
    else:
        yd = torch.full((A.m,), float("nan") if fill_nan else 7.0, dtype=xd.dtype, device="cuda")
    plan(xd, yd, alpha, beta)
    torch.cuda.synchronize()
    return yd.cpu().numpy()


def vectors(A, seed):
    x = synth.vector(A.n, synth.DIST_NORMAL, seed, synth.STREAM_X, A.dtype)
    y0 = synth.vector(A.m, synth.DIST_NORMAL, seed, synth.STREAM_Y, A.dtype)
    return x, y0


def without_rows(A, drop):
    """A with the rows in `drop` emptied (their nonzeros removed)."""
    lens = np.diff(A.row_ptr).astype(np.int64)
    keep = np.ones(A.nnz, dtype=bool)
    for i in drop:
        keep[A.row_ptr[i]:A.row_ptr[i + 1]] = False
        lens[i] = 0
    rp = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    return rp, A.col_idx[keep], A.vals[keep]


def skewed(m, n, seed, dtype, heavy):
    """Rows of 0..12 nonzeros plus the given {row: length} heavy rows."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(0, 13, size=m).astype(np.int32)
    lens[rng.random(m) < 0.15] = 0
    for r, L in heavy.items():
        lens[r] = min(L, n)
    return synth.fill_random(lens, n, dist=synth.DIST_NORMAL, seed=seed, dtype=dtype)


@pytest.mark.parametrize("dtype", ["f32", "f64"])
@pytest.mark.parametrize("G", [32, 64, 128, 256])
def test_rgcsr_layout_matches_oracle(dtype, G):
    """The plan's interleaved copy equals the oracle's slot by slot (no long
    rows: every row stays in the Row-grouped copy)."""
    A = synth.random_csr(10007, 3000, max_len=17, empty_frac=0.2, dist=synth.DIST_NORMAL, seed=G, dtype=dtype)
    plan, _ = make_plan(A, kernel="rgcsr", rgcsr_group=G)
    info = plan.info()
    assert info["kernel_name"] == "rgcsr" and info["rgcsr_group"] == G and info["num_long_rows"] == 0
    gp, rl, rg_col, rg_val = oracle.rgcsr_pack(A.row_ptr, A.col_idx, A.vals, G)
    np.testing.assert_array_equal(plan.export("rg_group_ptr"), gp)
    np.testing.assert_array_equal(plan.export("rg_row_len"), rl)
    np.testing.assert_array_equal(plan.export("rg_col"), rg_col)
    np.testing.assert_array_equal(plan.export("rg_val"), rg_val)
    assert info["rgcsr_slots"] == gp[-1] == info["stats"]["rg_slots"][{32: 0, 64: 1, 128: 2, 256: 3}[G]]
    plan.close()


@pytest.mark.parametrize("dtype", ["f32", "f64"])
@pytest.mark.parametrize("alpha,beta", [(1.0, 0.0), (1.5, 0.5), (-2.0, 0.0), (0.0, 1.0)])
def test_rgcsr_products(dtype, alpha, beta):
    for seed, (m, n, L, G) in enumerate([(20011, 20011, 9, 128), (777, 5000, 40, 32), (5000, 1, 1, 64),
                                         (33, 900, 300, 256)]):
        A = synth.random_csr(m, n, max_len=L, empty_frac=0.25, dist=synth.DIST_NORMAL, seed=seed, dtype=dtype)
        x, y0 = vectors(A, seed)
        plan, _ = make_plan(A, kernel="rgcsr", rgcsr_group=G)
        y = run_plan(plan, A, x, y0, alpha, beta)
        assert plan.device_status() == 0
        plan.close()
        assert_close_to_oracle(A, x, y, alpha, beta, y0, label=f"rgcsr {dtype} m={m} G={G}")


@pytest.mark.parametrize("dtype", ["f32", "f64"])
@pytest.mark.parametrize("kernel", ["long_rows", "rgcsr"])
def test_long_rows_split_off(dtype, kernel):
    """Rows at or above the threshold go to the long-row kernel: one segment
    (warp per row), a few segments, and hundreds of segments; the list and
    its segment starts equal the oracle's bin; the rest of the rows are
    computed by the thread-per-row or Row-grouped kernel."""
    heavy = {5: 600, 77: 4096, 78: 4097, 1000: 9000, 4242: 300000, 19998: 12345, 19999: 700}
    A = skewed(20000, 400000, 7, dtype, heavy)
    x, y0 = vectors(A, 7)
    for L in [512, 4097, 32]:
        plan, _ = make_plan(A, kernel=kernel, long_row_min=L)
        info = plan.info()
        ids, seg_begin = oracle.long_rows(A.row_ptr, L, SEG)
        assert info["num_long_rows"] == ids.size and info["long_row_min"] == L
        assert info["long_segment_nnz"] == SEG and info["num_long_segments"] == seg_begin[-1]
        np.testing.assert_array_equal(plan.export("long_rows"), ids)
        np.testing.assert_array_equal(plan.export("long_seg_begin"), seg_begin)
        assert info["launches_per_execute"] == 2
        if kernel == "rgcsr":
            G = info["rgcsr_group"]
            rp2, col2, val2 = without_rows(A, ids)
            gp, rl, rg_col, rg_val = oracle.rgcsr_pack(rp2, col2, val2, G)
            rl = rl.copy()
            rl[ids] = -1
            np.testing.assert_array_equal(plan.export("rg_group_ptr"), gp)
            np.testing.assert_array_equal(plan.export("rg_row_len"), rl)
            np.testing.assert_array_equal(plan.export("rg_col"), rg_col)
            np.testing.assert_array_equal(plan.export("rg_val"), rg_val)
        for alpha, beta in [(1.0, 0.0), (0.5, -1.5)]:
            y = run_plan(plan, A, x, y0, alpha, beta)
            assert_close_to_oracle(A, x, y, alpha, beta, y0, label=f"{kernel} {dtype} L={L}")
        assert plan.device_status() == 0
        plan.close()


@pytest.mark.parametrize("kernel", ["long_rows", "rgcsr"])
def test_row_kernels_deterministic_and_reusable(kernel):
    """Repeated products are bitwise equal (the long-row partials are added
    in a fixed order) and the arrival counters reset between products."""
    import torch
    A = skewed(30000, 500000, 3, "f32", {10: 450000, 20: 20000, 29999: 5000})
    x, y0 = vectors(A, 3)
    plan, _ = make_plan(A, kernel=kernel)
    xd = torch.from_numpy(x).cuda()
    outs = []
    for _ in range(4):
        yd = torch.zeros(A.m, dtype=torch.float32, device="cuda")
        plan(xd, yd, 1.0, 0.0)
        outs.append(yd.cpu().numpy())
    for o in outs[1:]:
        np.testing.assert_array_equal(o.view(np.uint32), outs[0].view(np.uint32))
    assert_close_to_oracle(A, x, outs[0], 1.0, 0.0, y0, label=kernel)
    plan.close()


@pytest.mark.parametrize("dtype", ["f32", "f64"])
def test_rgcsr_update_values_repacks(dtype):
    import torch
    A = skewed(9000, 9000, 5, dtype, {3: 3000})
    x, y0 = vectors(A, 5)
    plan, (rp, col, val) = make_plan(A, kernel="rgcsr", long_row_min=1024)
    assert plan.info()["num_long_rows"] == 1
    new_vals = synth.vector(A.nnz, synth.DIST_UNIFORM_PM1, 99, synth.STREAM_Y, dtype)
    vd = torch.from_numpy(new_vals).cuda()
    plan.update_values(vd)
    torch.cuda.synchronize()
    A2 = synth.CSR(A.m, A.n, A.row_ptr, A.col_idx, new_vals)
    rp2, col2, val2 = without_rows(A2, [3])
    _, _, _, rg_val = oracle.rgcsr_pack(rp2, col2, val2, plan.info()["rgcsr_group"])
    np.testing.assert_array_equal(plan.export("rg_val"), rg_val)
    y = run_plan(plan, A2, x, y0, 1.5, 0.5)
    assert_close_to_oracle(A2, x, y, 1.5, 0.5, y0, label="rgcsr after update_values")
    plan.close()


@pytest.mark.parametrize("kernel", ["rgcsr", "long_rows", "rgcsr_sorted"])
@pytest.mark.parametrize("dtype", ["f32", "f64"])
def test_row_kernels_degenerate_shapes(kernel, dtype):
    import torch
    cases = [
        ("all empty", np.zeros(3000, dtype=np.int32), 50),
        ("one long row", np.array([100000], dtype=np.int32), 200000),
        ("one column", np.ones(5000, dtype=np.int32), 1),
        ("single row short", np.array([7], dtype=np.int32), 10),
        ("no rows", np.zeros(0, dtype=np.int32), 10),
    ]
    for name, lens, n in cases:
        A = synth.fill_random(lens, n, dist=synth.DIST_NORMAL, seed=1, dtype=dtype)
        x, y0 = vectors(A, 1)
        plan, _ = make_plan(A, kernel=kernel)
        if A.m == 0:
            xd = torch.from_numpy(x).cuda()
            plan(xd, torch.empty(0, dtype=xd.dtype, device="cuda"), 1.0, 0.0)
            torch.cuda.synchronize()
            plan.close()
            continue
        for alpha, beta in [(1.0, 0.0), (2.0, 0.5)]:
            y = run_plan(plan, A, x, y0, alpha, beta)
            assert_close_to_oracle(A, x, y, alpha, beta, y0, label=f"{kernel} {dtype} {name}")
        assert plan.device_status() == 0
        plan.close()


def test_options_are_validated():
    import load_balanced_csr_gb300 as lb
    A = synth.random_csr(100, 100, max_len=5, seed=0, dtype="f32")
    for kw in [dict(kernel="rgcsr", rgcsr_group=48), dict(kernel="long_rows", long_row_min=16),
               dict(kernel="rgcsr", long_row_min=-1)]:
        with pytest.raises(lb.SpmvError):
            make_plan(A, **kw)


WINDOW = 1024


def permuted_without(A, perm, drop):
    """A's rows in the order perm, the rows in `drop` emptied."""
    lens = np.diff(A.row_ptr).astype(np.int64)
    dropped = np.zeros(A.m, dtype=bool)
    dropped[np.asarray(drop, dtype=np.int64)] = True
    cols, vals, new_lens = [], [], []
    for r in perm:
        if dropped[r]:
            new_lens.append(0)
            continue
        b, e = A.row_ptr[r], A.row_ptr[r + 1]
        cols.append(A.col_idx[b:e])
        vals.append(A.vals[b:e])
        new_lens.append(e - b)
    rp = np.concatenate([[0], np.cumsum(new_lens)]).astype(np.int32)
    col = np.concatenate(cols) if cols else np.zeros(0, np.int32)
    val = np.concatenate(vals) if vals else np.zeros(0, A.vals.dtype)
    return rp, col.astype(np.int32), val.astype(A.vals.dtype)


@pytest.mark.parametrize("dtype", ["f32", "f64"])
@pytest.mark.parametrize("L", [0, 512])
def test_rgcsr_sorted_layout_matches_oracle(dtype, L):
    """Row order equal to the oracle's window sort; the interleaved copy of
    the rows in that order (long rows emptied) equal to the oracle's copy."""
    heavy = {5: 600, 2047: 3000, 3000: 700} if L else {}
    A = skewed(3333, 5000, 21, dtype, heavy)
    plan, _ = make_plan(A, kernel="rgcsr_sorted", long_row_min=L or 1 << 30)
    info = plan.info()
    assert info["kernel_name"] == "rgcsr_sorted" and info["rgcsr_group"] == 32
    long_min = L if L else 0
    perm, eff = oracle.window_sort(A.row_ptr, WINDOW, long_min)
    np.testing.assert_array_equal(plan.export("rg_perm"), perm)
    np.testing.assert_array_equal(plan.export("rg_row_len"), eff)
    ids, _ = oracle.long_rows(A.row_ptr, L, SEG) if L else (np.zeros(0, np.int32), None)
    rp2, col2, val2 = permuted_without(A, perm, ids)
    gp, rl, rg_col, rg_val = oracle.rgcsr_pack(rp2, col2, val2, 32)
    np.testing.assert_array_equal(plan.export("rg_group_ptr"), gp)
    np.testing.assert_array_equal(plan.export("rg_col"), rg_col)
    np.testing.assert_array_equal(plan.export("rg_val"), rg_val)
    assert info["num_long_rows"] == len(ids)
    plan.close()


@pytest.mark.parametrize("dtype", ["f32", "f64"])
@pytest.mark.parametrize("alpha,beta", [(1.0, 0.0), (1.5, 0.5), (-2.0, 0.0), (0.0, 1.0)])
def test_rgcsr_sorted_products(dtype, alpha, beta):
    cases = [synth.random_csr(20011, 20011, max_len=9, empty_frac=0.25, dist=synth.DIST_NORMAL, seed=1, dtype=dtype),
             synth.random_csr(1000, 3000, max_len=40, empty_frac=0.1, dist=synth.DIST_NORMAL, seed=2, dtype=dtype),
             skewed(9000, 300000, 3, dtype, {4: 250000, 8999: 5000, 1024: 600}),
             synth.random_csr(31, 100, max_len=5, empty_frac=0.3, dist=synth.DIST_NORMAL, seed=4, dtype=dtype)]
    for k, A in enumerate(cases):
        x, y0 = vectors(A, k)
        plan, _ = make_plan(A, kernel="rgcsr_sorted")
        y = run_plan(plan, A, x, y0, alpha, beta)
        assert plan.device_status() == 0
        plan.close()
        assert_close_to_oracle(A, x, y, alpha, beta, y0, label=f"rgcsr_sorted {dtype} case {k}")


def test_rgcsr_sorted_update_values_and_determinism():
    import torch
    A = skewed(12000, 200000, 9, "f64", {77: 150000})
    x, y0 = vectors(A, 9)
    plan, _ = make_plan(A, kernel="rgcsr_sorted")
    new_vals = synth.vector(A.nnz, synth.DIST_UNIFORM_PM1, 5, synth.STREAM_Y, "f64")
    plan.update_values(torch.from_numpy(new_vals).cuda())
    A2 = synth.CSR(A.m, A.n, A.row_ptr, A.col_idx, new_vals)
    outs = [run_plan(plan, A2, x, y0, 1.5, 0.5) for _ in range(3)]
    for o in outs[1:]:
        np.testing.assert_array_equal(o.view(np.uint64), outs[0].view(np.uint64))
    assert_close_to_oracle(A2, x, outs[0], 1.5, 0.5, y0, label="rgcsr_sorted after update_values")
    plan.close()
