"""Every row structure of the smallest matrices, on every SpMV kernel: all
row-length vectors of m = 1..4 rows holding nnz = 0..6 nonzeros in total
(329 matrices, every place an empty row can sit), each with seeded columns
and values.  Each product is compared with the oracle row by row (and the
empty rows exactly), and the merge-path partition of each with the
oracle's, bit for bit.  A slip at a row boundary, an empty row or the last
row of a tile shows here first."""
import itertools

import numpy as np
import pytest

import oracle
import synth
from helpers import assert_close_to_oracle, to_gpu

pytestmark = pytest.mark.gpu

N_COLS = 6


def compositions(total, parts):
    """All vectors of `parts` non-negative integers summing to `total`."""
    for cuts in itertools.combinations_with_replacement(range(total + 1), parts - 1):
        bounds = (0,) + cuts + (total,)
        yield [bounds[i + 1] - bounds[i] for i in range(parts)]


def small_matrices(dtype):
    rng = np.random.default_rng(7)
    t = np.float64 if dtype == "f64" else np.float32
    for m in range(1, 5):
        for nnz in range(0, 7):
            for lens in compositions(nnz, m):
                rp = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
                col = np.concatenate([np.sort(rng.choice(N_COLS, size=L, replace=False)) for L in lens]
                                     + [np.zeros(0, np.int64)]).astype(np.int32)
                vals = rng.standard_normal(nnz).astype(t)
                yield synth.CSR(m, N_COLS, rp, col, vals)


def test_composition_count():
    assert sum(1 for _ in small_matrices("f64")) == 7 + 28 + 84 + 210


@pytest.mark.parametrize("dtype,kernels", [
    ("f64", ["auto", "merge_path", "thread_row", "rgcsr", "rgcsr_sorted", "group_mapped"]),
    ("f32", ["merge_path", "rgcsr"]),
])
def test_every_small_row_structure(dtype, kernels):
    import torch
    import load_balanced_csr_gb300 as lb
    t = torch.float64 if dtype == "f64" else torch.float32
    x = synth.vector(N_COLS, synth.DIST_NORMAL, 7, synth.STREAM_X, dtype)
    xd = torch.from_numpy(x).cuda()
    count = 0
    for A in small_matrices(dtype):
        y0 = synth.vector(A.m, synth.DIST_NORMAL, count, synth.STREAM_Y, dtype)
        rp, col, val = to_gpu(A)
        for kernel in kernels:
            with lb.Plan(rp, col, val, A.n, kernel=kernel) as plan:
                if kernel == "merge_path":
                    info = plan.info()
                    want = oracle.merge_path_partition(A.row_ptr, info["items_per_tile"], info["num_tiles"])
                    np.testing.assert_array_equal(plan.export("partition"), want)
                for alpha, beta in [(1.0, 0.0), (-1.5, 0.5)]:
                    yd = (torch.from_numpy(y0.copy()).cuda() if beta != 0
                          else torch.full((A.m,), float("nan"), dtype=t, device="cuda"))
                    plan(xd, yd, alpha, beta)
                    torch.cuda.synchronize()
                    assert_close_to_oracle(A, x, yd.cpu().numpy(), alpha, beta, y0 if beta != 0 else None,
                                           label=f"{kernel} {dtype} lens={np.diff(A.row_ptr).tolist()}")
                assert plan.device_status() == 0
        count += 1
    assert count == 329
