"""The five workloads at full size, with the plan the benchmark times
(kernel chosen automatically) and with merge path.  The oracle checks sampled rows one by one:
random rows, the first and last rows, the longest rows, the rows cut by
merge-path tile boundaries and empty rows.  Two properties check every row:
no row is skipped (y starts as NaN when beta = 0) and
1^T y = alpha (A^T 1)^T x + beta 1^T y_old within the summed tolerance."""
import numpy as np
import pytest

import synth
from helpers import TAU, assert_close_to_oracle, to_gpu

pytestmark = pytest.mark.gpu


def sample_rows(A, plan_info, part, seed=0):
    rng = np.random.default_rng(seed)
    m = A.m
    lens = np.diff(A.row_ptr)
    pick = [rng.integers(0, m, size=min(m, 20000)), np.arange(min(m, 1000)), np.arange(max(0, m - 1000), m)]
    pick.append(np.argsort(lens)[-min(m, 200):])  # longest rows
    if part is not None:
        pick.append(part[:, 0][part[:, 0] < m])  # rows open at a tile start
        pick.append(np.maximum(part[:, 0] - 1, 0))
    empty = np.flatnonzero(lens == 0)
    if len(empty):
        pick.append(empty[rng.integers(0, len(empty), size=min(len(empty), 5000))])
    return np.unique(np.concatenate(pick)).astype(np.int32)


@pytest.mark.parametrize("kernel", ["auto", "merge_path"])
@pytest.mark.parametrize("name", synth.WORKLOADS)
def test_full_size_workload(name, kernel):
    import torch
    import load_balanced_csr_gb300 as lb
    W = synth.workload(name)
    A = W.A
    rp, col, val = to_gpu(A)
    xd = torch.from_numpy(W.x).cuda()
    if W.beta != 0.0:
        yd = torch.from_numpy(W.y0.copy()).cuda()
    else:
        yd = torch.full((A.m,), float("nan"), dtype=val.dtype, device="cuda")
    with lb.Plan(rp, col, val, A.n, kernel=kernel) as plan:
        info = plan.info()
        if kernel == "auto" and info["kernel_name"] == "merge_path":
            pytest.skip("the plan chose merge path: covered by the merge_path case")
        plan(xd, yd, W.alpha, W.beta)
        torch.cuda.synchronize()
        part = plan.export("partition") if info["kernel_name"] == "merge_path" else None
    y = yd.cpu().numpy()
    assert np.all(np.isfinite(y)), "a row was not written"
    rows = sample_rows(A, info, part)
    assert_close_to_oracle(A, W.x, y, W.alpha, W.beta, W.y0, rows=rows, label=name)
    # every row at once: 1^T y against the column sums of A
    x64 = W.x.astype(np.float64)
    prod = A.vals.astype(np.float64) * x64[A.col_idx]
    colsum = np.bincount(A.col_idx, weights=A.vals.astype(np.float64), minlength=A.n)
    want = W.alpha * np.dot(colsum, x64)
    bound = abs(W.alpha) * np.abs(prod).sum()
    if W.beta != 0.0:
        want += W.beta * W.y0.astype(np.float64).sum()
        bound += np.abs(W.beta * W.y0.astype(np.float64)).sum()
    got = y.astype(np.float64).sum()
    assert abs(got - want) <= TAU[A.dtype] * bound + 1e-9 * bound
