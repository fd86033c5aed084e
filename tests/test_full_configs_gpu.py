"""The five workloads at full size, with the plan the benchmark times
(kernel chosen automatically) and with merge path: every row against the
oracle (computed once per workload, on blocks of rows in threads), with the
exact checks on empty rows; y starts as NaN when beta = 0, so a row that is
never written fails."""
import functools

import numpy as np
import pytest

import synth
from helpers import assert_all_rows_close, oracle_spmv_all, to_gpu

pytestmark = pytest.mark.gpu


@functools.lru_cache(maxsize=1)
def workload_and_reference(name):
    W = synth.workload(name)
    return W, oracle_spmv_all(W.A, W.x, W.alpha, W.beta, W.y0)


@pytest.mark.parametrize("kernel", ["auto", "merge_path"])
@pytest.mark.parametrize("name", synth.WORKLOADS)
def test_full_size_workload(name, kernel):
    import torch
    import load_balanced_csr_gb300 as lb
    W, ref = workload_and_reference(name)
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
        assert plan.device_status() == 0
    y = yd.cpu().numpy()
    assert np.all(np.isfinite(y)), "a row was not written"
    assert_all_rows_close(A, W.x, y, W.alpha, W.beta, W.y0, ref=ref, label=f"{name} {info['kernel_name']}")
