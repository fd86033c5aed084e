"""spmv_execute_noalloc: the product for callers that cannot allocate device
memory when they need it (a service that gives the whole device to its own
pool at start-up, a loop where cudaMalloc would synchronise the device).  It
keeps its scratch in a fixed array inside the library, so this test checks
two calls in a row -- the second one sees the scratch the first one left --
against the plan-based entry point, within the tests' accuracy bound.
Collected last so that a failure here does not hide any other test."""
import ctypes

import numpy as np
import pytest

import oracle
import synth
from helpers import TAU, to_gpu

pytestmark = pytest.mark.gpu


def _noalloc(A, x, y, alpha, beta):
    import torch
    import load_balanced_csr_gb300 as lb
    rp, col, val = to_gpu(A)
    status = lb.lib().spmv_execute_noalloc(
        A.m, A.n, A.nnz, rp.data_ptr(), col.data_ptr() if A.nnz else None, val.data_ptr() if A.nnz else None,
        1 if A.dtype == "f64" else 0, float(alpha), x.data_ptr(), float(beta), y.data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return status


def _with_plan(A, xd, y0, alpha, beta):
    import torch
    import load_balanced_csr_gb300 as lb
    rp, col, val = to_gpu(A)
    y = torch.from_numpy(y0.copy()).cuda()
    with lb.Plan(rp, col, val, A.n, kernel="merge_path") as plan:
        plan(xd, y, alpha, beta)
        torch.cuda.synchronize()
    return y.cpu().numpy()


@pytest.mark.parametrize("dtype", ["f32", "f64"])
def test_noalloc_matches_plan_entry_point_twice(dtype):
    import torch
    lens = synth.lengths_uniform(60000, 0, 20, 4)
    lens[123] = 50000  # a row cut across many tiles
    A = synth.fill_random(lens, 70000, dist=synth.DIST_NORMAL, seed=4, dtype=dtype)
    B = synth.random_csr(30000, 5000, max_len=9, empty_frac=0.3, dist=synth.DIST_NORMAL, seed=5, dtype=dtype)
    for M, alpha, beta in ((A, 1.0, 0.0), (B, -0.75, 1.25)):  # two calls in a row
        x = synth.vector(M.n, synth.DIST_NORMAL, 7, synth.STREAM_X, dtype)
        y0 = synth.vector(M.m, synth.DIST_NORMAL, 7, synth.STREAM_Y, dtype)
        xd = torch.from_numpy(x).cuda()
        yd = torch.from_numpy(y0.copy()).cuda()
        assert _noalloc(M, xd, yd, alpha, beta) == 0
        got = yd.cpu().numpy()
        want = _with_plan(M, xd, y0, alpha, beta)
        _, mag = oracle.spmv(M.row_ptr, M.col_idx, M.vals, x, alpha, beta, y0)
        err = np.abs(got.astype(np.float64) - want.astype(np.float64))
        assert np.all(err <= TAU[dtype] * mag + 1e-30)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import torch
    import load_balanced_csr_gb300 as lb
    L = lb.lib()
    fake = ctypes.c_void_p(0x1000)
    # 262,144 tiles of 1,024 units is the limit: one more unit is refused
    m = 262144 * 1024 + 1
    assert L.spmv_execute_noalloc(m, 1, 0, fake, None, None, 1, 1.0, None, 0.0, fake, None) == 1
    assert L.spmv_execute_noalloc(-1, 1, 0, fake, None, None, 0, 1.0, None, 0.0, fake, None) == 1
    assert L.spmv_execute_noalloc(0, 1, 0, None, None, None, 0, 1.0, None, 0.0, None, None) == 0
