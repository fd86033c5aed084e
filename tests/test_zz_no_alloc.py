"""spmv_execute_noalloc: the product for callers that cannot allocate device
memory when they need it (a service that gives the whole device to its own
pool at start-up, a loop where cudaMalloc would synchronise the device).  It
keeps its scratch in a fixed array inside the library, so this test checks
two calls in a row -- the second one sees the scratch the first one left --
against the oracle and against the plan-based entry point, within the
tests' accuracy bound; then calls whose arrays are not 16-byte aligned (the
kernel then loads its tiles lane by lane), a matrix with no nonzeros and
beta != 0, and the failure word that spmv_noalloc_device_status reads.
Collected last so that a failure here does not hide any other test."""
import ctypes

import numpy as np
import pytest

import oracle
import synth
from helpers import TAU, assert_close_to_oracle, to_gpu

pytestmark = pytest.mark.gpu


def _noalloc(m, n, nnz, rp, col, val, dtype, alpha, x, beta, y):
    import torch
    import load_balanced_csr_gb300 as lb
    status = lb.lib().spmv_execute_noalloc(
        m, n, nnz, rp.data_ptr(), col.data_ptr() if nnz else None, val.data_ptr() if nnz else None,
        1 if dtype == "f64" else 0, float(alpha), x.data_ptr() if nnz else None, float(beta), y.data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return status


def _device_status():
    import load_balanced_csr_gb300 as lb
    flags = ctypes.c_int32(-1)
    assert lb.lib().spmv_noalloc_device_status(ctypes.byref(flags)) == 0
    return flags.value


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
def test_noalloc_matches_oracle_and_plan_twice(dtype):
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
        rp, col, val = to_gpu(M)
        assert _noalloc(M.m, M.n, M.nnz, rp, col, val, dtype, alpha, xd, beta, yd) == 0
        assert _device_status() == 0
        got = yd.cpu().numpy()
        assert_close_to_oracle(M, x, got, alpha, beta, y0, label=f"noalloc {M.m}x{M.n}")
        want = _with_plan(M, xd, y0, alpha, beta)
        _, mag = oracle.spmv(M.row_ptr, M.col_idx, M.vals, x, alpha, beta, y0)
        err = np.abs(got.astype(np.float64) - want.astype(np.float64))
        assert np.all(err <= 2 * TAU[dtype] * mag + 1e-30)


@pytest.mark.parametrize("dtype", ["f32", "f64"])
def test_noalloc_unaligned_arrays(dtype):
    # every array starts one element past a 16-byte boundary; beta != 0 so
    # that y is read too
    import torch
    M = synth.random_csr(20000, 9000, max_len=30, empty_frac=0.2, dist=synth.DIST_NORMAL, seed=8, dtype=dtype)
    x = synth.vector(M.n, synth.DIST_NORMAL, 8, synth.STREAM_X, dtype)
    y0 = synth.vector(M.m, synth.DIST_NORMAL, 8, synth.STREAM_Y, dtype)

    def shifted(a):
        t = torch.empty(a.size + 1, dtype=torch.from_numpy(a).dtype, device="cuda")
        t[1:] = torch.from_numpy(a).cuda()
        return t[1:]

    rp, col, val, xd, yd = (shifted(a) for a in (M.row_ptr, M.col_idx, M.vals, x, y0))
    assert all(t.data_ptr() % 16 != 0 for t in (rp, col, val, xd, yd))
    assert _noalloc(M.m, M.n, M.nnz, rp, col, val, dtype, 1.5, xd, 0.5, yd) == 0
    assert _device_status() == 0
    assert_close_to_oracle(M, x, yd.cpu().numpy(), 1.5, 0.5, y0, label="noalloc unaligned")


@pytest.mark.parametrize("dtype", ["f32", "f64"])
def test_noalloc_no_nonzeros(dtype):
    import torch
    m = 5000
    M = synth.CSR(m, 7, np.zeros(m + 1, np.int32), np.zeros(0, np.int32),
                  np.zeros(0, np.float64 if dtype == "f64" else np.float32))
    y0 = synth.vector(m, synth.DIST_NORMAL, 9, synth.STREAM_Y, dtype)
    x = synth.vector(7, synth.DIST_NORMAL, 9, synth.STREAM_X, dtype)
    rp = torch.from_numpy(M.row_ptr).cuda()
    yd = torch.from_numpy(y0.copy()).cuda()
    assert _noalloc(m, 7, 0, rp, None, None, dtype, 2.0, torch.from_numpy(x).cuda(), -0.5, yd) == 0
    t = np.float64 if dtype == "f64" else np.float32
    np.testing.assert_array_equal(yd.cpu().numpy(), (t(-0.5) * y0).astype(t))


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import load_balanced_csr_gb300 as lb
    L = lb.lib()
    fake = ctypes.c_void_p(0x1000)
    # m + nnz <= 2^28 is the limit: one more unit is refused (before any
    # pointer is touched)
    assert L.spmv_execute_noalloc((1 << 28) + 1, 1, 0, fake, None, None, 1, 1.0, None, 0.0, fake, None) == 1
    assert L.spmv_execute_noalloc(1 << 27, 1, (1 << 27) + 1, fake, fake, fake, 1, 1.0, fake, 0.0, fake, None) == 1
    assert L.spmv_execute_noalloc(-1, 1, 0, fake, None, None, 0, 1.0, None, 0.0, fake, None) == 1
    assert L.spmv_execute_noalloc(0, 1, 0, None, None, None, 0, 1.0, None, 0.0, None, None) == 0
    assert L.spmv_noalloc_device_status(None) == 1
