"""spmv_execute_host: the product with x and y in host memory, copied
through the caller's device buffers by the library on the stream.  The
result is compared with the oracle and with spmv_execute on the same
device buffers (bit for bit: the same kernels run), for both value types,
beta zero (y_host never read: it starts as NaN) and not, page-locked and
pageable host buffers, on a side stream, with an empty matrix and the
argument checks."""
import numpy as np
import pytest

import synth
from helpers import assert_close_to_oracle, to_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", ["f32", "f64"])
@pytest.mark.parametrize("pinned", [True, False])
def test_execute_host_matches_device_path(dtype, pinned):
    import torch
    import load_balanced_csr_gb300 as lb
    A = synth.random_csr(20000, 15000, max_len=40, empty_frac=0.1, dist=synth.DIST_NORMAL, seed=31, dtype=dtype)
    x = synth.vector(A.n, synth.DIST_NORMAL, 31, synth.STREAM_X, dtype)
    y0 = synth.vector(A.m, synth.DIST_NORMAL, 31, synth.STREAM_Y, dtype)
    t = torch.float64 if dtype == "f64" else torch.float32
    rp, col, val = to_gpu(A)
    stream = torch.cuda.Stream()
    with lb.Plan(rp, col, val, A.n) as plan:
        x_dev = torch.empty(A.n, dtype=t, device="cuda")
        y_dev = torch.empty(A.m, dtype=t, device="cuda")
        for alpha, beta in [(1.0, 0.0), (-1.5, 0.5)]:
            x_h = torch.from_numpy(x.copy())
            y_h = torch.from_numpy(y0.copy()) if beta != 0 else torch.full((A.m,), float("nan"), dtype=t)
            if pinned:
                x_h, y_h = x_h.pin_memory(), y_h.pin_memory()
            y_dev.fill_(float("nan"))
            torch.cuda.synchronize()
            plan.execute_host(x_h, y_h, x_dev, y_dev, alpha, beta, stream=stream)
            stream.synchronize()
            got = y_h.numpy().copy()
            assert_close_to_oracle(A, x, got, alpha, beta, y0, label=f"execute_host {dtype} pinned={pinned}")
            # the device path on the same inputs gives the same bits
            xd = torch.from_numpy(x).cuda()
            yd = torch.from_numpy(y0.copy()).cuda()
            plan.execute(xd, yd, alpha, beta)
            torch.cuda.synchronize()
            ref = yd.cpu().numpy()
            np.testing.assert_array_equal(got.view(np.uint64 if dtype == "f64" else np.uint32),
                                          ref.view(np.uint64 if dtype == "f64" else np.uint32))
        assert plan.device_status() == 0


def test_execute_host_empty_and_checks():
    import torch
    import load_balanced_csr_gb300 as lb
    A = synth.fill_random(np.zeros(300, np.int32), 200, dist=synth.DIST_NORMAL, seed=2, dtype="f32")
    rp, col, val = to_gpu(A)
    with lb.Plan(rp, col, val, A.n) as plan:
        x_h = torch.ones(A.n).pin_memory()
        y_h = torch.full((A.m,), 3.0).pin_memory()
        x_dev, y_dev = torch.empty(A.n, device="cuda"), torch.empty(A.m, device="cuda")
        plan.execute_host(x_h, y_h, x_dev, y_dev, 1.0, 2.0)
        torch.cuda.synchronize()
        assert np.all(y_h.numpy() == 6.0)  # no nonzeros: y = beta * y
        with pytest.raises(TypeError):
            plan.execute_host(x_dev, y_h, x_dev, y_dev)
        with pytest.raises(ValueError):
            plan.execute_host(x_h[:10], y_h, x_dev, y_dev)
        L = lb.lib()
        assert L.spmv_execute_host(plan._h, 1.0, x_h.data_ptr(), 0.0, None, x_dev.data_ptr(), y_dev.data_ptr(),
                                   None) == 1
