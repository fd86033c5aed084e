"""The debug build (libspmv_debug.so, -DSPMV_DEBUG): every SpMV kernel
checks the column index of each gather against [0, n).  Plan creation
validates the indices, so the test changes some of them afterwards, on the
device, in the array the plan borrows; the checked kernels then flag bit 2
in the plan's device status and gather x[0] instead, so no read leaves x.
Every kernel that reads the original column indices is run: merge path,
thread per row, group-mapped, and the long-row kernel with thread per row.
The same plans on intact indices match the oracle with a clear status.
Only the debug build ever runs on the changed indices."""
import numpy as np
import pytest

import synth
from helpers import assert_close_to_oracle, to_gpu

pytestmark = pytest.mark.gpu

KERNELS = ["merge_path", "thread_row", "group_mapped", "long_rows"]


def _matrix(dtype):
    rng = np.random.default_rng(44)
    lens = rng.integers(0, 20, size=9000).astype(np.int32)
    lens[[10, 4000]] = [5000, 1200]  # long rows, for the long-row kernel
    return synth.fill_random(lens, 7000, dist=synth.DIST_NORMAL, seed=44, dtype=dtype)


@pytest.mark.parametrize("dtype", ["f32", "f64"])
@pytest.mark.parametrize("kernel", KERNELS)
def test_debug_build_flags_out_of_range_columns(kernel, dtype):
    import torch
    import load_balanced_csr_gb300 as lb
    A = _matrix(dtype)
    x = synth.vector(A.n, synth.DIST_NORMAL, 44, synth.STREAM_X, dtype)
    rp, col, val = to_gpu(A)
    opts = {"long_row_min": 1000} if kernel == "long_rows" else {}
    with lb.Plan(rp, col, val, A.n, kernel=kernel, debug=True, **opts) as plan:
        assert plan.info()["kernel_name"] == kernel
        xd = torch.from_numpy(x).cuda()
        yd = torch.full((A.m,), float("nan"), dtype=xd.dtype, device="cuda")
        plan(xd, yd)
        torch.cuda.synchronize()
        assert plan.device_status() == 0
        assert_close_to_oracle(A, x, yd.cpu().numpy(), 1.0, 0.0, None, label=f"debug build {kernel} {dtype}")
        # indices out of range, in short rows and in the long rows
        bad = [int(A.row_ptr[3]), int(A.row_ptr[10]) + 17, int(A.row_ptr[4000]) + 5, A.nnz - 1]
        col[bad[0]] = A.n + 7
        col[bad[1]] = -3
        col[bad[2]] = 2**31 - 1
        col[bad[3]] = A.n
        torch.cuda.synchronize()
        plan(xd, yd)
        torch.cuda.synchronize()
        assert plan.device_status() & 4, "an out-of-range column was not flagged"
        assert torch.isfinite(yd).all()


def test_debug_flag_is_not_set_by_the_release_build_path():
    """The release build on intact indices leaves bit 2 clear (the bit
    belongs to the debug build only)."""
    import torch
    import load_balanced_csr_gb300 as lb
    A = _matrix("f32")
    x = synth.vector(A.n, synth.DIST_NORMAL, 44, synth.STREAM_X, "f32")
    rp, col, val = to_gpu(A)
    with lb.Plan(rp, col, val, A.n) as plan:
        yd = torch.zeros(A.m, device="cuda")
        plan(torch.from_numpy(x).cuda(), yd)
        torch.cuda.synchronize()
        assert plan.device_status() == 0
