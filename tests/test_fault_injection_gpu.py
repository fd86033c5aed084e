"""Clean-up paths of plan and SpGEMM-handle creation, walked with host-side
fault injection (no GPU fault is involved): SPMV_FAULT=alloc:N makes the
N-th device allocation of a creation call fail as if the device were out of
memory, SPMV_FAULT=launch:N makes its N-th launch step fail before anything
is launched.  For every N up to the point where creation succeeds, the call
must return the matching status (ALLOC, CUDA), set *out to NULL, and free
everything it had allocated (the device's free memory is back where it was).
The plans cover every layout creation can build: merge path, Row-grouped
(with long rows), window-sorted Row-grouped, long rows + thread per row,
SpMM scratch and the transpose (with its own plan)."""
import ctypes
import os

import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

STATUS_ALLOC, STATUS_CUDA = 3, 4
MIB = 1 << 20


@pytest.fixture
def fault_env():
    yield
    os.environ.pop("SPMV_FAULT", None)


def _matrix():
    lens = synth.lengths_uniform(300000, 0, 12, 11)
    lens[1000] = 70000  # long rows for the long-row layouts
    lens[2000] = 9000
    return synth.fill_random(lens, 250000, dist=synth.DIST_NORMAL, seed=11, dtype="f32")


def _free_bytes():
    import torch
    torch.cuda.synchronize()
    return torch.cuda.mem_get_info()[0]


OPTIONS = [
    dict(kernel="merge_path"),
    dict(kernel="rgcsr"),
    dict(kernel="rgcsr_sorted"),
    dict(kernel="long_rows", long_row_min=64),
    dict(kernel="auto", with_spmm=True),
    dict(kernel="rgcsr", with_spmm=True),
    dict(kernel="auto", with_transpose=True),
]


@pytest.mark.parametrize("kind", ["alloc", "launch"])
@pytest.mark.parametrize("opts", OPTIONS, ids=lambda o: "-".join(f"{k}={v}" for k, v in o.items()))
def test_plan_creation_failures_clean_up(kind, opts, fault_env):
    import torch
    import load_balanced_csr_gb300 as lb
    A = _matrix()
    t = lambda a: torch.from_numpy(a).cuda()
    rp, col, val = t(A.row_ptr), t(A.col_idx), t(A.vals)
    o = lb.Options(lb.KERNELS[opts.get("kernel", "auto")], 0, 0, opts.get("long_row_min", 0),
                   int(opts.get("with_spmm", False)), int(opts.get("with_transpose", False)))
    L = lb.lib()
    stream = torch.cuda.current_stream().cuda_stream
    # one creation without faults first: the first launch of each kernel
    # loads its module, which takes device memory for good (not a leak)
    h = ctypes.c_void_p()
    assert L.spmv_plan_create_ex(ctypes.byref(h), A.m, A.n, A.nnz, rp.data_ptr(), col.data_ptr(), val.data_ptr(),
                                 0, ctypes.byref(o), stream) == 0
    assert L.spmv_plan_destroy(h) == 0
    free0 = _free_bytes()
    failures = 0
    for n in range(1, 200):
        os.environ["SPMV_FAULT"] = f"{kind}:{n}"
        h = ctypes.c_void_p(0xDEAD)
        st = L.spmv_plan_create_ex(ctypes.byref(h), A.m, A.n, A.nnz, rp.data_ptr(), col.data_ptr(), val.data_ptr(),
                                   0, ctypes.byref(o), stream)
        if st == 0:
            assert h.value
            assert L.spmv_plan_destroy(h) == 0
            break
        failures += 1
        assert st == (STATUS_ALLOC if kind == "alloc" else STATUS_CUDA), (n, st)
        assert not h.value, f"{kind}:{n}: *out not NULL on failure"
        assert abs(_free_bytes() - free0) < 2 * MIB, f"{kind}:{n}: device memory not freed"
    else:
        pytest.fail("creation never succeeded")
    assert failures >= 1  # at least one site was reached
    os.environ.pop("SPMV_FAULT")
    assert abs(_free_bytes() - free0) < 2 * MIB


@pytest.mark.parametrize("kind", ["alloc", "launch"])
def test_spgemm_creation_failures_clean_up(kind, fault_env):
    import torch
    import load_balanced_csr_gb300 as lb
    lens = synth.lengths_uniform(20000, 0, 10, 12)
    lens[5] = 6000  # a dense row of C: the dense-bin layout is built too
    A = synth.fill_random(lens, 20000, dist=synth.DIST_NORMAL, seed=12, dtype="f64")
    t = lambda a: torch.from_numpy(a).cuda()
    rp, col = t(A.row_ptr), t(A.col_idx)
    L = lb.lib()
    stream = torch.cuda.current_stream().cuda_stream
    h = ctypes.c_void_p()
    c_nnz = ctypes.c_int64(-1)
    assert L.spmv_spgemm_create(ctypes.byref(h), A.m, A.n, A.n, A.nnz, rp.data_ptr(), col.data_ptr(), A.nnz,
                                rp.data_ptr(), col.data_ptr(), 1, ctypes.byref(c_nnz), stream) == 0
    assert L.spmv_spgemm_destroy(h) == 0
    free0 = _free_bytes()
    failures = 0
    for n in range(1, 200):
        os.environ["SPMV_FAULT"] = f"{kind}:{n}"
        h = ctypes.c_void_p(0xDEAD)
        c_nnz = ctypes.c_int64(-1)
        st = L.spmv_spgemm_create(ctypes.byref(h), A.m, A.n, A.n, A.nnz, rp.data_ptr(), col.data_ptr(), A.nnz,
                                  rp.data_ptr(), col.data_ptr(), 1, ctypes.byref(c_nnz), stream)
        if st == 0:
            assert h.value and c_nnz.value > 0
            assert L.spmv_spgemm_destroy(h) == 0
            break
        failures += 1
        assert st == (STATUS_ALLOC if kind == "alloc" else STATUS_CUDA), (n, st)
        assert not h.value, f"{kind}:{n}: *out not NULL on failure"
        assert abs(_free_bytes() - free0) < 2 * MIB, f"{kind}:{n}: device memory not freed"
    else:
        pytest.fail("creation never succeeded")
    assert failures >= 1
