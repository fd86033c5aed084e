"""The C-ABI library loads without a GPU, exports every function the header
declares, and rejects bad arguments before touching the device."""
import ctypes

import load_balanced_csr_gb300 as lb


def test_library_exports_every_header_function():
    L = lb.lib()
    names = lb.header_functions()
    assert {"spmv_plan_create", "spmv_execute", "spmv_plan_destroy"} <= set(names)
    for name in names:
        assert hasattr(L, name), name


def test_debug_library_exports_every_header_function():
    """The debug build (device-side index checks) has the same interface."""
    L = lb.debug_lib()
    for name in lb.header_functions():
        assert hasattr(L, name), name
    assert L.spmv_status_string(0).decode() == lb.STATUS[0]


def test_status_strings():
    L = lb.lib()
    for code, text in lb.STATUS.items():
        assert L.spmv_status_string(code).decode() == text
    assert L.spmv_status_string(99).decode() == "unknown status"


def test_argument_errors_need_no_device():
    L = lb.lib()
    h = ctypes.c_void_p()
    fake = ctypes.c_void_p(0x1000)
    # out == NULL
    assert L.spmv_plan_create(None, 1, 1, 0, fake, None, None, 0, None) == 1
    # negative sizes
    assert L.spmv_plan_create(ctypes.byref(h), -1, 1, 0, fake, None, None, 0, None) == 1
    assert h.value is None
    assert L.spmv_plan_create(ctypes.byref(h), 1, -1, 0, fake, None, None, 0, None) == 1
    # m + nnz must stay below 2^31
    assert L.spmv_plan_create(ctypes.byref(h), 2**30, 1, 2**30, fake, fake, fake, 0, None) == 1
    # null row_ptr; null col/vals with nnz > 0; unknown dtype
    assert L.spmv_plan_create(ctypes.byref(h), 1, 1, 0, None, None, None, 0, None) == 1
    assert L.spmv_plan_create(ctypes.byref(h), 1, 1, 3, fake, None, fake, 0, None) == 1
    assert L.spmv_plan_create(ctypes.byref(h), 1, 1, 0, fake, None, None, 7, None) == 1
    assert b"dtype" in L.spmv_last_error()
    # bad options
    opt = lb.Options(9, 0, 0, 0)
    assert L.spmv_plan_create_ex(ctypes.byref(h), 1, 1, 0, fake, None, None, 0, ctypes.byref(opt), None) == 1
    opt = lb.Options(0, 6, 0, 0)
    assert L.spmv_plan_create_ex(ctypes.byref(h), 1, 1, 0, fake, None, None, 0, ctypes.byref(opt), None) == 1
    # execute / info / export / destroy on a null plan
    assert L.spmv_execute(None, 1.0, fake, 0.0, fake, None) == 1
    assert L.spmv_execute_host(None, 1.0, fake, 0.0, fake, fake, fake, None) == 1
    assert L.spmv_plan_info(None, None) == 1
    assert L.spmv_plan_export(None, 0, None, 0, None) == 1
    assert L.spmv_plan_update_values(None, fake, None) == 1
    assert L.spmv_plan_device_status(None, None) == 1
    assert L.spmv_plan_destroy(None) == 0
