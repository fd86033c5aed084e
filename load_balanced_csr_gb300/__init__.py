"""Load-balanced CSR SpMV for GB300 -- Python binding of ``libspmv.so``.

Argument marshalling only: every step of the product runs in the library's
CUDA kernels (include/spmv.h documents the C ABI).  PyTorch supplies device
memory and streams.  There is no CPU path: if the library cannot be loaded
the import of ``lib()`` raises.

    import torch, load_balanced_csr_gb300 as lb
    plan = lb.Plan(row_ptr, col_idx, vals, n)      # CUDA tensors: int32, int32, f32/f64
    plan(x, y, alpha=1.0, beta=0.0)               # y = alpha*A*x + beta*y on the current stream
"""
from __future__ import annotations

import ctypes
import os

from . import _build

__all__ = ["Plan", "SpGEMM", "spgemm", "SpmvError", "lib", "KERNELS", "EXPORTS", "header_functions",
           "gather_ceiling", "GATHER_PATHS"]

KERNELS = {"auto": 0, "merge_path": 1, "thread_row": 2, "rgcsr": 3, "long_rows": 4, "rgcsr_sorted": 5,
           "group_mapped": 6}
KERNEL_NAMES = {v: k for k, v in KERNELS.items()}
EXPORTS = {"partition": 0, "rg_group_ptr": 1, "rg_row_len": 2, "rg_col": 3, "rg_val": 4, "long_rows": 5,
           "long_seg_begin": 6, "rg_perm": 7, "t_ptr": 8, "t_idx": 9, "t_vals": 10, "t_src": 11}
STATUS = {0: "ok", 1: "invalid argument", 2: "invalid CSR matrix", 3: "allocation failed", 4: "CUDA error",
          5: "unsupported"}


class SpmvError(RuntimeError):
    def __init__(self, status: int, what: str, detail: str):
        super().__init__(f"{what}: {STATUS.get(status, status)} ({detail})")
        self.status = status


class Options(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int32), ("items_per_thread", ctypes.c_int32),
                ("rgcsr_group", ctypes.c_int32), ("long_row_min", ctypes.c_int32), ("with_spmm", ctypes.c_int32),
                ("with_transpose", ctypes.c_int32)]


class RowStats(ctypes.Structure):
    _fields_ = [("hist", ctypes.c_int64 * 32), ("sum_len", ctypes.c_int64), ("rg_slots", ctypes.c_int64 * 4),
                ("min_len", ctypes.c_int32), ("max_len", ctypes.c_int32), ("n_empty", ctypes.c_int32),
                ("flags", ctypes.c_int32), ("bandwidth", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class PlanInfo(ctypes.Structure):
    _fields_ = [("m", ctypes.c_int32), ("n", ctypes.c_int32), ("nnz", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("kernel", ctypes.c_int32), ("threads_per_tile", ctypes.c_int32),
                ("items_per_thread", ctypes.c_int32), ("rgcsr_group", ctypes.c_int32),
                ("items_per_tile", ctypes.c_int64), ("num_tiles", ctypes.c_int64),
                ("num_long_rows", ctypes.c_int32), ("launches_per_execute", ctypes.c_int32),
                ("workspace_bytes", ctypes.c_int64), ("stats", RowStats),
                ("long_row_min", ctypes.c_int32), ("long_segment_nnz", ctypes.c_int32),
                ("num_long_segments", ctypes.c_int64), ("rgcsr_slots", ctypes.c_int64),
                ("transposed_kernel", ctypes.c_int32), ("transposed_launches", ctypes.c_int32),
                ("merge_path_warps", ctypes.c_int64)]


class SpgemmInfo(ctypes.Structure):
    _fields_ = [("m", ctypes.c_int32), ("k", ctypes.c_int32), ("n", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("a_nnz", ctypes.c_int64), ("b_nnz", ctypes.c_int64), ("c_nnz", ctypes.c_int64),
                ("products", ctypes.c_int64), ("bin_rows", ctypes.c_int64 * 8), ("dense_slots", ctypes.c_int32),
                ("launches_per_compute", ctypes.c_int32), ("workspace_bytes", ctypes.c_int64),
                ("dense_pieces", ctypes.c_int64), ("dense_waves", ctypes.c_int64),
                ("numeric_bin_rows", ctypes.c_int64 * 8)]


_lib = None


def header_functions() -> list[str]:
    """Names of the functions include/spmv.h declares."""
    import re
    with open(os.path.join(_build.INCLUDE, "spmv.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"^(?:spmv_status_t|const char \*)\s*(spmv_\w+)\s*\(", text, re.M)))


def lib() -> ctypes.CDLL:
    """Load libspmv.so (building it first if its sources are newer)."""
    global _lib
    if _lib is None:
        _lib = _load(_build.build())
    return _lib


_debug_lib = None


def debug_lib() -> ctypes.CDLL:
    """Load libspmv_debug.so, the build with device-side checks of the column
    indices gathered with (-DSPMV_DEBUG), building it first if needed.  Same
    functions as lib(); an index outside [0, n) sets bit 2 of the plan's
    device status instead of reading outside x."""
    global _debug_lib
    if _debug_lib is None:
        _debug_lib = _load(_build.build(debug=True))
    return _debug_lib


def _load(path: str) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise RuntimeError(f"{os.path.basename(path)} is missing and could not be built")
    L = ctypes.CDLL(path)
    vp, i32, sz, dbl = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t, ctypes.c_double
    sigs = {
        "spmv_plan_create": [ctypes.POINTER(vp), i32, i32, i32, vp, vp, vp, ctypes.c_int, vp],
        "spmv_plan_create_ex": [ctypes.POINTER(vp), i32, i32, i32, vp, vp, vp, ctypes.c_int,
                                ctypes.POINTER(Options), vp],
        "spmv_execute": [vp, dbl, vp, dbl, vp, vp],
        "spmv_execute_host": [vp, dbl, vp, dbl, vp, vp, vp, vp],
        "spmv_plan_update_values": [vp, vp, vp],
        "spmv_plan_destroy": [vp],
        "spmv_plan_info": [vp, ctypes.POINTER(PlanInfo)],
        "spmv_plan_export": [vp, ctypes.c_int, vp, sz, ctypes.POINTER(sz)],
        "spmv_plan_device_status": [vp, ctypes.POINTER(i32)],
        "spmv_execute_noalloc": [i32, i32, i32, vp, vp, vp, ctypes.c_int, dbl, vp, dbl, vp, vp],
        "spmv_noalloc_device_status": [ctypes.POINTER(i32)],
        "spmv_execute_multi": [vp, i32, dbl, vp, ctypes.c_int64, dbl, vp, ctypes.c_int64, vp],
        "spmv_execute_transposed": [vp, dbl, vp, dbl, vp, vp],
        "spmv_spgemm_create": [ctypes.POINTER(vp), i32, i32, i32, i32, vp, vp, i32, vp, vp, ctypes.c_int,
                               ctypes.POINTER(ctypes.c_int64), vp],
        "spmv_spgemm_compute": [vp, vp, vp, vp, vp, vp, vp],
        "spmv_spgemm_info": [vp, ctypes.POINTER(SpgemmInfo)],
        "spmv_spgemm_device_status": [vp, ctypes.POINTER(i32)],
        "spmv_spgemm_destroy": [vp],
        "spmv_gather_ceiling": [i32, i32, vp, i32, vp, vp, ctypes.c_int, vp, vp, vp],
    }
    for name, args in sigs.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    L.spmv_status_string.argtypes = [ctypes.c_int]
    L.spmv_status_string.restype = ctypes.c_char_p
    L.spmv_last_error.argtypes = []
    L.spmv_last_error.restype = ctypes.c_char_p
    return L


def check(status: int, what: str, L: ctypes.CDLL | None = None) -> None:
    if status != 0:
        raise SpmvError(status, what, (L or lib()).spmv_last_error().decode())


def _stream_handle(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return 0
    if t.dtype == torch.float64:
        return 1
    raise TypeError(f"values must be float32 or float64, got {t.dtype}")


def _ptr(t) -> int | None:
    return t.data_ptr() if t is not None and t.numel() > 0 else None


class Plan:
    """A plan for y = alpha*A*x + beta*y with A in CSR (CUDA tensors).

    The plan borrows ``row_ptr``, ``col_idx`` and ``vals`` (kept referenced
    here so they stay alive) and owns a device workspace freed by
    ``close()``."""

    def __init__(self, row_ptr, col_idx, vals, n: int, *, kernel: str = "auto", items_per_thread: int = 0,
                 rgcsr_group: int = 0, long_row_min: int = 0, with_spmm: bool = False, with_transpose: bool = False,
                 stream=None, debug: bool = False):
        import torch
        for name, t, dt in (("row_ptr", row_ptr, torch.int32), ("col_idx", col_idx, torch.int32)):
            if t.dtype != dt or not t.is_cuda or not t.is_contiguous():
                raise TypeError(f"{name} must be a contiguous CUDA int32 tensor")
        if not vals.is_cuda or not vals.is_contiguous():
            raise TypeError("vals must be a contiguous CUDA tensor")
        m = row_ptr.numel() - 1
        nnz = col_idx.numel()
        if vals.numel() != nnz:
            raise ValueError("vals and col_idx differ in length")
        self._keep = (row_ptr, col_idx, vals)
        # debug: run on the build with device-side checks of the column
        # indices (an index outside [0, n) sets bit 2 of device_status())
        self._L = debug_lib() if debug else lib()
        self.m, self.n, self.nnz = m, int(n), nnz
        self.dtype = vals.dtype
        opts = Options(KERNELS[kernel], items_per_thread, rgcsr_group, long_row_min, int(bool(with_spmm)),
                       int(bool(with_transpose)))
        handle = ctypes.c_void_p()
        with torch.cuda.device(row_ptr.device):
            check(self._L.spmv_plan_create_ex(ctypes.byref(handle), m, self.n, nnz, _ptr(row_ptr), _ptr(col_idx),
                                            _ptr(vals), _dtype_code(vals), ctypes.byref(opts),
                                            _stream_handle(stream)), "spmv_plan_create", self._L)
        self._h = handle
        self.device = row_ptr.device

    def __call__(self, x, y, alpha: float = 1.0, beta: float = 0.0, stream=None):
        return self.execute(x, y, alpha, beta, stream)

    def execute(self, x, y, alpha: float = 1.0, beta: float = 0.0, stream=None):
        if self._h is None:
            raise RuntimeError("plan is closed")
        if x.dtype != self.dtype or y.dtype != self.dtype:
            raise TypeError("x and y must have the plan's value type")
        if x.numel() != self.n or y.numel() != self.m or not x.is_contiguous() or not y.is_contiguous():
            raise ValueError("x must have n and y m contiguous entries")
        if not x.is_cuda or not y.is_cuda:
            raise TypeError("x and y must be CUDA tensors")
        check(self._L.spmv_execute(self._h, float(alpha), _ptr(x), float(beta), _ptr(y), _stream_handle(stream)),
              "spmv_execute", self._L)
        return y

    def execute_host(self, x_host, y_host, x_dev, y_dev, alpha: float = 1.0, beta: float = 0.0, stream=None):
        """y_host = alpha*A*x_host + beta*y_host with x_host and y_host CPU
        tensors (pinned for asynchronous copies): the library copies them
        through the device buffers x_dev and y_dev on the stream.  y_host
        holds the result once the stream has been synchronised."""
        if self._h is None:
            raise RuntimeError("plan is closed")
        for t in (x_host, y_host, x_dev, y_dev):
            if t.dtype != self.dtype or not t.is_contiguous():
                raise TypeError("buffers must be contiguous and of the plan's value type")
        if x_host.numel() != self.n or x_dev.numel() != self.n or y_host.numel() != self.m or y_dev.numel() != self.m:
            raise ValueError("x buffers must have n and y buffers m entries")
        if x_host.is_cuda or y_host.is_cuda or not x_dev.is_cuda or not y_dev.is_cuda:
            raise TypeError("x_host and y_host must be CPU tensors, x_dev and y_dev CUDA tensors")
        check(self._L.spmv_execute_host(self._h, float(alpha), _ptr(x_host), float(beta), _ptr(y_host), _ptr(x_dev),
                                      _ptr(y_dev), _stream_handle(stream)), "spmv_execute_host", self._L)
        return y_host

    def execute_multi(self, X, Y, alpha: float = 1.0, beta: float = 0.0, stream=None):
        """Y = alpha*A*X + beta*Y for a row-major X (n-by-k) and Y (m-by-k);
        rows may be padded (a stride larger than k), columns must be
        contiguous.  The plan needs with_spmm=True."""
        if self._h is None:
            raise RuntimeError("plan is closed")
        if X.dtype != self.dtype or Y.dtype != self.dtype:
            raise TypeError("X and Y must have the plan's value type")
        if X.dim() != 2 or Y.dim() != 2 or X.shape[0] != self.n or Y.shape[0] != self.m or X.shape[1] != Y.shape[1]:
            raise ValueError("X must be n-by-k and Y m-by-k")
        if X.stride(1) != 1 or Y.stride(1) != 1:
            raise ValueError("X and Y must be row-major (unit column stride)")
        if not X.is_cuda or not Y.is_cuda:
            raise TypeError("X and Y must be CUDA tensors")
        k = X.shape[1]
        ldx = X.stride(0) if X.shape[0] > 1 else k
        ldy = Y.stride(0) if Y.shape[0] > 1 else k
        check(self._L.spmv_execute_multi(self._h, k, float(alpha), _ptr(X), ldx, float(beta), _ptr(Y), ldy,
                                       _stream_handle(stream)), "spmv_execute_multi", self._L)
        return Y

    def execute_transposed(self, x, y, alpha: float = 1.0, beta: float = 0.0, stream=None):
        """y = alpha*A^T*x + beta*y (x: m entries, y: n); needs with_transpose=True."""
        if self._h is None:
            raise RuntimeError("plan is closed")
        if x.dtype != self.dtype or y.dtype != self.dtype:
            raise TypeError("x and y must have the plan's value type")
        if x.numel() != self.m or y.numel() != self.n or not x.is_contiguous() or not y.is_contiguous():
            raise ValueError("x must have m and y n contiguous entries")
        if not x.is_cuda or not y.is_cuda:
            raise TypeError("x and y must be CUDA tensors")
        check(self._L.spmv_execute_transposed(self._h, float(alpha), _ptr(x), float(beta), _ptr(y),
                                            _stream_handle(stream)), "spmv_execute_transposed", self._L)
        return y

    def update_values(self, vals, stream=None):
        if vals.numel() != self.nnz or vals.dtype != self.dtype or not vals.is_contiguous():
            raise ValueError("vals must match the plan's nnz and value type")
        check(self._L.spmv_plan_update_values(self._h, _ptr(vals), _stream_handle(stream)), "spmv_plan_update_values",
              self._L)
        self._keep = (self._keep[0], self._keep[1], vals)

    def info(self) -> dict:
        inf = PlanInfo()
        check(self._L.spmv_plan_info(self._h, ctypes.byref(inf)), "spmv_plan_info", self._L)
        out = {f: getattr(inf, f) for f, _ in PlanInfo._fields_ if f != "stats"}
        s = inf.stats
        out["stats"] = {"hist": list(s.hist), "sum_len": s.sum_len, "rg_slots": list(s.rg_slots),
                        "min_len": s.min_len, "max_len": s.max_len, "n_empty": s.n_empty, "flags": s.flags,
                        "bandwidth": s.bandwidth}
        out["kernel_name"] = KERNEL_NAMES.get(inf.kernel, str(inf.kernel))
        return out

    def device_status(self) -> int:
        """Kernel-side failure flags (0 = none); waits for the device."""
        flags = ctypes.c_int32(0)
        check(self._L.spmv_plan_device_status(self._h, ctypes.byref(flags)), "spmv_plan_device_status", self._L)
        return flags.value

    def export(self, what: str):
        import numpy as np
        code = EXPORTS[what]
        need = ctypes.c_size_t(0)
        check(self._L.spmv_plan_export(self._h, code, None, 0, ctypes.byref(need)), "spmv_plan_export", self._L)
        dtype = {"partition": np.int32, "rg_group_ptr": np.int64, "rg_row_len": np.int32, "rg_col": np.int32,
                 "long_rows": np.int32, "long_seg_begin": np.int64, "rg_perm": np.int32, "t_ptr": np.int32,
                 "t_idx": np.int32, "t_src": np.int32,
                 "t_vals": np.float64 if str(self.dtype) == "torch.float64" else np.float32,
                 "rg_val": np.float64 if str(self.dtype) == "torch.float64" else np.float32}[what]
        buf = np.empty(need.value // np.dtype(dtype).itemsize, dtype=dtype)
        check(self._L.spmv_plan_export(self._h, code, buf.ctypes.data if buf.size else None, need.value, None),
              "spmv_plan_export", self._L)
        return buf.reshape(-1, 2) if what == "partition" else buf

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            check(self._L.spmv_plan_destroy(self._h), "spmv_plan_destroy", self._L)
        self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
        return False


class SpGEMM:
    """C = A*B for CSR matrices on the GPU (A m-by-k, B k-by-n; CUDA int32
    index tensors).  Creation runs the symbolic phase on the two patterns
    (borrowed: kept referenced here, their contents must not change) and
    fixes ``c_nnz``; ``compute`` runs the numeric phase for given values and
    returns C as (row_ptr, col_idx, vals) CUDA tensors, or fills the ones
    passed in."""

    def __init__(self, a_row_ptr, a_col_idx, b_row_ptr, b_col_idx, n: int, dtype, *, stream=None):
        import torch
        for name, t in (("a_row_ptr", a_row_ptr), ("a_col_idx", a_col_idx), ("b_row_ptr", b_row_ptr),
                        ("b_col_idx", b_col_idx)):
            if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
                raise TypeError(f"{name} must be a contiguous CUDA int32 tensor")
        if dtype not in (torch.float32, torch.float64):
            raise TypeError("dtype must be torch.float32 or torch.float64")
        self.m, self.k, self.n = a_row_ptr.numel() - 1, b_row_ptr.numel() - 1, int(n)
        self.a_nnz, self.b_nnz = a_col_idx.numel(), b_col_idx.numel()
        self.dtype = dtype
        self.device = a_row_ptr.device
        self._keep = (a_row_ptr, a_col_idx, b_row_ptr, b_col_idx)
        handle = ctypes.c_void_p()
        c_nnz = ctypes.c_int64(0)
        with torch.cuda.device(self.device):
            check(lib().spmv_spgemm_create(ctypes.byref(handle), self.m, self.k, self.n, self.a_nnz,
                                           _ptr(a_row_ptr), _ptr(a_col_idx), self.b_nnz, _ptr(b_row_ptr),
                                           _ptr(b_col_idx), 1 if dtype == torch.float64 else 0,
                                           ctypes.byref(c_nnz), _stream_handle(stream)), "spmv_spgemm_create")
        self._h = handle
        self.c_nnz = c_nnz.value

    def compute(self, a_vals, b_vals, out=None, stream=None):
        import torch
        if self._h is None:
            raise RuntimeError("SpGEMM handle is closed")
        if a_vals.numel() != self.a_nnz or b_vals.numel() != self.b_nnz:
            raise ValueError("a_vals and b_vals must match the patterns' nnz")
        for t in (a_vals, b_vals):
            if t.dtype != self.dtype or not t.is_cuda or not t.is_contiguous():
                raise TypeError("values must be contiguous CUDA tensors of the handle's dtype")
        if out is None:
            out = (torch.empty(self.m + 1, dtype=torch.int32, device=self.device),
                   torch.empty(self.c_nnz, dtype=torch.int32, device=self.device),
                   torch.empty(self.c_nnz, dtype=self.dtype, device=self.device))
        rp, col, val = out
        if rp.numel() != self.m + 1 or col.numel() != self.c_nnz or val.numel() != self.c_nnz:
            raise ValueError("output arrays must have m + 1, c_nnz and c_nnz entries")
        if rp.dtype != torch.int32 or col.dtype != torch.int32 or val.dtype != self.dtype:
            raise TypeError("outputs must be int32, int32 and the handle's dtype")
        check(lib().spmv_spgemm_compute(self._h, _ptr(a_vals), _ptr(b_vals), rp.data_ptr(), _ptr(col), _ptr(val),
                                        _stream_handle(stream)), "spmv_spgemm_compute")
        return rp, col, val

    def info(self) -> dict:
        inf = SpgemmInfo()
        check(lib().spmv_spgemm_info(self._h, ctypes.byref(inf)), "spmv_spgemm_info")
        out = {f: getattr(inf, f) for f, _ in SpgemmInfo._fields_}
        out["bin_rows"] = list(inf.bin_rows)[:7]
        out["numeric_bin_rows"] = list(inf.numeric_bin_rows)[:7]
        return out

    def device_status(self) -> int:
        flags = ctypes.c_int32(0)
        check(lib().spmv_spgemm_device_status(self._h, ctypes.byref(flags)), "spmv_spgemm_device_status")
        return flags.value

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            check(lib().spmv_spgemm_destroy(self._h), "spmv_spgemm_destroy")
        self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
        return False


def spgemm(a_row_ptr, a_col_idx, a_vals, b_row_ptr, b_col_idx, b_vals, n: int, stream=None):
    """C = A*B in one call: (row_ptr, col_idx, vals) CUDA tensors."""
    with SpGEMM(a_row_ptr, a_col_idx, b_row_ptr, b_col_idx, n, a_vals.dtype, stream=stream) as h:
        return h.compute(a_vals, b_vals, stream=stream)


GATHER_PATHS = {"stream": 0, "l1": 1, "l2": 2, "bulk16": 3, "tma4": 4, "l1_tma4": 5, "l1_tma4_quarter": 6,
                "tma4_16": 7, "stream_ldg": 8, "stream_bulk": 9, "stream_cpasync": 10, "stream_ldg_occ": 11,
                "stream_ldg_sts": 12, "stream_ldg_few": 13, **{f"stream_ldg_res{32 * k}k": 13 + k for k in range(1, 7)},
                "tex": 20}
GATHER_WITH_VALUES = tuple(k for k in GATHER_PATHS if k.startswith("stream_"))


def gather_ceiling(path: str, col_idx, x, checksum, error, stream=None, vals=None) -> None:
    """Diagnostic: gather x[col_idx[k]] for every k by one load path and add
    the values' bit patterns into ``checksum`` (a zeroed CUDA int64 tensor of
    one element; ``error`` likewise, int32).  The paths in
    GATHER_WITH_VALUES also stream ``vals`` (nnz entries of x's type) and add
    their bit patterns.  Asynchronous on ``stream``."""
    import torch
    if col_idx.dtype != torch.int32 or not col_idx.is_cuda or not col_idx.is_contiguous():
        raise TypeError("col_idx must be a contiguous CUDA int32 tensor")
    if not x.is_cuda or not x.is_contiguous():
        raise TypeError("x must be a contiguous CUDA tensor")
    if checksum.dtype != torch.int64 or error.dtype != torch.int32:
        raise TypeError("checksum must be int64 and error int32")
    if path in GATHER_WITH_VALUES and (vals is None or vals.dtype != x.dtype or vals.numel() != col_idx.numel()
                                       or not vals.is_cuda or not vals.is_contiguous()):
        raise TypeError("this path needs vals: a contiguous CUDA tensor of x's type with one entry per column")
    check(lib().spmv_gather_ceiling(GATHER_PATHS[path], col_idx.numel(), _ptr(col_idx), x.numel(), _ptr(x),
                                    _ptr(vals) if vals is not None else None, _dtype_code(x), checksum.data_ptr(),
                                    error.data_ptr(), _stream_handle(stream)),
          f"spmv_gather_ceiling({path})")
