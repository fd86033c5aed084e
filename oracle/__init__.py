"""CPU oracle for the load-balanced CSR SpMV library -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product library never does.

The arithmetic lives in ``oracle.c`` (plain single-threaded C, long double
accumulation); this module compiles it with gcc and wraps it with ctypes.
Every function is pinned by the CPU tests against closed forms, brute force
on tiny inputs, a dense product and the worked example of the Row-grouped
CSR page (``tests/test_oracle_pins.py``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
_LIB = os.path.join(_HERE, "_liboracle.so")


def build(force: bool = False) -> str:
    """Compile oracle.c (gcc -O2, no FMA contraction) into an in-tree library."""
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= newest:
        return _LIB
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_HERE)
    os.close(fd)
    try:
        subprocess.run(["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-ffp-contract=off",
                        "-fno-fast-math", _SRC, "-o", tmp], check=True, capture_output=True, text=True)
        os.replace(tmp, _LIB)
    finally:
        if os.path.exists(tmp):
            os.unlink(tmp)
    return _LIB


class _Stats(ctypes.Structure):
    _fields_ = [("hist", ctypes.c_int64 * 32), ("sum_len", ctypes.c_int64),
                ("rg_slots", ctypes.c_int64 * 4), ("min_len", ctypes.c_int32),
                ("max_len", ctypes.c_int32), ("n_empty", ctypes.c_int32), ("flags", ctypes.c_int32),
                ("bandwidth", ctypes.c_int32), ("reserved", ctypes.c_int32)]


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = _bind(ctypes.CDLL(build()))
    return _lib


def compile_variant(source_text: str, out_path: str) -> str:
    """Compile a modified copy of the oracle source (used by the mutation
    tests, which plant slips in the oracle to show that the pins catch them)."""
    src = out_path + ".c"
    with open(src, "w") as f:
        f.write(source_text)
    subprocess.run(["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-ffp-contract=off", "-I", _HERE,
                    src, "-o", out_path], check=True, capture_output=True, text=True)
    return out_path


class use_library:
    """Context manager: route this module's calls to another compiled copy."""

    def __init__(self, path: str):
        self.path = path

    def __enter__(self):
        global _lib
        self.saved = lib()
        _lib = _bind(ctypes.CDLL(self.path))
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self.saved
        return False


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


def _bind(cdll):
    i32, i64, dbl, vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
    spmv_args = [i32, i32, vp, vp, vp, vp, dbl, dbl, vp, vp, i64, vp, vp]
    sig = {
        "oracle_spmv_f64": spmv_args,
        "oracle_spmv_f32": spmv_args,
        "oracle_merge_path_partition": [i32, i32, vp, i64, i64, vp],
        "oracle_row_stats": [i32, i32, i32, vp, vp, ctypes.POINTER(_Stats)],
        "oracle_rgcsr_layout": [i32, vp, i32, vp, vp],
        "oracle_rgcsr_pack_f64": [i32, vp, vp, vp, i32, vp, vp, vp],
        "oracle_rgcsr_pack_f32": [i32, vp, vp, vp, i32, vp, vp, vp],
        "oracle_long_rows": [i32, vp, i32, i32, vp, vp, ctypes.POINTER(i64)],
        "oracle_window_sort": [i32, vp, i32, i32, vp, vp],
        "oracle_spmm_f64": [i32, i32, i32, vp, vp, vp, vp, i64, dbl, dbl, vp, i64, vp, vp],
        "oracle_spmm_f32": [i32, i32, i32, vp, vp, vp, vp, i64, dbl, dbl, vp, i64, vp, vp],
        "oracle_transpose_f64": [i32, i32, vp, vp, vp, vp, vp, vp, vp],
        "oracle_transpose_f32": [i32, i32, vp, vp, vp, vp, vp, vp, vp],
        "oracle_spmv_transposed_f64": [i32, i32, vp, vp, vp, vp, dbl, dbl, vp, vp, vp],
        "oracle_spmv_transposed_f32": [i32, i32, vp, vp, vp, vp, dbl, dbl, vp, vp, vp],
        "oracle_spgemm_f64": [i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp],
        "oracle_spgemm_f32": [i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp],
    }
    for name, argtypes in sig.items():
        f = getattr(cdll, name)
        f.argtypes = argtypes
        f.restype = ctypes.c_int
    return cdll


def _p(a):
    return None if a is None else a.ctypes.data


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def spmv(row_ptr, col_idx, vals, x, alpha=1.0, beta=0.0, y_old=None, rows=None, n=None):
    """y = alpha*A*x + beta*y_old for all rows (or only ``rows``); returns (y, mag).

    The value type (float32 or float64) follows ``vals``; y has that type and
    mag (the tolerance scale |alpha| sum|a x| + |beta y_old|) is float64."""
    row_ptr = _i32(row_ptr)
    col_idx = _i32(col_idx)
    f64 = np.asarray(vals).dtype == np.float64
    t = np.float64 if f64 else np.float32
    vals = np.ascontiguousarray(vals, dtype=t)
    x = np.ascontiguousarray(x, dtype=t)
    m = len(row_ptr) - 1
    n = len(x) if n is None else n
    if beta != 0.0:
        y_old = np.ascontiguousarray(y_old, dtype=t)
    else:
        y_old = None
    if rows is not None:
        rows = _i32(rows)
        count = len(rows)
    else:
        count = m
    y = np.empty(count, dtype=t)
    mag = np.empty(count, dtype=np.float64)
    fn = lib().oracle_spmv_f64 if f64 else lib().oracle_spmv_f32
    rc = fn(m, n, _p(row_ptr), _p(col_idx), _p(vals), _p(x), float(alpha), float(beta), _p(y_old),
            _p(rows), count, _p(y), _p(mag))
    if rc:
        raise ValueError("oracle_spmv: bad arguments")
    return y, mag


def merge_path_partition(row_ptr, T: int, P: int | None = None) -> np.ndarray:
    """(P+1, 2) int32 array of (row, nonzero) splits of diagonals min(p*T, m+nnz)."""
    row_ptr = _i32(row_ptr)
    m = len(row_ptr) - 1
    nnz = int(row_ptr[-1])
    if P is None:
        P = max(1, -(-(m + nnz) // T))
    part = np.empty((P + 1, 2), dtype=np.int32)
    if lib().oracle_merge_path_partition(m, nnz, _p(row_ptr), T, P, _p(part)):
        raise ValueError("oracle_merge_path_partition: bad arguments")
    return part


def row_stats(row_ptr, col_idx, n: int, nnz: int | None = None) -> dict:
    row_ptr = _i32(row_ptr)
    col_idx = _i32(col_idx)
    m = len(row_ptr) - 1
    nnz = len(col_idx) if nnz is None else nnz
    s = _Stats()
    if lib().oracle_row_stats(m, n, nnz, _p(row_ptr), _p(col_idx), ctypes.byref(s)):
        raise ValueError("oracle_row_stats: bad arguments")
    return {"hist": list(s.hist), "sum_len": s.sum_len, "rg_slots": list(s.rg_slots),
            "min_len": s.min_len, "max_len": s.max_len, "n_empty": s.n_empty, "flags": s.flags,
            "bandwidth": s.bandwidth}


def rgcsr_layout(row_ptr, G: int):
    row_ptr = _i32(row_ptr)
    m = len(row_ptr) - 1
    ng = -(-m // G)
    gp = np.empty(ng + 1, dtype=np.int64)
    rl = np.empty(m, dtype=np.int32)
    if lib().oracle_rgcsr_layout(m, _p(row_ptr), G, _p(gp), _p(rl)):
        raise ValueError("oracle_rgcsr_layout: bad arguments")
    return gp, rl


def rgcsr_pack(row_ptr, col_idx, vals, G: int):
    """(group_ptr, row_len, rg_col, rg_val) of the Row-grouped CSR layout."""
    row_ptr = _i32(row_ptr)
    col_idx = _i32(col_idx)
    gp, rl = rgcsr_layout(row_ptr, G)
    m = len(row_ptr) - 1
    f64 = np.asarray(vals).dtype == np.float64
    t = np.float64 if f64 else np.float32
    vals = np.ascontiguousarray(vals, dtype=t)
    rg_col = np.empty(int(gp[-1]), dtype=np.int32)
    rg_val = np.empty(int(gp[-1]), dtype=t)
    fn = lib().oracle_rgcsr_pack_f64 if f64 else lib().oracle_rgcsr_pack_f32
    if fn(m, _p(row_ptr), _p(col_idx), _p(vals), G, _p(gp), _p(rg_col), _p(rg_val)):
        raise ValueError("oracle_rgcsr_pack: bad arguments")
    return gp, rl, rg_col, rg_val


def long_rows(row_ptr, min_len: int, seg_nnz: int):
    """(ids, seg_begin): rows with at least min_len nonzeros, ascending, and
    the first segment of each (segments of seg_nnz nonzeros)."""
    row_ptr = _i32(row_ptr)
    m = len(row_ptr) - 1
    count = ctypes.c_int64(0)
    if lib().oracle_long_rows(m, _p(row_ptr), min_len, seg_nnz, None, None, ctypes.byref(count)):
        raise ValueError("oracle_long_rows: bad arguments")
    ids = np.empty(count.value, dtype=np.int32)
    seg_begin = np.empty(count.value + 1, dtype=np.int64)
    if lib().oracle_long_rows(m, _p(row_ptr), min_len, seg_nnz, _p(ids), _p(seg_begin), ctypes.byref(count)):
        raise ValueError("oracle_long_rows: bad arguments")
    return ids, seg_begin


def window_sort(row_ptr, window: int, long_min: int = 0):
    """(perm, eff_len) of the window-sorted row order (quadratic: small inputs)."""
    row_ptr = _i32(row_ptr)
    m = len(row_ptr) - 1
    perm = np.empty(m, dtype=np.int32)
    eff = np.empty(m, dtype=np.int32)
    if lib().oracle_window_sort(m, _p(row_ptr), window, long_min, _p(perm), _p(eff)):
        raise ValueError("oracle_window_sort: bad arguments")
    return perm, eff


def spmm(row_ptr, col_idx, vals, X, alpha=1.0, beta=0.0, Y_old=None, n=None):
    """Y = alpha*A*X + beta*Y_old for a row-major X (n-by-k); returns (Y, mag),
    Y m-by-k of the value type, mag float64."""
    row_ptr = _i32(row_ptr)
    col_idx = _i32(col_idx)
    f64 = np.asarray(vals).dtype == np.float64
    t = np.float64 if f64 else np.float32
    vals = np.ascontiguousarray(vals, dtype=t)
    X = np.ascontiguousarray(X, dtype=t)
    m = len(row_ptr) - 1
    k = X.shape[1]
    n = X.shape[0] if n is None else n
    yo = np.ascontiguousarray(Y_old, dtype=t) if beta != 0.0 else None
    Y = np.empty((m, k), dtype=t)
    mag = np.empty((m, k), dtype=np.float64)
    fn = lib().oracle_spmm_f64 if f64 else lib().oracle_spmm_f32
    if fn(m, n, k, _p(row_ptr), _p(col_idx), _p(vals), _p(X), k, float(alpha), float(beta), _p(yo), k,
          _p(Y), _p(mag)):
        raise ValueError("oracle_spmm: bad arguments")
    return Y, mag


def transpose(row_ptr, col_idx, vals, n: int):
    """(t_ptr, t_idx, t_vals, t_src): A^T in CSR form, rows of each column in
    increasing order, t_src the entry's position in A."""
    row_ptr = _i32(row_ptr)
    col_idx = _i32(col_idx)
    f64 = np.asarray(vals).dtype == np.float64
    t = np.float64 if f64 else np.float32
    vals = np.ascontiguousarray(vals, dtype=t)
    m = len(row_ptr) - 1
    nnz = int(row_ptr[-1])
    tp = np.empty(n + 1, dtype=np.int32)
    ti = np.empty(nnz, dtype=np.int32)
    tv = np.empty(nnz, dtype=t)
    ts = np.empty(nnz, dtype=np.int32)
    fn = lib().oracle_transpose_f64 if f64 else lib().oracle_transpose_f32
    if fn(m, n, _p(row_ptr), _p(col_idx), _p(vals), _p(tp), _p(ti), _p(tv), _p(ts)):
        raise ValueError("oracle_transpose: bad arguments")
    return tp, ti, tv, ts


def spmv_transposed(row_ptr, col_idx, vals, x, n: int, alpha=1.0, beta=0.0, y_old=None):
    """y = alpha*A^T*x + beta*y_old (x: m entries, y: n); returns (y, mag)."""
    row_ptr = _i32(row_ptr)
    col_idx = _i32(col_idx)
    f64 = np.asarray(vals).dtype == np.float64
    t = np.float64 if f64 else np.float32
    vals = np.ascontiguousarray(vals, dtype=t)
    x = np.ascontiguousarray(x, dtype=t)
    m = len(row_ptr) - 1
    yo = np.ascontiguousarray(y_old, dtype=t) if beta != 0.0 else None
    y = np.empty(n, dtype=t)
    mag = np.empty(n, dtype=np.float64)
    fn = lib().oracle_spmv_transposed_f64 if f64 else lib().oracle_spmv_transposed_f32
    if fn(m, n, _p(row_ptr), _p(col_idx), _p(vals), _p(x), float(alpha), float(beta), _p(yo), _p(y), _p(mag)):
        raise ValueError("oracle_spmv_transposed: bad arguments")
    return y, mag


def spgemm(a_ptr, a_col, a_val, b_ptr, b_col, b_val, n: int, c_row_ptr=None):
    """C = A*B (A m-by-k, B k-by-n, CSR): (c_row_ptr int64, c_col, c_val),
    columns in increasing order in each row, sums in long double.  A first
    call sizes the rows; c_row_ptr, when given (the row pointers of an
    earlier call on the same patterns), takes its place."""
    a_ptr, a_col, b_ptr, b_col = _i32(a_ptr), _i32(a_col), _i32(b_ptr), _i32(b_col)
    f64 = np.asarray(a_val).dtype == np.float64
    t = np.float64 if f64 else np.float32
    a_val = np.ascontiguousarray(a_val, dtype=t)
    b_val = np.ascontiguousarray(b_val, dtype=t)
    m, k = len(a_ptr) - 1, len(b_ptr) - 1
    fn = lib().oracle_spgemm_f64 if f64 else lib().oracle_spgemm_f32
    if c_row_ptr is not None:
        rp = np.array(c_row_ptr, dtype=np.int64)
        assert len(rp) == m + 1
    else:
        rp = np.empty(m + 1, dtype=np.int64)
        if fn(m, k, n, _p(a_ptr), _p(a_col), _p(a_val), _p(b_ptr), _p(b_col), _p(b_val), _p(rp), None, None):
            raise ValueError("oracle_spgemm: bad arguments")
    col = np.empty(int(rp[-1]), dtype=np.int32)
    val = np.empty(int(rp[-1]), dtype=t)
    if fn(m, k, n, _p(a_ptr), _p(a_col), _p(a_val), _p(b_ptr), _p(b_col), _p(b_val), _p(rp), _p(col), _p(val)):
        raise ValueError("oracle_spgemm: bad arguments")
    return rp, col, val
