"""Seeded synthetic inputs: CSR matrices and dense vectors.

Shared by the tests, the benchmark and the oracle checks.  Nothing here
computes a matrix-vector product: the C file draws row lengths, sorted
distinct column sets and values, and this module forms row pointers as the
running sum of the lengths and wraps the results in numpy arrays.

The five workloads of the benchmark (``WORKLOADS``) follow the matrix
families the load-balancing pages measure SpMV on (a regular stencil, a
power-law graph, very short irregular rows, extreme skew); the pages'
SuiteSparse corpus is not available here, and these seeded matrices stand in
for it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB = os.path.join(_HERE, "_libsynth.so")

DIST_UNIFORM_PM1 = 0
DIST_NORMAL = 1
DIST_SMALL_INT = 2

# vector stream ids (each vector draws from its own stream)
STREAM_X = 1
STREAM_Y = 2


def build(force: bool = False) -> str:
    """Compile gen.c into an in-tree shared library (gcc, OpenMP if present)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_HERE)
    os.close(fd)
    base = ["gcc", "-O2", "-fPIC", "-shared", "-std=gnu11", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    try:
        r = subprocess.run(base[:1] + ["-fopenmp"] + base[1:], capture_output=True, text=True)
        if r.returncode != 0:
            subprocess.run(base, check=True, capture_output=True, text=True)
        os.replace(tmp, _LIB)
    finally:
        if os.path.exists(tmp):
            os.unlink(tmp)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        i32, i64, u64, dbl, vp, ip = (ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64,
                                      ctypes.c_double, ctypes.c_void_p, ctypes.c_void_p)
        sig = {
            "synth_vector": [i64, ctypes.c_int, u64, u64, ctypes.c_int, vp],
            "synth_lengths_uniform": [i32, i32, i32, u64, ip],
            "synth_lengths_powerlaw": [i32, dbl, i32, dbl, dbl, u64, ip, ctypes.POINTER(dbl)],
            "synth_lengths_skew": [i32, i32, i32, i32, ip, u64, ip, ip],
            "synth_fill_random": [i32, i32, ip, i32, ctypes.c_int, u64, ctypes.c_int, ip, vp],
            "synth_laplace2d_lengths": [i32, i32, ip],
            "synth_laplace2d_fill": [i32, i32, ip, ctypes.c_int, ip, vp],
            "synth_stencil27_lengths": [i32, ip],
            "synth_stencil27_fill": [i32, ip, ctypes.c_int, dbl, u64, ctypes.c_int, ip, vp],
        }
        for name, argtypes in sig.items():
            f = getattr(_lib, name)
            f.argtypes = argtypes
            f.restype = ctypes.c_int
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise RuntimeError(f"{what} failed with code {rc}")


def _np_dtype(dtype: str):
    return {"f32": np.float32, "f64": np.float64}[dtype]


@dataclass
class CSR:
    """A CSR matrix (row_ptr[m+1], col_idx[nnz], vals[nnz]) with m rows, n columns."""

    m: int
    n: int
    row_ptr: np.ndarray
    col_idx: np.ndarray
    vals: np.ndarray
    meta: dict = field(default_factory=dict)

    @property
    def nnz(self) -> int:
        return int(self.row_ptr[-1]) if self.m >= 0 else 0

    @property
    def dtype(self) -> str:
        return "f64" if self.vals.dtype == np.float64 else "f32"


def row_ptr_from_lengths(lengths: np.ndarray) -> np.ndarray:
    rp = np.zeros(len(lengths) + 1, dtype=np.int64)
    np.cumsum(lengths, out=rp[1:])
    if rp[-1] >= 2**31:
        raise ValueError("nnz does not fit int32")
    return rp.astype(np.int32)


def vector(n: int, dist: int, seed: int, stream: int, dtype: str) -> np.ndarray:
    out = np.empty(n, dtype=_np_dtype(dtype))
    _check(lib().synth_vector(n, dist, seed, stream, int(dtype == "f64"), _ptr(out)), "synth_vector")
    return out


def fill_random(lengths: np.ndarray, n: int, *, band: int = -1, dist: int = DIST_UNIFORM_PM1,
                seed: int = 0, dtype: str = "f64", meta=None) -> CSR:
    """Columns uniform without repetition (within +-band of the diagonal if band >= 0),
    sorted in each row; values from ``dist``."""
    lengths = np.ascontiguousarray(lengths, dtype=np.int32)
    m = len(lengths)
    rp = row_ptr_from_lengths(lengths)
    nnz = int(rp[-1])
    col = np.empty(nnz, dtype=np.int32)
    val = np.empty(nnz, dtype=_np_dtype(dtype))
    _check(lib().synth_fill_random(m, n, _ptr(rp), band, dist, seed, int(dtype == "f64"),
                                   _ptr(col), _ptr(val)), "synth_fill_random")
    return CSR(m, n, rp, col, val, dict(meta or {}))


def lengths_uniform(m: int, lo: int, hi: int, seed: int) -> np.ndarray:
    out = np.empty(m, dtype=np.int32)
    _check(lib().synth_lengths_uniform(m, lo, hi, seed, _ptr(out)), "synth_lengths_uniform")
    return out


def lengths_powerlaw(m: int, exponent: float, cap: int, mean: float, seed: int, tol: float = 0.01):
    out = np.empty(m, dtype=np.int32)
    s = ctypes.c_double(0.0)
    _check(lib().synth_lengths_powerlaw(m, exponent, cap, mean, tol, seed, _ptr(out), ctypes.byref(s)),
           "synth_lengths_powerlaw")
    return out, s.value


def lengths_skew(m: int, lo: int, hi: int, heavy: list[int], seed: int):
    out = np.empty(m, dtype=np.int32)
    heavy_a = np.ascontiguousarray(heavy, dtype=np.int32)
    rows = np.empty(len(heavy), dtype=np.int32)
    _check(lib().synth_lengths_skew(m, lo, hi, len(heavy), _ptr(heavy_a), seed, _ptr(out), _ptr(rows)),
           "synth_lengths_skew")
    return out, rows


def laplace2d(nx: int, ny: int, dtype: str = "f64") -> CSR:
    m = nx * ny
    lengths = np.empty(m, dtype=np.int32)
    _check(lib().synth_laplace2d_lengths(nx, ny, _ptr(lengths)), "synth_laplace2d_lengths")
    rp = row_ptr_from_lengths(lengths)
    col = np.empty(int(rp[-1]), dtype=np.int32)
    val = np.empty(int(rp[-1]), dtype=_np_dtype(dtype))
    _check(lib().synth_laplace2d_fill(nx, ny, _ptr(rp), int(dtype == "f64"), _ptr(col), _ptr(val)),
           "synth_laplace2d_fill")
    return CSR(m, m, rp, col, val, {"structure": f"5-point Laplacian {nx}x{ny}"})


def stencil27(g: int, *, dist: int = DIST_UNIFORM_PM1, diag: float = 27.0, seed: int = 0,
              dtype: str = "f32") -> CSR:
    m = g * g * g
    lengths = np.empty(m, dtype=np.int32)
    _check(lib().synth_stencil27_lengths(g, _ptr(lengths)), "synth_stencil27_lengths")
    rp = row_ptr_from_lengths(lengths)
    col = np.empty(int(rp[-1]), dtype=np.int32)
    val = np.empty(int(rp[-1]), dtype=_np_dtype(dtype))
    _check(lib().synth_stencil27_fill(g, _ptr(rp), dist, diag, seed, int(dtype == "f64"), _ptr(col), _ptr(val)),
           "synth_stencil27_fill")
    return CSR(m, m, rp, col, val, {"structure": f"27-point stencil {g}^3"})


# --------------------------------------------------------------------------
# workloads


@dataclass
class Workload:
    name: str
    A: CSR
    x: np.ndarray
    y0: np.ndarray | None
    alpha: float
    beta: float
    description: str


def _vectors(A: CSR, dist: int, seed: int, y_dist: int | None):
    x = vector(A.n, dist, seed, STREAM_X, A.dtype)
    y0 = vector(A.m, y_dist, seed, STREAM_Y, A.dtype) if y_dist is not None else None
    return x, y0


def workload(name: str, scale: int = 1, seed: int = 0) -> Workload:
    """Build one of the five workloads; ``scale`` > 1 shrinks the large ones
    (m and the heavy rows divided by ``scale``) for oracle-sized parity runs."""
    if name == "laplace2d_64":
        A = laplace2d(64, 64, "f64")
        x, y0 = _vectors(A, DIST_UNIFORM_PM1, seed, None)
        return Workload(name, A, x, y0, 1.0, 0.0,
                        "2-D 5-point Laplacian 64x64, fp64, x U[-1,1], alpha=1, beta=0")
    if name == "stencil27_128":
        g = max(4, 128 // scale)
        A = stencil27(g, dist=DIST_UNIFORM_PM1, diag=27.0, seed=seed, dtype="f32")
        x, y0 = _vectors(A, DIST_UNIFORM_PM1, seed, None)
        return Workload(name, A, x, y0, 1.0, 0.0,
                        f"3-D 27-point stencil {g}^3, fp32 U[-1,1] off-diagonal, diagonal 27, alpha=1, beta=0")
    if name == "powerlaw_4M":
        m = max(1024, 4_194_304 // scale)
        cap = max(64, 200_000 // scale)
        lens, s = lengths_powerlaw(m, 2.1, cap, 16.0, seed)
        A = fill_random(lens, m, band=-1, dist=DIST_NORMAL, seed=seed, dtype="f32",
                        meta={"structure": "power law 2.1", "scale": s, "cap": cap})
        x, y0 = _vectors(A, DIST_NORMAL, seed, None)
        return Workload(name, A, x, y0, 1.0, 0.0,
                        f"power-law rows (exponent 2.1, clip [1,{cap}], mean 16), m=n={m}, fp32 N(0,1)")
    if name == "short_rows_16M":
        m = max(1024, 16_777_216 // scale)
        lens = lengths_uniform(m, 0, 4, seed)
        A = fill_random(lens, m, band=1024, dist=DIST_UNIFORM_PM1, seed=seed, dtype="f64",
                        meta={"structure": "lengths U{0..4}, band +-1024"})
        x, y0 = _vectors(A, DIST_UNIFORM_PM1, seed, DIST_NORMAL)
        return Workload(name, A, x, y0, 1.5, 0.5,
                        f"short rows U{{0..4}}, band +-1024, m=n={m}, fp64, alpha=1.5, beta=0.5")
    if name == "skew_8M":
        m = max(4096, 8_388_608 // scale)
        heavy = [max(64, 4_000_000 // scale)] + [max(16, 100_000 // scale)] * 64
        lens, rows = lengths_skew(m, 1, 8, heavy, seed)
        A = fill_random(lens, m, band=-1, dist=DIST_NORMAL, seed=seed, dtype="f64",
                        meta={"structure": "skew", "heavy_rows": rows})
        x, y0 = _vectors(A, DIST_NORMAL, seed, None)
        return Workload(name, A, x, y0, 1.0, 0.0,
                        f"extreme skew: one row of {heavy[0]}, 64 rows of {heavy[1]}, others U[1,8], m=n={m}, fp64")
    raise KeyError(name)


WORKLOADS = ["laplace2d_64", "stencil27_128", "powerlaw_4M", "short_rows_16M", "skew_8M"]


def random_csr(m: int, n: int, *, max_len: int, empty_frac: float = 0.0, dist: int = DIST_UNIFORM_PM1,
               seed: int = 0, dtype: str = "f64") -> CSR:
    """Small random CSR for tests: lengths U[0, max_len] (capped at n), then a
    seeded fraction of rows forced empty."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(0, max_len + 1, size=m).astype(np.int32)
    lens = np.minimum(lens, n).astype(np.int32)
    if empty_frac > 0:
        lens[rng.random(m) < empty_frac] = 0
    return fill_random(lens, n, band=-1, dist=dist, seed=seed, dtype=dtype)
