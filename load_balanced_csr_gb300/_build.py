"""Build the CUDA library in-tree: nvcc for sm_103a, one object per source,
compiled in parallel, linked into ``libspmv.so`` beside this file."""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(HERE, "libspmv.so")
OBJDIR = os.path.join(HERE, "_build")
# the debug build (-DSPMV_DEBUG: device-side checks of the column indices
# gathered with) sits beside it, from objects of its own
DEBUG_LIB = os.path.join(HERE, "libspmv_debug.so")
DEBUG_OBJDIR = os.path.join(OBJDIR, "debug")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2", "--expt-relaxed-constexpr",
              "-Xptxas", "-warn-spills"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libspmv.so")
    return cand


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs() -> list[str]:
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h"))


def _stamp(objdir: str) -> str:
    return os.path.join(objdir, "flags.txt")


def _flags_used(objdir: str = OBJDIR) -> str | None:
    try:
        with open(_stamp(objdir)) as f:
            return f.read()
    except OSError:
        return None


def stale(extra: list[str] | None = None, lib: str = LIB, objdir: str = OBJDIR) -> bool:
    """The library is missing, older than a source, or built with other
    extra nvcc flags."""
    if not os.path.exists(lib):
        return True
    if (_flags_used(objdir) or "") != " ".join(extra or []):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(f) > t for f in _inputs())


def build(force: bool = False, verbose: bool = False, extra: list[str] | None = None, debug: bool = False) -> str:
    """Compile every source for sm_103a and link libspmv.so (debug:
    libspmv_debug.so, with -DSPMV_DEBUG).  Extra nvcc flags come from
    `extra` and the SPMV_NVCC_EXTRA environment variable (compile-time tuning
    parameters, e.g. -DLBCSR_MP_STAGES=1)."""
    extra = (extra or []) + os.environ.get("SPMV_NVCC_EXTRA", "").split() + (["-DSPMV_DEBUG"] if debug else [])
    lib, objdir = (DEBUG_LIB, DEBUG_OBJDIR) if debug else (LIB, OBJDIR)
    if not force and not stale(extra, lib, objdir):
        return lib
    os.makedirs(objdir, exist_ok=True)
    cc = nvcc()
    flags = NVCC_FLAGS + ARCH + ["-I", INCLUDE, "-I", CSRC] + extra

    def compile_one(src: str) -> str:
        obj = os.path.join(objdir, os.path.basename(src) + ".o")
        cmd = [cc, "-c", src, "-o", obj] + flags
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr}")
        if verbose and r.stderr.strip():
            print(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, sources()))
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=HERE)
    os.close(fd)
    try:
        cmd = [cc, "-shared", *ARCH, "-o", tmp, *objs, "-Xcompiler", "-fPIC"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr}")
        os.replace(tmp, lib)
        with open(_stamp(objdir), "w") as f:
            f.write(" ".join(extra))
    finally:
        if os.path.exists(tmp):
            os.unlink(tmp)
    return lib


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True, debug="--debug" in sys.argv))
