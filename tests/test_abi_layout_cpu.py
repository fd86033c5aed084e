"""The ctypes structures of the Python binding against the C header: a
small C program compiled here with gcc prints the size of every structure
include/spmv.h declares and the offset of every field, and the binding's
ctypes mirrors must agree byte for byte (a mismatch would hand the library
garbage options or read garbage statistics on the GPU)."""
import ctypes
import os
import re
import shutil
import subprocess

import pytest

import load_balanced_csr_gb300 as lb
from load_balanced_csr_gb300 import _build

STRUCTS = {
    "spmv_options_t": lb.Options,
    "spmv_row_stats_t": lb.RowStats,
    "spmv_plan_info_t": lb.PlanInfo,
    "spmv_spgemm_info_t": lb.SpgemmInfo,
}


def c_layout(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "spmv.h"', "int main(void) {"]
    for cname, py in STRUCTS.items():
        lines.append(f'    printf("{cname} size %zu\\n", sizeof({cname}));')
        for field, _ in py._fields_:
            if field == "reserved":
                continue
            lines.append(f'    printf("{cname} {field} %zu\\n", offsetof({cname}, {field}));')
    lines += ["    return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-I", _build.INCLUDE, str(src), "-o", str(exe)], check=True, capture_output=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    got = {}
    for line in out.splitlines():
        cname, field, value = line.split()
        got[(cname, field)] = int(value)
    return got


def test_ctypes_structures_match_the_header(tmp_path):
    got = c_layout(tmp_path)
    for cname, py in STRUCTS.items():
        assert got[(cname, "size")] == ctypes.sizeof(py), \
            f"{cname}: size {got[(cname, 'size')]} in C, {ctypes.sizeof(py)} in ctypes"
        for field, _ in py._fields_:
            if field == "reserved":
                continue
            assert got[(cname, field)] == getattr(py, field).offset, \
                f"{cname}.{field}: offset {got[(cname, field)]} in C, {getattr(py, field).offset} in ctypes"


def test_header_kernel_and_export_codes_match_the_binding():
    """The enum values the binding passes by name."""
    with open(os.path.join(_build.INCLUDE, "spmv.h")) as f:
        text = f.read()
    kernels = {m.group(1).lower(): int(m.group(2))
               for m in re.finditer(r"SPMV_KERNEL_([A-Z_]+)\s*=\s*(\d+)", text)}
    assert kernels == lb.KERNELS
    exports = {m.group(1).lower(): int(m.group(2))
               for m in re.finditer(r"SPMV_EXPORT_([A-Z_]+)\s*=\s*(\d+)", text)}
    assert exports == lb.EXPORTS
