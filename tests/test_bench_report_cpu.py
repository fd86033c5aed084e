"""The benchmark's report arithmetic on the CPU: the compulsory bytes of a
product, counted by hand on a small matrix, and the SpMM path label, which
restates the library's choice of path (first applicable of: the Row-grouped
copy with rare long rows, CSR for short rows or rare long rows with at most
two column slices, the merge-path partition)."""
import numpy as np

import bench
import synth


def test_compulsory_bytes_by_hand():
    # 3 x 5, rows of 2, 0 and 3 nonzeros, fp32: indices and values 5 * (4 + 4),
    # row_ptr 4 * 4, x 5 * 4, y read and written 2 * 3 * 4 (the roofline's
    # count); the beta-aware count drops the y read when beta == 0
    A = synth.CSR(3, 5, np.array([0, 2, 2, 5], np.int32), np.array([0, 4, 1, 2, 3], np.int32),
                  np.ones(5, np.float32))
    assert bench.compulsory_bytes(A) == 40 + 16 + 20 + 24
    assert bench.compulsory_bytes(A, 0.0) == 40 + 16 + 20 + 12
    assert bench.compulsory_bytes(A, 0.5) == 40 + 16 + 20 + 24
    B = synth.CSR(3, 5, A.row_ptr, A.col_idx, np.ones(5, np.float64))
    assert bench.compulsory_bytes(B) == 5 * 12 + 16 + 40 + 48
    assert bench.compulsory_bytes(B, 0.0) == 5 * 12 + 16 + 40 + 24


def test_roofline_fractions():
    # 1e9 bytes in 1e6 us (1 s) is 1 GB/s; the beta-aware count is half of it
    r = bench.roofline(10**9, 5 * 10**8, 10**6, "none", "none")
    assert r["achieved"] == 1.0 and r["unit"] == "GB/s"
    assert abs(r["frac"] - 1.0 / r["peak"]) < 1e-4
    assert abs(r["frac_beta_aware"] - 0.5 / r["peak"]) < 1e-4


def _info(kernel, m, num_long=0, max_len=8, group=32):
    return {"kernel_name": kernel, "rgcsr_group": group, "num_long_rows": num_long, "m": m,
            "stats": {"max_len": max_len}}


def test_spmm_path_label_follows_the_choice():
    short = np.arange(0, 4 * 10001, 4, dtype=np.int64)           # 10,000 rows of 4
    name, launches = bench.spmm_path_of(_info("rgcsr", 10000), 40, 4, short)
    assert name.startswith("Row-grouped") and launches == 2       # slices of 32 (fp32)
    name, launches = bench.spmm_path_of(_info("rgcsr", 10000), 40, 8, short)
    assert name.startswith("Row-grouped") and launches == 3       # slices of 16 (fp64)
    name, launches = bench.spmm_path_of(_info("merge_path", 10000), 40, 4, short)
    assert name.startswith("short-row") and launches == 2         # 32 + 8
    name, _ = bench.spmm_path_of(_info("merge_path", 10000), 7, 4, short)
    assert name.startswith("merge-path")                          # k not a multiple of 4
    # one row of 100 among 10,000 (rare): the CSR path with long rows up to two slices
    lens = np.full(10000, 4, dtype=np.int64)
    lens[5] = 100
    rp = np.concatenate([[0], np.cumsum(lens)])
    name, launches = bench.spmm_path_of(_info("merge_path", 10000, max_len=100), 32, 4, rp)
    assert "4096-nonzero segment" in name and launches == 2
    name, _ = bench.spmm_path_of(_info("merge_path", 10000, max_len=100), 128, 4, rp)
    assert name.startswith("merge-path")                          # four slices: merge path
    # many long rows: merge path
    lens[:100] = 100
    rp = np.concatenate([[0], np.cumsum(lens)])
    name, _ = bench.spmm_path_of(_info("merge_path", 10000, max_len=100), 32, 4, rp)
    assert name.startswith("merge-path")
    # a Row-grouped plan whose long rows are not rare
    name, _ = bench.spmm_path_of(_info("rgcsr", 10000, num_long=10), 32, 4, rp)
    assert name.startswith("merge-path")
