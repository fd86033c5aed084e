"""The plan's kernel choice, pinned at each rule's boundary.  The rules, in
order (the first that applies wins):

1. n == 1 and rows of at most 32 nonzeros -> thread per row (the single-column
   case that "A GPU load-balancing programming model", section 6.1, names:
   perfectly balanced work needs no balancing);
2. (m < 500 or n < 500) and nnz < 10,000 and rows of at most 256 -> thread per
   row (the same paper's small-matrix rule, section 6.2);
3. m <= 65,536 and rows of at most 64 -> thread per row (latency-bound sizes);
4. a Row-grouped copy with groups of 32 rows pads at most 10 % -> Row-grouped
   CSR (the Row-grouped CSR page, section 4: padding is the format's cost);
5. otherwise merge path.

Each case builds a matrix on one side of a boundary (duplicate columns are
allowed by the ABI, which is how n == 1 gets rows longer than one), plans it
on the GPU (the statistics come from the plan's own kernels) and checks the
kernel the plan reports.  A threshold that slipped by one would fail here
even where every product stays correct."""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu


def _csr(lens, n, seed=0):
    """Rows of the given lengths, columns drawn uniformly in [0, n) (with
    repeats when a row is longer than n), sorted within each row."""
    rng = np.random.default_rng(seed)
    lens = np.asarray(lens, dtype=np.int64)
    rp = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    col = rng.integers(0, n, size=int(rp[-1]), dtype=np.int64).astype(np.int32)
    for i in range(len(lens)):
        col[rp[i]:rp[i + 1]].sort()
    vals = rng.standard_normal(int(rp[-1])).astype(np.float32)
    return synth.CSR(len(lens), n, rp, col, vals)


def _kernel(A):
    import torch
    import load_balanced_csr_gb300 as lb
    t = lambda a: torch.from_numpy(a).cuda()
    with lb.Plan(t(A.row_ptr), t(A.col_idx), t(A.vals), A.n) as plan:
        info = plan.info()
    return info["kernel_name"], info["stats"]


def test_rule1_single_column():
    # n == 1: rows of 32 (duplicates) take thread per row even at m > 65,536
    k, s = _kernel(_csr(np.full(70000, 32), 1))
    assert s["max_len"] == 32 and k == "thread_row"
    # rows of 33: rule 1 no longer applies; uniform rows pad nothing -> Row-grouped
    k, s = _kernel(_csr(np.full(70000, 33), 1))
    assert s["max_len"] == 33 and k == "rgcsr"


def _small(m, n, nnz, longest, seed=1):
    lens = np.zeros(m, dtype=np.int64)
    lens[0] = longest
    rest = nnz - longest
    lens[1:] = rest // (m - 1)
    lens[1:1 + rest % (m - 1)] += 1
    assert lens.sum() == nnz and lens.max() == longest
    return _csr(lens, n, seed)


def test_rule2_small_matrices():
    # m = 499 < 500, nnz = 9,999 < 10,000, longest row 256: thread per row
    assert _kernel(_small(499, 100000, 9999, 256))[0] == "thread_row"
    # n = 499 < 500 instead of m
    assert _kernel(_small(600, 499, 9999, 256))[0] == "thread_row"
    # each boundary crossed on its own: merge path (rows too uneven for rule 4,
    # a row longer than 64 for rule 3)
    assert _kernel(_small(499, 100000, 10000, 256))[0] == "merge_path"
    assert _kernel(_small(499, 100000, 9999, 257))[0] == "merge_path"
    assert _kernel(_small(500, 500, 9999, 256))[0] == "merge_path"


def test_rule3_latency_bound_sizes():
    rng = np.random.default_rng(3)
    lens = rng.integers(0, 9, size=65536)
    lens[7] = 64
    assert _kernel(_csr(lens, 65536, 3))[0] == "thread_row"
    lens[7] = 65  # one row too long
    assert _kernel(_csr(lens, 65536, 3))[0] == "merge_path"
    lens = rng.integers(0, 9, size=65537)
    lens[7] = 64  # one row too many
    assert _kernel(_csr(lens, 65537, 3))[0] == "merge_path"


def test_rule4_row_grouped_padding():
    # groups of 32 rows: 31 rows of 10 and one of L.  The copy holds 32 * L
    # slots per group for 310 + L nonzeros: L = 11 pads 9.66 %, L = 12 pads
    # 19.3 % (beyond 10 %)
    groups = 4096
    for L, want in ((11, "rgcsr"), (12, "merge_path")):
        lens = np.tile(np.concatenate([np.full(31, 10), [L]]), groups)
        k, s = _kernel(_csr(lens, 200000, 4))
        assert s["rg_slots"][0] == 32 * L * groups
        assert k == want, (L, k)


def test_plan_log_names_the_rule():
    """SPMV_LOG=1 prints one line per plan on stderr: the statistics and
    the kernel with the rule that chose it (checked in a child process, so
    that the variable is read at plan creation there)."""
    import os
    import subprocess
    import sys
    code = (
        "import sys; sys.path.insert(0, 'tests'); import numpy as np, torch, synth\n"
        "import load_balanced_csr_gb300 as lb\n"
        "from helpers import to_gpu\n"
        "A = synth.fill_random(np.full(300, 3, np.int32), 200, seed=1, dtype='f32')\n"
        "rp, col, val = to_gpu(A)\n"
        "lb.Plan(rp, col, val, A.n).close()\n"
        "B = synth.fill_random(synth.lengths_uniform(200000, 0, 80, 2), 200000, seed=2, dtype='f64')\n"
        "rp, col, val = to_gpu(B)\n"
        "lb.Plan(rp, col, val, B.n).close()\n"
    )
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, SPMV_LOG="1")
    r = subprocess.run([sys.executable, "-c", code], cwd=root, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stderr.splitlines() if ln.startswith("spmv plan:")]
    assert len(lines) == 2, r.stderr[-2000:]
    assert "m=300 n=200 nnz=900 f32" in lines[0] and "kernel=thread_row (small matrix" in lines[0]
    assert "kernel=merge_path (default)" in lines[1] and "f64" in lines[1]
