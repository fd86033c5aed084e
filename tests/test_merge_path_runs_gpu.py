"""Merge path when each warp owns a long run of tiles, at sizes where every
row can still be checked against the oracle.

The warps of the merge-path kernel each take a contiguous run of about
num_tiles / W tiles (W = the plan's merge_path_warps).  The state carried
from tile to tile -- the sum of the open row in a register, the lanes'
shares of a row that fills whole tiles, the reuse of the copy stages -- is
only exercised when runs are long, so these matrices hold at least 8 W
tiles; long rows cross many tiles and many warps (their partial sums meet in
the cut-row protocol).  The last test makes runs long enough that the plan
must add warps beyond the GPU's resident ones to keep each run within the
summation-depth cap (120 - 2 (items per lane + 1) tiles)."""
import numpy as np
import pytest

import synth
from helpers import assert_all_rows_close, to_gpu

pytestmark = pytest.mark.gpu


def _run(A, alpha, beta, ipt, seed):
    import torch
    import load_balanced_csr_gb300 as lb
    x = synth.vector(A.n, synth.DIST_NORMAL, seed, synth.STREAM_X, A.dtype)
    y0 = synth.vector(A.m, synth.DIST_NORMAL, seed, synth.STREAM_Y, A.dtype)
    rp, col, val = to_gpu(A)
    xd = torch.from_numpy(x).cuda()
    yd = torch.from_numpy(y0.copy()).cuda() if beta != 0 else \
        torch.full((A.m,), float("nan"), dtype=val.dtype, device="cuda")
    with lb.Plan(rp, col, val, A.n, kernel="merge_path", items_per_thread=ipt) as plan:
        info = plan.info()
        plan(xd, yd, alpha, beta)
        plan(xd, yd, alpha, beta) if beta == 0 else None  # a second product reuses the counters
        torch.cuda.synchronize()
        assert plan.device_status() == 0
    return info, x, y0, yd.cpu().numpy()


@pytest.mark.parametrize("dtype", ["f32", "f64"])
def test_many_tiles_per_warp(dtype):
    m = 1_300_000
    lens = synth.lengths_uniform(m, 0, 12, 21)
    lens[[5, 400_000, 1_299_990]] = 300_000   # each crosses over a thousand tiles of 256
    lens[700_000:700_040] = 20_000
    A = synth.fill_random(lens, 2_000_000, dist=synth.DIST_NORMAL, seed=21, dtype=dtype)
    for alpha, beta in ((1.0, 0.0), (1.5, 0.5)):
        info, x, y0, y = _run(A, alpha, beta, 8, 21)
        P, W = info["num_tiles"], info["merge_path_warps"]
        assert W > 0 and P >= 8 * W, (P, W)
        assert -(-P // W) <= 120 - 2 * 9
        assert np.all(np.isfinite(y)), "a row was not written"
        assert_all_rows_close(A, x, y, alpha, beta, y0, label=f"{dtype} alpha={alpha} beta={beta}")


def test_runs_capped_by_summation_depth():
    # ~102M rows + nonzeros in tiles of 256: the resident warps alone would
    # each run over 102 tiles, so the plan adds warps
    m = 12_000_000
    lens = synth.lengths_uniform(m, 0, 15, 22)
    lens[3] = 2_000_000  # one row across ~7,800 tiles
    A = synth.fill_random(lens, m, dist=synth.DIST_NORMAL, seed=22, dtype="f32")
    info, x, y0, y = _run(A, 1.0, 0.0, 8, 22)
    P, W = info["num_tiles"], info["merge_path_warps"]
    assert -(-P // W) <= 120 - 2 * 9 and P > 102 * 152 * 24, (P, W)
    assert np.all(np.isfinite(y))
    assert_all_rows_close(A, x, y, 1.0, 0.0, y0, label="capped runs")
