"""The gather-ceiling diagnostic (spmv_gather_ceiling): every load path must
gather exactly x[col_idx[k]] for every k.  The check is the sum, modulo 2^64,
of the gathered values' bit patterns, computed here with numpy from the same
seeded columns and x; columns reach the last entries of x (past the 32-byte
rows the tensor gather covers), and nnz is not a multiple of a warp's chunk."""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

PATHS = None  # every path the binding lists


@pytest.mark.parametrize("dtype", ["f32", "f64"])
@pytest.mark.parametrize("n,nnz", [(37, 3 * 4096 + 77), (1000, 3 * 4096 + 77), (123457, 3 * 4096 + 77),
                                   (5000, 40 * 256)])
def test_gather_checksum(dtype, n, nnz):
    import torch
    import load_balanced_csr_gb300 as lb
    rng = np.random.default_rng(n)
    col = rng.integers(0, n, size=nnz).astype(np.int32)
    col[:5] = n - 1  # the tail of x
    x = synth.vector(n, synth.DIST_NORMAL, n, synth.STREAM_X, dtype)
    bits = x.view(np.uint64 if dtype == "f64" else np.uint32)
    want = int(np.sum(bits[col].astype(np.uint64), dtype=np.uint64))
    want_stream = int(np.sum(col.astype(np.uint64), dtype=np.uint64))
    vals = synth.vector(nnz, synth.DIST_NORMAL, n + 1, synth.STREAM_Y, dtype)
    vbits = vals.view(np.uint64 if dtype == "f64" else np.uint32)
    want_vals = (want + int(np.sum(vbits.astype(np.uint64), dtype=np.uint64))) & (2**64 - 1)
    cd, xd, vd = torch.from_numpy(col).cuda(), torch.from_numpy(x).cuda(), torch.from_numpy(vals).cuda()
    for path in lb.GATHER_PATHS:
        for rep in range(2):
            cs = torch.zeros(1, dtype=torch.int64, device="cuda")
            err = torch.zeros(1, dtype=torch.int32, device="cuda")
            lb.gather_ceiling(path, cd, xd, cs, err, vals=vd)
            torch.cuda.synchronize()
            assert int(err.item()) == 0, path
            got = int(cs.item()) & (2**64 - 1)
            expect = want_stream if path == "stream" else want_vals if path in lb.GATHER_WITH_VALUES else want
            assert got == expect, (path, rep)


def test_gather_rejects_misaligned_x():
    import torch
    import load_balanced_csr_gb300 as lb
    col = torch.zeros(100, dtype=torch.int32, device="cuda")
    xbuf = torch.zeros(1001, dtype=torch.float32, device="cuda")
    x = xbuf[1:]  # 4 bytes past a 16-byte boundary
    cs = torch.zeros(1, dtype=torch.int64, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for path in ("bulk16", "tma4", "l1_tma4", "l1_tma4_quarter", "tma4_16"):
        with pytest.raises(lb.SpmvError):
            lb.gather_ceiling(path, col, x, cs, err)
    lb.gather_ceiling("l1", col, x, cs, err)  # plain loads take any alignment
    torch.cuda.synchronize()
    assert int(err.item()) == 0
