"""The allocation-free SpMV entry point against the regular one.

evocg_spmv_noalloc serves callers that cannot let a library allocate device memory at call
time (allocation may synchronise the device, is forbidden during stream capture, and is
off limits to programs that own all device memory through their own pool). It keeps its
scratch in a fixed array of the loaded library. This file runs last on purpose, so a failure
here never hides the results of the other GPU tests.
"""
import numpy as np
import pytest

import oracle
from helpers import row_rel_err
from mixed_precision_sparse_gb300 import evocg
from mixed_precision_sparse_gb300 import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _tiles_with_map(m, T, seed):
    n, rp, ci, v = m
    G = evocg.tile_build(n, rp, ci, v, T)
    trow, ex = G.tile_rows()
    evocg.set_tile_precision(G, W.tile_map(trow, ex["tileColIdx"], G.nrb, seed))
    return G


@pytest.mark.parametrize("name,m,T", [
    ("lap2d_64", W.laplace2d_5pt(64), 16),
    ("diff3d_24", W.diffusion3d_7pt(24, 3), 32),
    ("banded_30k", W.banded_spd(30000, 4, band=900), 64),
])
def test_noalloc_matches_regular_spmv_twice(name, m, T):
    """Two calls in a row (they share the fixed scratch): the same kernel as evocg_spmv_ex
    forcing the kernel the allocation-free entry point runs (the direct kernel for tiles of 16,
    the default otherwise), so the same bits; and every row against the oracle at the
    mixed-map tolerance (1e-6 of the row's absolute sum)."""
    n, rp, ci, v = m
    G = _tiles_with_map(m, T, 11)
    A = oracle.CSR(n, rp, ci, v)
    t = oracle.Tiles(A, T)
    mp = W.tile_map(t.tile_rows(), t.tileColIdx, t.nrb, 11)
    absA = oracle.CSR(n, rp, ci, np.abs(v))
    rng = np.random.default_rng(5)
    for call in range(2):
        xh = rng.uniform(-1, 1, G.n) * 10.0 ** rng.uniform(-3, 3, G.n)
        x = torch.from_numpy(xh).cuda()
        y_ref = torch.empty_like(x)
        y_new = torch.full_like(x, float("nan"))
        evocg.spmv_ex(G, x, y_ref, evocg.SPMV_DIRECT if T == 16 else 0)
        evocg.spmv_noalloc(G, x, y_new)
        torch.cuda.synchronize()
        assert torch.equal(y_new.view(torch.int64), y_ref.view(torch.int64)), call
        want = oracle.mixed_spmv(A, t, mp, xh)
        err = row_rel_err(y_new.cpu().numpy(), want, oracle.mixed_spmv(absA, t, mp, np.abs(xh)))
        assert err.max() <= 1e-6, (call, err.max())
    G.free()


def test_noalloc_rejects_sizes_beyond_its_scratch_and_host_pointers():
    n, rp, ci, v = W.laplace2d_5pt(1025, 1024)          # n = 1,049,600 > 2^20
    G = evocg.tile_build(n, rp, ci, v, 32)
    x = torch.zeros(n, dtype=torch.float64, device="cuda")
    y = torch.empty_like(x)
    with pytest.raises(evocg.EvocgError) as e:
        evocg.spmv_noalloc(G, x, y)
    assert e.value.code == evocg.EINVAL and "1048576" in str(e.value)
    G.free()
    G = _tiles_with_map(W.laplace2d_5pt(32), 16, 1)
    with pytest.raises(evocg.EvocgError) as e:
        evocg.spmv_noalloc(G, np.zeros(G.n), np.zeros(G.n))
    assert e.value.code == evocg.EINVAL
    G.free()
