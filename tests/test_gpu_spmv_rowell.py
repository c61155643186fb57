"""GPU parity of the row-ELL SpMV kernel (tiles of 64 holding about one entry per row) against
the oracle: every row, per-row relative error, small banded matrices, per-tile and
per-column-block maps, a ragged last row block and the full banded workload; and against the
direct kernel to rounding."""
import numpy as np
import pytest

import oracle
from helpers import Pair, row_rel_err
from mixed_precision_sparse_gb300 import evocg
from mixed_precision_sparse_gb300 import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL64 = 1e-12
TOLMIX = 1e-6

CASES = [("banded_20k", W.banded_spd(20000, 6, band=700)),
         ("banded_ragged", W.banded_spd(5003, 3, band=3000)),
         ("banded_wide", W.banded_spd(30000, 4, band=4096))]


def _run(P, x, mp, kind=evocg.MAP_PER_TILE, flags=evocg.SPMV_ROWELL):
    evocg.set_tile_precision(P.G, mp, kind)
    y = torch.full((P.n,), np.nan, dtype=torch.float64, device="cuda")
    evocg.spmv_ex(P.G, x, y, flags)
    torch.cuda.synchronize()
    return y.cpu().numpy()


@pytest.mark.parametrize("name,m", CASES, ids=[c[0] for c in CASES])
def test_rowell_spmv_parity(name, m):
    P = Pair(m, 64)
    rng = np.random.default_rng(5)
    xh = rng.uniform(-1, 1, P.n) * 10.0 ** rng.uniform(-3, 3, P.n)
    x = torch.from_numpy(xh).cuda()
    for mp in (np.zeros(P.t.ntiles, np.uint8), P.tile_map(1), P.tile_map(2, (0, 0, 1)),
               P.tile_map(3, (0, 1, 0)), P.tile_map(4, (0.2, 0.3, 0.5))):
        y = _run(P, x, mp)
        want = oracle.mixed_spmv(P.A, P.t, mp, xh)
        den = P.abs_sum(mp, xh)
        assert np.all(np.isfinite(y))
        assert row_rel_err(y, want, den).max() <= (TOL64 if not mp.any() else TOLMIX)
        yd = _run(P, x, mp, flags=evocg.SPMV_DIRECT)
        assert row_rel_err(y, yd, den).max() <= 1e-12
    # a per-column-block map (what the controllers write)
    cb = np.random.default_rng(2).integers(0, 3, P.t.nrb).astype(np.uint8)
    y = _run(P, x, cb, evocg.MAP_PER_COLBLOCK)
    tm = cb[P.t.tileColIdx]
    assert row_rel_err(y, oracle.mixed_spmv(P.A, P.t, tm, xh), P.abs_sum(tm, xh)).max() <= TOLMIX


def test_rowell_spmv_parity_full_size():
    w = W.workload(4)
    P = Pair((w.n, w.rp, w.ci, w.v), w.T)
    xh = np.random.default_rng(4).uniform(-1, 1, P.n)
    x = torch.from_numpy(xh).cuda()
    for mp, tol in ((np.zeros(P.t.ntiles, np.uint8), TOL64), (P.tile_map(4), TOLMIX)):
        y = _run(P, x, mp)
        want = oracle.mixed_spmv(P.A, P.t, mp, xh)
        assert row_rel_err(y, want, P.abs_sum(mp, xh)).max() <= tol


def test_rowell_fp64_variants_in_a_solve():
    """A banded solve with the FP64 finish runs the kernel's all-FP64 and p.q variants: it
    reaches rtol in the oracle's FP64 residual with an iteration count within 3% of the
    oracle's (same map)."""
    n, rp, ci, v = W.banded_spd(20000, 6, band=700)
    P = Pair((n, rp, ci, v), 64)
    mp = P.tile_map(6)
    evocg.set_tile_precision(P.G, mp)
    b = np.random.default_rng(3).standard_normal(n)
    x = np.empty(n)
    info = evocg.cg_solve(P.G, b, x, 1e-8, 20000, False, None, True)
    ref = oracle.cg(P.A, P.t, b, 1e-8, 20000, tile_map=mp, finish_fp64=True)
    assert info["status"] == evocg.OK == ref["status"], info
    assert abs(info["iters"] - ref["iters"]) <= max(2, 0.03 * ref["iters"]), (info["iters"], ref["iters"])
    assert oracle.true_residual(P.A, b, x) <= 1e-8


def test_rowell_row_order_depends_only_on_the_map():
    """Setting a per-tile map puts every row's slots in (precision, column) order, whatever
    order an earlier map left: the same map gives bit-identical products before and after
    other maps (per tile and per column block), and the all-FP64 map restores column order
    (its products equal the ones taken before any mixed map, bit for bit)."""
    P = Pair(W.banded_spd(20000, 6, band=700), 64)
    xh = np.random.default_rng(9).standard_normal(P.n)
    x = torch.from_numpy(xh).cuda()
    z = np.zeros(P.t.ntiles, np.uint8)
    y64 = _run(P, x, z)
    a, b = P.tile_map(11), P.tile_map(12, (0.2, 0.3, 0.5))
    ya = _run(P, x, a)
    _run(P, x, b)
    _run(P, x, np.random.default_rng(3).integers(0, 3, P.t.nrb).astype(np.uint8), evocg.MAP_PER_COLBLOCK)
    assert np.array_equal(_run(P, x, a).view(np.uint64), ya.view(np.uint64))
    assert np.array_equal(_run(P, x, z).view(np.uint64), y64.view(np.uint64))
