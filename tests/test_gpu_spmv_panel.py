"""GPU parity of the panel SpMV kernel (tiles of 16 and 32) against the oracle: every row,
per-row relative error, on the small matrices, the edge cases and the full-size workloads."""
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

CASES = [
    ("lap2d_64", W.laplace2d_5pt(64), 16),
    ("lap2d_ragged", W.laplace2d_5pt(37, 29), 16),
    ("rand61_t16", W.random_spd_small(61, 1, 0.2), 16),
    ("rand100_t32", W.random_spd_small(100, 2, 0.1), 32),
    ("diff3d_20", W.diffusion3d_7pt(20, 4), 32),
    ("fe3d_12", W.fe3d_q1_27pt(12, 5), 32),
    ("aniso_70", W.aniso2d_q1_9pt(70), 32),
    ("tiny_n5", W.random_spd_small(5, 7, 0.5), 16),
    ("dense_t32", W.dense_to_csr(np.random.default_rng(0).standard_normal((100, 100)) + 200 * np.eye(100)), 32),
    ("wide_rows_t16", W.dense_to_csr(np.random.default_rng(1).standard_normal((70, 70)) + 100 * np.eye(70)), 16),
]


def _panel(P, x, mp, kind=evocg.MAP_PER_TILE):
    evocg.set_tile_precision(P.G, mp, kind)
    y = torch.full((P.n,), np.nan, dtype=torch.float64, device="cuda")
    evocg.spmv_ex(P.G, x, y, evocg.SPMV_PANEL)
    torch.cuda.synchronize()
    return y.cpu().numpy()


@pytest.mark.parametrize("name,m,T", CASES, ids=[c[0] for c in CASES])
def test_panel_spmv_parity(name, m, T):
    P = Pair(m, T)
    rng = np.random.default_rng(5)
    xh = rng.uniform(-1, 1, P.n) * 10.0 ** rng.uniform(-3, 3, P.n)
    x = torch.from_numpy(xh).cuda()
    for mp in (np.zeros(P.t.ntiles, np.uint8), P.tile_map(1), P.tile_map(2, (0, 0, 1)),
               P.tile_map(3, (0, 1, 0)), P.tile_map(4, (0.2, 0.3, 0.5))):
        y = _panel(P, x, mp)
        want = oracle.mixed_spmv(P.A, P.t, mp, xh)
        err = row_rel_err(y, want, P.abs_sum(mp, xh))
        assert np.all(np.isfinite(y))
        assert err.max() <= (TOL64 if not mp.any() else TOLMIX), (err.max(), int(err.argmax()))


def test_panel_spmv_colblock_map_and_edge_cases():
    P = Pair(W.diffusion3d_7pt(16, 9), 32)
    xh = np.random.default_rng(1).standard_normal(P.n)
    x = torch.from_numpy(xh).cuda()
    cb = np.random.default_rng(2).integers(0, 3, P.t.nrb).astype(np.uint8)
    y = _panel(P, x, cb, evocg.MAP_PER_COLBLOCK)
    tm = cb[P.t.tileColIdx]
    want = oracle.mixed_spmv(P.A, P.t, tm, xh)
    assert row_rel_err(y, want, P.abs_sum(tm, xh)).max() <= TOLMIX
    # empty rows, a column block with no tiles, n not a multiple of T, n < T
    M = np.zeros((45, 45))
    M[np.arange(45), np.arange(45)] = np.arange(1, 46)
    M[7] = 0.0
    M[:, 20:32] = 0.0
    M[44, 0] = M[0, 44] = -0.5
    for T in (16, 32):
        P = Pair(W.dense_to_csr(M), T)
        xh = np.random.default_rng(T).standard_normal(45)
        x = torch.from_numpy(xh).cuda()
        for mp in (np.zeros(P.t.ntiles, np.uint8), P.tile_map(1), P.tile_map(2, (0, 0, 1))):
            y = _panel(P, x, mp)
            want = oracle.mixed_spmv(P.A, P.t, mp, xh)
            assert row_rel_err(y, want, P.abs_sum(mp, xh)).max() <= (TOL64 if not mp.any() else TOLMIX)


@pytest.mark.parametrize("cfg", [2, 3, 5])
def test_panel_spmv_parity_full_size(cfg):
    w = W.workload(cfg)
    P = Pair((w.n, w.rp, w.ci, w.v), w.T)
    xh = np.random.default_rng(cfg).uniform(-1, 1, P.n)
    x = torch.from_numpy(xh).cuda()
    for mp, tol in ((np.zeros(P.t.ntiles, np.uint8), TOL64), (P.tile_map(cfg), TOLMIX)):
        y = _panel(P, x, mp)
        want = oracle.mixed_spmv(P.A, P.t, mp, xh)
        err = row_rel_err(y, want, P.abs_sum(mp, xh))
        assert err.max() <= tol, (err.max(), int(err.argmax()))


def test_lost_stage_wait_is_reported_and_the_context_stays_usable():
    """The panel kernel's stage waits are bounded in time. Under the test hook one warp
    withholds its first arrival, so its wait runs out (after 2 ms): the call returns
    EVOCG_ETIMEOUT instead of hanging, and the next call on the same handle is correct."""
    P = Pair(W.diffusion3d_7pt(16, 9), 32)
    mp = P.tile_map(3)
    evocg.set_tile_precision(P.G, mp)
    xh = np.random.default_rng(4).standard_normal(P.n)
    y = np.empty(P.n)
    with pytest.raises(evocg.EvocgError) as e:
        evocg.spmv_ex(P.G, xh, y, evocg.SPMV_PANEL | evocg.SPMV_TEST_LOST_WAIT)
    assert e.value.code == evocg.ETIMEOUT
    evocg.spmv_ex(P.G, xh, y, evocg.SPMV_PANEL)
    want = oracle.mixed_spmv(P.A, P.t, mp, xh)
    assert row_rel_err(y, want, P.abs_sum(mp, xh)).max() <= TOLMIX
