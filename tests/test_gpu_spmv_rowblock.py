"""GPU parity of the row-block SpMV kernel (tiles of 32) against the oracle: every row, per-row
relative error, on the small matrices, a matrix built for the kernel's less common paths, the
edge cases and the full-size workloads; and against the direct kernel to rounding."""
import numpy as np
import pytest

import oracle
from helpers import Pair, many_tiles_t32, row_rel_err
from mixed_precision_sparse_gb300 import evocg
from mixed_precision_sparse_gb300 import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL64 = 1e-12
TOLMIX = 1e-6

CASES = [
    ("rand100", W.random_spd_small(100, 2, 0.1)),
    ("diff3d_20", W.diffusion3d_7pt(20, 4)),
    ("fe3d_12", W.fe3d_q1_27pt(12, 5)),
    ("aniso_70", W.aniso2d_q1_9pt(70)),
    ("lap2d_ragged", W.laplace2d_5pt(37, 29)),
    ("tiny_n5", W.random_spd_small(5, 7, 0.5)),
    ("dense_100", W.dense_to_csr(np.random.default_rng(0).standard_normal((100, 100)) + 200 * np.eye(100))),
    ("many_tiles", many_tiles_t32()),
]


def _run(P, x, mp, kind=evocg.MAP_PER_TILE, flags=evocg.SPMV_ROWBLOCK):
    evocg.set_tile_precision(P.G, mp, kind)
    y = torch.full((P.n,), np.nan, dtype=torch.float64, device="cuda")
    evocg.spmv_ex(P.G, x, y, flags)
    torch.cuda.synchronize()
    return y.cpu().numpy()


@pytest.mark.parametrize("name,m", CASES, ids=[c[0] for c in CASES])
def test_rowblock_spmv_parity(name, m):
    P = Pair(m, 32)
    rng = np.random.default_rng(5)
    xh = rng.uniform(-1, 1, P.n) * 10.0 ** rng.uniform(-3, 3, P.n)
    x = torch.from_numpy(xh).cuda()
    for mp in (np.zeros(P.t.ntiles, np.uint8), P.tile_map(1), P.tile_map(2, (0, 0, 1)),
               P.tile_map(3, (0, 1, 0)), P.tile_map(4, (0.2, 0.3, 0.5))):
        y = _run(P, x, mp)
        want = oracle.mixed_spmv(P.A, P.t, mp, xh)
        den = P.abs_sum(mp, xh)
        err = row_rel_err(y, want, den)
        assert np.all(np.isfinite(y))
        assert err.max() <= (TOL64 if not mp.any() else TOLMIX), (err.max(), int(err.argmax()))
        yd = _run(P, x, mp, flags=evocg.SPMV_DIRECT)
        assert row_rel_err(y, yd, den).max() <= 1e-12


def test_rowblock_spmv_colblock_map_and_edge_cases():
    P = Pair(many_tiles_t32(3), 32)
    xh = np.random.default_rng(1).standard_normal(P.n)
    x = torch.from_numpy(xh).cuda()
    for seed in range(3):
        cb = np.random.default_rng(seed).integers(0, 3, P.t.nrb).astype(np.uint8)
        y = _run(P, x, cb, evocg.MAP_PER_COLBLOCK)
        tm = cb[P.t.tileColIdx]
        want = oracle.mixed_spmv(P.A, P.t, tm, xh)
        assert row_rel_err(y, want, P.abs_sum(tm, xh)).max() <= TOLMIX
    # empty rows, a column block with no tiles, n not a multiple of 32, n < 32
    M = np.zeros((45, 45))
    M[np.arange(45), np.arange(45)] = np.arange(1, 46)
    M[7] = 0.0
    M[:, 20:32] = 0.0
    M[44, 0] = M[0, 44] = -0.5
    for mat in (M, M[:20, :20]):
        P = Pair(W.dense_to_csr(mat), 32)
        xh = np.random.default_rng(len(mat)).standard_normal(P.n)
        x = torch.from_numpy(xh).cuda()
        for mp in (np.zeros(P.t.ntiles, np.uint8), P.tile_map(1), P.tile_map(2, (0, 0, 1))):
            y = _run(P, x, mp)
            want = oracle.mixed_spmv(P.A, P.t, mp, xh)
            assert row_rel_err(y, want, P.abs_sum(mp, xh)).max() <= (TOL64 if not mp.any() else TOLMIX)


@pytest.mark.parametrize("cfg", [2, 3, 5])
def test_rowblock_spmv_parity_full_size(cfg):
    w = W.workload(cfg)
    P = Pair((w.n, w.rp, w.ci, w.v), w.T)
    xh = np.random.default_rng(cfg).uniform(-1, 1, P.n)
    x = torch.from_numpy(xh).cuda()
    for mp, tol in ((np.zeros(P.t.ntiles, np.uint8), TOL64), (P.tile_map(cfg), TOLMIX)):
        y = _run(P, x, mp)
        want = oracle.mixed_spmv(P.A, P.t, mp, xh)
        err = row_rel_err(y, want, P.abs_sum(mp, xh))
        assert err.max() <= tol, (err.max(), int(err.argmax()))


def test_rowblock_fp64_variants_in_a_solve():
    """A solve with the FP64 finish runs the kernel's all-FP64 variants (the restart product
    q = A x and the FP64 true residual) besides the mixed one, here on a matrix whose row
    blocks have single-entry tiles: the solve reaches rtol in the oracle's FP64 residual."""
    n, rp, ci, v = W.aniso2d_q1_9pt(70)
    P = Pair((n, rp, ci, v), 32)
    evocg.set_tile_precision(P.G, P.tile_map(2, (0.2, 0.3, 0.5)))
    b = np.random.default_rng(3).uniform(-1, 1, n)
    x = np.empty(n)
    info = evocg.cg_solve(P.G, b, x, 1e-8, 20000, True, None, True)
    assert info["status"] == evocg.OK, info
    assert oracle.true_residual(P.A, b, x) <= 1e-8
    for it in range(2):   # and the all-FP64 product alone, against the oracle
        xh = np.random.default_rng(it).standard_normal(n)
        y = _run(P, torch.from_numpy(xh).cuda(), np.zeros(P.t.ntiles, np.uint8))
        want = oracle.mixed_spmv(P.A, P.t, None, xh)
        assert row_rel_err(y, want, P.abs_sum(np.zeros(P.t.ntiles, np.uint8), xh)).max() <= TOL64
