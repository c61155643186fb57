"""The seeded synthetic workloads against the recipes they implement: sizes, exact symmetry,
the value law of each construction, and reproducibility from the seed. These generators
stand in for the SuiteSparse SPD matrices of EvoCG §4.1 (not available here); both the
oracle and the GPU library are fed from them."""
import numpy as np
import pytest

from mixed_precision_sparse_gb300 import workloads as W

SIZES = {1: (4096, 20224), 2: (2097152, 14581760), 3: (884736, 23393656),
         4: (4000000, 67999928), 5: (16777216, 150945796)}
SETTINGS = {1: (16, 1e-10, 20000, False, "static"), 2: (32, 1e-8, 10000, True, "threshold"),
            3: (32, 1e-8, 10000, True, "mlp"), 4: (64, 1e-8, 10000, False, "static"),
            5: (32, 1e-8, 5000, True, "static")}


def _rows(w):
    return np.repeat(np.arange(w.n, dtype=np.int64), np.diff(w.rp))


def _asymmetry_ulps(w):
    """Largest |a_ij - a_ji| in units of the last place of |a_ij| (None when the pattern is
    not symmetric): the entries sorted by (row, col) and by (col, row) pair a_ij with a_ji."""
    r, c = _rows(w), w.ci.astype(np.int64)
    o1 = np.lexsort((c, r))
    o2 = np.lexsort((r, c))
    if not (np.array_equal(r[o1], c[o2]) and np.array_equal(c[o1], r[o2])):
        return None
    a, t = w.v[o1], w.v[o2]
    return float(np.max(np.abs(a - t) / np.spacing(np.abs(a))))


def _diag(w):
    r = _rows(w)
    d = np.zeros(w.n)
    on = w.ci == r
    d[r[on]] = w.v[on]
    return d, on


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_full_size_and_settings(cfg):
    w = W.workload(cfg)
    assert (w.n, w.nnz) == SIZES[cfg]
    assert (w.T, w.rtol, w.maxit, w.jacobi, w.ctrl) == SETTINGS[cfg]
    assert w.b.shape == (w.n,) and np.all(np.isfinite(w.b)) and np.all(np.isfinite(w.v))
    assert np.all(np.diff(w.rp) >= 1)
    d, on = _diag(w)
    assert np.count_nonzero(on) == w.n and np.all(d > 0)      # a positive diagonal everywhere
    if cfg == 1:
        assert set(np.unique(w.v)) == {4.0, -1.0}
        assert np.array_equal(w.b, W.csr_matvec(w.n, w.rp, w.ci, w.v, w.extra["x_true"]))
    if cfg == 4:
        r = _rows(w)
        off = ~on
        assert np.all(np.abs(r[off] - w.ci[off]) <= 4096)      # inside the band
        absum = np.bincount(r[off], weights=np.abs(w.v[off]), minlength=w.n)
        assert np.allclose(d, 1.05 * absum, rtol=1e-12, atol=0)   # 1.05 x row abs-sum


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_symmetry_and_reproducibility(cfg):
    """Exactly symmetric where both triangles are produced by the same operations (the
    Laplacian, the face-coefficient diffusion, the mirrored banded entries); within 2 units
    in the last place where floating point orders them differently: D A D computes
    (d_i a_ij) d_j, and the anisotropic stencil sums its element contributions in another
    order for the opposite offset."""
    w = W.workload(cfg, scale=0.125 if cfg > 1 else 1.0)
    ulps = _asymmetry_ulps(w)
    assert ulps is not None                                   # symmetric pattern
    assert ulps == 0.0 if cfg in (1, 2, 4) else ulps <= 2.0
    w2 = W.workload(cfg, scale=0.125 if cfg > 1 else 1.0)
    assert np.array_equal(w.rp, w2.rp) and np.array_equal(w.ci, w2.ci)
    assert np.array_equal(w.v.view(np.uint64), w2.v.view(np.uint64))
    assert np.array_equal(w.b.view(np.uint64), w2.b.view(np.uint64))


def test_diffusion_value_law():
    """7-point finite volumes: off-diagonals -k with k = 10^U[-2, 2]; the diagonal is the sum
    of the cell's six face coefficients, so it exceeds the off-diagonal magnitudes by the
    boundary faces only (interior rows: equal to within rounding)."""
    w = W.workload(2, scale=0.125)
    N = w.extra["grid"]
    r = _rows(w)
    d, on = _diag(w)
    k = -w.v[~on]
    assert np.all(k >= 1e-2) and np.all(k <= 1e2)
    offsum = np.bincount(r[~on], weights=k, minlength=w.n)
    deg = np.bincount(r[~on], minlength=w.n)
    inner = deg == 6
    assert np.allclose(d[inner], offsum[inner], rtol=1e-13)
    assert np.all(d[~inner] > offsum[~inner])                   # Dirichlet ghost faces
    assert w.n == N ** 3


def test_fe_scaling_law():
    """Q1 27-point stiffness + h^2 mass, then D A D with D = 10^U[-3, 0]: the unscaled
    diagonal is 8/3 + 8 h^2 / 27, so d_i = sqrt(a_ii / that) lies in [1e-3, 1], and
    a_ij / (d_i d_j) recovers the unscaled stencil value of the offset."""
    w = W.workload(3, scale=0.125)
    N = w.extra["grid"]
    h = 1.0 / (N + 1)
    d, on = _diag(w)
    di = np.sqrt(d / (8.0 / 3.0 + h * h * 8.0 / 27.0))
    assert np.all(di >= 1e-3 * (1 - 1e-12)) and np.all(di <= 1.0 * (1 + 1e-12))
    r = _rows(w)
    c = w.ci.astype(np.int64)
    raw = w.v / (di[r] * di[c])
    vals = {0: 8 / 3 + h * h * 8 / 27, 1: 0.0 + h * h * 2 / 27, 2: -1 / 6 + h * h / 54,
            3: -1 / 12 + h * h / 216}
    dx = np.abs(c % N - r % N)
    dy = np.abs((c // N) % N - (r // N) % N)
    dz = np.abs(c // (N * N) - r // (N * N))
    m = (dx > 0).astype(int) + (dy > 0) + (dz > 0)
    want = np.array([vals[int(k)] for k in range(4)])[m]
    assert np.allclose(raw, want, rtol=1e-10, atol=1e-14)


def test_anisotropic_rows_sum_to_zero_inside():
    """-div(K grad u) annihilates constants: every row whose nine neighbours all exist sums
    to zero (to rounding); rows at the Dirichlet boundary sum to a positive number."""
    w = W.workload(5, scale=0.0625)
    r = _rows(w)
    s = np.bincount(r, weights=w.v, minlength=w.n)
    scale = np.bincount(r, weights=np.abs(w.v), minlength=w.n)
    full = np.diff(w.rp) == 9
    assert np.all(np.abs(s[full]) <= 1e-13 * scale[full])
    assert np.all(s[~full] > 0)
