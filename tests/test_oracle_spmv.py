"""Pins of the oracle's SpMV, plain and mixed-precision, against results fixed outside it:
dense brute force, exact integer products, and exact rational sums of exactly rounded terms."""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle
from mixed_precision_sparse_gb300 import workloads as W


def _csr(m):
    return oracle.CSR(*m)


@pytest.mark.parametrize("n,seed", [(7, 1), (33, 2), (64, 3)])
def test_csr_spmv_matches_dense(n, seed):
    m = W.random_spd_small(n, seed, 0.4)
    A = _csr(m)
    x = np.random.default_rng(seed).standard_normal(n)
    want = W.csr_to_dense(*m) @ x
    got = oracle.csr_spmv(A, x)
    scale = np.abs(W.csr_to_dense(*m)) @ np.abs(x)
    assert np.all(np.abs(got - want) <= 1e-14 * scale)


def test_all_fp64_map_is_plain_csr_spmv():
    m = W.aniso2d_q1_9pt(40)
    A = _csr(m)
    t = oracle.Tiles(A, 32)
    x = np.random.default_rng(0).uniform(-1, 1, A.n)
    y1 = oracle.mixed_spmv(A, t, np.zeros(t.ntiles, np.uint8), x)
    y2 = oracle.csr_spmv(A, x)
    assert np.array_equal(y1, y2)
    assert np.array_equal(oracle.mixed_spmv(A, t, None, x), y2)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_mixed_spmv_exact_on_representable_inputs(seed):
    """The 64x64 Laplacian holds 4 and -1, exact in BF16 and FP32, and integers |x| <= 256
    are exact in both: every precision map must give exactly A x (integer arithmetic)."""
    m = W.laplace2d_5pt(64)
    A = _csr(m)
    t = oracle.Tiles(A, 16)
    rng = np.random.default_rng(seed)
    x = rng.integers(-256, 257, A.n)
    want = W.csr_to_dense(*m).astype(np.int64) @ x
    trow = t.tile_rows()
    for fr in [(1, 0, 0), (0, 1, 0), (0, 0, 1), (0.4, 0.4, 0.2)]:
        mp = W.tile_map(trow, t.tileColIdx, t.nrb, seed, fr)
        got = oracle.mixed_spmv(A, t, mp, x.astype(np.float64))
        assert np.array_equal(got, want.astype(np.float64))


def _bf16_round_table(v):
    """Nearest BF16 value (ties to even pattern) by exhaustive search, for one float."""
    bits = np.arange(0, 0x7F80, dtype=np.uint32)
    vals = (bits << 16).view(np.float32).astype(np.float64)
    a = abs(v)
    i = np.searchsorted(vals, a)
    if i < len(vals) and vals[i] == a:
        r = vals[i]
    else:
        lo, hi = vals[i - 1], vals[i]
        if a - lo < hi - a or (a - lo == hi - a and bits[i - 1] % 2 == 0):
            r = lo
        else:
            r = hi
    return math.copysign(r, v)


@pytest.mark.parametrize("T,seed", [(16, 5), (32, 6)])
def test_mixed_spmv_exact_rational(T, seed):
    """Each term is rebuilt exactly (the column exponent from frexp, FP32 rounding from
    numpy's cast, BF16 from the exhaustive table), summed in exact rationals, and the
    oracle's FP64 row sum must lie within its own summation error of that exact sum."""
    m = W.random_spd_small(45, seed, 0.3)
    n, rp, ci, v = m
    rng = np.random.default_rng(seed)
    v = v * 10.0 ** rng.uniform(-6, 6, v.size)          # spread the magnitudes
    A = oracle.CSR(n, rp, ci, v)
    t = oracle.Tiles(A, T)
    x = rng.standard_normal(n) * 10.0 ** rng.uniform(-3, 3, n)
    mp = W.tile_map(t.tile_rows(), t.tileColIdx, t.nrb, seed)
    got = oracle.mixed_spmv(A, t, mp, x)
    colmax = np.zeros(n)
    np.maximum.at(colmax, ci, np.abs(v))
    for i in range(n):
        exact, absum = Fraction(0), Fraction(0)
        for k in range(rp[i], rp[i + 1]):
            j = int(ci[k])
            tt = int(np.nonzero((t.tile_rows() == i // T) & (t.tileColIdx == j // T))[0][0])
            p = int(mp[tt])
            if p == 0:
                term = Fraction(float(v[k] * x[j]))          # the FP64 product, rounded once
            else:
                e = math.frexp(colmax[j])[1] - 1
                s = math.ldexp(v[k], -e)
                if p == 1:
                    at, xt = float(np.float32(s)), float(np.float32(x[j]))
                else:
                    at, xt = _bf16_round_table(s), _bf16_round_table(x[j])
                term = Fraction(at) * Fraction(xt) * Fraction(2) ** e
            exact += term
            absum += abs(term)
        nterms = int(rp[i + 1] - rp[i])
        err = abs(Fraction(float(got[i])) - exact)
        assert err <= Fraction(nterms) * Fraction(2) ** -52 * absum + Fraction(2) ** -1074


def test_mixed_spmv_perturbation_size():
    """Eq. 2/5 perturbation: an all-BF16 map changes A x by at most about 2^-8 per term
    (value and x each rounded once), an all-FP32 map by about 2^-23."""
    m = W.diffusion3d_7pt(8, 3)
    A = _csr(m)
    t = oracle.Tiles(A, 32)
    x = np.random.default_rng(1).uniform(-1, 1, A.n)
    y = oracle.csr_spmv(A, x)
    absum = np.abs(W.csr_to_dense(*m)) @ np.abs(x)
    for p, bound in [(1, 2.0 ** -23), (2, 2.0 ** -7)]:
        yt = oracle.mixed_spmv(A, t, np.full(t.ntiles, p, np.uint8), x)
        rel = np.abs(yt - y) / absum
        assert rel.max() <= bound * 1.01
        assert rel.max() > bound / 64  # the rounding is really applied
