"""GPU parity: tile layout (bit-exact), rounding (bit-exact) and the mixed-precision SpMV
(per-row relative error against the oracle) through the C ABI."""
import numpy as np
import pytest

import oracle
from helpers import Pair, row_rel_err
from test_host_layout import same_csc
from mixed_precision_sparse_gb300 import evocg
from mixed_precision_sparse_gb300 import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL64 = 1e-12   # all-FP64 map
TOLMIX = 1e-6   # mixed maps


def _small_cases():
    return [
        ("lap2d_64", W.laplace2d_5pt(64), 16),
        ("lap2d_ragged", W.laplace2d_5pt(37, 29), 16),
        ("rand61_t16", W.random_spd_small(61, 1, 0.2), 16),
        ("rand100_t32", W.random_spd_small(100, 2, 0.1), 32),
        ("rand200_t64", W.random_spd_small(200, 3, 0.04), 64),
        ("diff3d_20", W.diffusion3d_7pt(20, 4), 32),
        ("fe3d_12", W.fe3d_q1_27pt(12, 5), 32),
        ("aniso_70", W.aniso2d_q1_9pt(70), 32),
        ("banded_20k", W.banded_spd(20000, 6, band=700), 64),
        ("tiny_n5", W.random_spd_small(5, 7, 0.5), 16),
    ]


CASES = _small_cases()


@pytest.mark.parametrize("pad", [1, 2])
@pytest.mark.parametrize("name,m,T", CASES, ids=[c[0] for c in CASES])
def test_layout_bit_exact(name, m, T, pad):
    """The device-resident structure, copied back and written as EvoCG's Tile-CSC, equals the
    oracle's independent Tile-CSC bit for bit (both paddings)."""
    P = Pair(m, T)
    same_csc(P.G.export_csc(pad), oracle.Tiles(P.A, T, pad))


def test_rounding_bit_exact():
    rng = np.random.default_rng(11)
    x = np.ldexp(rng.uniform(1, 2, 200000), rng.integers(-160, 140, 200000)) * rng.choice([-1, 1], 200000)
    f = rng.uniform(-1e3, 1e3, 20000).astype(np.float32).astype(np.float64)
    ulp = np.spacing(np.abs(f).astype(np.float32)).astype(np.float64)
    bv = ((rng.integers(1, 0x7F7F, 20000).astype(np.uint32) << 16).view(np.float32)).astype(np.float64)
    ulpb = np.ldexp(1.0, np.frexp(bv)[1] - 8)
    x = np.concatenate([x, f + ulp / 2, f - ulp / 2, bv + ulpb / 2, bv - ulpb / 2,
                        [0.0, -0.0, np.inf, -np.inf, np.nan, 1e-320, 3.5e38, -3.5e38]])
    o32 = np.empty(x.size, np.float32)
    o16 = np.empty(x.size, np.uint16)
    evocg.round_fp(x, o32, o16)
    w32 = oracle.round_f32(x)
    w16 = oracle.round_bf16_bits(x)
    nan = np.isnan(x)
    assert np.array_equal(o32[~nan].view(np.uint32), w32[~nan].view(np.uint32))
    assert np.array_equal(o16[~nan], w16[~nan])
    assert np.all(np.isnan(o32[nan])) and np.all((o16[nan] & 0x7FFF) > 0x7F80)


def _check_spmv(P, tile_map, x, tol, dev=True):
    evocg.set_tile_precision(P.G, tile_map if tile_map is not None else np.zeros(P.t.ntiles, np.uint8))
    want = oracle.mixed_spmv(P.A, P.t, tile_map, x)
    if dev:
        xd = torch.from_numpy(x).cuda()
        yd = torch.full((P.n,), np.nan, dtype=torch.float64, device="cuda")
        evocg.spmv(P.G, xd, yd)
        torch.cuda.synchronize()
        y = yd.cpu().numpy()
    else:
        y = np.full(P.n, np.nan)
        evocg.spmv(P.G, x, y)
    err = row_rel_err(y, want, P.abs_sum(tile_map, x))
    assert np.all(np.isfinite(y))
    assert err.max() <= tol, (err.max(), int(err.argmax()))
    return err.max()


@pytest.mark.parametrize("name,m,T", CASES, ids=[c[0] for c in CASES])
def test_spmv_parity_small(name, m, T):
    P = Pair(m, T)
    rng = np.random.default_rng(3)
    x = rng.uniform(-1, 1, P.n) * 10.0 ** rng.uniform(-3, 3, P.n)
    _check_spmv(P, None, x, TOL64)
    for seed, fr in [(1, (0.4, 0.4, 0.2)), (2, (0, 1, 0)), (3, (0, 0, 1)), (4, (0.2, 0.3, 0.5))]:
        _check_spmv(P, P.tile_map(seed, fr), x, TOLMIX)


def test_spmv_mixed_is_exact_on_representable_inputs():
    """Values 4 and -1 and integers |x| <= 256 are exact in every format: any map must give
    exactly A x, the same bits on both sides."""
    P = Pair(W.laplace2d_5pt(64), 16)
    x = np.random.default_rng(0).integers(-256, 257, P.n).astype(np.float64)
    for seed in range(3):
        mp = P.tile_map(seed)
        evocg.set_tile_precision(P.G, mp)
        y = np.empty(P.n)
        evocg.spmv(P.G, x, y)
        assert np.array_equal(y, oracle.mixed_spmv(P.A, P.t, mp, x))


def test_spmv_host_pointers_and_colblock_map():
    P = Pair(W.diffusion3d_7pt(16, 9), 32)
    x = np.random.default_rng(1).standard_normal(P.n)
    _check_spmv(P, P.tile_map(7), x, TOLMIX, dev=False)
    cb = np.random.default_rng(2).integers(0, 3, P.t.nrb).astype(np.uint8)
    evocg.set_tile_precision(P.G, cb, evocg.MAP_PER_COLBLOCK)
    tm = cb[P.t.tileColIdx]
    assert np.array_equal(evocg.get_tile_precision(P.G), tm)
    y = np.empty(P.n)
    evocg.spmv(P.G, x, y)
    want = oracle.mixed_spmv(P.A, P.t, tm, x)
    assert row_rel_err(y, want, P.abs_sum(tm, x)).max() <= TOLMIX


def test_spmv_edge_cases():
    # empty rows, a column block with no tiles, n not a multiple of T, n < T
    M = np.zeros((45, 45))
    M[np.arange(45), np.arange(45)] = np.arange(1, 46)
    M[7] = 0.0
    M[:, 20:32] = 0.0
    M[44, 0] = M[0, 44] = -0.5
    for T in (16, 32, 64):
        P = Pair(W.dense_to_csr(M), T)
        x = np.random.default_rng(T).standard_normal(45)
        for mp in (None, P.tile_map(1), P.tile_map(2, (0, 0, 1))):
            _check_spmv(P, mp, x, TOL64 if mp is None else TOLMIX)
    # diagonal-only matrix (one tile per row block), values across the FP64 range
    d = 10.0 ** np.random.default_rng(5).uniform(-200, 200, 300)
    P = Pair(W.dense_to_csr(np.diag(d)), 32)
    x = np.random.default_rng(6).standard_normal(300)
    _check_spmv(P, None, x, TOL64)


def test_spmv_rejects_bad_maps():
    P = Pair(W.laplace2d_5pt(20), 16)
    with pytest.raises(evocg.EvocgError) as e:
        evocg.set_tile_precision(P.G, np.full(P.t.ntiles, 3, np.uint8))
    assert e.value.code == evocg.EINVAL
    with pytest.raises(evocg.EvocgError) as e:
        evocg.set_tile_precision(P.G, np.zeros(P.t.ntiles + 1, np.uint8))
    assert e.value.code == evocg.EINVAL
    n, rp, ci, v = W.laplace2d_5pt(8)
    with pytest.raises(evocg.EvocgError) as e:
        evocg.tile_build(n, rp, ci, v, 48)
    assert e.value.code == evocg.EINVAL
    ci2 = ci.copy()
    ci2[1], ci2[2] = ci2[2], ci2[1]  # unsorted row
    with pytest.raises(evocg.EvocgError):
        evocg.tile_build(n, rp, ci2, v, 16)
    v2 = v.copy()
    v2[3] = np.nan
    with pytest.raises(evocg.EvocgError):
        evocg.tile_build(n, rp, ci, v2, 16)


@pytest.mark.parametrize("cfg", [2, 3, 5, 4])
def test_spmv_parity_full_size(cfg):
    """Full-size workloads in the benchmark's launch configuration: the uploaded structure
    against the oracle's Tile-CSC, then every row of the SpMV."""
    w = W.workload(cfg)
    P = Pair((w.n, w.rp, w.ci, w.v), w.T)
    same_csc(P.G.export_csc(1), P.t)
    x = np.random.default_rng(cfg).uniform(-1, 1, P.n)
    _check_spmv(P, None, x, TOL64)
    _check_spmv(P, P.tile_map(cfg), x, TOLMIX)


@pytest.mark.parametrize("name,m,T", CASES + [
    ("dense_t32", W.dense_to_csr(np.random.default_rng(0).standard_normal((100, 100)) + 200 * np.eye(100)), 32),
    ("dense_t64", W.dense_to_csr(np.random.default_rng(1).standard_normal((200, 200)) + 300 * np.eye(200)), 64),
], ids=[c[0] for c in CASES] + ["dense_t32", "dense_t64"])
def test_spmv_kernels_agree(name, m, T):
    """The panel kernel (the default for tiles of 16 and 32) and the direct kernel sum the same
    exactly rounded-operand products in different orders: they agree to rounding, and each
    matches the oracle. Dense tiles exercise the panel kernel's path for a tile larger than a
    stage; n not a multiple of T the partial last x segment."""
    P = Pair(m, T)
    rng = np.random.default_rng(5)
    x = torch.from_numpy(rng.uniform(-1, 1, P.n) * 10.0 ** rng.uniform(-3, 3, P.n)).cuda()
    for mp in (np.zeros(P.t.ntiles, np.uint8), P.tile_map(1), P.tile_map(2, (0, 0, 1)), P.tile_map(3, (0, 1, 0))):
        evocg.set_tile_precision(P.G, mp)
        ys = {}
        for k, flag in (("direct", evocg.SPMV_DIRECT), ("default", 0)):
            ys[k] = torch.full((P.n,), np.nan, dtype=torch.float64, device="cuda")
            evocg.spmv_ex(P.G, x, ys[k], flag)
        torch.cuda.synchronize()
        want = oracle.mixed_spmv(P.A, P.t, mp, x.cpu().numpy())
        den = P.abs_sum(mp, x.cpu().numpy())
        assert row_rel_err(ys["default"].cpu().numpy(), ys["direct"].cpu().numpy(), den).max() <= 1e-12
        for k in ys:
            err = row_rel_err(ys[k].cpu().numpy(), want, den)
            assert err.max() <= (TOL64 if not mp.any() else TOLMIX), k


def test_spmv_misaligned_x():
    """An x that is not 16-byte aligned cannot be a bulk-copy source: the panel kernel copies
    its FP64 segments entry by entry instead, with the same result bit for bit."""
    P = Pair(W.diffusion3d_7pt(16, 2), 32)
    for mp in (P.tile_map(4), np.zeros(P.t.ntiles, np.uint8)):
        evocg.set_tile_precision(P.G, mp)
        buf = torch.from_numpy(np.random.default_rng(9).standard_normal(P.n + 1)).cuda()
        xa = buf[1:]                       # 8 bytes past a 256-byte boundary
        xb = buf[1:].clone()               # aligned copy of the same values
        assert xa.data_ptr() % 16 == 8 and xb.data_ptr() % 16 == 0
        ya = torch.empty(P.n, dtype=torch.float64, device="cuda")
        yb = torch.empty_like(ya)
        evocg.spmv(P.G, xa, ya)
        evocg.spmv(P.G, xb, yb)
        torch.cuda.synchronize()
        assert torch.equal(ya.view(torch.int64), yb.view(torch.int64))
