"""The library's host tile builder against the oracle's, bit for bit, without a GPU
(evocg_tile_layout_host: the builder evocg_tile_build runs before it uploads). The GPU suite
checks the uploaded copy the same way."""
import numpy as np
import pytest

import oracle
from mixed_precision_sparse_gb300 import build, evocg
from mixed_precision_sparse_gb300 import workloads as W


def _cases():
    yield "lap2d_16", W.laplace2d_5pt(16), 16
    yield "lap2d_ragged", W.laplace2d_5pt(37, 29), 16
    yield "rand61_t16", W.random_spd_small(61, 1, 0.2), 16
    yield "rand100_t32", W.random_spd_small(100, 2, 0.1), 32
    yield "rand200_t64", W.random_spd_small(200, 3, 0.04), 64
    yield "diff3d_20", W.diffusion3d_7pt(20, 4), 32
    yield "fe3d_12", W.fe3d_q1_27pt(12, 5), 32
    yield "aniso_70", W.aniso2d_q1_9pt(70), 32
    yield "banded_20k", W.banded_spd(20000, 6, band=700), 64
    yield "tiny_n5", W.random_spd_small(5, 7, 0.5), 16
    yield "dense_t64", W.dense_to_csr(np.random.default_rng(1).standard_normal((130, 130)) + 300 * np.eye(130)), 64


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()


def _same(h, t):
    assert (h["ntiles"], h["nslots"]) == (t.ntiles, t.nslots)
    for k in ["tileRowPtr", "tileColIdx", "tileNnzOff", "rowMask", "tileWidth", "colIdx", "v16",
              "colExp"]:
        assert np.array_equal(h[k], getattr(t, k)), k
    assert np.array_equal(h["v64"].view(np.uint64), t.v64.view(np.uint64))
    assert np.array_equal(h["v32"].view(np.uint32), t.v32.view(np.uint32))


@pytest.mark.parametrize("name,m,T", list(_cases()), ids=[c[0] for c in _cases()])
def test_host_builder_equals_oracle(name, m, T):
    n, rp, ci, v = m
    _same(evocg.tile_layout_host(n, rp, ci, v, T), oracle.Tiles(oracle.CSR(n, rp, ci, v), T))


@pytest.mark.parametrize("cfg", [2, 4])
def test_host_builder_equals_oracle_full_size(cfg):
    """The 128^3 diffusion (stencil tiles) and the 4M banded workload (sparse 64 x 64 tiles
    with second levels)."""
    w = W.workload(cfg)
    _same(evocg.tile_layout_host(w.n, w.rp, w.ci, w.v, w.T),
          oracle.Tiles(oracle.CSR(w.n, w.rp, w.ci, w.v), w.T))


def test_host_builder_rejects_bad_input():
    n, rp, ci, v = W.laplace2d_5pt(8)
    with pytest.raises(evocg.EvocgError):
        evocg.tile_layout_host(n, rp, ci, v, 24)                 # tile sizes are 16, 32, 64
    v2 = np.array(v, copy=True)
    v2[3] = np.inf
    with pytest.raises(evocg.EvocgError):
        evocg.tile_layout_host(n, rp, ci, v2, 16)                # values must be finite
    ci2 = np.array(ci, copy=True)
    ci2[1], ci2[2] = ci2[2], ci2[1]
    with pytest.raises(evocg.EvocgError):
        evocg.tile_layout_host(n, rp, ci2, v, 16)                # columns ascending per row


@pytest.mark.parametrize("name,m,T", list(_cases()), ids=[c[0] for c in _cases()])
@pytest.mark.parametrize("warps", [1, 7, 2432])
def test_staged_plan_passes_its_checks(name, m, T, warps):
    """The staged SpMV's plan, built as the library builds it, passes the checks the library
    applies before using it, for one warp, a few warps, and the 128^3 solve's 2432 consumer
    warps (more warps than row blocks leaves warps without work)."""
    n, rp, ci, v = m
    nb, ok = evocg.staged_plan_host(n, rp, ci, v, T, warps)
    assert ok and nb >= (1 if n > 0 else 0)


@pytest.mark.parametrize("cfg", [1, 2, 3])
def test_staged_plan_of_the_stencil_workloads(cfg):
    w = W.workload(cfg)
    for warps in (1216 * 2, 152 * 4 * 4):   # the T = 32 and T = 16 kernels' consumer warps
        nb, ok = evocg.staged_plan_host(w.n, w.rp, w.ci, w.v, w.T, warps)
        assert ok and nb > 0
    if cfg == 2:   # the 128^3 solve's plan: 65,294 batches of at most 16 tiles
        nb, _ = evocg.staged_plan_host(w.n, w.rp, w.ci, w.v, w.T, 2432)
        assert 423936 / 16 <= nb <= 423936


def test_empty_matrix():
    z64, z32, zf = np.zeros(1, np.int64), np.zeros(0, np.int32), np.zeros(0)
    h = evocg.tile_layout_host(0, z64, z32, zf, 16)
    assert (h["ntiles"], h["nslots"]) == (0, 0) and list(h["tileRowPtr"]) == [0]
    assert evocg.staged_plan_host(0, z64, z32, zf, 32, 4) == (0, True)
