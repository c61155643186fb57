"""The library's tile builder against the oracle's, bit for bit, without a GPU: the Tile-CSC
of EvoCG Fig. 4 written from the library's builder (evocg_tile_csc_host) equals the oracle's
independent Tile-CSC builder for both paddings; the library's own slot-major interior
(evocg_tile_layout_host, the arrays the SpMV kernels read) holds exactly the CSR entries. The
GPU suite checks the uploaded copy the same way (evocg_tiles_export_csc)."""
import numpy as np
import pytest

import oracle
from helpers import many_tiles_t32, rowblock_counts
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


def same_csc(h, t):
    """Library Tile-CSC arrays h against the oracle's Tiles t, bit for bit."""
    assert (h["ntiles"], h["nnz_p"]) == (t.ntiles, t.nnz_p)
    for k in ["tileRowPtr", "tileColIdx", "tileNnzOff", "colPtr", "rowIdx", "v16", "colExp"]:
        assert np.array_equal(h[k], getattr(t, k)), k
    assert np.array_equal(h["v64"].view(np.uint64), t.v64.view(np.uint64))
    assert np.array_equal(h["v32"].view(np.uint32), t.v32.view(np.uint32))


@pytest.mark.parametrize("pad", [1, 2])
@pytest.mark.parametrize("name,m,T", list(_cases()), ids=[c[0] for c in _cases()])
def test_host_tile_csc_equals_oracle(name, m, T, pad):
    n, rp, ci, v = m
    same_csc(evocg.tile_csc_host(n, rp, ci, v, T, pad), oracle.Tiles(oracle.CSR(n, rp, ci, v), T, pad))


@pytest.mark.parametrize("cfg", [2, 4])
def test_host_tile_csc_equals_oracle_full_size(cfg):
    """The 128^3 diffusion (stencil tiles) and the 4M banded workload (sparse 64 x 64 tiles)."""
    w = W.workload(cfg)
    same_csc(evocg.tile_csc_host(w.n, w.rp, w.ci, w.v, w.T, 1),
             oracle.Tiles(oracle.CSR(w.n, w.rp, w.ci, w.v), w.T, 1))


def test_host_tile_csc_fig4b():
    """The library reproduces the Fig. 4(b) fragment (colPtr 0, 4, 6 ... x, x+2; column 0
    padded with the sentinel row index R) from its own builder."""
    from test_oracle_tiles import fig4b_matrix
    g, T, (n, rp, ci, v) = fig4b_matrix()
    h = evocg.tile_csc_host(n, rp, ci, v, T, int(g["pad"]))
    assert list(h["colPtr"][0][:3]) == [int(s) for s in g["colPtr_head"].split()]
    assert list(h["colPtr"][0][-2:]) == [int(s) for s in g["colPtr_tail"].split()]
    assert list(h["rowIdx"]) == [int(s) for s in g["rowIdx"].split()]


def slot_layout_holds_the_csr(h, n, rp, ci, v, T):
    """The kernels' slot-major interior (row mask, width, w x h slots, pads at local column T)
    rebuilt into CSR with numpy equals the input; every pad is +0 in all three streams. A tile
    with more than one slot starts on a multiple of 16 slots and is followed by pads up to a
    multiple of 16; every row block's slots start on a multiple of 16."""
    rows, cols, vals = [], [], []
    trow = np.repeat(np.arange(len(h["tileRowPtr"]) - 1), np.diff(h["tileRowPtr"]))
    first = h["tileNnzOff"][h["tileRowPtr"][:-1][np.diff(h["tileRowPtr"]) > 0]]
    assert np.all(first % 16 == 0)
    real = np.zeros(h["nslots"], bool)
    for t in range(h["ntiles"]):
        m, w, off = int(h["rowMask"][t]), int(h["tileWidth"][t]), int(h["tileNnzOff"][t])
        rr = [r for r in range(T) if (m >> r) & 1]
        if w * len(rr) > 1:
            assert off % 16 == 0 and h["tileNnzOff"][t + 1] - off >= (w * len(rr) + 15) // 16 * 16
        else:
            assert h["tileNnzOff"][t + 1] - off >= 1
        real[off:off + w * len(rr)] = True
        for k in range(w):
            for j, r in enumerate(rr):
                s = off + k * len(rr) + j
                if h["colIdx"][s] == T:
                    assert h["v64"][s] == 0 and h["v32"][s] == 0 and h["v16"][s] == 0
                    continue
                rows.append(trow[t] * T + r)
                cols.append(int(h["tileColIdx"][t]) * T + int(h["colIdx"][s]))
                vals.append(h["v64"][s])
    gaps = ~real            # slots outside every tile's rectangle: pads
    assert np.all(h["colIdx"][gaps] == T) and np.all(h["v64"][gaps] == 0) and np.all(h["v16"][gaps] == 0)
    rows, cols, vals = np.array(rows), np.array(cols), np.array(vals)
    o = np.lexsort((cols, rows))
    assert np.array_equal(cols[o], ci) and np.array_equal(vals[o].view(np.uint64), np.asarray(v).view(np.uint64))
    assert np.array_equal(np.searchsorted(rows[o], np.arange(n + 1)), rp)


@pytest.mark.parametrize("name,m,T", list(_cases()), ids=[c[0] for c in _cases()])
def test_slot_layout_holds_the_csr(name, m, T):
    n, rp, ci, v = m
    slot_layout_holds_the_csr(evocg.tile_layout_host(n, rp, ci, v, T), n, rp, ci, v, T)


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


@pytest.mark.parametrize("name,m,T", [c for c in _cases() if c[2] <= 32], ids=[c[0] for c in _cases() if c[2] <= 32])
@pytest.mark.parametrize("warps,stage", [(1, 4096), (7, 3072), (3648, 4096), (4864, 2560)])
def test_panel_plan_passes_its_checks(name, m, T, warps, stage):
    """The panel SpMV's batch plan, built as the library builds it, passes the checks the
    library applies before using it, for one warp, a few warps and the grids of the kernel
    variants (more warps than panels leaves warps without work), with stages from 2.5 to 4 KB
    (a dense tile larger than a stage becomes a direct batch)."""
    n, rp, ci, v = m
    nb, ok = evocg.panel_plan_host(n, rp, ci, v, T, warps, stage)
    assert ok, evocg.last_error()
    assert nb >= (n + T - 1) // T   # at least one batch per panel


@pytest.mark.parametrize("cfg", [1, 2, 3])
def test_panel_plan_of_the_stencil_workloads(cfg):
    w = W.workload(cfg)
    nb, ok = evocg.panel_plan_host(w.n, w.rp, w.ci, w.v, w.T, 3648, 4096)
    assert ok, evocg.last_error()
    if cfg == 2:   # every 128^3 panel's tiles fit one 4 KB stage sized for FP64
        assert nb == w.n // 32


def test_panel_plan_rejects_tiles_of_64():
    n, rp, ci, v = W.laplace2d_5pt(70)
    nb, ok = evocg.panel_plan_host(n, rp, ci, v, 64, 8, 4096)
    assert not ok and nb == 0


@pytest.mark.parametrize("name,m", [(c[0], c[1]) for c in _cases() if c[2] == 32] +
                         [("many_tiles", many_tiles_t32()), ("lap2d_t32", W.laplace2d_5pt(100))],
                         ids=[c[0] for c in _cases() if c[2] == 32] + ["many_tiles", "lap2d_t32"])
def test_rowblock_plan_passes_its_checks(name, m):
    """The row-block SpMV's plan, built as the library builds it, passes the checks the library
    applies before using it, and its descriptor and single-entry ELL counts equal those counted
    from the CSR with numpy."""
    n, rp, ci, v = m
    nd, ns, ok = evocg.rowblock_plan_host(n, rp, ci, v, 32)
    assert ok, evocg.last_error()
    assert (nd, ns) == rowblock_counts(n, rp, ci)


@pytest.mark.parametrize("cfg", [2, 3])
def test_rowblock_plan_of_the_stencil_workloads(cfg):
    w = W.workload(cfg)
    nd, ns, ok = evocg.rowblock_plan_host(w.n, w.rp, w.ci, w.v, w.T)
    assert ok, evocg.last_error()
    assert (nd, ns) == rowblock_counts(w.n, w.rp, w.ci)


def test_rowblock_plan_is_for_tiles_of_32():
    n, rp, ci, v = W.laplace2d_5pt(70)
    for T in (16, 64):
        assert evocg.rowblock_plan_host(n, rp, ci, v, T) == (0, 0, False)


def _rowell_slots(n, rp, ci, T=64):
    """ELL slots of the row-ELL plan counted from the CSR with numpy: per row block, T times
    its longest row."""
    per = np.diff(rp)
    nrb = (n + T - 1) // T
    return int(sum(T * per[b * T:(b + 1) * T].max(initial=0) for b in range(nrb)))


@pytest.mark.parametrize("name,m", [("banded_20k", W.banded_spd(20000, 6, band=700)),
                                    ("banded_ragged", W.banded_spd(5003, 3, band=3000)),
                                    ("banded_wide", W.banded_spd(30000, 4, band=4096))])
def test_rowell_plan_passes_its_checks(name, m):
    """The row-ELL plan of a matrix of sparse 64 x 64 tiles passes the checks the library
    applies before using it, with the ELL size counted from the CSR."""
    n, rp, ci, v = m
    ns, ok = evocg.rowell_plan_host(n, rp, ci, v, 64)
    assert ok, evocg.last_error()
    assert ns == _rowell_slots(n, rp, ci)


def test_rowell_plan_only_for_sparse_tiles_of_64():
    dense = W.dense_to_csr(np.random.default_rng(1).standard_normal((130, 130)) + 300 * np.eye(130))
    assert evocg.rowell_plan_host(*dense, 64) == (0, False)                 # dense tiles
    n, rp, ci, v = W.banded_spd(20000, 6, band=700)
    assert evocg.rowell_plan_host(n, rp, ci, v, 32)[1] is False            # tiles of 32


def test_empty_matrix():
    z64, z32, zf = np.zeros(1, np.int64), np.zeros(0, np.int32), np.zeros(0)
    h = evocg.tile_layout_host(0, z64, z32, zf, 16)
    assert (h["ntiles"], h["nslots"]) == (0, 0) and list(h["tileRowPtr"]) == [0]
    assert evocg.panel_plan_host(0, z64, z32, zf, 32, 4) == (0, True)
    assert evocg.rowblock_plan_host(0, z64, z32, zf, 32) == (0, 0, True)
