"""Pins of the oracle's Tile-CSC layout (EvoCG §3.3.1 Fig. 4(a), §3.3.2 Fig. 4(b)): round
trip to CSR, structural invariants of the CSC interior and its padding, counts taken another
way (distinct row-block/column-block pairs, closed forms for stencils), the column scale,
and the worked examples of Fig. 4(a) and Fig. 4(b)."""
import os

import numpy as np
import pytest

import oracle
from mixed_precision_sparse_gb300 import workloads as W

GOLD_A = os.path.join(os.path.dirname(__file__), "golden", "fig4a_tile_lists.txt")
GOLD_B = os.path.join(os.path.dirname(__file__), "golden", "fig4b_tile_csc.txt")


def _csr(m):
    return oracle.CSR(*m)


def _cases():
    yield "lap2d_16", W.laplace2d_5pt(16), 16
    yield "lap2d_ragged", W.laplace2d_5pt(13, 11), 16
    yield "rand50_t16", W.random_spd_small(50, 1, 0.2), 16
    yield "rand70_t32", W.random_spd_small(70, 2, 0.1), 32
    yield "rand130_t64", W.random_spd_small(130, 3, 0.05), 64
    yield "diff3d_6", W.diffusion3d_7pt(6, 4), 32
    yield "fe3d_5", W.fe3d_q1_27pt(5, 5), 32
    yield "aniso_20", W.aniso2d_q1_9pt(20), 32
    yield "banded", W.banded_spd(9000, 6, band=300), 64


def _check_csc(t, A):
    """Every tile: colPtr starts at 0, ascends and ends at the tile's stream length; inside a
    column the stored entries come first with strictly ascending rows below T (rows past n
    never appear), then at most one sentinel (row T, +0 in every stream), present exactly
    when pad = 2 and the column's count is odd; the stored entries are the CSR's."""
    T = t.T
    assert t.tileNnzOff[0] == 0 and t.tileNnzOff[-1] == t.nnz_p
    assert np.all(np.diff(t.tileNnzOff) >= 1)
    trow = t.tile_rows()
    n_real = 0
    for tt in range(t.ntiles):
        cp = t.colPtr[tt].astype(np.int64)
        off = int(t.tileNnzOff[tt])
        assert cp[0] == 0 and cp[-1] == t.tileNnzOff[tt + 1] - off and np.all(np.diff(cp) >= 0)
        rows_here = min(T, t.n - int(trow[tt]) * T)
        for c in range(T):
            r = t.rowIdx[off + cp[c]: off + cp[c + 1]].astype(np.int64)
            real = r < T
            k = int(real.sum())
            assert np.all(real[:k]) and not np.any(real[k:])        # sentinels last
            assert np.all(np.diff(r[:k]) > 0) and np.all(r[:k] < rows_here)
            npads = r.size - k
            assert npads == (k % 2 if t.pad == 2 else 0)
            if npads:
                s = slice(off + cp[c] + k, off + cp[c + 1])
                assert np.all(r[k:] == T)
                assert np.all(t.v64[s].view(np.uint64) == 0)
                assert np.all(t.v32[s].view(np.uint32) == 0) and np.all(t.v16[s] == 0)
            n_real += k
        assert np.any(np.diff(cp) > 0)                                # no empty tile
    assert n_real == A.rp[-1] == t.nnz == int(t.tile_entries().sum())


@pytest.mark.parametrize("pad", [1, 2])
@pytest.mark.parametrize("name,m,T", list(_cases()), ids=[c[0] for c in _cases()])
def test_round_trip_and_invariants(name, m, T, pad):
    A = _csr(m)
    assert oracle.csr_check(A) == 0
    t = oracle.Tiles(A, T, pad)
    back = t.to_csr()
    assert np.array_equal(back.rp, A.rp)
    assert np.array_equal(back.ci, A.ci)
    assert np.array_equal(back.v.view(np.uint64), A.v.view(np.uint64))
    assert t.tileRowPtr[0] == 0 and np.all(np.diff(t.tileRowPtr) >= 0)
    for rb in range(t.nrb):
        cbs = t.tileColIdx[t.tileRowPtr[rb]:t.tileRowPtr[rb + 1]]
        assert np.all(np.diff(cbs) > 0)
    _check_csc(t, A)
    # counts taken another way: distinct (row block, column block) pairs; with pad = 2 the
    # stream length is the sum over (row block, column) groups of the count rounded up to even
    rows = np.repeat(np.arange(A.n), np.diff(A.rp))
    key = (rows // T).astype(np.int64) * A.n + A.ci
    pairs = np.unique((rows // T) * ((A.n + T - 1) // T) + A.ci // T)
    assert pairs.size == t.ntiles
    _, cnt = np.unique(key, return_counts=True)
    assert t.nnz_p == (int(cnt.sum()) if pad == 1 else int((cnt + cnt % 2).sum()))


def test_value_streams_follow_column_scale():
    A = _csr(W.fe3d_q1_27pt(5, 7))      # column maxima far from 1 after D A D
    t = oracle.Tiles(A, 32)
    colmax = np.zeros(A.n)
    np.maximum.at(colmax, A.ci, np.abs(A.v))
    e = np.frexp(colmax)[1] - 1
    assert np.array_equal(t.colExp.astype(int), np.clip(e, -100, 100))
    j, idx = [], []
    for tt in range(t.ntiles):
        for r, c, s in t.entries(tt):
            if r < 32:
                j.append(int(t.tileColIdx[tt]) * 32 + c)
                idx.append(s)
    j, idx = np.array(j), np.array(idx)
    scaled = np.ldexp(t.v64[idx], -t.colExp[j].astype(int))
    assert np.array_equal(t.v32[idx], scaled.astype(np.float32))     # numpy's RNE cast
    smax = np.zeros(A.n)
    np.maximum.at(smax, j, np.abs(scaled))
    assert np.all((smax >= 1.0) & (smax < 2.0))  # each column's largest scaled entry is in [1, 2)
    assert idx.size == t.nnz


def test_empty_rows_and_columns():
    # rows 3 and 5 empty, n = 20 not a multiple of T = 16
    M = np.zeros((20, 20))
    M[np.arange(20), np.arange(20)] = 2.0
    M[3, 3] = 0.0
    M[5, 5] = 0.0
    M[0, 19] = M[19, 0] = -1.0
    A = _csr(W.dense_to_csr(M))
    for pad in (1, 2):
        t = oracle.Tiles(A, 16, pad)
        assert t.nrb == 2
        assert list(t.tileRowPtr) == [0, 2, 4]
        assert list(t.tileColIdx) == [0, 1, 0, 1]
        # tile (0, 0): the diagonal without columns 3 and 5; (0, 1): row 0 at local column 3;
        # (1, 0): row 3 (global 19) at column 0; (1, 1): rows 0..3 on the diagonal
        cp0 = [0, 1, 2, 3, 3, 4, 4] + list(range(5, 15))
        step = 1 if pad == 1 else 2
        assert list(t.colPtr[0]) == [step * c for c in cp0]
        assert list(t.colPtr[1]) == [0, 0, 0, 0] + [step] * 13
        assert list(t.colPtr[2]) == [0] + [step] * 16
        assert list(t.colPtr[3]) == [0] + [step * k for k in (1, 2, 3, 4)] + [4 * step] * 12
        assert list(t.rowIdx[t.tileNnzOff[1]:t.tileNnzOff[2]]) == [0] + [16] * (step - 1)
        assert t.to_csr().ci.tolist() == A.ci.tolist()


def _golden(path):
    d = {}
    for line in open(path):
        if line.startswith("#") or not line.strip():
            continue
        k, rest = line.split(None, 1)
        d[k] = rest.strip()
    return d


@pytest.mark.parametrize("T", [16, 32, 64])
def test_fig4a_inter_tile_lists(T):
    """Row blocks 1, 2 and 4 of Fig. 4(a); the figure's row blocks 0 and 3, drawn with N/C
    placeholders only, are not part of the pin (three of its five row blocks are used)."""
    g = _golden(GOLD_A)
    groups = [[int(c) for c in grp.split(",")] for grp in g["rowblock_colblocks"].split("|")]
    n = T * 9
    M = np.zeros((n, n))
    for rb, cbs in enumerate(groups):
        for cb in cbs:
            M[rb * T + (cb % T), cb * T + (rb % T)] = 1.0 + cb
    A = _csr(W.dense_to_csr(M))
    t = oracle.Tiles(A, T)
    want_ptr = [int(s) for s in g["tileRowPtr"].split()]
    want_idx = [int(s) for s in g["tileColIdx"].split()]
    assert list(t.tileRowPtr[:4]) == want_ptr
    assert list(t.tileColIdx) == want_idx
    assert np.all(t.tileRowPtr[4:] == want_ptr[-1])


def fig4b_matrix():
    """The matrix of the Fig. 4(b) fixture: one tile whose listed columns hold the listed
    rows (values 1, 2, 3, ... in column-major order)."""
    g = _golden(GOLD_B)
    T = int(g["tile_size"])
    M = np.zeros((T, T))
    val = 1.0
    for grp in g["column_rows"].split("|"):
        c, rows = grp.split(":")
        for r in rows.split(","):
            M[int(r), int(c)] = val
            val += 1.0
    return g, T, W.dense_to_csr(M)


def test_fig4b_intra_tile_fragment():
    g, T, m = fig4b_matrix()
    t = oracle.Tiles(_csr(m), T, int(g["pad"]))
    assert t.ntiles == 1
    head = [int(s) for s in g["colPtr_head"].split()]
    tail = [int(s) for s in g["colPtr_tail"].split()]
    assert list(t.colPtr[0][:len(head)]) == head
    assert list(t.colPtr[0][-len(tail):]) == tail
    assert list(t.rowIdx) == [int(s) for s in g["rowIdx"].split()]
    assert t.rowIdx[3] == T and t.v64[3] == 0.0          # the sentinel row index R = T
    assert list(t.v64[t.rowIdx < T]) == [1.0, 2.0, 3.0, 4.0, 5.0, 6.0, 7.0]
    t1 = oracle.Tiles(_csr(m), T, 1)                      # no padding: no sentinel
    assert list(t1.rowIdx) == [0, 3, 63, 2, 5, 2, 4] and t1.colPtr[0][1] == 3


def _count_5pt(nx, ny, T):
    """Closed form for the 5-point stencil with T | nx: every row block is T points of one
    grid line; it touches its own block, the left/right blocks of its line (if any) and the
    same block of the lines above and below (if any)."""
    nb = nx // T
    return nb * ny + 2 * (nb - 1) * ny + 2 * nb * (ny - 1)


def _padded_5pt(nx, ny, T):
    """Entries of the padded (pad = 2) streams of the 5-point stencil with T | nx: the own
    tile's interior columns hold rows c-1, c, c+1 (3, padded to 4), its first and last
    columns 2; a left / right tile holds 1 entry (padded to 2); a tile of the line above or
    below holds one entry in each of its T columns (each padded to 2)."""
    nb = nx // T
    return nb * ny * (4 * T - 4) + 2 * (nb - 1) * ny * 2 + 2 * nb * (ny - 1) * 2 * T


def _count_7pt(N, T):
    nb = N // T
    lines = N * N
    return nb * lines + 2 * (nb - 1) * lines + 2 * 2 * nb * (N - 1) * N


def _padded_7pt(N, T):
    nb = N // T
    lines = N * N
    return nb * lines * (4 * T - 4) + 2 * (nb - 1) * lines * 2 + 2 * 2 * nb * (N - 1) * N * 2 * T


def test_stencil_tile_counts_closed_form():
    t1 = oracle.Tiles(_csr(W.laplace2d_5pt(64)), 16, 2)
    assert t1.ntiles == _count_5pt(64, 64, 16) == 1144         # the 64x64 Laplacian workload
    assert t1.nnz_p == _padded_5pt(64, 64, 16) == 32256
    t2 = oracle.Tiles(_csr(W.laplace2d_5pt(96, 40)), 32, 2)
    assert t2.ntiles == _count_5pt(96, 40, 32)
    assert t2.nnz_p == _padded_5pt(96, 40, 32)
    t3 = oracle.Tiles(_csr(W.diffusion3d_7pt(32, 1)), 32, 2)
    assert t3.ntiles == _count_7pt(32, 32) and t3.nnz_p == _padded_7pt(32, 32)
    t4 = oracle.Tiles(_csr(W.diffusion3d_7pt(64, 1)), 32, 2)
    assert t4.ntiles == _count_7pt(64, 32) and t4.nnz_p == _padded_7pt(64, 32)
    assert _count_7pt(128, 32) == 423936                        # the 128^3 workload
    assert _padded_7pt(128, 32) == 24969216                     # 1.71 x its 14,581,760 entries


def test_worked_example_by_hand():
    """A 4 x 4 tile worked out by hand from the CSC definition: column 0 holds rows 0, 3;
    column 1 rows 2, 3; column 2 row 0; column 3 row 3. With pad = 2, column 2 and column 3
    end with the sentinel row 4."""
    M = np.zeros((4, 4))
    M[0, 0], M[0, 2] = 1.0, 2.0
    M[2, 1] = 3.0
    M[3, 0], M[3, 1], M[3, 3] = 4.0, 5.0, 6.0
    t = oracle.Tiles(_csr(W.dense_to_csr(M)), 4, 2)
    assert t.ntiles == 1 and t.nnz == 6 and t.nnz_p == 8
    assert list(t.colPtr[0]) == [0, 2, 4, 6, 8]
    assert list(t.rowIdx) == [0, 3, 2, 3, 0, 4, 3, 4]
    assert list(t.v64) == [1.0, 4.0, 3.0, 5.0, 2.0, 0.0, 6.0, 0.0]
    t1 = oracle.Tiles(_csr(W.dense_to_csr(M)), 4, 1)
    assert list(t1.colPtr[0]) == [0, 2, 4, 5, 6] and list(t1.rowIdx) == [0, 3, 2, 3, 0, 3]
