"""Pins of the oracle's tile layout: round trip, structural invariants, counts taken
another way, and the inter-tile worked example of EvoCG Fig. 4(a)."""
import os

import numpy as np
import pytest

import oracle
from mixed_precision_sparse_gb300 import workloads as W

GOLD = os.path.join(os.path.dirname(__file__), "golden", "fig4a_tile_lists.txt")


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


def _check_slots(t, A):
    """Slot invariants: every tile is a w x h rectangle over its nonempty rows; in each
    row the real entries come first with strictly ascending local columns, then pads
    (column T, value +0 in every stream); some row fills the width; the real entries
    are exactly the CSR entries."""
    T = t.T
    h = np.array([bin(int(m)).count("1") for m in t.rowMask], np.int64)
    assert np.all(h >= 1) and np.all(t.tileWidth >= 1)
    assert np.array_equal(np.diff(t.tileNnzOff), h * t.tileWidth.astype(np.int64))
    assert t.tileNnzOff[-1] == t.nslots and t.tileNnzOff[0] == 0
    n_real = 0
    last_rb = (t.n - 1) // T if t.n else -1
    for tt in range(t.ntiles):
        w, hh, off = int(t.tileWidth[tt]), int(h[tt]), int(t.tileNnzOff[tt])
        if t.tile_rows()[tt] == last_rb and t.n % T:
            assert int(t.rowMask[tt]) >> (t.n % T) == 0        # no rows past n
        c = t.colIdx[off:off + w * hh].reshape(w, hh).astype(np.int64)
        real = c < T
        assert np.all(real[0])                                 # listed rows are nonempty
        assert np.all(real[:-1] >= real[1:])                   # pads only after entries
        assert np.any(real[-1])                                # the width is attained
        cc = np.where(real, c, 10 ** 6)
        assert np.all(np.diff(cc, axis=0)[real[1:]] > 0)       # ascending columns
        pads = ~real.ravel()
        sl = slice(off, off + w * hh)
        assert np.all(c.ravel()[pads] == T)
        assert np.all(t.v64[sl][pads].view(np.uint64) == 0)
        assert np.all(t.v32[sl][pads].view(np.uint32) == 0) and np.all(t.v16[sl][pads] == 0)
        n_real += int(real.sum())
    assert n_real == A.rp[-1] == t.nnz
    assert np.array_equal(t.tile_entries().sum(), t.nnz)


@pytest.mark.parametrize("name,m,T", list(_cases()), ids=[c[0] for c in _cases()])
def test_round_trip_and_invariants(name, m, T):
    A = _csr(m)
    assert oracle.csr_check(A) == 0
    t = oracle.Tiles(A, T)
    back = t.to_csr()
    assert np.array_equal(back.rp, A.rp)
    assert np.array_equal(back.ci, A.ci)
    assert np.array_equal(back.v.view(np.uint64), A.v.view(np.uint64))
    # structure
    assert t.tileRowPtr[0] == 0 and np.all(np.diff(t.tileRowPtr) >= 0)
    for rb in range(t.nrb):
        cbs = t.tileColIdx[t.tileRowPtr[rb]:t.tileRowPtr[rb + 1]]
        assert np.all(np.diff(cbs) > 0)
    _check_slots(t, A)
    # tile count taken another way: distinct (row block, column block) pairs
    rows = np.repeat(np.arange(A.n), np.diff(A.rp))
    pairs = np.unique((rows // T) * ((A.n + T - 1) // T) + A.ci // T)
    assert pairs.size == t.ntiles


def test_value_streams_follow_column_scale():
    A = _csr(W.fe3d_q1_27pt(5, 7))      # column maxima far from 1 after D A D
    t = oracle.Tiles(A, 32)
    rows = np.repeat(np.arange(A.n), np.diff(A.rp))
    colmax = np.zeros(A.n)
    np.maximum.at(colmax, A.ci, np.abs(A.v))
    e = np.frexp(colmax)[1] - 1
    assert np.array_equal(t.colExp.astype(int), np.clip(e, -100, 100))
    # every stored entry: its global column through the slots of its tile
    back_cols, idx = [], []
    for tt in range(t.ntiles):
        for r, s in t.slots(tt):
            if t.colIdx[s] < 32:
                back_cols.append(int(t.tileColIdx[tt]) * 32 + int(t.colIdx[s]))
                idx.append(s)
    j, idx = np.array(back_cols), np.array(idx)
    scaled = np.ldexp(t.v64[idx], -t.colExp[j].astype(int))
    assert np.array_equal(t.v32[idx], scaled.astype(np.float32))
    smax = np.zeros(A.n)
    np.maximum.at(smax, j, np.abs(scaled))
    assert np.all((smax >= 1.0) & (smax < 2.0))  # each column's largest scaled entry is in [1, 2)
    assert rows.size == t.nnz


def test_empty_rows_and_columns():
    # rows 3 and 5 empty, tile (0,1) absent, n not a multiple of T
    M = np.zeros((20, 20))
    M[np.arange(20), np.arange(20)] = 2.0
    M[3, 3] = 0.0
    M[5, 5] = 0.0
    M[0, 19] = M[19, 0] = -1.0
    A = _csr(W.dense_to_csr(M))
    t = oracle.Tiles(A, 16)
    assert t.nrb == 2
    assert list(t.tileRowPtr) == [0, 2, 4]
    assert list(t.tileColIdx) == [0, 1, 0, 1]
    m = [int(x) for x in t.rowMask]
    assert (m[0] >> 3) & 1 == 0 and (m[0] >> 5) & 1 == 0        # empty local rows
    assert m[0] == 0xFFFF & ~(1 << 3) & ~(1 << 5) and m[1] == 1   # row 0 reaches column 19
    assert m[3] == 0xF and m[2] == 1 << 3                         # rows past n are absent
    assert list(t.tileWidth) == [1, 1, 1, 1]
    back = t.to_csr()
    assert np.array_equal(back.ci, A.ci)


def _golden():
    d = {}
    for line in open(GOLD):
        if line.startswith("#") or not line.strip():
            continue
        k, rest = line.split(None, 1)
        d[k] = rest.strip()
    return d


@pytest.mark.parametrize("T", [16, 32, 64])
def test_fig4a_inter_tile_lists(T):
    g = _golden()
    groups = [[int(c) for c in grp.split(",")] for grp in g["rowblock_colblocks"].split("|")]
    n = T * 9
    M = np.zeros((n, n))
    for rb, cbs in enumerate(groups):
        for cb in cbs:
            M[rb * T + (cb % T), cb * T + (rb % T)] = 1.0 + cb
    # rows of row blocks 3.. are empty
    A = _csr(W.dense_to_csr(M))
    t = oracle.Tiles(A, T)
    want_ptr = [int(s) for s in g["tileRowPtr"].split()]
    want_idx = [int(s) for s in g["tileColIdx"].split()]
    assert list(t.tileRowPtr[:4]) == want_ptr
    assert list(t.tileColIdx) == want_idx
    assert np.all(t.tileRowPtr[4:] == want_ptr[-1])


def _count_5pt(nx, ny, T):
    """Closed form for the 5-point stencil with T | nx: every row block is T points of one
    grid line; it touches its own block, the left/right blocks of its line (if any) and the
    same block of the lines above and below (if any)."""
    nb = nx // T
    return nb * ny + 2 * (nb - 1) * ny + 2 * nb * (ny - 1)


def _slots_5pt(nx, ny, T):
    """Slots of the 5-point stencil with T | nx and T >= 3: a row block's own tile holds
    x-1, x, x+1 (width 3 over all T rows; its first and last rows have two entries and
    one pad each), the left / right tiles one entry each, the tiles of the lines above and
    below one entry in every row."""
    nb = nx // T
    return nb * ny * 3 * T + 2 * (nb - 1) * ny + 2 * nb * (ny - 1) * T


def _count_7pt(N, T):
    nb = N // T
    lines = N * N
    return nb * lines + 2 * (nb - 1) * lines + 2 * 2 * nb * (N - 1) * N


def test_stencil_tile_counts_closed_form():
    t1 = oracle.Tiles(_csr(W.laplace2d_5pt(64)), 16)
    assert t1.ntiles == _count_5pt(64, 64, 16) == 1144        # the 64x64 Laplacian workload
    assert t1.nslots == _slots_5pt(64, 64, 16)
    assert t1.nslots - t1.nnz == 2 * (64 // 16) * 64           # two pads per own tile
    t2 = oracle.Tiles(_csr(W.laplace2d_5pt(96, 40)), 32)
    assert t2.ntiles == _count_5pt(96, 40, 32)
    assert t2.nslots == _slots_5pt(96, 40, 32)
    t3 = oracle.Tiles(_csr(W.diffusion3d_7pt(32, 1)), 32)
    assert t3.ntiles == _count_7pt(32, 32)
    t4 = oracle.Tiles(_csr(W.diffusion3d_7pt(64, 1)), 32)
    assert t4.ntiles == _count_7pt(64, 32)
    assert _count_7pt(128, 32) == 423936                       # the 128^3 workload


def test_slot_order_worked_example():
    """A 4 x 4 tile worked out by hand from the slot definition: rows 0, 2, 3 are
    nonempty (mask 0b1101, h = 3), row 3 is the longest (w = 3). Slot (k, j) at k*h + j
    holds the k-th entry of the j-th nonempty row, else a pad (column 4):
        k = 0: row 0 -> col 0, row 2 -> col 1, row 3 -> col 0
        k = 1: row 0 -> col 2, row 2 -> pad,   row 3 -> col 1
        k = 2: row 0 -> pad,   row 2 -> pad,   row 3 -> col 3"""
    M = np.zeros((4, 4))
    M[0, 0], M[0, 2] = 1.0, 2.0
    M[2, 1] = 3.0
    M[3, 0], M[3, 1], M[3, 3] = 4.0, 5.0, 6.0
    t = oracle.Tiles(_csr(W.dense_to_csr(M)), 4)
    assert t.ntiles == 1 and int(t.rowMask[0]) == 0b1101 and int(t.tileWidth[0]) == 3
    assert list(t.colIdx) == [0, 1, 0, 2, 4, 1, 4, 4, 3]
    assert list(t.v64) == [1.0, 3.0, 4.0, 2.0, 0.0, 5.0, 0.0, 0.0, 6.0]
    assert t.nslots == 9 and t.nnz == 6
