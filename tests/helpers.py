"""Shared helpers of the GPU parity tests: the same seeded inputs go to the oracle and to
the GPU library; no expected value is ever taken from the GPU side."""
import numpy as np

import oracle
from mixed_precision_sparse_gb300 import evocg
from mixed_precision_sparse_gb300 import workloads as W


class Pair:
    """A matrix held by both sides: the oracle (CSR + its own tile layout) and the GPU."""

    def __init__(self, m, T):
        n, rp, ci, v = m
        self.n, self.T = n, T
        self.A = oracle.CSR(n, rp, ci, v)
        self.t = oracle.Tiles(self.A, T)
        self.G = evocg.tile_build(n, rp, ci, v, T)
        self.absA = oracle.CSR(n, rp, ci, np.abs(v))

    def tile_map(self, seed, fracs=(0.4, 0.4, 0.2)):
        """Per-tile map from the seeded counter generator, keyed by the oracle's own tile
        list (the GPU's list is checked bit-exact against it separately)."""
        return W.tile_map(self.t.tile_rows(), self.t.tileColIdx, self.t.nrb, seed, fracs)

    def abs_sum(self, tile_map, x):
        """Per-row sum of |a~_ij x~_j| (the denominator of the per-row relative error)."""
        return oracle.mixed_spmv(self.absA, self.t, tile_map, np.abs(x))


def row_rel_err(y, want, denom):
    return np.abs(y - want) / np.maximum(denom, 1e-300)


def many_tiles_t32(seed=0):
    """A 2048 x 2048 matrix (64 column blocks) built to reach the row-block SpMV's less common
    paths with tiles of 32: besides the diagonal tiles, row block 0 has 40 regular tiles (two
    entries each, in two rows: more than one warp's worth of descriptors), seven single-entry
    tiles in row 5 and three in row 9 (an ELL block of odd width, with pads); row block 1 has
    only its diagonal tile and single-entry tiles (two per row, one in the last two rows)."""
    rng = np.random.default_rng(seed)
    n = 2048
    ent = {(i, i): 4.0 + rng.random() for i in range(n)}
    for cb in range(1, 41):                       # regular tiles of row block 0
        ent[(cb % 32, cb * 32 + 3)] = rng.standard_normal()
        ent[((cb + 7) % 32, cb * 32 + 17)] = rng.standard_normal()
    for k, cb in enumerate(range(41, 48)):        # singles of row 5
        ent[(5, cb * 32 + 1 + k)] = rng.standard_normal()
    for cb in (50, 55, 60):                       # singles of row 9
        ent[(9, cb * 32 + 30)] = rng.standard_normal()
    for i in range(32, 64):                       # row block 1: singles in distinct column blocks
        k = i - 32
        ent[(i, (2 + k) * 32 + k)] = rng.standard_normal()
        if k < 30:
            ent[(i, (34 + (7 * k) % 30) * 32 + 31 - k)] = rng.standard_normal()
    keys = sorted(ent)
    rows = np.array([k[0] for k in keys], np.int64)
    rp = np.searchsorted(rows, np.arange(n + 1)).astype(np.int64)
    ci = np.array([k[1] for k in keys], np.int32)
    v = np.array([ent[k] for k in keys], np.float64)
    return n, rp, ci, v


def rowblock_counts(n, rp, ci, T=32):
    """Descriptors and single-entry ELL slots of the row-block SpMV plan, counted from the
    CSR with numpy: a tile with two or more entries gets a descriptor; per row block, the
    rows with single-entry tiles times the largest number of them in one row."""
    rows = np.repeat(np.arange(n), np.diff(rp))
    ncb = (n + T - 1) // T
    tile = (rows // T) * ncb + ci // T
    tiles, cnt = np.unique(tile, return_counts=True)
    ndesc = int(np.sum(cnt >= 2))
    single = np.isin(tile, tiles[cnt == 1])
    rb, r = rows[single] // T, rows[single] % T
    slots = 0
    for b in np.unique(rb):
        per = np.bincount(r[rb == b], minlength=T)
        slots += int(per.max()) * int(np.count_nonzero(per))
    return ndesc, slots
