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
