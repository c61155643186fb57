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


def oracle_envelope(A, tiles, b, nperturb=8, seed=0, **kw):
    """Iteration counts of the oracle's solve of A x = b and of `nperturb` solves whose
    right-hand side differs in the last bit of one random entry.

    The mixed-precision operator rounds each x entry to its tile's format, a function
    that jumps at rounding boundaries, so a last-bit change anywhere (an input, or the
    summation order of a dot product) can move the iteration count by several percent.
    The counts of these equally valid runs bound what a correct implementation may give.
    Returns (reference run, (min iters, max iters), (min rec, max rec))."""
    ref = oracle.cg(A, tiles, b, **kw)
    its, recs = [ref["iters"]], [ref["iters_rec"]]
    rng = np.random.default_rng(seed)
    for _ in range(nperturb):
        b2 = np.array(b, dtype=np.float64, copy=True)
        i = int(rng.integers(0, b2.size))
        b2[i] = np.nextafter(b2[i], np.inf)
        r = oracle.cg(A, tiles, b2, **kw)
        its.append(r["iters"])
        recs.append(r["iters_rec"])
    return ref, (min(its), max(its)), (min(recs), max(recs))


def within_envelope(value, env, frac=0.03, slack=2):
    lo, hi = env
    return lo - max(slack, frac * lo) <= value <= hi + max(slack, frac * hi)
