"""Row-block sharding of the solve over ranks, one GPU each: host planning and the halo
exchange.

The pages run one GPU (EvoCG §4.1, one A100). Across ranks the path splits along its row
blocks: a rank owns a contiguous range of row blocks (its rows of A, b, x, r, z and p) and
everything per row stays on it; per CG iteration it needs (1) the entries of p its rows read
in columns it does not own (its halo) before its SpMV, and (2) three FP64 sums over all rows
(p.q, r.z, r.r). This module plans (1) once per matrix and carries it out each iteration:

  partition()   contiguous row-block ranges, balanced by stored entries;
  local_part()  a rank's local matrix: its rows, columns renumbered with its own rows first
                and then its halo (the off-rank columns it reads, ascending), as a square CSR
                of size n_own + n_halo whose halo rows are empty (so the single-GPU tile
                builder and SpMV take it as it is: y's first n_own entries are the rank's rows
                of A p); the halo positions each peer fills, and the own rows each peer needs;
  HaloExchange  one exchange: every rank sends each peer the p entries that peer reads and
                receives its own halo, with point-to-point messages of torch.distributed
                (gloo on the host, NCCL between GPUs).

The three sums are all_reduce(SUM) of FP64 scalars. No collective touches the matrix.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


def partition(n: int, row_ptr, T: int, world: int) -> np.ndarray:
    """Row bounds (world + 1 entries) of contiguous row-block ranges, one per rank, balanced
    by stored entries: rank r owns rows bounds[r] .. bounds[r + 1] - 1; every bound but the
    last is a multiple of T (a row block is never split)."""
    if world < 1:
        raise ValueError("world must be at least 1")
    rp = np.asarray(row_ptr, np.int64)
    nrb = (n + T - 1) // T
    ends = np.minimum(np.arange(1, nrb + 1, dtype=np.int64) * T, n)
    cum = rp[ends] if nrb else np.zeros(0, np.int64)        # entries up to each row block's end
    total = int(rp[n])
    cuts = [0]
    for r in range(1, world):
        target = total * r / world
        k = int(np.searchsorted(cum, target, side="left"))  # first row block reaching the target
        if k < nrb and k > 0 and abs(cum[k - 1] - target) <= abs(cum[k] - target):
            k -= 1
        cuts.append(max(cuts[-1], min(k + 1, nrb)))
    cuts.append(nrb)
    return np.minimum(np.asarray(cuts, np.int64) * T, n)


@dataclass
class LocalPart:
    """One rank's share: rows [r0, r1) of the global matrix, renumbered."""
    rank: int
    r0: int
    r1: int
    halo: np.ndarray                  # global columns of the halo, ascending
    row_ptr: np.ndarray               # square local CSR of size n_ext (halo rows empty)
    col_idx: np.ndarray
    vals: np.ndarray
    recv: dict = field(default_factory=dict)   # peer -> (first, end) halo positions it fills
    send: dict = field(default_factory=dict)   # peer -> own-row indices (local) it reads

    @property
    def n_own(self) -> int:
        return self.r1 - self.r0

    @property
    def n_ext(self) -> int:
        return self.n_own + int(self.halo.size)


def _halo(rp, ci, r0, r1):
    cols = ci[rp[r0]:rp[r1]]
    return np.unique(cols[(cols < r0) | (cols >= r1)])


def local_part(n: int, row_ptr, col_idx, vals, bounds, rank: int) -> LocalPart:
    """Rank `rank`'s local matrix and exchange lists under the row bounds of partition()."""
    rp = np.asarray(row_ptr, np.int64)
    ci = np.asarray(col_idx, np.int32)
    v = np.asarray(vals, np.float64)
    bounds = np.asarray(bounds, np.int64)
    world = bounds.size - 1
    r0, r1 = int(bounds[rank]), int(bounds[rank + 1])
    n_own = r1 - r0
    halo = _halo(rp, ci, r0, r1)
    a, b = int(rp[r0]), int(rp[r1])
    cols = ci[a:b].astype(np.int64)
    own = (cols >= r0) & (cols < r1)
    new = np.where(own, cols - r0, n_own + np.searchsorted(halo, cols))
    rows = np.repeat(np.arange(n_own, dtype=np.int64), np.diff(rp[r0:r1 + 1]))
    order = np.lexsort((new, rows))                     # ascending columns within each row
    lrp = np.concatenate([rp[r0:r1 + 1] - a, np.full(halo.size, b - a, np.int64)])
    part = LocalPart(rank, r0, r1, halo, lrp, new[order].astype(np.int32), v[a:b][order])
    for q in range(world):
        if q == rank:
            continue
        q0, q1 = int(bounds[q]), int(bounds[q + 1])
        lo, hi = int(np.searchsorted(halo, q0)), int(np.searchsorted(halo, q1))
        if hi > lo:
            part.recv[q] = (lo, hi)
        theirs = _halo(rp, ci, q0, q1)                  # what peer q reads ...
        mine = theirs[(theirs >= r0) & (theirs < r1)]   # ... of my rows, in q's halo order
        if mine.size:
            part.send[q] = (mine - r0).astype(np.int64)
    return part


class HaloExchange:
    """Fills x_ext[n_own:] (the halo) from the peers' own entries, sending each peer the
    entries of x_ext[:n_own] it reads. x_ext: a 1-D float64 torch tensor of n_ext entries on
    the device the process group's backend serves (CPU for gloo)."""

    def __init__(self, part: LocalPart, dist):
        import torch
        self.part, self.dist = part, dist
        self._send_idx = {q: torch.from_numpy(ix) for q, ix in part.send.items()}

    def __call__(self, x_ext):
        import torch
        p, dist = self.part, self.dist
        reqs, keep = [], []
        for q, (lo, hi) in sorted(p.recv.items()):
            buf = torch.empty(hi - lo, dtype=x_ext.dtype, device=x_ext.device)
            keep.append((lo, hi, buf))
            reqs.append(dist.irecv(buf, src=q))
        for q, ix in sorted(self._send_idx.items()):
            out = x_ext[:p.n_own].index_select(0, ix.to(x_ext.device)).contiguous()
            keep.append((None, None, out))
            reqs.append(dist.isend(out, dst=q))
        for r in reqs:
            r.wait()
        for lo, hi, buf in keep:
            if lo is not None:
                x_ext[p.n_own + lo:p.n_own + hi] = buf
        return x_ext
