"""Run and time the mixed-precision SpMV alone on the synthetic workloads.

    python -m mixed_precision_sparse_gb300.spmv_run [--workloads 2,3,5] [--reps 50]
                                                    [--maps mixed,fp64] [--launches K]
                                                    [--kernel default|direct|panel|rowblock|rowell]

For each workload: build the tile structure, set the seeded 40/40/20 per-tile map (or the
all-FP64 map), and launch the SpMV kernel back to back on device-resident x and y (every
workload's matrix streams are larger than L2 except the 64 x 64 Laplacian's), timed with
CUDA events on the launching stream. Prints one JSON line per (workload, map) with the
microseconds per launch and the algorithmic bytes of the launch over EvoCG's Tile-CSC layout
(the active value stream of each tile, the row indices, column pointers and descriptors, x
read once and y written once).

`--launches K` skips the timing and issues exactly K SpMV launches after one x-copy launch,
for use under a profiler.
"""
from __future__ import annotations

import argparse
import json
import os
import sys

import numpy as np

if __package__ in (None, ""):
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

from mixed_precision_sparse_gb300 import evocg  # noqa: E402
from mixed_precision_sparse_gb300 import workloads as W  # noqa: E402


def spmv_bytes(n, ntiles, nrb, nnz_by_prec, T):
    """Algorithmic bytes of one SpMV launch over EvoCG's Tile-CSC layout: the active value
    stream of every stored entry (sentinels not counted), one row-index byte per entry, per
    tile its column pointers (2(T+1) bytes) and a 12-byte descriptor, the tile row pointers,
    x read once and y written once."""
    vals = 8 * int(nnz_by_prec[0]) + 4 * int(nnz_by_prec[1]) + 2 * int(nnz_by_prec[2])
    return (vals + int(sum(nnz_by_prec)) + (2 * (int(T) + 1) + 12) * int(ntiles) +
            8 * (int(nrb) + 1) + 16 * int(n))


def tile_entries(ex, T):
    """Stored entries (slots that are not pads) of every tile, from an export."""
    real = (ex["colIdx"] < T).astype(np.int64)
    c = np.concatenate([[0], np.cumsum(real)])
    off = ex["tileNnzOff"]
    return c[off[1:]] - c[off[:-1]]


def main(argv=None):
    import torch

    ap = argparse.ArgumentParser()
    ap.add_argument("--workloads", default="2,3,5")
    ap.add_argument("--maps", default="mixed,fp64")
    ap.add_argument("--reps", type=int, default=50)
    ap.add_argument("--launches", type=int, default=0)
    ap.add_argument("--kernel", default="default", choices=["default", "direct", "panel", "rowblock", "rowell"],
                    help="SpMV kernel to time (default: the library's choice)")
    a = ap.parse_args(argv)
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    for cfg in [int(c) for c in a.workloads.split(",") if c]:
        w = W.workload(cfg)
        G = evocg.tile_build(w.n, w.rp, w.ci, w.v, w.T)
        trow, ex = G.tile_rows()
        tnnz = tile_entries(ex, G.T)
        x = torch.from_numpy(np.random.default_rng(7).uniform(-1, 1, w.n)).to(dev)
        y = torch.empty_like(x)
        for label in a.maps.split(","):
            if label == "mixed":
                mp = W.tile_map(trow, ex["tileColIdx"], G.nrb, 12345)
            elif label == "fp32":
                mp = np.ones(G.ntiles, np.uint8)
            elif label == "bf16":
                mp = np.full(G.ntiles, 2, np.uint8)
            else:
                mp = np.zeros(G.ntiles, np.uint8)
            evocg.set_tile_precision(G, mp)
            kflag = {"default": 0, "direct": evocg.SPMV_DIRECT, "panel": evocg.SPMV_PANEL,
                     "rowblock": evocg.SPMV_ROWBLOCK, "rowell": evocg.SPMV_ROWELL}[a.kernel]
            evocg.spmv_ex(G, x, y, kflag)   # makes the x copies the kernel reads, if any
            flags = evocg.SPMV_REUSE_XCOPIES | kflag
            if a.launches:
                for _ in range(a.launches):
                    evocg.spmv_ex(G, x, y, flags)
                torch.cuda.synchronize()
                continue
            for _ in range(5):
                evocg.spmv_ex(G, x, y, flags)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record(stream)
            for _ in range(a.reps):
                evocg.spmv_ex(G, x, y, flags)
            e1.record(stream)
            torch.cuda.synchronize()
            us = e0.elapsed_time(e1) * 1000.0 / a.reps
            per = np.bincount(mp, weights=tnnz, minlength=3).astype(np.int64)
            B = spmv_bytes(G.n, G.ntiles, G.nrb, per, G.T)
            print(json.dumps({"workload": w.name, "map": label,
                              "kernel": a.kernel, "n": w.n, "nnz": w.nnz,
                              "ntiles": int(G.ntiles), "us": round(us, 2), "bytes": B,
                              "gbs": round(B / us / 1e3, 1)}), flush=True)
        G.free()
    return 0


if __name__ == "__main__":
    sys.exit(main())
