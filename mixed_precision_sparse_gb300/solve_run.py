"""Run one CG / Jacobi-PCG solve of a synthetic workload through the C ABI and print its info.

    python -m mixed_precision_sparse_gb300.solve_run [--workload 5] [--maxit K] [--fp64]
                                                     [--no-finish] [--relative]

The workload's own settings (preconditioner, controller or static map, rtol, maxit) are used
unless overridden: --maxit caps the iterations (a short run of the same per-iteration kernels,
for profilers), --fp64 sets every tile to FP64 with no controller, --no-finish skips the FP64
finish, --relative scales the threshold rule's cut points by ||b||_inf. Prints one JSON line:
status, iterations, true residual, precision census, seconds (wall clock of the call,
including the graph build on first use). With EVOCG_GRAPH=0 in the
environment every kernel of the solve is a plain launch.
"""
from __future__ import annotations

import argparse
import json
import os
import sys
import time

import numpy as np

if __package__ in (None, ""):
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

from mixed_precision_sparse_gb300 import evocg  # noqa: E402
from mixed_precision_sparse_gb300 import workloads as W  # noqa: E402


def main(argv=None):
    import torch

    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", type=int, default=5)
    ap.add_argument("--maxit", type=int, default=0)
    ap.add_argument("--fp64", action="store_true")
    ap.add_argument("--no-finish", action="store_true")
    ap.add_argument("--relative", action="store_true",
                    help="threshold controller with cut points scaled by ||b||_inf (an option)")
    a = ap.parse_args(argv)
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w = W.workload(a.workload)
    G = evocg.tile_build(w.n, w.rp, w.ci, w.v, w.T)
    ctrl = None
    if a.fp64 or (w.ctrl == "static" and w.map_seed is None):
        evocg.set_tile_precision(G, np.zeros(G.ntiles, np.uint8))
    elif w.ctrl == "threshold":
        ctrl = evocg.Ctrl.threshold(w.eps, relative=a.relative)
    elif w.ctrl == "mlp":
        ctrl = evocg.Ctrl.mlp(W.mlp_weights(w.T, w.mlp_seed), 1, w.delta)
    else:
        trow, ex = G.tile_rows()
        evocg.set_tile_precision(G, W.tile_map(trow, ex["tileColIdx"], G.nrb, w.map_seed))
    b = torch.from_numpy(np.ascontiguousarray(w.b)).to(dev)
    x = torch.empty_like(b)
    maxit = a.maxit if a.maxit > 0 else w.maxit
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    info = evocg.cg_solve(G, b, x, w.rtol, maxit, w.jacobi, ctrl, not a.no_finish)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    print(json.dumps({"workload": w.name, "n": w.n, "nnz": w.nnz, "maxit": maxit, "fp64": a.fp64,
                      "relative": a.relative,
                      "status": info["status"], "iters": info["iters"],
                      "iters_recursive": info["iters_recursive"], "true_res": info["true_res"],
                      "prec_nnz": [int(c) for c in info["prec_nnz"]], "seconds": dt}))
    G.free()
    return 0


if __name__ == "__main__":
    sys.exit(main())
