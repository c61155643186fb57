"""Write oracle_iterations.json: the CPU oracle's full-solve iteration count per workload.

The benchmark's reference arm times the oracle on a bounded sample of iterations and
extrapolates with this count; the GPU tests compare the GPU solve's counts with it. For each
workload the file also keeps the first `HEAD` entries of the oracle's residual history
(||r_k|| / ||r_0||) and its recursive-convergence count, which the GPU tests compare on the
large workloads. Only the oracle and the input generator are called here.
Usage: python tests/golden/make_oracle_iterations.py [workload ...]   (default: 2)
"""
import fcntl
import json
import os
import sys
import time

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from mixed_precision_sparse_gb300 import workloads as W  # noqa: E402

HEAD = 201


def _store(path, key, value):
    """Read-modify-write one key of a JSON file under an exclusive lock (several workloads
    may run as separate processes)."""
    with open(path + ".lock", "w") as lk:
        fcntl.flock(lk, fcntl.LOCK_EX)
        out = json.load(open(path)) if os.path.exists(path) else {}
        out[key] = value
        tmp = path + f".tmp{os.getpid()}"
        with open(tmp, "w") as f:
            json.dump(out, f, indent=1, sort_keys=True)
        os.replace(tmp, path)


def main(cfgs):
    path = os.path.join(HERE, "oracle_iterations.json")
    for cfg in cfgs:
        w = W.workload(cfg)
        A = oracle.CSR(w.n, w.rp, w.ci, w.v)
        t = oracle.Tiles(A, w.T)
        kw = dict(jacobi=w.jacobi, finish_fp64=True)
        if w.ctrl == "threshold":
            kw.update(ctrl="threshold", eps=w.eps)
        elif w.ctrl == "mlp":
            kw.update(ctrl="mlp", weights=W.mlp_weights(w.T, w.mlp_seed), delta=w.delta)
        else:
            kw.update(tile_map=W.tile_map(t.tile_rows(), t.tileColIdx, t.nrb, w.map_seed))
        t0 = time.time()
        r = oracle.cg(A, t, w.b, w.rtol, w.maxit, **kw)
        rec = dict(workload=w.name, iters=r["iters"], iters_rec=r["iters_rec"],
                   restarts=r["restarts"], status=r["status"], true_res=r["true_res"],
                   seconds=round(time.time() - t0, 1),
                   hist_head=[float(h) for h in r["hist"][:HEAD]])
        print(cfg, {k: v for k, v in rec.items() if k != "hist_head"}, flush=True)
        _store(path, str(cfg), rec)


if __name__ == "__main__":
    main([int(a) for a in sys.argv[1:]] or [2])
