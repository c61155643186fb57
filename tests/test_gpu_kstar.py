"""GPU checks of the per-iteration decision log (the profiling run of EvoCG §3.4 interval
reuse) through the C ABI: row k is the column-block map the SpMV of iteration k used, so the
log, weighted by the stored entries of each column block, must reproduce the solve's own
precision census exactly; the reuse interval chosen from it is the oracle's choice on the same
log; a device log and a host log record the same rows; a solve with the chosen interval still
converges."""
import numpy as np
import pytest

import oracle
from helpers import Pair
from mixed_precision_sparse_gb300 import evocg
from mixed_precision_sparse_gb300 import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _entries_per_colblock(P):
    e = np.zeros(P.t.nrb, np.int64)
    np.add.at(e, P.t.tileColIdx.astype(np.int64), P.t.tile_entries())
    return e


def _case(kind):
    if kind == "threshold":
        w = W.workload(2, scale=0.25)      # 32^3 diffusion, Jacobi-PCG, threshold rule
        return w, (lambda: evocg.Ctrl.threshold(w.eps, 1))
    w = W.workload(3, scale=0.25)          # 24^3 FE, Jacobi-PCG, seeded policy
    wts = W.mlp_weights(w.T, w.mlp_seed)
    return w, (lambda: evocg.Ctrl.mlp(wts, 1, w.delta))


@pytest.mark.parametrize("kind", ["threshold", "mlp"])
def test_decision_log_reproduces_the_census(kind):
    w, make = _case(kind)
    P = Pair((w.n, w.rp, w.ci, w.v), w.T)
    rows = w.maxit
    log = np.full((rows, P.t.nrb), 255, np.uint8)             # 255: never written
    bd = torch.from_numpy(w.b).cuda()
    xd = torch.empty(P.n, dtype=torch.float64, device="cuda")
    info = evocg.cg_solve(P.G, bd, xd, w.rtol, w.maxit, True, make().log_to(log), True)
    torch.cuda.synchronize()
    rec = info["iters_recursive"]
    assert info["status"] == evocg.OK and rec > 0
    assert np.all(log[:rec] <= 2) and np.all(log[rec:] == 255)   # the controlled phase only
    ent = _entries_per_colblock(P)
    want = np.zeros(3, np.int64)
    for c in range(3):
        want[c] = int(((log[:rec] == c) * ent[None, :]).sum())
    want[0] += (info["iters"] - rec) * int(ent.sum())          # FP64 finish: every tile FP64
    assert list(info["prec_nnz"]) == list(want)
    # the device log path records the same rows
    logd = torch.full((rows, P.t.nrb), 255, dtype=torch.uint8, device="cuda")
    info2 = evocg.cg_solve(P.G, bd, xd, w.rtol, w.maxit, True, make().log_to(logd), True)
    torch.cuda.synchronize()
    assert info2["iters"] == info["iters"]
    assert np.array_equal(logd.cpu().numpy(), log)
    # the interval chosen from the log: the library's host selection equals the oracle's
    ks, f = evocg.kstar_select(log[:rec])
    ko, fo = oracle.kstar_select(log[:rec])
    assert ks == ko and np.array_equal(f, fo)
    # a solve with the chosen interval converges to the same tolerance
    info3 = evocg.cg_solve(P.G, bd, xd, w.rtol, w.maxit, True, make() if ks == 1 else
                           (evocg.Ctrl.threshold(w.eps, ks) if kind == "threshold" else
                            evocg.Ctrl.mlp(W.mlp_weights(w.T, w.mlp_seed), ks, w.delta)), True)
    torch.cuda.synchronize()
    assert info3["status"] == evocg.OK
    assert oracle.true_residual(P.A, w.b, xd.cpu().numpy()) <= w.rtol
