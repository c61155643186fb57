"""Pins of the oracle's CG / Jacobi-PCG and of its two precision controllers.

CG: the dense Cholesky solution (scipy) within n iterations, monotone A-norm error, the
history against the true residual, exact invariances under power-of-two scalings, and the
status codes. Controllers: boundary cases of the threshold rule, closed-form special
cases and invariances of the MLP, and numpy's matmul forward pass."""
import numpy as np
import pytest
import scipy.linalg as sl

import oracle
from mixed_precision_sparse_gb300 import workloads as W


def _setup(m, T):
    A = oracle.CSR(*m)
    return A, oracle.Tiles(A, T)


@pytest.mark.parametrize("n,seed", [(12, 1), (40, 2), (64, 3)])
def test_cg_reaches_cholesky_solution_within_n_iterations(n, seed):
    m = W.random_spd_small(n, seed, 0.3, shift=1.0)
    A, t = _setup(m, 16)
    M = W.csr_to_dense(*m)
    b = np.random.default_rng(seed).standard_normal(n)
    xs = sl.cho_solve(sl.cho_factor(M), b)
    res = oracle.cg(A, t, b, rtol=1e-13, maxit=4 * n)
    assert res["status"] == oracle.OK
    assert res["iters"] <= n
    assert np.linalg.norm(res["x"] - xs) <= 1e-10 * np.linalg.norm(xs)


def test_cg_a_norm_error_monotone():
    m = W.random_spd_small(50, 7, 0.2, shift=0.2)
    A, t = _setup(m, 16)
    M = W.csr_to_dense(*m)
    b = np.random.default_rng(7).standard_normal(50)
    xs = sl.cho_solve(sl.cho_factor(M), b)
    errs = []
    for k in range(1, 40):
        r = oracle.cg(A, t, b, rtol=0.0, maxit=k)
        e = r["x"] - xs
        errs.append(float(e @ M @ e))
    assert all(errs[i + 1] <= errs[i] * (1 + 1e-12) for i in range(len(errs) - 1))


def test_cg_history_is_relative_residual():
    m = W.laplace2d_5pt(12)
    A, t = _setup(m, 16)
    b = np.random.default_rng(1).uniform(-1, 1, A.n)
    M = W.csr_to_dense(*m)
    full = oracle.cg(A, t, b, rtol=1e-10, maxit=500)
    assert full["status"] == oracle.OK and full["hist"][0] == 1.0
    for k in (1, 5, 10, 20):
        r = oracle.cg(A, t, b, rtol=0.0, maxit=k)
        true = np.linalg.norm(b - M @ r["x"]) / np.linalg.norm(b)
        assert abs(full["hist"][k] - true) <= 1e-12
    assert full["hist"][-1] <= 1e-10 < full["hist"][-2]
    assert full["true_res"] <= 1e-9


def test_jacobi_with_constant_power_of_two_diagonal_equals_cg():
    """Diagonal 4 everywhere: z = r/4 is an exact scaling, so PCG and CG produce the same
    alpha*p and beta at every step and identical histories, bit for bit."""
    w = W.workload(1)
    A, t = _setup((w.n, w.rp, w.ci, w.v), w.T)
    a = oracle.cg(A, t, w.b, rtol=1e-10, maxit=2000, jacobi=False)
    b = oracle.cg(A, t, w.b, rtol=1e-10, maxit=2000, jacobi=True)
    assert a["iters"] == b["iters"]
    assert np.array_equal(a["hist"], b["hist"])
    assert np.array_equal(a["x"], b["x"])


def test_jacobi_pcg_invariant_under_power_of_two_diagonal_scaling():
    """Jacobi-PCG on D A D with right-hand side D b runs the same iteration as on A with b
    (x' = D^-1 x). With D a power of two every operation scales exactly, so the iterates
    agree bit for bit."""
    m = W.diffusion3d_7pt(7, 2)
    n, rp, ci, v = m
    d = 2.0 ** np.random.default_rng(3).integers(-20, 20, n).astype(float)
    rows = np.repeat(np.arange(n), np.diff(rp))
    A, t = _setup(m, 32)
    As, ts = _setup((n, rp, ci, d[rows] * v * d[ci]), 32)
    b = np.random.default_rng(4).uniform(-1, 1, n)
    # the stopping test measures ||r|| unscaled, so compare a fixed number of steps
    for k in (1, 7, 40):
        r1 = oracle.cg(A, t, b, rtol=0.0, maxit=k, jacobi=True)
        r2 = oracle.cg(As, ts, d * b, rtol=0.0, maxit=k, jacobi=True)
        assert r1["iters"] == r2["iters"] == k
        assert np.array_equal(r1["x"], d * r2["x"])


def test_status_codes():
    m = W.dense_to_csr(np.diag([1.0, -1.0, 2.0]))
    A, t = _setup(m, 16)
    r = oracle.cg(A, t, np.array([0.0, 1.0, 0.0]), 1e-10, 10)
    assert r["status"] == oracle.EBREAKDOWN
    m = W.laplace2d_5pt(20)
    A, t = _setup(m, 16)
    b = np.ones(A.n)
    r = oracle.cg(A, t, b, 1e-12, 5)
    assert r["status"] == oracle.ENOTCONV and r["iters"] == 5
    r = oracle.cg(A, t, np.zeros(A.n), 1e-12, 5)
    assert r["status"] == oracle.OK and r["iters"] == 0
    r = oracle.cg(A, t, b, 1e-12, 5, jacobi=True)
    assert r["status"] != oracle.EINVAL
    m = W.dense_to_csr(np.array([[0.0, 1.0], [1.0, 2.0]]))
    A, t = _setup(m, 16)
    assert oracle.cg(A, t, np.ones(2), 1e-10, 10, jacobi=True)["status"] == oracle.EINVAL


def test_finish_fp64_restores_true_residual():
    m = W.diffusion3d_7pt(10, 5)
    A, t = _setup(m, 32)
    b = np.random.default_rng(5).uniform(-1, 1, A.n)
    bf = np.full(t.ntiles, 2, np.uint8)
    plain = oracle.cg(A, t, b, 1e-10, 3000, jacobi=True, tile_map=bf)
    fin = oracle.cg(A, t, b, 1e-10, 3000, jacobi=True, tile_map=bf, finish_fp64=True)
    assert plain["status"] == oracle.OK and plain["true_res"] > 1e-10
    assert fin["status"] == oracle.OK and fin["restarts"] >= 1
    assert fin["true_res"] <= 1e-10
    assert fin["iters_rec"] == plain["iters"] and fin["iters"] > plain["iters"]


def test_precision_census():
    w = W.workload(1)
    A, t = _setup((w.n, w.rp, w.ci, w.v), w.T)
    mp = W.tile_map(t.tile_rows(), t.tileColIdx, t.nrb, 1)
    r = oracle.cg(A, t, w.b, 1e-10, 3000, tile_map=mp)
    per = np.bincount(mp, weights=t.tile_entries(), minlength=3)
    assert np.array_equal(r["prec_nnz"], (per * r["iters"]).astype(np.int64))


# ---------------------------------------------------------------- controllers

def test_threshold_rule_boundaries():
    eps = 1e-8
    lo = 0.1 * eps
    T = 4
    segs = [[lo, 0, 0, 0],                   # m == 0.1 eps -> FP32 (BF16 needs m < 0.1 eps)
            [np.nextafter(lo, 0), 0, 0, 0],  # just below -> BF16
            [0, -eps, 0, 0],                 # m == eps -> FP64
            [0, 0, np.nextafter(-eps, 0), 0],  # just below eps -> FP32
            [0, 0, 0, 0],                    # zero segment -> BF16
            [1e-30, -2e-9, 3e-10, 0],        # m = 2e-9 -> FP32
            [np.nan, 0, 0, 0]]               # not-a-number never passes a '<' test -> FP64
    p = np.array(sum(segs, []), dtype=np.float64)
    assert list(oracle.ctrl_threshold(p, T, eps)) == [1, 2, 0, 1, 2, 1, 0]
    # partial last segment
    assert list(oracle.ctrl_threshold(np.array([1.0, 0, 0, 0, 1e-20]), T, eps)) == [0, 2]


def _forward_np(p, T, w, delta):
    W1, b1, W2, b2, W3, b3 = [np.asarray(a, np.float64) for a in w]
    ncb = (p.size + T - 1) // T
    seg = np.zeros(ncb * T)
    seg[: p.size] = p
    seg = seg.reshape(ncb, T)
    phi = seg / np.maximum(np.linalg.norm(seg, axis=1), delta)[:, None]
    h1 = np.maximum(phi @ W1.T + b1, 0)
    h2 = np.maximum(h1 @ W2.T + b2, 0)
    return h2 @ W3.T + b3


def test_mlp_matches_numpy_forward():
    T = 32
    w = W.mlp_weights(T, 3)
    p = W.p_snapshot(32 * 50 + 7, T, 3)
    mp, lg = oracle.ctrl_mlp(p, T, w, 1e-30)
    want = _forward_np(p, T, w, 1e-30)
    assert np.allclose(lg, want, rtol=0, atol=1e-12)
    assert np.array_equal(mp, np.argmax(lg, axis=1))


def test_mlp_special_cases():
    T = 16
    w = list(W.mlp_weights(T, 4))
    w[4] = np.zeros_like(w[4])                       # W3 = 0: logits are the bias
    for b3, want in [([0.1, 0.5, 0.2], 1), ([0.3, 0.3, 0.1], 0), ([0.1, 0.4, 0.4], 1),
                     ([-1.0, -2.0, 0.0], 2)]:
        w[5] = np.array(b3, np.float32)
        mp, _ = oracle.ctrl_mlp(np.random.default_rng(0).standard_normal(64), T, w, 1e-30)
        assert np.all(mp == want)                    # ties go to the lower code


def test_mlp_normalisation_invariance_and_delta():
    T = 32
    w = W.mlp_weights(T, 5)
    p = np.random.default_rng(6).standard_normal(T * 40)
    s = 2.0 ** np.random.default_rng(7).integers(-30, 30, 40).repeat(T)
    a, la = oracle.ctrl_mlp(p, T, w, 1e-30)
    b, lb = oracle.ctrl_mlp(p * s, T, w, 1e-30)
    assert np.array_equal(a, b) and np.array_equal(la, lb)   # phi is scale free above delta
    tiny = p * 1e-40                                           # ||p_i|| < delta: phi = p/delta
    c, lc = oracle.ctrl_mlp(tiny, T, w, 1e-30)
    want = _forward_np(tiny, T, w, 1e-30)
    assert np.allclose(lc, want, atol=1e-12)
    assert not np.allclose(lc, la)


# ---------------------------------------------------------------- decision log and replay

@pytest.mark.parametrize("kind", ["threshold", "mlp"])
def test_replaying_the_decision_log_reproduces_the_controlled_solve(kind):
    """Row k of the oracle's decision log is the column-block map of iteration k: feeding the
    log back as a fixed schedule must give the controlled solve again, bit for bit, and the
    log weighted by each block's stored entries must give the solve's precision census."""
    if kind == "threshold":
        w = W.workload(2, scale=0.125)
        kw = dict(ctrl="threshold", eps=w.eps)
    else:
        w = W.workload(3, scale=0.125)
        kw = dict(ctrl="mlp", weights=W.mlp_weights(w.T, w.mlp_seed), delta=w.delta)
    A, t = _setup((w.n, w.rp, w.ci, w.v), w.T)
    ref = oracle.cg(A, t, w.b, w.rtol, w.maxit, jacobi=True, finish_fp64=True,
                    log_rows=w.maxit, **kw)
    rec = ref["iters_rec"]
    log = ref["log"]
    assert rec > 0 and np.all(log[:rec] <= 2) and np.all(log[rec:] == 255)
    rep = oracle.cg(A, t, w.b, w.rtol, w.maxit, jacobi=True, finish_fp64=True,
                    ctrl="replay", replay=log[:rec])
    assert rep["iters"] == ref["iters"] and rep["iters_rec"] == rec
    assert np.array_equal(rep["hist"].view(np.uint64), ref["hist"].view(np.uint64))
    assert np.array_equal(rep["x"].view(np.uint64), ref["x"].view(np.uint64))
    ent = np.zeros(t.nrb, np.int64)
    np.add.at(ent, t.tileColIdx.astype(np.int64), t.tile_entries())
    want = np.array([((log[:rec] == c) * ent[None, :]).sum() for c in range(3)], np.int64)
    want[0] += (ref["iters"] - rec) * ent.sum()
    assert np.array_equal(ref["prec_nnz"], want)


def test_replay_of_an_all_fp64_log_is_the_fp64_solve():
    w = W.workload(1)
    A, t = _setup((w.n, w.rp, w.ci, w.v), w.T)
    plain = oracle.cg(A, t, w.b, w.rtol, w.maxit)
    rep = oracle.cg(A, t, w.b, w.rtol, w.maxit, ctrl="replay",
                    replay=np.zeros((3, t.nrb), np.uint8))     # shorter than the solve
    assert rep["iters"] == plain["iters"]
    assert np.array_equal(rep["hist"].view(np.uint64), plain["hist"].view(np.uint64))
