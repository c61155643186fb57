"""Row-block sharding over ranks, on the host: the partition and the local matrices against
the global CSR, and with world size 2 on gloo (127.0.0.1) a distributed SpMV and a
distributed Jacobi-PCG (halo exchange before every SpMV, FP64 all_reduce of the three sums)
against the oracle's single-process SpMV and CG."""
import os
import socket

import numpy as np
import pytest

import oracle
from mixed_precision_sparse_gb300 import shard
from mixed_precision_sparse_gb300 import workloads as W

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


CASES = [("diff3d_12", W.diffusion3d_7pt(12, 4), 32), ("fe3d_8", W.fe3d_q1_27pt(8, 2), 32),
         ("lap2d_ragged", W.laplace2d_5pt(37, 29), 16), ("banded", W.banded_spd(5000, 3, band=300), 64)]


@pytest.mark.parametrize("name,m,T", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("world", [1, 2, 3, 5])
def test_partition_is_contiguous_and_balanced(name, m, T, world):
    n, rp, ci, v = m
    b = shard.partition(n, rp, T, world)
    assert b[0] == 0 and b[-1] == n and np.all(np.diff(b) >= 0)
    assert np.all(b[:-1] % T == 0)                       # row blocks are never split
    per = rp[b[1:]] - rp[b[:-1]]
    rb_max = max(int(rp[min(n, (k + 1) * T)] - rp[k * T]) for k in range((n + T - 1) // T))
    assert per.max() - rp[n] / world <= rb_max           # within one row block of the ideal


@pytest.mark.parametrize("name,m,T", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("world", [2, 3])
def test_local_parts_hold_the_matrix(name, m, T, world):
    """Every rank's local rows, mapped back through its halo, are the global rows; the halo is
    exactly the off-rank columns read; what a rank sends a peer is what the peer receives."""
    n, rp, ci, v = m
    b = shard.partition(n, rp, T, world)
    parts = [shard.local_part(n, rp, ci, v, b, r) for r in range(world)]
    for p in parts:
        back = np.concatenate([np.arange(p.r0, p.r1), p.halo])   # local column -> global
        assert np.all(np.diff(p.row_ptr[p.n_own:]) == 0)         # halo rows empty
        for i in range(p.n_own):
            a, e = p.row_ptr[i], p.row_ptr[i + 1]
            lc = p.col_idx[a:e]
            assert np.all(np.diff(lc) > 0)                       # ascending local columns
            g = back[lc]
            o = np.argsort(g)
            ga, ge = rp[p.r0 + i], rp[p.r0 + i + 1]
            assert np.array_equal(g[o], ci[ga:ge]) and np.array_equal(p.vals[a:e][o], v[ga:ge])
        cols = ci[rp[p.r0]:rp[p.r1]]
        assert np.array_equal(p.halo, np.unique(cols[(cols < p.r0) | (cols >= p.r1)]))
        for q, (lo, hi) in p.recv.items():
            assert np.array_equal(parts[q].send[p.rank] + parts[q].r0, p.halo[lo:hi])
        assert sum(hi - lo for lo, hi in p.recv.values()) == p.halo.size


def _dist_main(rank, world, port, name, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        m, T = {c[0]: (c[1], c[2]) for c in CASES}[name]
        n, rp, ci, v = m
        b = shard.partition(n, rp, T, world)
        p = shard.local_part(n, rp, ci, v, b, rank)
        ex = shard.HaloExchange(p, dist)
        Aloc = oracle.CSR(p.n_ext, p.row_ptr, p.col_idx, p.vals)
        A = oracle.CSR(n, rp, ci, v)

        def allsum(a):
            t = torch.tensor([float(a)], dtype=torch.float64)
            dist.all_reduce(t)
            return float(t.item())

        def spmv(xown):
            xe = torch.zeros(p.n_ext, dtype=torch.float64)
            xe[:p.n_own] = torch.from_numpy(xown)
            ex(xe)
            return oracle.csr_spmv(Aloc, xe.numpy())[:p.n_own]

        # distributed SpMV against the global one, every row
        xg = np.random.default_rng(3).uniform(-1, 1, n)
        y = spmv(xg[p.r0:p.r1].copy())
        want = oracle.csr_spmv(A, xg)[p.r0:p.r1]
        den = oracle.csr_spmv(oracle.CSR(n, rp, ci, np.abs(v)), np.abs(xg))[p.r0:p.r1]
        spmv_err = float(np.max(np.abs(y - want) / np.maximum(den, 1e-300), initial=0.0))
        # distributed Jacobi-PCG (the oracle's order: x0 = 0, stop on ||r|| / ||r0|| <= rtol)
        bg = np.random.default_rng(5).uniform(-1, 1, n)
        diag = np.array([v[rp[i]:rp[i + 1]][ci[rp[i]:rp[i + 1]] == i][0] for i in range(p.r0, p.r1)])
        dinv = 1.0 / diag
        rtol, maxit = 1e-10, 2000
        x = np.zeros(p.n_own)
        r = bg[p.r0:p.r1].copy()
        z = dinv * r
        pv = z.copy()
        rho, rr = allsum(r @ z), allsum(r @ r)
        nr0 = np.sqrt(rr)
        hist = [1.0]
        for _ in range(maxit):
            q = spmv(pv)
            alpha = rho / allsum(pv @ q)
            x += alpha * pv
            r -= alpha * q
            z = dinv * r
            rz, rr = allsum(r @ z), allsum(r @ r)
            hist.append(np.sqrt(rr) / nr0)
            if hist[-1] <= rtol:
                break
            beta = rz / rho
            rho = rz
            pv = z + beta * pv
        ref = oracle.cg(A, oracle.Tiles(A, T), bg, rtol, maxit, jacobi=True)
        k = min(len(hist), len(ref["hist"]))
        hist_err = float(np.max(np.abs(np.array(hist[:k]) - ref["hist"][:k]) / ref["hist"][:k]))
        x_err = float(np.linalg.norm(x - ref["x"][p.r0:p.r1]) / np.linalg.norm(ref["x"]))
        out[rank] = dict(spmv=spmv_err, iters=len(hist) - 1, ref_iters=ref["iters"],
                         hist=hist_err, x=x_err, halo=int(p.halo.size))
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("name", ["diff3d_12", "fe3d_8", "banded"])
def test_distributed_spmv_and_pcg_gloo_world2(name):
    world = 2
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_dist_main, args=(world, _free_port(), name, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        r = res[rank]
        assert r["halo"] > 0                              # the split really exchanges entries
        assert r["spmv"] <= 1e-14, r                      # the same products, another order
        assert abs(r["iters"] - r["ref_iters"]) <= 1, r
        assert r["hist"] <= 1e-8, r
        assert r["x"] <= 1e-9, r
    assert res[0]["iters"] == res[1]["iters"]
