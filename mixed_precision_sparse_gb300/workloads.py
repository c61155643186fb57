"""Seeded synthetic inputs: SPD matrices, right-hand sides, precision maps, policy weights.

This module only DRAWS inputs. It holds none of the solver's arithmetic (no tiling, no
rounding, no SpMV, no CG), so the GPU library and the CPU oracle can both be fed from it
without sharing any of the method's code. Random numbers the method itself would draw
(static precision maps, policy weights) are produced here and passed in as inputs.

The five workloads stand in for the 47 SuiteSparse SPD matrices of "EvoCG: Self-Evolving
Precision Control for Faster Conjugate Gradient" (§4.1 Datasets), which are not available:
SPD, 10^4..10^7 rows, stencil / finite-element / banded structure, ill-conditioned cases.

Matrices are returned as (n, row_ptr int64, col_idx int32 ascending per row, values FP64).
"""
from __future__ import annotations

import itertools
import math
from dataclasses import dataclass, field

import numpy as np

FP64, FP32, BF16 = 0, 1, 2



def splitmix64(x):
    """SplitMix64 finaliser (Steele, Lea, Flood 2014), vectorised over uint64 arrays."""
    z = np.asarray(x, dtype=np.uint64) + np.uint64(0x9E3779B97F4A7C15)
    z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
    return z ^ (z >> np.uint64(31))


def counter_uniform(keys, seed: int):
    """U[0,1) per integer key: the top 53 bits of splitmix64(key xor mixed seed)."""
    s = splitmix64(np.array([seed], dtype=np.uint64))[0]
    h = splitmix64(np.asarray(keys, dtype=np.uint64) ^ s)
    return (h >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)


# --------------------------------------------------------------------------------------
# matrices
# --------------------------------------------------------------------------------------

def _stencil_csr(dims, offsets, coefs):
    """CSR of a stencil operator on a grid with x fastest (natural order), Dirichlet
    (neighbours outside the grid dropped). offsets: list of integer tuples (dx, dy[, dz]);
    coefs: list of scalars or arrays over the grid nodes (length n)."""
    dims = tuple(int(d) for d in dims)
    n = int(np.prod(dims))
    strides = [1]
    for d in dims[:-1]:
        strides.append(strides[-1] * d)
    lin = [sum(o[a] * strides[a] for a in range(len(dims))) for o in offsets]
    order = np.argsort(lin, kind="stable")
    idx = np.arange(n, dtype=np.int64)
    coord = []
    rem = idx
    for d in dims:
        coord.append((rem % d).astype(np.int32))
        rem = rem // d
    counts = np.zeros(n, np.int64)
    masks, cols, vals = [], [], []
    for s in order:
        o = offsets[s]
        m = np.ones(n, bool)
        for a, d in enumerate(dims):
            if o[a] != 0:
                c = coord[a] + o[a]
                m &= (c >= 0) & (c < d)
        masks.append(m)
        counts += m
    rp = np.zeros(n + 1, np.int64)
    np.cumsum(counts, out=rp[1:])
    nnz = int(rp[-1])
    ci = np.empty(nnz, np.int32)
    v = np.empty(nnz, np.float64)
    fill = rp[:-1].copy()
    for m, s in zip(masks, order):
        rows = idx[m]
        pos = fill[m]
        ci[pos] = (rows + lin[s]).astype(np.int32)
        c = coefs[s]
        v[pos] = c[m] if np.ndim(c) else float(c)
        fill[m] += 1
    return n, rp, ci, v


def laplace2d_5pt(nx: int, ny: int | None = None):
    """2D 5-point Laplacian, Dirichlet: 4 on the diagonal, -1 to each grid neighbour."""
    ny = nx if ny is None else ny
    offs = [(0, -1), (-1, 0), (0, 0), (1, 0), (0, 1)]
    return _stencil_csr((nx, ny), offs, [-1.0, -1.0, 4.0, -1.0, -1.0])


def diffusion3d_7pt(N: int, seed: int, lo: float = -2.0, hi: float = 2.0):
    """3D 7-point finite-volume diffusion on N^3 cells. Every cell face carries one
    coefficient 10^U[lo,hi]; boundary faces couple to a Dirichlet ghost and only add to
    the diagonal. A_ii = sum of the cell's six face coefficients, A_ij = -k_face."""
    rng = np.random.default_rng(seed)
    kx = 10.0 ** rng.uniform(lo, hi, size=(N, N, N + 1))   # [z][y][x-face]
    ky = 10.0 ** rng.uniform(lo, hi, size=(N, N + 1, N))
    kz = 10.0 ** rng.uniform(lo, hi, size=(N + 1, N, N))
    west, east = kx[:, :, :-1].ravel(), kx[:, :, 1:].ravel()
    south, north = ky[:, :-1, :].ravel(), ky[:, 1:, :].ravel()
    down, up = kz[:-1].ravel(), kz[1:].ravel()
    diag = west + east + south + north + down + up
    offs = [(0, 0, -1), (0, -1, 0), (-1, 0, 0), (0, 0, 0), (1, 0, 0), (0, 1, 0), (0, 0, 1)]
    return _stencil_csr((N, N, N), offs, [-down, -south, -west, diag, -east, -north, -up])


def fe3d_q1_27pt(N: int, seed: int, dlo: float = -3.0, dhi: float = 0.0):
    """Trilinear (Q1) finite elements for -Lap(u) + u on the unit cube, N^3 interior nodes
    (h = 1/(N+1)), Dirichlet, divided by h: stencil = stiffness + h^2 * mass, 27 points.
    Then a symmetric random diagonal scaling D A D with D_ii = 10^U[dlo, dhi]."""
    h = 1.0 / (N + 1)
    stiff = {0: 8.0 / 3.0, 1: 0.0, 2: -1.0 / 6.0, 3: -1.0 / 12.0}
    mass = {0: 8.0 / 27.0, 1: 2.0 / 27.0, 2: 1.0 / 54.0, 3: 1.0 / 216.0}
    offs = [o[::-1] for o in itertools.product((-1, 0, 1), repeat=3)]
    coefs = []
    for o in offs:
        m = sum(1 for c in o if c != 0)
        coefs.append(stiff[m] + h * h * mass[m])
    n, rp, ci, v = _stencil_csr((N, N, N), offs, coefs)
    d = 10.0 ** np.random.default_rng(seed).uniform(dlo, dhi, size=n)
    rows = np.repeat(np.arange(n), np.diff(rp))
    v = d[rows] * v * d[ci]
    return n, rp, ci, v


def aniso2d_q1_9pt(N: int, eps: float = 1e-3, theta_deg: float = 30.0):
    """Bilinear (Q1) finite elements for -div(K grad u) on N^2 interior nodes, Dirichlet,
    K = R(theta) diag(1, eps) R(theta)^T. The element matrix is integrated with 2x2 Gauss
    points (exact here) and assembled into the 9-point interior stencil."""
    t = math.radians(theta_deg)
    R = np.array([[math.cos(t), -math.sin(t)], [math.sin(t), math.cos(t)]])
    K = R @ np.diag([1.0, eps]) @ R.T
    g = [0.5 - 0.5 / math.sqrt(3.0), 0.5 + 0.5 / math.sqrt(3.0)]
    nodes = [(0, 0), (1, 0), (0, 1), (1, 1)]

    def grad(a, x, y):
        ax, ay = nodes[a]
        fx = x if ax else 1.0 - x
        fy = y if ay else 1.0 - y
        return np.array([(1.0 if ax else -1.0) * fy, fx * (1.0 if ay else -1.0)])

    Ke = np.zeros((4, 4))
    for x in g:
        for y in g:
            for a in range(4):
                for b in range(4):
                    Ke[a, b] += 0.25 * grad(a, x, y) @ K @ grad(b, x, y)
    sten = {}
    for ex in (-1, 0):
        for ey in (-1, 0):
            pa = nodes.index((-ex, -ey))
            for b, (lx, ly) in enumerate(nodes):
                o = (ex + lx, ey + ly)
                sten[o] = sten.get(o, 0.0) + Ke[pa, b]
    offs = sorted(sten, key=lambda o: (o[1], o[0]))
    return _stencil_csr((N, N), offs, [sten[o] for o in offs])


def banded_spd(n: int, seed: int, per_row: int = 8, band: int = 4096, blk: int = 64,
               ulo: float = -4.0, uhi: float = 0.0, dom: float = 1.05):
    """Random banded SPD: row i draws `per_row` distinct columns in (i, i+band] (fewer near
    the end), each mirrored to (j, i); values N(0,1) * 10^u with u ~ U[ulo,uhi] drawn per
    `blk`-row block of the upper entry's row; diagonal = dom * row abs-sum."""
    rng = np.random.default_rng(seed)
    avail = np.minimum(band, n - 1 - np.arange(n, dtype=np.int64))
    offs = np.zeros((n, per_row), np.int64)
    m = avail >= per_row
    wide = np.nonzero(avail >= 8 * per_row)[0]
    o = 1 + np.floor(rng.random((wide.size, per_row)) * avail[wide, None]).astype(np.int64)
    todo = np.arange(wide.size)
    while todo.size:  # redraw the rows that drew a column twice
        s = np.sort(o[todo], axis=1)
        todo = todo[(s[:, 1:] == s[:, :-1]).any(axis=1)]
        o[todo] = 1 + np.floor(rng.random((todo.size, per_row))
                               * avail[wide[todo], None]).astype(np.int64)
    offs[wide] = o
    for i in np.nonzero(m & (avail < 8 * per_row))[0]:  # narrow rows near the end
        offs[i] = 1 + rng.permutation(int(avail[i]))[:per_row]
    for i in np.nonzero(~m & (avail > 0))[0]:  # the last rows take every column left
        a = int(avail[i])
        offs[i, :a] = np.arange(1, a + 1)
    cnt = np.where(m, per_row, np.maximum(avail, 0))
    valid = np.arange(per_row)[None, :] < cnt[:, None]
    ui = np.repeat(np.arange(n, dtype=np.int64), per_row).reshape(n, per_row)[valid]
    uj = (np.arange(n, dtype=np.int64)[:, None] + offs)[valid]
    ublk = rng.uniform(ulo, uhi, size=(n + blk - 1) // blk)
    uv = rng.standard_normal(ui.size) * 10.0 ** ublk[ui // blk]
    rows = np.concatenate([ui, uj])
    cols = np.concatenate([uj, ui])
    vals = np.concatenate([uv, uv])
    absum = np.bincount(rows, weights=np.abs(vals), minlength=n)
    diag_i = np.arange(n, dtype=np.int64)
    rows = np.concatenate([rows, diag_i])
    cols = np.concatenate([cols, diag_i])
    vals = np.concatenate([vals, dom * absum])
    order = np.argsort(rows * n + cols, kind="stable")
    rows, cols, vals = rows[order], cols[order], vals[order]
    rp = np.zeros(n + 1, np.int64)
    np.cumsum(np.bincount(rows, minlength=n), out=rp[1:])
    return n, rp, cols.astype(np.int32), vals


def random_spd_small(n: int, seed: int, density: float = 0.3, shift: float = 0.5):
    """Small random sparse SPD matrix (symmetric pattern, diagonally dominant)."""
    rng = np.random.default_rng(seed)
    M = rng.standard_normal((n, n)) * (rng.random((n, n)) < density)
    M = np.triu(M, 1)
    M = M + M.T
    M[np.arange(n), np.arange(n)] = np.abs(M).sum(1) + shift + rng.random(n)
    return dense_to_csr(M)


def dense_to_csr(M):
    M = np.asarray(M, dtype=np.float64)
    n = M.shape[0]
    rows, cols = np.nonzero(M)
    rp = np.zeros(n + 1, np.int64)
    np.cumsum(np.bincount(rows, minlength=n), out=rp[1:])
    return n, rp, cols.astype(np.int32), M[rows, cols]


def csr_to_dense(n, rp, ci, v):
    M = np.zeros((n, n))
    rows = np.repeat(np.arange(n), np.diff(rp))
    M[rows, ci] = v
    return M


def csr_matvec(n, rp, ci, v, x):
    """Plain matrix-vector product used only to form right-hand sides (b = A x_true)."""
    import scipy.sparse as sp
    return sp.csr_matrix((v, ci, rp), shape=(n, n)) @ np.asarray(x, np.float64)


# --------------------------------------------------------------------------------------
# precision maps and policy weights
# --------------------------------------------------------------------------------------

def tile_map(tile_rb, tile_cb, ncb: int, seed: int, fracs=(0.4, 0.4, 0.2)):
    """Static per-tile precision map, i.i.d. per tile from a counter-based uniform keyed
    by (row block, column block): u < f0 -> FP64, u < f0+f1 -> FP32, else BF16."""
    key = np.asarray(tile_rb, np.uint64) * np.uint64(ncb) + np.asarray(tile_cb, np.uint64)
    u = counter_uniform(key, seed)
    out = np.full(u.shape, BF16, np.uint8)
    out[u < fracs[0] + fracs[1]] = FP32
    out[u < fracs[0]] = FP64
    return out


def mlp_weights(C: int, seed: int, hidden=(64, 64), n_out: int = 3):
    """Policy-MLP weights for input size C: W ~ U(-1/sqrt(fan_in), 1/sqrt(fan_in)),
    biases likewise; FP32, each W row-major (out, in). Returns (W1, b1, W2, b2, W3, b3)."""
    rng = np.random.default_rng(seed)
    sizes = [C, *hidden, n_out]
    out = []
    for fi, fo in zip(sizes[:-1], sizes[1:]):
        bnd = 1.0 / math.sqrt(fi)
        out.append(rng.uniform(-bnd, bnd, size=(fo, fi)).astype(np.float32))
        out.append(rng.uniform(-bnd, bnd, size=fo).astype(np.float32))
    return tuple(out)


def p_snapshot(n: int, C: int, seed: int, lo: float = -12.0, hi: float = 1.0):
    """A search-direction-like vector: N(0,1) entries whose segments of C are scaled by
    10^U[lo,hi], so segment maxima straddle the threshold rule's cut points."""
    rng = np.random.default_rng(seed)
    ns = (n + C - 1) // C
    scale = np.repeat(10.0 ** rng.uniform(lo, hi, size=ns), C)[:n]
    return rng.standard_normal(n) * scale


# --------------------------------------------------------------------------------------
# the five workloads
# --------------------------------------------------------------------------------------

@dataclass
class Workload:
    name: str
    n: int
    rp: np.ndarray
    ci: np.ndarray
    v: np.ndarray
    b: np.ndarray
    T: int
    rtol: float
    maxit: int
    jacobi: bool
    ctrl: str                   # 'static' (map_seed set, or all FP64), 'threshold', 'mlp'
    eps: float = 0.0            # threshold rule epsilon (= rtol)
    kstar: int = 1
    map_seed: int | None = None  # static 40/40/20 per-tile map
    mlp_seed: int | None = None
    delta: float = 1e-30
    extra: dict = field(default_factory=dict)

    @property
    def nnz(self):
        return int(self.rp[-1])


WORKLOADS = {
    1: "laplace2d_5pt_64x64",
    2: "diffusion3d_7pt_128cubed",
    3: "fe3d_q1_27pt_96cubed_dad",
    4: "banded_spd_4M_bw4096",
    5: "aniso2d_q1_9pt_4096sq",
}


def workload(cfg: int, seed: int | None = None, scale: float = 1.0) -> Workload:
    """Build workload `cfg` (1..5). `scale` < 1 shrinks the grid (tests only; the
    structure, value law and solver settings are those of the full workload)."""
    seed = cfg if seed is None else seed
    rng = np.random.default_rng(1000 + seed)
    if cfg == 1:
        nx = max(4, int(round(64 * scale)))
        n, rp, ci, v = laplace2d_5pt(nx)
        x_true = rng.uniform(-1.0, 1.0, size=n)
        b = csr_matvec(n, rp, ci, v, x_true)
        return Workload(WORKLOADS[1], n, rp, ci, v, b, 16, 1e-10, 20000, False, "static",
                        map_seed=seed, extra=dict(x_true=x_true, grid=nx))
    if cfg == 2:
        N = max(4, int(round(128 * scale)))
        n, rp, ci, v = diffusion3d_7pt(N, seed)
        b = rng.uniform(-1.0, 1.0, size=n)
        return Workload(WORKLOADS[2], n, rp, ci, v, b, 32, 1e-8, 10000, True, "threshold",
                        eps=1e-8, extra=dict(grid=N))
    if cfg == 3:
        N = max(4, int(round(96 * scale)))
        n, rp, ci, v = fe3d_q1_27pt(N, seed)
        b = csr_matvec(n, rp, ci, v, np.ones(n))
        return Workload(WORKLOADS[3], n, rp, ci, v, b, 32, 1e-8, 10000, True, "mlp",
                        mlp_seed=seed, extra=dict(grid=N))
    if cfg == 4:
        n0 = max(8192, int(round(4_000_000 * scale)))
        n, rp, ci, v = banded_spd(n0, seed)
        b = rng.standard_normal(n)
        return Workload(WORKLOADS[4], n, rp, ci, v, b, 64, 1e-8, 10000, False, "static",
                        map_seed=seed)
    if cfg == 5:
        N = max(4, int(round(4096 * scale)))
        n, rp, ci, v = aniso2d_q1_9pt(N)
        b = rng.uniform(-1.0, 1.0, size=n)
        return Workload(WORKLOADS[5], n, rp, ci, v, b, 32, 1e-8, 5000, True, "static",
                        map_seed=seed, extra=dict(grid=N))
    raise ValueError(f"unknown workload {cfg}")
