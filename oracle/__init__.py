"""CPU oracle for the tile-wise mixed-precision CG hot path (test infrastructure).

Only the test-suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this package. It wraps ``oracle.c`` (plain, single-threaded C, FP64) with
ctypes and numpy; it shares no code with the GPU library and never imports it.

The method is the one of "EvoCG: Self-Evolving Precision Control for Faster Conjugate
Gradient" (arXiv 2611.04469); each C function cites the section it restates.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

FP64, FP32, BF16 = 0, 1, 2
OK, EINVAL, ENOMEM, ENOTCONV, EBREAKDOWN = 0, 1, 2, 4, 5


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (-O2, no fused multiply-add) into _build/liboracle.so."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = C.CDLL(_SO)
            P = C.c_void_p
            i64, i32, dbl = C.c_int64, C.c_int, C.c_double
            lib.ora_round_to_format.restype = dbl
            lib.ora_round_to_format.argtypes = [dbl, i32, i32, i32]
            lib.ora_round_f32_array.argtypes = [i64, P, P]
            lib.ora_round_bf16_array.argtypes = [i64, P, P]
            lib.ora_csr_spmv.argtypes = [i64, P, P, P, P, P]
            lib.ora_csr_check.argtypes = [i64, P, P, P]
            lib.ora_csr_check.restype = i32
            lib.ora_col_exp.argtypes = [i64, P, P, P, P]
            lib.ora_tile_csc_count.argtypes = [i64, P, P, i32, i32, P, P, P]
            lib.ora_tile_csc_count.restype = i32
            lib.ora_tile_csc_build.argtypes = [i64, P, P, P, i32, i32] + [P] * 9
            lib.ora_tile_csc_build.restype = i32
            lib.ora_kstar_select.argtypes = [P, i64, i64, C.c_double, P, P, i32]
            lib.ora_kstar_select.restype = i32
            lib.ora_mixed_spmv.argtypes = [i64, P, P, P, i32, P, P, P, P, P, P]
            lib.ora_ctrl_threshold.argtypes = [i64, i32, P, dbl, P]
            lib.ora_ctrl_mlp.argtypes = [i64, i32, P, i32, i32, P, P, P, P, P, P, dbl, P, P]
            lib.ora_true_residual.argtypes = [i64, P, P, P, P, P]
            lib.ora_true_residual.restype = dbl
            lib.ora_cg_flat.argtypes = ([i64, P, P, P, i32, P, P, P, P, P, dbl, i32, i32,
                                         i32, P, dbl, i32, i32, i32] + [P] * 6 +
                                        [dbl, i32, P, P, P, P, P, i64, P, i64])
            lib.ora_cg_flat.restype = i32
            _lib = lib
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


class CSR:
    """A square CSR matrix: int64 row pointers, int32 sorted columns, FP64 values."""

    def __init__(self, n, rp, ci, v):
        self.n = int(n)
        self.rp = _c(rp, np.int64)
        self.ci = _c(ci, np.int32)
        self.v = _c(v, np.float64)


def round_to_format(x: float, frac_bits: int, emin: int, emax: int) -> float:
    return _load().ora_round_to_format(float(x), frac_bits, emin, emax)


def round_f32(x):
    """FP64 -> FP32, round-to-nearest-even, as an FP32 array."""
    x = _c(x, np.float64)
    out = np.empty(x.shape, np.float32)
    _load().ora_round_f32_array(x.size, _p(x), _p(out))
    return out


def round_bf16_bits(x):
    """FP64 -> BF16 (single rounding, nearest-even), as uint16 bit patterns."""
    x = _c(x, np.float64)
    out = np.empty(x.shape, np.uint16)
    _load().ora_round_bf16_array(x.size, _p(x), _p(out))
    return out


def csr_check(A: CSR) -> int:
    return _load().ora_csr_check(A.n, _p(A.rp), _p(A.ci), _p(A.v))


def csr_spmv(A: CSR, x):
    x = _c(x, np.float64)
    y = np.empty(A.n, np.float64)
    _load().ora_csr_spmv(A.n, _p(A.rp), _p(A.ci), _p(A.v), _p(x), _p(y))
    return y


def col_exp(A: CSR):
    e = np.empty(A.n, np.int8)
    _load().ora_col_exp(A.n, _p(A.rp), _p(A.ci), _p(A.v), _p(e))
    return e


class Tiles:
    """The Tile-CSC layout of EvoCG §3.3 (Fig. 4): CSR over row blocks of T x T tiles
    (tileRowPtr, tileColIdx), and inside every tile a CSC: colPtr[t] (T + 1 offsets from
    the tile's first entry tileNnzOff[t]), rowIdx (row within the row block; T is the
    sentinel of a pad), and the FP64 / FP32 / BF16 value streams over the same entries.
    pad = 2 pads every column to even length as the paper does; pad = 1 stores no pads."""

    def __init__(self, A: CSR, T: int, pad: int = 1):
        lib = _load()
        nt, nz, nzp = C.c_int64(), C.c_int64(), C.c_int64()
        st = lib.ora_tile_csc_count(A.n, _p(A.rp), _p(A.ci), int(T), int(pad), C.byref(nt),
                                    C.byref(nz), C.byref(nzp))
        if st != OK:
            raise ValueError(f"tile count failed: status {st}")
        self.n, self.T, self.pad = A.n, int(T), int(pad)
        self.nrb = (A.n + T - 1) // T
        self.ntiles, self.nnz, self.nnz_p = nt.value, nz.value, nzp.value
        self.tileRowPtr = np.empty(self.nrb + 1, np.int64)
        self.tileColIdx = np.empty(max(self.ntiles, 1), np.int32)
        self.tileNnzOff = np.empty(self.ntiles + 1, np.int64)
        self.colPtr = np.empty((max(self.ntiles, 1), T + 1), np.uint16)
        self.rowIdx = np.empty(max(self.nnz_p, 1), np.uint8)
        self.v64 = np.empty(max(self.nnz_p, 1), np.float64)
        self.v32 = np.empty(max(self.nnz_p, 1), np.float32)
        self.v16 = np.empty(max(self.nnz_p, 1), np.uint16)
        self.colExp = np.empty(max(A.n, 1), np.int8)
        st = lib.ora_tile_csc_build(A.n, _p(A.rp), _p(A.ci), _p(A.v), int(T), int(pad),
                                    _p(self.tileRowPtr), _p(self.tileColIdx), _p(self.tileNnzOff),
                                    _p(self.colPtr), _p(self.rowIdx), _p(self.v64), _p(self.v32),
                                    _p(self.v16), _p(self.colExp))
        if st != OK:
            raise ValueError(f"tile build failed: status {st}")
        self.tileColIdx = self.tileColIdx[: self.ntiles]
        self.colPtr = self.colPtr[: self.ntiles]
        self.rowIdx, self.v64 = self.rowIdx[: self.nnz_p], self.v64[: self.nnz_p]
        self.v32, self.v16 = self.v32[: self.nnz_p], self.v16[: self.nnz_p]
        self.colExp = self.colExp[: A.n]

    def tile_rows(self):
        """Row-block index of every tile."""
        return np.repeat(np.arange(self.nrb, dtype=np.int64), np.diff(self.tileRowPtr))

    def tile_entries(self):
        """Stored entries (not sentinels) of every tile."""
        real = (self.rowIdx < self.T).astype(np.int64)
        c = np.concatenate([[0], np.cumsum(real)])
        return c[self.tileNnzOff[1:]] - c[self.tileNnzOff[:-1]]

    def entries(self, t):
        """(local row, local column, stream index) of every entry of tile t in storage
        order, sentinels included (local row T)."""
        off, cp = int(self.tileNnzOff[t]), self.colPtr[t]
        return [(int(self.rowIdx[off + e]), c, off + e)
                for c in range(self.T) for e in range(int(cp[c]), int(cp[c + 1]))]

    def to_csr(self) -> CSR:
        """Rebuild CSR (FP64 stream) from the layout: the round-trip check."""
        T = self.T
        rows, cols, vals = [], [], []
        trow = self.tile_rows()
        for t in range(self.ntiles):
            for r, c, s in self.entries(t):
                if r == T:
                    continue
                rows.append(trow[t] * T + r)
                cols.append(int(self.tileColIdx[t]) * T + c)
                vals.append(self.v64[s])
        rows, cols, vals = np.array(rows, np.int64), np.array(cols, np.int64), np.array(vals)
        order = np.lexsort((cols, rows))
        rows, cols, vals = rows[order], cols[order], vals[order]
        rp = np.zeros(self.n + 1, np.int64)
        np.add.at(rp, rows + 1, 1)
        return CSR(self.n, np.cumsum(rp), cols.astype(np.int32), vals)


def mixed_spmv(A: CSR, tiles: Tiles, tile_prec, x):
    """Emulated mixed-precision SpMV (tile_prec None = every tile FP64)."""
    x = _c(x, np.float64)
    y = np.empty(A.n, np.float64)
    tp = None if tile_prec is None else _c(tile_prec, np.uint8)
    _load().ora_mixed_spmv(A.n, _p(A.rp), _p(A.ci), _p(A.v), tiles.T, _p(tiles.colExp),
                           _p(tiles.tileRowPtr), _p(tiles.tileColIdx), _p(tp), _p(x), _p(y))
    return y


def ctrl_threshold(p, T: int, eps: float):
    p = _c(p, np.float64)
    ncb = (p.size + T - 1) // T
    out = np.empty(ncb, np.uint8)
    _load().ora_ctrl_threshold(p.size, T, _p(p), float(eps), _p(out))
    return out


def ctrl_mlp(p, T: int, weights, delta: float):
    """weights = (W1, b1, W2, b2, W3, b3), FP32, W row-major (out, in). Returns (map, logits)."""
    p = _c(p, np.float64)
    W1, b1, W2, b2, W3, b3 = [_c(w, np.float32) for w in weights]
    H1, H2 = b1.size, b2.size
    ncb = (p.size + T - 1) // T
    out = np.empty(ncb, np.uint8)
    logits = np.empty(ncb * 3, np.float64)
    _load().ora_ctrl_mlp(p.size, T, _p(p), H1, H2, _p(W1), _p(b1), _p(W2), _p(b2), _p(W3),
                         _p(b3), float(delta), _p(out), _p(logits))
    return out, logits.reshape(ncb, 3)


def true_residual(A: CSR, b, x) -> float:
    b, x = _c(b, np.float64), _c(x, np.float64)
    return _load().ora_true_residual(A.n, _p(A.rp), _p(A.ci), _p(A.v), _p(b), _p(x))


def cg(A: CSR, tiles: Tiles, b, rtol: float, maxit: int, jacobi: bool = False,
       ctrl: str = "static", tile_map=None, eps: float = 0.0, kstar: int = 1,
       weights=None, delta: float = 1e-30, finish_fp64: bool = False, replay=None,
       log_rows: int = 0):
    """CG / Jacobi-PCG with a static map, an in-loop controller ('threshold', 'mlp'), or a
    replayed sequence of column-block maps ('replay': row k of `replay` at iteration k, the
    last row past its end).

    Returns a dict: status, x, iters, iters_rec, restarts, hist (iters+1 entries),
    rel_res (recursive), true_res (FP64 recomputed), prec_nnz (entries per precision), and
    with log_rows > 0 `log`: the column-block map in force at each of the first log_rows
    iterations of the controlled phase (rows it did not reach hold 255).
    """
    b = _c(b, np.float64)
    x = np.zeros(A.n, np.float64)
    hist = np.zeros(maxit + 1, np.float64)
    out = np.zeros(3, np.int64)
    fout = np.zeros(2, np.float64)
    pn = np.zeros(3, np.int64)
    kind = {"static": 0, "threshold": 1, "mlp": 2, "replay": 3}[ctrl]
    rp_log = None if replay is None else _c(replay, np.uint8)
    if kind == 3 and (rp_log is None or rp_log.ndim != 2 or rp_log.shape[1] != tiles.nrb):
        raise ValueError("replay needs a (rows, nrb) uint8 map log")
    logo = np.full((max(int(log_rows), 0), tiles.nrb), 255, np.uint8) if log_rows > 0 else None
    tm = None if tile_map is None else _c(tile_map, np.uint8)
    if weights is not None:
        W = [_c(w, np.float32) for w in weights]
        H1, H2 = W[1].size, W[3].size
    else:
        W, H1, H2 = [None] * 6, 0, 0
    st = _load().ora_cg_flat(A.n, _p(A.rp), _p(A.ci), _p(A.v), tiles.T, _p(tiles.tileRowPtr),
                             _p(tiles.tileColIdx), _p(tiles.colExp), _p(b), _p(x), float(rtol),
                             int(maxit), int(bool(jacobi)), kind, _p(tm), float(eps), int(kstar),
                             H1, H2, *[_p(w) for w in W], float(delta), int(bool(finish_fp64)),
                             _p(hist), _p(out), _p(fout), _p(pn), _p(rp_log),
                             0 if rp_log is None else int(rp_log.shape[0]), _p(logo),
                             0 if logo is None else int(logo.shape[0]))
    it = int(out[0])
    res = dict(status=st, x=x, iters=it, iters_rec=int(out[1]), restarts=int(out[2]),
               hist=hist[: it + 1].copy(), rel_res=float(fout[0]), true_res=float(fout[1]),
               prec_nnz=pn.copy())
    if logo is not None:
        res["log"] = logo
    return res


def kstar_select(log, limit: float = 0.1):
    """Reuse interval of EvoCG §3.4 from a (rows, ncb) uint8 decision log: (K*, fractions of
    delayed upward transitions for K = 1, 2, 4, ...)."""
    log = _c(log, np.uint8)
    rows, ncb = log.shape
    ks = C.c_int()
    frac = np.zeros(64)
    nc = _load().ora_kstar_select(_p(log), int(rows), int(ncb), float(limit), C.byref(ks),
                                  _p(frac), 64)
    return ks.value, frac[:nc]
