"""Thin ctypes binding of libevocg.so (C ABI: include/evocg.h). Argument marshalling only:
every step of the solver runs in the library's CUDA kernels.

Arrays may be torch tensors (CUDA or CPU) or numpy arrays; they are passed as raw pointers
and the library detects host vs device memory itself. Streams default to torch's current
CUDA stream. If the library is missing or cannot load, every call raises: there is no
fallback path.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libevocg.so")

OK, EINVAL, ENOMEM, ECUDA, ENOTCONV, EBREAKDOWN, ETIMEOUT, EDEVICE = range(8)
FP64, FP32, BF16 = 0, 1, 2
MAP_PER_TILE, MAP_PER_COLBLOCK = 0, 1
CTRL_STATIC, CTRL_THRESHOLD, CTRL_MLP = 0, 1, 2

_lock = threading.Lock()
_lib = None


class EvocgError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"evocg error {code}: {msg}")
        self.code = code


class TilesDesc(C.Structure):
    _fields_ = [("n", C.c_int64), ("nrb", C.c_int64), ("ntiles", C.c_int64), ("nnz", C.c_int64),
                ("tile_size", C.c_int32), ("map_kind", C.c_int32), ("bytes_index", C.c_int64),
                ("bytes_v64", C.c_int64), ("bytes_v32", C.c_int64), ("bytes_v16", C.c_int64),
                ("bytes_colexp", C.c_int64), ("nslots", C.c_int64)]


class Ctrl(C.Structure):
    _fields_ = [("kind", C.c_int), ("kstar", C.c_int), ("eps", C.c_double),
                ("hidden1", C.c_int), ("hidden2", C.c_int), ("weights", C.c_void_p),
                ("delta", C.c_double), ("map_log", C.c_void_p), ("map_log_rows", C.c_int64),
                ("eps_relative", C.c_int)]

    def log_to(self, log) -> "Ctrl":
        """Record the per-iteration column-block maps into `log` (rows x nrb uint8, a numpy
        array or a CUDA tensor) during the next solves with this controller."""
        self.map_log = _ptr(log)
        self.map_log_rows = int(log.shape[0])
        self._keep_log = log
        return self

    @staticmethod
    def threshold(eps: float, kstar: int = 1, relative: bool = False) -> "Ctrl":
        """EvoCG §4.7's rule with eps absolute, or (relative=True, an option beside the paper's
        rule) with both cut points scaled by ||b||_inf."""
        return Ctrl(kind=CTRL_THRESHOLD, kstar=kstar, eps=eps, eps_relative=int(bool(relative)))

    @staticmethod
    def mlp(weights, kstar: int = 1, delta: float = 1e-30) -> "Ctrl":
        """weights = (W1, b1, W2, b2, W3, b3) as FP32 arrays, W row-major (out, in)."""
        ws = [np.ascontiguousarray(w, dtype=np.float32).ravel() for w in weights]
        packed = np.concatenate(ws)
        c = Ctrl(kind=CTRL_MLP, kstar=kstar, hidden1=int(ws[1].size), hidden2=int(ws[3].size),
                 weights=packed.ctypes.data, delta=delta)
        c._keep = packed  # keep the packed weights alive with the struct
        return c


class SolveInfo(C.Structure):
    _fields_ = [("status", C.c_int), ("iters", C.c_int), ("iters_recursive", C.c_int),
                ("restarts", C.c_int), ("rel_res", C.c_double), ("true_res", C.c_double),
                ("prec_nnz", C.c_int64 * 3), ("ctrl_calls", C.c_int64)]

    def as_dict(self):
        return dict(status=self.status, iters=self.iters, iters_recursive=self.iters_recursive,
                    restarts=self.restarts, rel_res=self.rel_res, true_res=self.true_res,
                    prec_nnz=[int(v) for v in self.prec_nnz], ctrl_calls=int(self.ctrl_calls))


def lib():
    """Load libevocg.so (raises if it is missing: build it with build.build())."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise EvocgError(EDEVICE, f"{LIB_PATH} is missing; run "
                                 "mixed_precision_sparse_gb300.build.build() first")
            try:
                import torch  # noqa: F401  (loads the CUDA runtime the library shares)
            except Exception:
                pass
            L = C.CDLL(LIB_PATH)
            P, i64, i32, dbl = C.c_void_p, C.c_int64, C.c_int, C.c_double
            sig = {
                "evocg_tile_build": [i64, P, P, P, i32, C.POINTER(C.c_void_p)],
                "evocg_tiles_free": [P],
                "evocg_tiles_info": [P, C.POINTER(TilesDesc)],
                "evocg_tiles_export": [P] + [P] * 10,
                "evocg_set_tile_precision": [P, P, i64, i32, P],
                "evocg_get_tile_precision": [P, P, i64, P],
                "evocg_spmv": [P, P, P, P],
                "evocg_spmv_ex": [P, P, P, i32, P],
                "evocg_spmv_noalloc": [P, P, P, P],
                "evocg_cg_solve": [P, P, P, dbl, i32, i32, C.POINTER(Ctrl), i32, P,
                                   C.POINTER(SolveInfo), P],
                "evocg_ctrl_decide": [P, C.POINTER(Ctrl), P, P, P, P],
                "evocg_round": [P, i64, P, P, P],
                "evocg_kstar_select": [P, i64, i64, dbl, C.POINTER(C.c_int), P, i32,
                                       C.POINTER(C.c_int)],
                "evocg_tile_layout_host": [i64, P, P, P, i32, C.POINTER(C.c_int64),
                                           C.POINTER(C.c_int64)] + [P] * 10,
                "evocg_panel_plan_host": [i64, P, P, P, i32, i64, i32, C.POINTER(C.c_int64),
                                          C.POINTER(C.c_int)],
                "evocg_rowblock_plan_host": [i64, P, P, P, i32, C.POINTER(C.c_int64),
                                             C.POINTER(C.c_int64), C.POINTER(C.c_int)],
                "evocg_rowell_plan_host": [i64, P, P, P, i32, C.POINTER(C.c_int64), C.POINTER(C.c_int)],
                "evocg_tile_csc_host": [i64, P, P, P, i32, i32, C.POINTER(C.c_int64),
                                        C.POINTER(C.c_int64)] + [P] * 9,
                "evocg_tiles_export_csc": [P, i32, C.POINTER(C.c_int64)] + [P] * 9,
                "evocg_version": [],
            }
            for name, args in sig.items():
                f = getattr(L, name)
                f.argtypes = args
                f.restype = i32
            L.evocg_last_error.argtypes = []
            L.evocg_last_error.restype = C.c_char_p
            _lib = L
    return _lib


def last_error() -> str:
    return lib().evocg_last_error().decode()


def _check(code, allow=(OK,)):
    if code not in allow:
        raise EvocgError(code, last_error())
    return code


def _ptr(a):
    """Raw pointer of a torch tensor or numpy array (None -> NULL)."""
    if a is None:
        return None
    if hasattr(a, "data_ptr"):
        if not a.is_contiguous():
            raise ValueError("arrays must be contiguous")
        return a.data_ptr()
    if isinstance(a, np.ndarray):
        if not a.flags["C_CONTIGUOUS"]:
            raise ValueError("arrays must be contiguous")
        return a.ctypes.data
    raise TypeError(f"unsupported array type {type(a)}")


def _stream(stream):
    if stream is not None:
        return stream if isinstance(stream, int) else stream.cuda_stream
    try:
        import torch
        if torch.cuda.is_available():
            return torch.cuda.current_stream().cuda_stream
    except Exception:
        pass
    return None


def _np(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


class Tiles:
    """Handle of a tile structure on the current CUDA device."""

    def __init__(self, handle):
        self.h = C.c_void_p(handle)
        d = TilesDesc()
        _check(lib().evocg_tiles_info(self.h, C.byref(d)))
        self.n, self.nrb, self.ntiles, self.nnz = d.n, d.nrb, d.ntiles, d.nnz
        self.nslots = d.nslots
        self.T = d.tile_size
        self.desc = d

    def info(self) -> TilesDesc:
        d = TilesDesc()
        _check(lib().evocg_tiles_info(self.h, C.byref(d)))
        return d

    def free(self):
        if self.h:
            lib().evocg_tiles_free(self.h)
            self.h = C.c_void_p(0)

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass

    def export(self) -> dict:
        ns = self.nslots
        out = dict(tileRowPtr=np.empty(self.nrb + 1, np.int64),
                   tileColIdx=np.empty(self.ntiles, np.int32),
                   tileNnzOff=np.empty(self.ntiles + 1, np.int64),
                   rowMask=np.empty(self.ntiles, np.uint64),
                   tileWidth=np.empty(self.ntiles, np.uint8),
                   colIdx=np.empty(ns, np.uint8), v64=np.empty(ns, np.float64),
                   v32=np.empty(ns, np.float32), v16=np.empty(ns, np.uint16),
                   colExp=np.empty(self.n, np.int8))
        ks = ["tileRowPtr", "tileColIdx", "tileNnzOff", "rowMask", "tileWidth", "colIdx", "v64",
              "v32", "v16", "colExp"]
        _check(lib().evocg_tiles_export(self.h, *[_ptr(out[k]) for k in ks]))
        return out

    def tile_rows(self):
        ex = self.export()
        return np.repeat(np.arange(self.nrb, dtype=np.int64), np.diff(ex["tileRowPtr"])), ex

    def export_csc(self, pad: int = 1) -> dict:
        """The device-resident structure rewritten as EvoCG's Tile-CSC (evocg_tiles_export_csc)."""
        nzp = C.c_int64()
        _check(lib().evocg_tiles_export_csc(self.h, int(pad), C.byref(nzp), *[None] * 9))
        out = _csc_arrays(self.n, self.T, self.ntiles, nzp.value)
        _check(lib().evocg_tiles_export_csc(self.h, int(pad), None, *[_ptr(out[k]) for k in _CSC_KEYS]))
        out["ntiles"], out["nnz_p"] = self.ntiles, nzp.value
        return out


_CSC_KEYS = ["tileRowPtr", "tileColIdx", "tileNnzOff", "colPtr", "rowIdx", "v64", "v32", "v16",
             "colExp"]


def _csc_arrays(n, T, ntiles, nnz_p):
    nrb = (int(n) + T - 1) // T
    return dict(tileRowPtr=np.empty(nrb + 1, np.int64), tileColIdx=np.empty(ntiles, np.int32),
                tileNnzOff=np.empty(ntiles + 1, np.int64),
                colPtr=np.empty((ntiles, T + 1), np.uint16), rowIdx=np.empty(nnz_p, np.uint8),
                v64=np.empty(nnz_p, np.float64), v32=np.empty(nnz_p, np.float32),
                v16=np.empty(nnz_p, np.uint16), colExp=np.empty(int(n), np.int8))


def tile_csc_host(n, row_ptr, col_idx, vals, tile_size: int, pad: int = 1) -> dict:
    """EvoCG's Tile-CSC written by the library's builder on the host (no GPU): a dict of
    tileRowPtr, tileColIdx, tileNnzOff, colPtr (ntiles x (T+1)), rowIdx, v64, v32, v16,
    colExp, plus ntiles and nnz_p."""
    rp, ci, v = _np(row_ptr, np.int64), _np(col_idx, np.int32), _np(vals, np.float64)
    nt, nzp = C.c_int64(), C.c_int64()
    T = int(tile_size)
    _check(lib().evocg_tile_csc_host(int(n), _ptr(rp), _ptr(ci), _ptr(v), T, int(pad),
                                     C.byref(nt), C.byref(nzp), *[None] * 9))
    out = _csc_arrays(n, T, nt.value, nzp.value)
    _check(lib().evocg_tile_csc_host(int(n), _ptr(rp), _ptr(ci), _ptr(v), T, int(pad), None, None,
                                     *[_ptr(out[k]) for k in _CSC_KEYS]))
    out["ntiles"], out["nnz_p"] = nt.value, nzp.value
    return out


def tile_build(n, row_ptr, col_idx, vals, tile_size: int) -> Tiles:
    rp, ci, v = _np(row_ptr, np.int64), _np(col_idx, np.int32), _np(vals, np.float64)
    h = C.c_void_p()
    _check(lib().evocg_tile_build(int(n), _ptr(rp), _ptr(ci), _ptr(v), int(tile_size),
                                  C.byref(h)))
    return Tiles(h.value)


def tile_layout_host(n, row_ptr, col_idx, vals, tile_size: int) -> dict:
    """The tile layout evocg_tile_build would make, computed on the host (no GPU): a dict of
    the arrays evocg_tiles_export returns, plus ntiles and nslots."""
    rp, ci, v = _np(row_ptr, np.int64), _np(col_idx, np.int32), _np(vals, np.float64)
    nt, ns = C.c_int64(), C.c_int64()
    nul = [None] * 10
    _check(lib().evocg_tile_layout_host(int(n), _ptr(rp), _ptr(ci), _ptr(v), int(tile_size),
                                        C.byref(nt), C.byref(ns), *nul))
    T = int(tile_size)
    nrb = (int(n) + T - 1) // T
    out = dict(tileRowPtr=np.empty(nrb + 1, np.int64), tileColIdx=np.empty(nt.value, np.int32),
               tileNnzOff=np.empty(nt.value + 1, np.int64), rowMask=np.empty(nt.value, np.uint64),
               tileWidth=np.empty(nt.value, np.uint8), colIdx=np.empty(ns.value, np.uint8),
               v64=np.empty(ns.value, np.float64), v32=np.empty(ns.value, np.float32),
               v16=np.empty(ns.value, np.uint16), colExp=np.empty(int(n), np.int8))
    ks = ["tileRowPtr", "tileColIdx", "tileNnzOff", "rowMask", "tileWidth", "colIdx", "v64",
          "v32", "v16", "colExp"]
    _check(lib().evocg_tile_layout_host(int(n), _ptr(rp), _ptr(ci), _ptr(v), T, None, None,
                                        *[_ptr(out[k]) for k in ks]))
    out["ntiles"], out["nslots"] = nt.value, ns.value
    return out


def panel_plan_host(n, row_ptr, col_idx, vals, tile_size: int, warps: int, stage_bytes: int = 4096):
    """(batches, valid) of the panel SpMV's plan for `warps` warps and stages of stage_bytes,
    on the host."""
    rp, ci, v = _np(row_ptr, np.int64), _np(col_idx, np.int32), _np(vals, np.float64)
    nb, ok = C.c_int64(), C.c_int()
    _check(lib().evocg_panel_plan_host(int(n), _ptr(rp), _ptr(ci), _ptr(v), int(tile_size),
                                       int(warps), int(stage_bytes), C.byref(nb), C.byref(ok)))
    return nb.value, bool(ok.value)


def rowblock_plan_host(n, row_ptr, col_idx, vals, tile_size: int):
    """(descriptors, single-entry ELL slots, valid) of the row-block SpMV's plan, on the host."""
    rp, ci, v = _np(row_ptr, np.int64), _np(col_idx, np.int32), _np(vals, np.float64)
    nd, ns, ok = C.c_int64(), C.c_int64(), C.c_int()
    _check(lib().evocg_rowblock_plan_host(int(n), _ptr(rp), _ptr(ci), _ptr(v), int(tile_size),
                                          C.byref(nd), C.byref(ns), C.byref(ok)))
    return nd.value, ns.value, bool(ok.value)


def rowell_plan_host(n, row_ptr, col_idx, vals, tile_size: int):
    """(ELL slots, valid) of the row-ELL SpMV's plan, on the host."""
    rp, ci, v = _np(row_ptr, np.int64), _np(col_idx, np.int32), _np(vals, np.float64)
    ns, ok = C.c_int64(), C.c_int()
    _check(lib().evocg_rowell_plan_host(int(n), _ptr(rp), _ptr(ci), _ptr(v), int(tile_size),
                                        C.byref(ns), C.byref(ok)))
    return ns.value, bool(ok.value)


def set_tile_precision(A: Tiles, prec_map, map_kind: int = MAP_PER_TILE, stream=None):
    m = prec_map if hasattr(prec_map, "data_ptr") else _np(prec_map, np.uint8)
    n = m.numel() if hasattr(m, "numel") else m.size
    _check(lib().evocg_set_tile_precision(A.h, _ptr(m), int(n), int(map_kind), _stream(stream)))


def get_tile_precision(A: Tiles, stream=None):
    out = np.empty(A.ntiles, np.uint8)
    _check(lib().evocg_get_tile_precision(A.h, _ptr(out), A.ntiles, _stream(stream)))
    return out


SPMV_REUSE_XCOPIES = 1
SPMV_DIRECT = 2
SPMV_PANEL = 8
SPMV_TEST_LOST_WAIT = 16
SPMV_ROWBLOCK = 32
SPMV_ROWELL = 64


def spmv(A: Tiles, x, y, stream=None):
    _check(lib().evocg_spmv(A.h, _ptr(x), _ptr(y), _stream(stream)))
    return y


def spmv_noalloc(A: Tiles, x, y, stream=None):
    """evocg_spmv_noalloc: the same product with no allocation (device x, y; n <= 2^20)."""
    _check(lib().evocg_spmv_noalloc(A.h, _ptr(x), _ptr(y), _stream(stream)))
    return y


def spmv_ex(A: Tiles, x, y, flags: int = 0, stream=None):
    _check(lib().evocg_spmv_ex(A.h, _ptr(x), _ptr(y), int(flags), _stream(stream)))
    return y


def cg_solve(A: Tiles, b, x, rtol: float, maxit: int, jacobi: bool = False, ctrl: Ctrl = None,
             finish_fp64: bool = False, res_hist=None, stream=None) -> dict:
    """Returns the solve info as a dict (status OK, ENOTCONV or EBREAKDOWN; other codes raise)."""
    info = SolveInfo()
    code = lib().evocg_cg_solve(A.h, _ptr(b), _ptr(x), float(rtol), int(maxit), int(bool(jacobi)),
                                C.byref(ctrl) if ctrl is not None else None,
                                int(bool(finish_fp64)), _ptr(res_hist), C.byref(info),
                                _stream(stream))
    _check(code, allow=(OK, ENOTCONV, EBREAKDOWN))
    return info.as_dict()


def ctrl_decide(A: Tiles, ctrl: Ctrl, p, cb_prec, logits=None, stream=None):
    _check(lib().evocg_ctrl_decide(A.h, C.byref(ctrl), _ptr(p), _ptr(cb_prec), _ptr(logits),
                                   _stream(stream)))
    return cb_prec


def kstar_select(map_log, limit: float = 0.1):
    """Reuse interval K* (EvoCG §3.4) from a (rows, nrb) host decision log: (K*, fractions of
    delayed upward transitions for K = 1, 2, 4, ...)."""
    log = _np(map_log, np.uint8)
    rows, ncb = log.shape
    ks, nc = C.c_int(), C.c_int()
    frac = np.zeros(64)
    _check(lib().evocg_kstar_select(_ptr(log), int(rows), int(ncb), float(limit), C.byref(ks),
                                    _ptr(frac), 64, C.byref(nc)))
    return ks.value, frac[: nc.value]


def round_fp(x, out32=None, out16=None, stream=None):
    n = x.numel() if hasattr(x, "numel") else x.size
    _check(lib().evocg_round(_ptr(x), int(n), _ptr(out32), _ptr(out16), _stream(stream)))


def version() -> int:
    return lib().evocg_version()
