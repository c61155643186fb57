"""Arithmetic rates of the GPU the kernels run on (probe/rates.cu; not part of the solver).

    python -m mixed_precision_sparse_gb300.rates [--blocks-per-sm 4] [--ms 10]

Prints one JSON line per operation: FP64 FMA, FP32 FMA, the hardware FP64->FP32 and
FP32->FP64 conversions, and the integer-pipe FP64->FP32 rounding the kernels use instead,
each as operations per second (CUDA events) and per clock per SM at the maximum SM clock. The
conversion probes carry one 64-bit integer add and one FP32 add (or an integer OR and add)
per conversion, so their figures are lower bounds on the conversion alone.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import sys

if __package__ in (None, ""):
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

from mixed_precision_sparse_gb300 import build as B  # noqa: E402

KINDS = ["fp64_fma", "fp32_fma", "cvt_f64_to_f32", "cvt_f32_to_f64", "int_round_f64_to_f32"]


def probe(lib, kind, bps, iters):
    ops, per_clk, ms = ctypes.c_double(), ctypes.c_double(), ctypes.c_double()
    rc = lib.evocg_rate_probe(kind, bps, iters, ctypes.byref(ops), ctypes.byref(per_clk), ctypes.byref(ms))
    if rc:
        raise RuntimeError(f"evocg_rate_probe({KINDS[kind]}) failed with CUDA error {rc}")
    return ops.value, per_clk.value, ms.value


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--blocks-per-sm", type=int, default=4)
    ap.add_argument("--ms", type=float, default=10.0, help="target duration of the timed launch")
    a = ap.parse_args(argv)
    lib = ctypes.CDLL(B.build_probe())
    lib.evocg_rate_probe.restype = ctypes.c_int
    lib.evocg_rate_probe.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int] + [ctypes.POINTER(ctypes.c_double)] * 3
    for k, name in enumerate(KINDS):
        it, ms = 64, 0.0
        while it < 2_000_000:   # grow until the launch is long enough to scale from
            _, _, ms = probe(lib, k, a.blocks_per_sm, it)
            if ms >= 1.0:
                break
            it *= 4
        it = int(max(64, min(2_000_000, it * a.ms / max(ms, 1e-3))))
        ops, per_clk, ms = probe(lib, k, a.blocks_per_sm, it)
        print(json.dumps({"op": name, "ops_per_clk_per_sm_at_max_clock": round(per_clk, 3), "ops_per_s": ops,
                          "ms": round(ms, 3), "iters": it, "blocks_per_sm": a.blocks_per_sm,
                          "threads_per_block": 256, "chains_per_thread": 8}), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
