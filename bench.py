"""Benchmark: CG time-to-solution of the tile-wise mixed-precision solver on one GB300.

Workload (default): Q1 bilinear 9-point anisotropic diffusion on a 4096 x 4096 grid
(n = 16,777,216, nnz = 150,945,796; the largest single-GPU configuration), ratio 1e3 rotated
30 degrees, b ~ U[-1,1], 32 x 32 tiles, Jacobi-PCG, rtol 1e-8, maxit 5000, the seeded
40/40/20 FP64/FP32/BF16 per-tile map, FP64 finish. A step is one full solve (mixed SpMV with
fused p.q, fused updates, the graph-driven loop and the FP64 true-residual check), inputs
resident in HBM. `--workload N` selects another of the five configurations.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload N]

N > 1 runs N independent replicas (one solve per rank per step, weak scaling); launch it
with torch.distributed.run. `--impl reference` times the CPU oracle on the host cores on a
bounded sample of the same workload and prints the same JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "CG time-to-solution (s) and mixed-precision SpMV HBM GB/s vs GB300 peak"
REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
           0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
           0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
           0x100: "display_clock_setting"}


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi SM clock and throttle reasons, sampled every 200 ms in the background; the
    timed region starts once the first sample has arrived (at most 3 s of waiting)."""

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.t = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index),
                 "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            t0 = time.time()
            while not self.lines and self.proc.poll() is None and time.time() - t0 < 3.0:
                time.sleep(0.01)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            if self.t:
                self.t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], None, set()
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 3:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
                bits = int(parts[2], 16)
            except ValueError:
                continue
            for b, name in REASONS.items():
                if bits & b:
                    reasons.add(name)
        reasons.discard("gpu_idle")
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def _workload(cfg):
    from mixed_precision_sparse_gb300 import workloads as W
    return W.workload(cfg)


def _traffic_for(kernel_src_hash, workload):
    """Per-launch DRAM bytes of the SpMV from the committed ncu summary, if it was taken on
    this workload and on the current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", "spmv_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if d.get("kernel_src_sha256") != kernel_src_hash or d.get("workload", "").split(",")[0] != workload:
        return None
    return d.get("bytes_per_launch_full_size")


def _spmv_kernel_label(G, dev):
    """Which SpMV kernel the solve runs on this structure (the library's automatic choice):
    the row-block kernel for tiles of 32, the panel kernel for 16, and for 64 the row-ELL
    kernel when its plan exists (tiles holding about one entry per row), else the direct one."""
    import torch

    from mixed_precision_sparse_gb300 import evocg
    if G.T == 32:
        return "spmv_rowblock_kernel (warp per 32-row block, lane per row; single-entry tiles staged by cp.async)"
    if G.T == 16:
        return "spmv_panel_kernel (tiles of 16)"
    x = torch.zeros(G.n, dtype=torch.float64, device=dev)
    y = torch.empty_like(x)
    try:
        evocg.spmv_ex(G, x, y, evocg.SPMV_ROWELL)
        return "spmv_rowell_kernel (row-ELL interior for tiles of 64 holding about one entry per row)"
    except evocg.EvocgError:
        return "spmv_kernel (direct, tiles of 64)"


def _src_hash():
    """Hash of what the SpMV kernels are built from: the kernel sources, the host planner and
    builder whose layout they read, and the internal header."""
    csrc = os.path.join(ROOT, "mixed_precision_sparse_gb300", "csrc")
    h = hashlib.sha256()
    for name in ("spmv_rowblock.cu", "rowblock_plan.cpp", "tile_build.cpp", "spmv.cu", "fpconv.cuh",
                 "evocg_internal.h"):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


# --------------------------------------------------------------------------------------
# CPU oracle (reference arm and cpu_baseline)
# --------------------------------------------------------------------------------------

def _oracle_iterations(cfg):
    p = os.path.join(ROOT, "tests", "golden", "oracle_iterations.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        v = d.get(str(cfg))
        if v:
            return int(v["iters"])
    return None


def default_sample_iters(w):
    """Oracle iterations for about 10-20 s of single-core CPU work (the oracle runs at roughly
    25 ns per stored entry and iteration)."""
    return max(2, min(40, int(round(15.0 / (2.6e-8 * max(w.nnz, 1))))))


def oracle_sample(w, sample_iters):
    """Time `sample_iters` iterations of the oracle's solve of workload w (single thread), with
    the workload's own map or controller. Returns seconds per iteration."""
    import oracle
    from mixed_precision_sparse_gb300 import workloads as W
    A = oracle.CSR(w.n, w.rp, w.ci, w.v)
    t = oracle.Tiles(A, w.T)
    kw = dict(jacobi=w.jacobi)
    if w.ctrl == "threshold":
        kw.update(ctrl="threshold", eps=w.eps)
    elif w.ctrl == "mlp":
        kw.update(ctrl="mlp", weights=W.mlp_weights(w.T, w.mlp_seed), delta=w.delta)
    else:
        kw.update(tile_map=W.tile_map(t.tile_rows(), t.tileColIdx, t.nrb, w.map_seed))
    t0 = time.perf_counter()
    r = oracle.cg(A, t, w.b, 0.0, sample_iters, **kw)
    el = time.perf_counter() - t0
    return el / max(1, r["iters"]), r


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    w = _workload(args.workload)
    iters_full = _oracle_iterations(args.workload)
    sample = args.cpu_sample_iters or max(1, default_sample_iters(w) // 2)
    times = []
    for _ in range(args.warmup):
        oracle_sample(w, 1)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        sec_it, _ = oracle_sample(w, sample)
        times.append(sec_it)
    wall = time.perf_counter() - t0
    sec_it = statistics.median(times)
    value = sec_it * iters_full if iters_full else None
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * wall / max(1, args.steps), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "n": w.n, "nnz": w.nnz, "tile": w.T,
                   "solver": "jacobi-pcg" if w.jacobi else "cg", "rtol": w.rtol,
                   "controller": w.ctrl, "parallelism": "replicas"},
        "cpu_baseline": {"value": value, "unit": "s", "cores": 1, "kind": "oracle",
                         "sample": f"{sample} iterations per step, seconds/iteration x "
                                   f"{iters_full} iterations of the oracle's full solve"},
        "e2e": {"value": value, "unit": "s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------------------

def max_over_ranks(v, dist, device):
    """The largest of the ranks' values (the job's clock is its slowest replica); v itself
    on a single process (dist None)."""
    if not dist:
        return float(v)
    import torch
    t = torch.tensor([float(v)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_seconds_per_solve(ms_per_step, world):
    """Whole-job time per solve: every rank runs one solve per step (independent replicas),
    so a step of ms_per_step milliseconds completes `world` solves."""
    return ms_per_step / 1000.0 / world


def spmv_measure(G, w, dev, stream, peak, reps=50, cold_reps=10):
    """SpMV alone on workload w's structure G: microseconds per launch warm and with L2
    flushed, algorithmic bytes, GB/s and fractions of the peak, for the seeded 40/40/20 map
    and the all-FP64 map (the latter also against the FP64 pipe's rate)."""
    import numpy as np
    import torch

    from mixed_precision_sparse_gb300 import evocg, spmv_run
    from mixed_precision_sparse_gb300 import workloads as W
    trow, ex = G.tile_rows()
    tnnz = spmv_run.tile_entries(ex, G.T)
    xs = torch.from_numpy(np.random.default_rng(7).uniform(-1, 1, w.n)).to(dev)
    ys = torch.empty_like(xs)
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0)) or (128 << 20)
    flush = torch.empty(2 * l2 // 4, dtype=torch.float32, device=dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    out = {}
    for label, mp in (("mixed_40_40_20", W.tile_map(trow, ex["tileColIdx"], G.nrb, 12345)),
                      ("fp64", np.zeros(G.ntiles, np.uint8))):
        evocg.set_tile_precision(G, mp)
        evocg.spmv(G, xs, ys)
        for _ in range(5):
            evocg.spmv_ex(G, xs, ys, evocg.SPMV_REUSE_XCOPIES)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(reps):
            evocg.spmv_ex(G, xs, ys, evocg.SPMV_REUSE_XCOPIES)
        e1.record(stream)
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1000.0 / reps
        cold = []
        for _ in range(cold_reps):
            flush.fill_(1.0)
            e0.record(stream)
            evocg.spmv_ex(G, xs, ys, evocg.SPMV_REUSE_XCOPIES)
            e1.record(stream)
            torch.cuda.synchronize()
            cold.append(e0.elapsed_time(e1) * 1000.0)
        per = np.bincount(mp, weights=tnnz, minlength=3).astype(np.int64)
        B = spmv_run.spmv_bytes(w.n, G.ntiles, G.nrb, per, G.T)
        cus = statistics.median(cold)
        out[label] = {"us": us, "bytes": int(B), "gbs": B / us / 1e3,
                      "frac_of_peak": B / us / 1e3 / peak, "frac_of_8tbs": B / us / 1e3 / 8000.0,
                      "cold": {"us": cus, "gbs": B / cus / 1e3, "frac_of_peak": B / cus / 1e3 / peak}}
    # all-FP64: one FP64 fused multiply-add per stored entry, against the FP64 pipe's rate
    out["fp64"]["fp64_fma_per_s"] = int(per.sum()) / (out["fp64"]["us"] * 1e-6)
    return out


def extra_workload(cfg, dev, stream, peak, steps=3):
    """The solve and the SpMV of another configuration, outside the timed region."""
    import torch

    from mixed_precision_sparse_gb300 import evocg
    from mixed_precision_sparse_gb300 import workloads as W
    w = _workload(cfg)
    G = evocg.tile_build(w.n, w.rp, w.ci, w.v, w.T)
    ctrl = None
    if w.ctrl == "threshold":
        ctrl = evocg.Ctrl.threshold(w.eps, w.kstar)
    elif w.ctrl == "mlp":
        ctrl = evocg.Ctrl.mlp(W.mlp_weights(w.T, w.mlp_seed), w.kstar, w.delta)
    else:
        trow, ex = G.tile_rows()
        evocg.set_tile_precision(G, W.tile_map(trow, ex["tileColIdx"], G.nrb, w.map_seed))
    b = torch.from_numpy(w.b).to(dev)
    x = torch.empty_like(b)
    info = evocg.cg_solve(G, b, x, w.rtol, w.maxit, w.jacobi, ctrl, True)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(steps):
        info = evocg.cg_solve(G, b, x, w.rtol, w.maxit, w.jacobi, ctrl, True)
    e1.record(stream)
    torch.cuda.synchronize()
    tts = e0.elapsed_time(e1) / 1000.0 / steps
    spmv = spmv_measure(G, w, dev, stream, peak)
    G.free()
    return {"tts_s": tts, "iters": info["iters"], "status": info["status"],
            "true_res": info["true_res"], "spmv": spmv}


def run_ours(args):
    import numpy as np
    import torch

    from mixed_precision_sparse_gb300 import evocg, spmv_run
    from mixed_precision_sparse_gb300 import workloads as W

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()

    w = _workload(args.workload)
    t0 = time.perf_counter()
    G = evocg.tile_build(w.n, w.rp, w.ci, w.v, w.T)
    build_s = time.perf_counter() - t0
    if w.ctrl == "threshold":
        ctrl = evocg.Ctrl.threshold(w.eps, w.kstar)
    elif w.ctrl == "mlp":
        ctrl = evocg.Ctrl.mlp(W.mlp_weights(w.T, w.mlp_seed), w.kstar, w.delta)
    else:
        ctrl = None
        trow, ex = G.tile_rows()
        evocg.set_tile_precision(G, W.tile_map(trow, ex["tileColIdx"], G.nrb, w.map_seed))
    b = torch.from_numpy(w.b).to(dev)
    x = torch.empty_like(b)
    hist = torch.empty(w.maxit + 1, dtype=torch.float64, device=dev)

    def solve():
        return evocg.cg_solve(G, b, x, w.rtol, w.maxit, w.jacobi, ctrl, True, hist)

    for _ in range(max(3, args.warmup)):
        info = solve()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    infos = []
    with ClockSampler(local) as clk:
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(args.steps):
            infos.append(solve())
        e1.record(stream)
        torch.cuda.synchronize()
    if dist:
        dist.barrier()
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, dist, dev)
    info = infos[-1]
    value = job_seconds_per_solve(ms, world)
    launches = 0
    for inf in infos:
        # init + 3 kernels per iteration (+1 policy kernel per iteration with the MLP),
        # true-residual check 2 per check, each restart graph: SpMV + init
        per_it = 3 + (1 if w.ctrl == "mlp" else 0)
        launches += 1 + per_it * inf["iters"] + 2 * (1 + inf["restarts"]) + 2 * inf["restarts"]

    # ---- end to end through the C ABI with pinned host buffers
    bh = torch.from_numpy(w.b).pin_memory()
    xh = torch.empty(w.n, dtype=torch.float64).pin_memory()
    hh = torch.empty(w.maxit + 1, dtype=torch.float64).pin_memory()
    evocg.cg_solve(G, bh, xh, w.rtol, w.maxit, w.jacobi, ctrl, True, hh)
    e2e_steps = max(1, min(args.steps, 5))
    torch.cuda.synchronize()
    e0.record(stream)
    e2e_infos = [evocg.cg_solve(G, bh, xh, w.rtol, w.maxit, w.jacobi, ctrl, True, hh)
                 for _ in range(e2e_steps)]
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, dist, dev)
    h2d = 8 * w.n
    d2h = 8 * w.n + 8 * (e2e_infos[-1]["iters"] + 1)

    # ---- the same solve with every tile in FP64 and no controller (the all-FP64 GPU path the
    # mixed-precision solve is compared with), outside the timed region
    evocg.set_tile_precision(G, np.zeros(G.ntiles, np.uint8))
    fp64_info = evocg.cg_solve(G, b, x, w.rtol, w.maxit, w.jacobi, None, True, hist)
    torch.cuda.synchronize()
    fp64_steps = max(1, min(args.steps, 3))
    e0.record(stream)
    for _ in range(fp64_steps):
        fp64_info = evocg.cg_solve(G, b, x, w.rtol, w.maxit, w.jacobi, None, True, hist)
    e1.record(stream)
    torch.cuda.synchronize()
    fp64_s = e0.elapsed_time(e1) / 1000.0 / fp64_steps
    fp64_solve = {"s": fp64_s, "iters": fp64_info["iters"], "true_res": fp64_info["true_res"],
                  "mixed_over_fp64": value * world / fp64_s}

    # ---- the dominant kernel (the SpMV) timed alone on the solve's stream with CUDA events,
    # with the seeded 40/40/20 mixed map and all-FP64: warm (back-to-back launches; every
    # launch streams more than L2 on the large workloads) and cold (L2 flushed by writing a
    # buffer of twice its size before each launch, each launch timed on its own)
    peak, peak_kind = _peaks()
    spmv = spmv_measure(G, w, dev, stream, peak)
    src_hash = _src_hash()
    traffic = _traffic_for(src_hash, w.name)
    mixed = spmv["mixed_40_40_20"]
    roofline = {"bound": "hbm", "achieved": mixed["gbs"], "peak": peak, "unit": "GB/s",
                "frac": mixed["frac_of_peak"], "traffic": traffic,
                "kernel": _spmv_kernel_label(G, dev) + "; mixed 40/40/20 map",
                "peak_kind": peak_kind, "frac_of_8tbs": mixed["frac_of_8tbs"],
                "bytes_per_launch": mixed["bytes"], "us_per_launch": mixed["us"],
                "bytes_rule": "Tile-CSC algorithmic bytes: active value stream + 1 row-index "
                              "byte per entry + 2(T+1)+12 bytes per tile + x and y once",
                "cold_l2": {k: spmv[k]["cold"] for k in spmv}, "fp64_map": spmv["fp64"]}
    extra = {}
    if args.workload != 2 and not args.no_extra:
        extra["diffusion3d_7pt_128cubed"] = extra_workload(2, dev, stream, peak)

    # ---- CPU oracle on the host cores, a bounded sample (rank 0, N = 1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        ns = args.cpu_sample_iters or default_sample_iters(w)
        sec_it, _ = oracle_sample(w, ns)
        cpu = {"value": sec_it * info["iters"], "unit": "s", "cores": 1, "kind": "oracle",
               "sample": f"first {ns} iterations of the same solve, "
                         f"seconds/iteration x the GPU solve's {info['iters']} iterations"}

    # what one iteration streams (the SpMV's algorithmic bytes with the map in force plus the
    # vector kernels' ~105 bytes per row) against the L2 size: no flush is needed when it is
    # larger than L2; a smaller workload is L2-resident and says so
    d = G.info()
    it_bytes = int(d.bytes_index) + 8 * int(d.nnz) + 105 * w.n
    l2_bytes = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0))
    l2_note = (f"inputs larger than L2 (up to {it_bytes / 1e6:.0f} MB streamed per iteration, "
               f"L2 {l2_bytes / 1e6:.0f} MB); no flush" if it_bytes > l2_bytes else
               f"L2-resident workload ({it_bytes / 1e6:.1f} MB per iteration, "
               f"L2 {l2_bytes / 1e6:.0f} MB); not flushed, reported as a latency case")

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "s", "n_gpus": world,
            "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64+f32+bf16 (tile-wise), f64 vectors", "data": "synthetic",
            "config": {"workload": w.name, "n": w.n, "nnz": w.nnz, "tile": w.T,
                       "solver": "jacobi-pcg" if w.jacobi else "cg", "rtol": w.rtol,
                       "maxit": w.maxit, "controller": w.ctrl, "finish_fp64": True,
                       "parallelism": f"replicas x{world}",
                       "l2": l2_note},
            "solve": {"iters": info["iters"], "iters_recursive": info["iters_recursive"],
                      "restarts": info["restarts"], "true_res": info["true_res"],
                      "prec_nnz": info["prec_nnz"], "ctrl_calls": info["ctrl_calls"],
                      "status": info["status"], "tile_build_s": build_s,
                      "s_per_iter": value / max(1, info["iters"]) * world},
            "fp64_solve": fp64_solve,
            "clocks": clk.summary(),
            "e2e": {"value": e2e_ms / 1000.0 / world, "unit": "s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "gpu_launches": launches,
            "roofline": roofline,
            "cpu_baseline": cpu,
            "other_workloads": extra,
        }
        print(json.dumps(line), flush=True)
    G.free()
    if dist:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=5)
    ap.add_argument("--cpu-sample-iters", type=int, default=0,
                    help="oracle iterations per CPU sample (0: about 10-20 s of CPU work)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="skip the 128^3 workload's summary")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
