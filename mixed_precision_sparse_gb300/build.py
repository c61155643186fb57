"""Build libevocg.so in-tree for sm_103a (GB300) with nvcc; no cmake, no torch extension.

Objects go to mixed_precision_sparse_gb300/_build/, the library next to this file.
Translation units compile in parallel; a unit is rebuilt when it or a header changed.
build_probe() builds librates.so, the arithmetic-rate probe (probe/rates.cu; rates.py).
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INC = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libevocg.so")
PROBE_SRC = os.path.join(HERE, "probe", "rates.cu")
PROBE_LIB = os.path.join(HERE, "librates.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc():
    p = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(p):
        raise RuntimeError("nvcc not found (CUDA 13 toolkit required)")
    return p


def _headers():
    return glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(INC, "*.h"))


def _stale(obj, src, deps):
    if not os.path.exists(obj):
        return True
    stamp = obj + ".flags"
    flags = os.environ.get("EVOCG_NVCC_FLAGS", "")
    if not os.path.exists(stamp) or open(stamp).read() != flags:
        return True
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(d) > t for d in [src, *deps])


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False) -> str:
    os.makedirs(OUT_DIR, exist_ok=True)
    nvcc = _nvcc()
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))
    deps = _headers()
    common = ["-std=c++17", "-O3", "-I", INC, "-I", CSRC, "-Xcompiler", "-fPIC"]
    # extra nvcc flags from EVOCG_NVCC_FLAGS (none by default; e.g. -Xptxas=-v for register and
    # spill counts); recorded in each object's stamp so that a change of flags rebuilds it
    extra = os.environ.get("EVOCG_NVCC_FLAGS", "").split()
    common += extra
    jobs = []
    objs = []
    for s in srcs:
        obj = os.path.join(OUT_DIR, os.path.basename(s) + ".o")
        objs.append(obj)
        if force or _stale(obj, s, deps):
            cmd = [nvcc, *common, "-c", s, "-o", obj]
            if s.endswith(".cu"):
                cmd[1:1] = [*ARCH, "-lineinfo", "-rdc=true"]
                if ptxas_verbose:
                    cmd.insert(1, "-Xptxas=-v")
            else:
                cmd[1:1] = ["-x", "c++"]
            jobs.append(cmd)

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    failed = []
    with ThreadPoolExecutor(max_workers=min(8, max(1, len(jobs)))) as ex:
        for cmd, r in ex.map(run, jobs):
            if verbose or ptxas_verbose or r.returncode:
                sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
            if r.returncode:
                failed.append(cmd[-3])
            else:
                with open(cmd[-1] + ".flags", "w") as f:
                    f.write(os.environ.get("EVOCG_NVCC_FLAGS", ""))
    if failed:
        raise RuntimeError(f"nvcc failed for {failed}")
    if force or jobs or not os.path.exists(LIB):
        tmp = LIB + f".tmp{os.getpid()}"
        cudalib = os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "lib64")
        link = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs, "-lcudadevrt",
                "-lpthread", "-Xlinker", "-rpath", "-Xlinker", cudalib]
        r = subprocess.run(link, capture_output=True, text=True)
        if r.returncode:
            raise RuntimeError("link failed:\n" + r.stdout + r.stderr)
        os.replace(tmp, LIB)
    return LIB


def build_probe(force: bool = False) -> str:
    """The arithmetic-rate probe library (not part of the solver)."""
    deps = [PROBE_SRC, os.path.join(CSRC, "fpconv.cuh")]
    if not force and os.path.exists(PROBE_LIB) and \
            all(os.path.getmtime(d) <= os.path.getmtime(PROBE_LIB) for d in deps):
        return PROBE_LIB
    tmp = PROBE_LIB + f".tmp{os.getpid()}"
    cmd = [_nvcc(), *ARCH, "-std=c++17", "-O3", "-lineinfo", "-I", CSRC, "-Xcompiler", "-fPIC", "-shared",
           "-cudart", "shared", "-o", tmp, PROBE_SRC]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode:
        raise RuntimeError("probe build failed:\n" + r.stdout + r.stderr)
    os.replace(tmp, PROBE_LIB)
    return PROBE_LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                ptxas_verbose="--ptxas" in sys.argv))
