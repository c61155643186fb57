"""The C ABI from a plain C program: tests/c_abi_host.c is compiled with gcc as C99 against
include/evocg.h, linked to libevocg.so, and run on the host (it calls only the entry points
that need no GPU). Its printed results are checked against the oracle and hand counts."""
import os
import subprocess

import numpy as np
import pytest

import oracle
from mixed_precision_sparse_gb300 import build
from mixed_precision_sparse_gb300 import workloads as W

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


@pytest.fixture(scope="module")
def c_output():
    lib = build.build()
    libdir = os.path.dirname(lib)
    os.makedirs(build.OUT_DIR, exist_ok=True)
    exe = os.path.join(build.OUT_DIR, "c_abi_host")   # the library's own build directory
    subprocess.check_call(["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                           "-I", os.path.join(ROOT, "include"), os.path.join(HERE, "c_abi_host.c"),
                           "-o", exe, "-L", libdir, "-levocg", f"-Wl,-rpath,{libdir}"])
    out = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stdout + out.stderr
    return {ln.split()[0]: ln.split()[1:] for ln in out.stdout.splitlines()}


def test_layout_from_c_matches_the_oracle(c_output):
    """Sizes of the library's slot-major interior printed by the C program, against counts
    taken from the CSR with numpy (tiles and entries also against the oracle's Tile-CSC)."""
    n, rp, ci, v = W.laplace2d_5pt(20)
    T = 16
    t = oracle.Tiles(oracle.CSR(n, rp, ci, v), T)
    got = dict(zip(c_output["layout"][0::2], map(int, c_output["layout"][1::2])))
    assert got["ntiles"] == t.ntiles and got["nnz"] == t.nnz
    assert got["tiles_in_last_rowblock"] == int(t.tileRowPtr[-1] - t.tileRowPtr[-2])
    rows = np.repeat(np.arange(n), np.diff(rp))
    tile = (rows // T) * ((n + T - 1) // T) + ci // T        # tile of every entry
    rt, per_row = np.unique(tile * n + rows, return_counts=True)   # entries of (tile, row)
    width = np.zeros(tile.max() + 1, np.int64)
    np.maximum.at(width, rt // n, per_row)
    nrows = np.bincount(rt // n, minlength=tile.max() + 1)
    assert got["widest"] == int(width.max())
    assert int(c_output["rows_in_masks"][0]) == rt.size
    # slots: a tile of m > 1 slots starts on a multiple of 16 and takes m rounded up to 16; a
    # single-entry tile takes one slot; each row block's slots are rounded up to 16
    m = width * nrows
    nrb = (n + T - 1) // T
    slots = 0
    for rb in range(nrb):
        pos = 0
        for tt in range(rb * nrb, (rb + 1) * nrb):
            if tt < m.size and m[tt] > 1:
                pos = (pos + 15) // 16 * 16 + (m[tt] + 15) // 16 * 16
            elif tt < m.size:
                pos += m[tt]
        slots += (pos + 15) // 16 * 16
    assert got["nslots"] == slots


def test_plan_and_kstar_from_c(c_output):
    assert c_output["plan"][2:] == ["valid", "1"] and int(c_output["plan"][1]) > 0
    ks = c_output["kstar"]
    assert ks[0] == "1" and ks[2] == "4"
    assert [float(f) for f in ks[4:8]] == [0.0, 1.0, 1.0, 1.0]
    assert oracle.kstar_select(np.array([2, 2, 2, 1, 1, 0, 0, 0], np.uint8).reshape(-1, 1))[0] == 1


def test_error_message_reaches_c(c_output):
    assert "tile_size" in " ".join(c_output["error"])
