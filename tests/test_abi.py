"""CPU checks of the C ABI: the library builds for sm_103a, loads, and exports every
function include/evocg.h declares. No compute call is made (no GPU here)."""
import os
import re

import pytest

from mixed_precision_sparse_gb300 import build, evocg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "evocg.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(evocg_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return evocg.lib()


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 12
    for name in names:
        assert hasattr(lib, name), name


def test_version_and_error_string(lib):
    assert evocg.version() >= 1
    assert isinstance(evocg.last_error(), str)


def test_no_gpu_is_reported_not_faked(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    from mixed_precision_sparse_gb300 import workloads as W
    n, rp, ci, v = W.laplace2d_5pt(8)
    with pytest.raises(evocg.EvocgError) as e:
        evocg.tile_build(n, rp, ci, v, 16)
    assert e.value.code == evocg.EDEVICE


def test_rate_probe_builds_and_exports():
    """The arithmetic-rate probe (a measuring tool beside the library) builds for sm_103a and
    exports its one entry point; with no GPU a call returns a CUDA error code, not rates."""
    import ctypes
    p = build.build_probe()
    lib = ctypes.CDLL(p)
    assert hasattr(lib, "evocg_rate_probe")
    lib.evocg_rate_probe.restype = ctypes.c_int
    d = [ctypes.c_double() for _ in range(3)]
    assert lib.evocg_rate_probe(9, 4, 64, *[ctypes.byref(x) for x in d]) != 0   # unknown kind
