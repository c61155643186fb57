"""Pins of the oracle's FP64 -> FP32 / BF16 rounding against references outside it.

FP32: numpy's float64 -> float32 cast (IEEE round-to-nearest-even in hardware).
BF16: an exhaustive table of every finite BF16 value, nearest by search with ties to the
even pattern, and the hand-derived cases of tests/golden/bf16_rounding_cases.txt.
"""
import os
import struct

import numpy as np
import pytest

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden", "bf16_rounding_cases.txt")


def _hex_to_f64(h):
    return struct.unpack(">d", int(h, 16).to_bytes(8, "big"))[0]


def _bf16_table():
    bits = np.arange(0, 0x7F80, dtype=np.uint32)  # all finite non-negative patterns
    vals = (bits << 16).view(np.float32).astype(np.float64)
    return bits.astype(np.uint16), vals


def _bf16_bruteforce(x):
    """Nearest finite BF16 by table search; ties to the even pattern; IEEE overflow."""
    bits, vals = _bf16_table()
    out = np.empty(x.shape, np.uint16)
    top, below = vals[-1], vals[-2]
    for idx, xv in np.ndenumerate(x):
        if np.isnan(xv):
            out[idx] = 0x7FC0
            continue
        sign = 0x8000 if np.signbit(xv) else 0
        a = abs(xv)
        if a >= top + (top - below) / 2:  # at or beyond the overflow tie -> inf
            out[idx] = sign | 0x7F80
            continue
        i = np.searchsorted(vals, a)
        if i < len(vals) and vals[i] == a:
            out[idx] = sign | bits[i]
            continue
        lo, hi = i - 1, i
        dlo, dhi = a - vals[lo], vals[hi] - a
        if dlo < dhi or (dlo == dhi and bits[lo] % 2 == 0):
            out[idx] = sign | bits[lo]
        else:
            out[idx] = sign | bits[hi]
    return out


def _samples(seed, n=4000):
    rng = np.random.default_rng(seed)
    mant = rng.uniform(1.0, 2.0, n)
    ex = rng.integers(-150, 130, n)
    x = np.ldexp(mant, ex) * rng.choice([-1.0, 1.0], n)
    # exact halfway points of FP32 and BF16 spacings, and their neighbours
    f = rng.uniform(-100, 100, 500).astype(np.float32).astype(np.float64)
    ulp32 = np.spacing(np.abs(f).astype(np.float32)).astype(np.float64)
    b = _bf16_table()[1][rng.integers(1, 0x7F7F, 500)]
    ulpb = np.ldexp(1.0, np.frexp(b)[1] - 8)
    ties = np.concatenate([f + ulp32 / 2, f - ulp32 / 2, b + ulpb / 2, b + ulpb / 2 * (1 + 2**-40),
                           b + ulpb / 2 * (1 - 2**-40)])
    return np.concatenate([x, ties, [0.0, -0.0, 1.0, 3.4028234663852886e38, 1e-45, 1e-300]])


def test_round_f32_matches_hardware_cast():
    x = _samples(1)
    with np.errstate(over="ignore"):
        want = x.astype(np.float32)
    got = oracle.round_f32(x)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_round_f32_special():
    x = np.array([np.inf, -np.inf, 1e39, -1e39, np.nan])
    got = oracle.round_f32(x)
    assert got[0] == np.inf and got[1] == -np.inf and got[2] == np.inf and got[3] == -np.inf
    assert np.isnan(got[4])


def test_round_bf16_matches_exhaustive_table():
    x = _samples(2)
    got = oracle.round_bf16_bits(x)
    want = _bf16_bruteforce(x)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(x[i], hex(got[i]), hex(want[i])) for i in bad[:5]]


def test_round_bf16_golden_cases():
    rows = []
    for line in open(GOLD):
        if line.startswith("#") or not line.strip():
            continue
        h, e, *_ = line.split()
        rows.append((_hex_to_f64(h), int(e, 16), line.strip()))
    x = np.array([r[0] for r in rows])
    got = oracle.round_bf16_bits(x)
    for g, (xv, e, txt) in zip(got, rows):
        assert g == e, f"{txt}: got {hex(g)}"


def test_bf16_single_rounding_differs_from_double_rounding():
    # the reading is one rounding from FP64; rounding through FP32 would give 0x3f80 here
    x = np.array([_hex_to_f64("0x3ff0100000010000")])
    assert oracle.round_bf16_bits(x)[0] == 0x3F81
    via32 = oracle.round_bf16_bits(x.astype(np.float32).astype(np.float64))[0]
    assert via32 == 0x3F80


@pytest.mark.parametrize("frac,emin,emax", [(23, -126, 127), (7, -126, 127), (10, -14, 15)])
def test_round_to_format_is_idempotent_and_monotone(frac, emin, emax):
    x = np.sort(_samples(3))
    r = np.array([oracle.round_to_format(v, frac, emin, emax) for v in x])
    rr = np.array([oracle.round_to_format(v, frac, emin, emax) for v in r])
    assert np.array_equal(r, rr)
    finite = np.isfinite(r)
    assert np.all(np.diff(r[finite]) >= 0)


def test_fp16_format_matches_numpy_half():
    # the same routine with binary16 parameters must agree with numpy's float16 cast
    x = np.random.default_rng(4).uniform(-70000, 70000, 3000)
    x = np.concatenate([x, np.ldexp(np.random.default_rng(5).uniform(1, 2, 500),
                                    np.random.default_rng(6).integers(-26, -10, 500))])
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).astype(np.float64)
    got = np.array([oracle.round_to_format(v, 10, -14, 15) for v in x])
    assert np.array_equal(got, want)
