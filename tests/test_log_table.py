"""The FP64 volume kernel's table-driven logarithm, checked on the host.

The kernel (csrc/log_fp64.cuh) reduces x = 2^k m with m in [0.75, 1.5) to the
nearest point F of a 1/128 grid (1/256 below 1) and evaluates
    ln x = k ln 2 + ln F + ln(1 + r),  r = (m - F)/F,
with 1/F and ln F (lead and trail) from log_table.inc and ln(1 + r) by its
Taylor series to r^7 (P. T. P. Tang, ACM TOMS 16(4), 1990).  These tests pin
the committed table to 50-digit arithmetic and run the same steps in Python,
with exactly rounded fused multiply-adds, against the host's log.  The GPU
test of the compiled function is test_gpu_numerics.py.
"""
import math
import os
import re
import struct
from fractions import Fraction

import numpy as np
import pytest

mpmath = pytest.importorskip("mpmath")

INC = os.path.join(os.path.dirname(__file__), "..", "flux_differencing_gb300", "csrc", "log_table.inc")


def _table():
    txt = open(INC).read()
    pairs = [(float.fromhex(a), float.fromhex(b))
             for a, b in re.findall(r"\{(-?0x[0-9a-fp.+-]+), (-?0x[0-9a-fp.+-]+)\}", txt)]
    tail_block = txt[txt.index("kLogTail"):]
    tail = [float.fromhex(v) for v in re.findall(r"^\s+(-?0x[0-9a-fp.+-]+),$", tail_block, re.M)]
    hi = float.fromhex(re.search(r"kLn2Hi = (-?0x[^;]+);", txt).group(1))
    lo = float.fromhex(re.search(r"kLn2Lo = (-?0x[^;]+);", txt).group(1))
    return pairs, tail, hi, lo


def _grid_point(idx):
    """F of table entry idx (0..64: 1 + j/128; 65..129: (1 + j/128)/2, j = idx - 1)."""
    if idx <= 64:
        return mpmath.mpf(1) + mpmath.mpf(idx) / 128
    return (mpmath.mpf(1) + mpmath.mpf(idx - 1) / 128) / 2


def test_table_entries_are_correctly_rounded():
    mpmath.mp.dps = 50
    pairs, tail, hi, lo = _table()
    assert len(pairs) == 130 and len(tail) == 130
    for idx, ((inv_f, ln_f), ln_t) in enumerate(zip(pairs, tail)):
        F = _grid_point(idx)
        assert inv_f == float(1 / F), idx
        assert ln_f == float(mpmath.log(F)), idx
        # lead + trail carries ln F to ~106 bits
        assert abs(mpmath.mpf(ln_f) + mpmath.mpf(ln_t) - mpmath.log(F)) <= mpmath.mpf(2) ** -100, idx
    ln2 = mpmath.log(2)
    assert hi == float(mpmath.floor(ln2 * 2 ** 42) / 2 ** 42)
    assert hi * 2 ** 42 == int(hi * 2 ** 42)  # k ln2_hi exact for |k| < 2^11
    assert abs(mpmath.mpf(hi) + mpmath.mpf(lo) - ln2) < mpmath.mpf(2) ** -95


def _fma(a, b, c):
    return float(Fraction(a) * Fraction(b) + Fraction(c))


def _hilo(x):
    u = struct.unpack("<Q", struct.pack("<d", x))[0]
    hi, lo = u >> 32, u & 0xFFFFFFFF
    return hi - (1 << 32) if hi >= 1 << 31 else hi, lo


def _from_hilo(hi, lo):
    return struct.unpack("<d", struct.pack("<Q", ((hi & 0xFFFFFFFF) << 32) | (lo & 0xFFFFFFFF)))[0]


def _log_steps(x, pairs, tail, ln2_hi, ln2_lo):
    """The kernel's steps, integer manipulations included, in Python."""
    hi, lo = _hilo(x)
    mant = hi & 0x000FFFFF
    half = 1 if mant >= 0x80000 else 0
    j = (mant + 0x1000) >> 13
    ebits = 0x3FF00000 - (half << 20)
    m = _from_hilo(ebits | mant, lo)
    F = _from_hilo(ebits + (j << 13), 0)
    inv_f, ln_f = pairs[j + half]
    ln_t = tail[j + half]
    k = ((hi >> 20) & 0x7FF) - 1023 + half
    kd = _from_hilo(0x43300000, k + 1024) - 4503599627371520.0
    assert kd == k
    assert m - F == float(Fraction(m) - Fraction(F))  # exact (Sterbenz)
    r = (m - F) * inv_f
    assert abs(r) <= 2.0 ** -8 * 1.0001
    r2 = r * r
    q = _fma(r, 1.0 / 7.0, -1.0 / 6.0)
    q = _fma(q, r, 1.0 / 5.0)
    q = _fma(q, r, -0.25)
    q = _fma(q, r, 1.0 / 3.0)
    q = _fma(q, r, -0.5)
    p = _fma(r2, q, r)
    return _fma(kd, ln2_hi, ln_f) + (_fma(kd, ln2_lo, p) + ln_t)


def test_method_within_one_ulp_of_host_log():
    pairs, tail, hi, lo = _table()
    rng = np.random.default_rng(5)
    xs = np.concatenate([
        np.exp(rng.uniform(np.log(1e-300), np.log(1e300), 1500)),
        1.0 + rng.uniform(-2.0 ** -8, 2.0 ** -8, 500),   # around 1: relative accuracy
        rng.uniform(0.75, 1.0, 400),                      # halved branch, ln F < 0
        rng.uniform(0.97, 1.03, 400),                     # cancellation of ln F against ln(1 + r)
        0.75 * (1.0 + rng.uniform(-1e-6, 1e-6, 100)),     # reduction boundaries
        1.5 * (1.0 + rng.uniform(-1e-6, 1e-6, 100)),
        1.0 + np.arange(-50, 51) * 2.0 ** -52,
        rng.uniform(1e-6, 1e-4, 200),                     # 2b = rho/p of the workloads
    ])
    worst = 0.0
    for x in xs:
        x = float(x)
        y = _log_steps(x, pairs, tail, hi, lo)
        ref = math.log(x)
        if ref == 0.0:
            assert y == 0.0
            continue
        worst = max(worst, abs(y - ref) / np.spacing(abs(ref)))
    assert worst <= 1.0, worst
