"""The FP64 volume kernel's table-driven logarithm, checked on the host.

The kernel (csrc/log_fp64.cuh) reduces x = 2^k m with m in [0.75, 1.5) to the
nearest point F of a 1/512 grid (1/1024 below 1) and evaluates
    ln x = k ln 2 + ln F + ln(1 + r),  r = (m - F)/F,
with 1/F and ln F from log_table.inc and ln(1 + r) by its Taylor series to
r^5 (P. T. P. Tang, ACM TOMS 16(4), 1990), summed as k ln2 + (ln F + ln(1 + r))
with ln 2 and ln F each rounded once.  The kernel uses the logarithms only in
differences of two nodes' values, where the rounding of ln 2 cancels.  These
tests pin the committed table to 50-digit arithmetic and run the same steps
in Python, with exactly rounded fused multiply-adds, against 50-digit
logarithms: the absolute value, and the difference of two of them.  The GPU
test of the compiled function (test_gpu_numerics.py) checks it bit for bit
against these steps.
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
    ln2 = float.fromhex(re.search(r"kLn2 = (-?0x[^;]+);", txt).group(1))
    return pairs, ln2


def _grid_point(idx):
    """F of table entry idx (0..256: 1 + j/512; 257..513: (1 + j/512)/2, j = idx - 1)."""
    if idx <= 256:
        return mpmath.mpf(1) + mpmath.mpf(idx) / 512
    return (mpmath.mpf(1) + mpmath.mpf(idx - 1) / 512) / 2


def test_table_entries_are_correctly_rounded():
    mpmath.mp.dps = 50
    pairs, ln2 = _table()
    assert len(pairs) == 514
    for idx, (inv_f, ln_f) in enumerate(pairs):
        F = _grid_point(idx)
        assert inv_f == float(1 / F), idx
        assert ln_f == float(mpmath.log(F)), idx
    assert ln2 == float(mpmath.log(2))
    assert abs(mpmath.mpf(ln2) - mpmath.log(2)) < mpmath.mpf(2) ** -55


def _fma(a, b, c):
    return float(Fraction(a) * Fraction(b) + Fraction(c))


def _hilo(x):
    u = struct.unpack("<Q", struct.pack("<d", x))[0]
    hi, lo = u >> 32, u & 0xFFFFFFFF
    return hi - (1 << 32) if hi >= 1 << 31 else hi, lo


def _from_hilo(hi, lo):
    return struct.unpack("<d", struct.pack("<Q", ((hi & 0xFFFFFFFF) << 32) | (lo & 0xFFFFFFFF)))[0]


def log_steps(x, pairs, ln2):
    """The kernel's steps, integer manipulations included, in Python."""
    hi, lo = _hilo(x)
    mant = hi & 0x000FFFFF
    half = 1 if mant >= 0x80000 else 0
    j = (mant + 0x400) >> 11
    ebits = 0x3FF00000 - (half << 20)
    m = _from_hilo(ebits | mant, lo)
    F = _from_hilo(ebits + (j << 11), 0)
    inv_f, ln_f = pairs[j + half]
    k = ((hi >> 20) & 0x7FF) - 1023 + half
    kd = _from_hilo(0x43300000, k + 1024) - 4503599627371520.0
    assert kd == k
    assert m - F == float(Fraction(m) - Fraction(F))  # exact (Sterbenz)
    r = (m - F) * inv_f
    assert abs(r) <= 2.0 ** -10 * 1.0001
    r2 = r * r
    q = _fma(r, 1.0 / 5.0, -0.25)
    q = _fma(q, r, 1.0 / 3.0)
    q = _fma(q, r, -0.5)
    p = _fma(r2, q, r)
    return _fma(kd, ln2, ln_f + p), k


def sample_points(rng, n=1):
    return np.concatenate([
        np.exp(rng.uniform(np.log(1e-300), np.log(1e300), 1500 * n)),
        1.0 + rng.uniform(-2.0 ** -10, 2.0 ** -10, 500 * n),  # around 1: relative accuracy
        rng.uniform(0.75, 1.0, 400 * n),                      # halved branch, ln F < 0
        rng.uniform(0.97, 1.03, 400 * n),                     # ln F against ln(1 + r)
        0.75 * (1.0 + rng.uniform(-1e-6, 1e-6, 100 * n)),     # reduction boundaries
        1.5 * (1.0 + rng.uniform(-1e-6, 1e-6, 100 * n)),
        1.0 + np.arange(-50, 51) * 2.0 ** -52,
        rng.uniform(1e-6, 1e-4, 200 * n),                     # 2b = rho/p of the workloads
        rng.uniform(0.01, 2.0, 200 * n),                      # densities
    ])


def _ulp(x):
    return float(np.spacing(abs(x)))


def test_method_absolute_error():
    """|L(x) - ln x| <= half an ulp of the result + |k| 2^-55 + 2^-54 (the
    roundings of ln 2, ln F and the inner sum)."""
    mpmath.mp.dps = 50
    pairs, ln2 = _table()
    rng = np.random.default_rng(5)
    worst = 0.0
    for x in sample_points(rng):
        x = float(x)
        y, k = log_steps(x, pairs, ln2)
        ref = mpmath.log(mpmath.mpf(x))
        if x == 1.0:
            assert y == 0.0
            continue
        err = abs(mpmath.mpf(y) - ref)
        bound = 0.5 * _ulp(y) + abs(k) * 2.0 ** -55 + 2.0 ** -54
        worst = max(worst, float(err / bound))
    assert worst <= 1.0, worst


def test_method_differences_within_one_ulp():
    """The kernel's use: ln a+ - ln a- for two nodes.  Pairs at the relative
    distances of neighbouring nodes (1e-12 .. 0.5) and across powers of two:
    |L(y) - L(x) - ln(y/x)| <= one ulp of the larger result, plus |k_y - k_x|
    2^-55 when the two straddle a power of two, plus the roundings of ln F and
    the inner sums (2^-53)."""
    mpmath.mp.dps = 50
    pairs, ln2 = _table()
    rng = np.random.default_rng(6)
    xs = sample_points(rng)
    worst = 0.0
    for x in xs:
        x = float(x)
        for rel in (1e-12, 1e-6, 3e-3, 0.02, 0.3):
            y = x * (1.0 + rel * rng.uniform(-1.0, 1.0))
            if not (0.0 < y < 1.7e308):
                continue
            lx, kx = log_steps(x, pairs, ln2)
            ly, ky = log_steps(y, pairs, ln2)
            ref = mpmath.log(mpmath.mpf(y)) - mpmath.log(mpmath.mpf(x))
            err = abs(mpmath.mpf(ly) - mpmath.mpf(lx) - ref)
            bound = max(_ulp(lx), _ulp(ly)) + abs(ky - kx) * 2.0 ** -55 + 2.0 ** -53
            worst = max(worst, float(err / bound))
    assert worst <= 1.0, worst
