"""The FP32 volume kernel's logarithmic means (no GPU).

The FP32 pair evaluation forms {{a}}_log = (a+ + a-) f/(2 atanh f) and
1/{{a}}_log = (2 atanh(f)/f)/(a+ + a-), f = (a+ - a-)/(a+ + a-), from degree-4
polynomials in u = f^2 on u <= 0.16 (csrc/logmean_poly.inc, written by
csrc/gen_logmean_poly.py) in every CTA whose densities and values of b lie
within a factor 2.25 of one another; in other CTAs, the pairs beyond the
polynomials' range take the logarithm of their ratio.  Checked
here against 40-digit arithmetic: the committed coefficients (as the FP32
values the kernel uses, evaluated by Horner in FP32 like the kernel) stay
within 2e-7 relative of the exact ratios on the whole range, at u = 0.16 and
near 0, and the identities they stand for hold (the log mean of a and c
computed from them equals (c - a)/(ln c - ln a)).
"""
import os
import re

import numpy as np
import pytest

mp = pytest.importorskip("mpmath")
mp.mp.dps = 40

INC = os.path.join(os.path.dirname(__file__), "..", "flux_differencing_gb300", "csrc", "logmean_poly.inc")


def _coeffs():
    txt = open(INC).read()
    out = {}
    for name in ("kLogMeanRatio", "kInvLogMeanRatio"):
        body = re.search(name + r"\[5\] = \{([^}]*)\}", txt).group(1)
        out[name] = [np.float32(float(v.strip().rstrip("f"))) for v in body.split(",")]
    out["U"] = float(re.search(r"kLogMeanPolyU = ([0-9.e+-]+)f", txt).group(1))
    return out


def _horner32(c, u):
    h = np.float32(c[-1])
    for cc in reversed(c[:-1]):
        h = np.float32(np.float32(h * np.float32(u)) + cc)  # FMA in the kernel: at most as accurate
    return float(h)


def test_polynomials_against_exact_ratios():
    c = _coeffs()
    assert c["U"] == pytest.approx(0.16)
    us = [c["U"] * k / 400 for k in range(401)] + [1e-12, 1e-6, c["U"]]
    worst1 = worst2 = 0.0
    for u in us:
        u32 = float(np.float32(u))
        f = mp.sqrt(mp.mpf(u32))
        g1 = mp.mpf("0.5") if u32 == 0 else f / (2 * mp.atanh(f))
        g2 = mp.mpf(2) if u32 == 0 else 2 * mp.atanh(f) / f
        worst1 = max(worst1, abs(float((_horner32(c["kLogMeanRatio"], u32) - g1) / g1)))
        worst2 = max(worst2, abs(float((_horner32(c["kInvLogMeanRatio"], u32) - g2) / g2)))
    assert worst1 < 2e-7, worst1
    assert worst2 < 2e-7, worst2


def test_log_mean_identity():
    """(a + c) g1(u) = (c - a)/(ln c - ln a) and g2(u)/(a + c) its inverse, for
    pairs up to the polynomials' limit (c/a = 2.33)."""
    c = _coeffs()
    rng = np.random.default_rng(3)
    for _ in range(200):
        a = mp.mpf(float(rng.uniform(0.1, 10.0)))
        ratio = mp.mpf(float(rng.uniform(1.0, 2.3)))
        cc = a * ratio
        f = (cc - a) / (cc + a)
        u = float(f * f)
        assert u <= c["U"]
        exact = (cc - a) / (mp.log(cc) - mp.log(a))
        approx = (a + cc) * mp.mpf(float(_horner32(c["kLogMeanRatio"], u)))
        assert abs((approx - exact) / exact) < 2e-7
        inv = mp.mpf(float(_horner32(c["kInvLogMeanRatio"], u))) / (a + cc)
        assert abs(inv * exact - 1) < 2e-7


def test_committed_table_is_the_generator_output():
    """logmean_poly.inc is exactly what gen_logmean_poly.py writes (about 40 s
    of 40-digit Remez iterations)."""
    import subprocess
    import sys
    gen = os.path.join(os.path.dirname(INC), "gen_logmean_poly.py")
    out = subprocess.run([sys.executable, gen], capture_output=True, text=True, check=True).stdout
    assert out == open(INC).read()
