"""Accuracy of the volume kernel's reciprocal and logarithms (GPU required).

FP64 reciprocal: hardware estimate refined by one third-order Newton-Raphson
step; it must stay within 2 ulp of correctly rounded division.  FP32: the
hardware estimate alone, within 2^-22 relative.  Reference values are numpy's
IEEE division on the host.  FP64 logarithm (Tang's table-driven reduction):
bit for bit the host emulation of its steps, and close to the host's log.
Float-float building blocks against FP64 error bounds.
"""
import ctypes

import numpy as np
import pytest
import torch

import flux_differencing_gb300 as fd

pytestmark = pytest.mark.gpu


def _run(lib, x, fp64, mode=None):
    dt = torch.float64 if fp64 else torch.float32
    xd = torch.from_numpy(x).to("cuda", dt)
    yd = torch.empty_like(xd)
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    m = mode if mode is not None else (1 if fp64 else 0)
    assert lib.esdg_selftest_rcp(m, xd.numel(), ctypes.c_void_p(xd.data_ptr()),
                                 ctypes.c_void_p(yd.data_ptr()), s) == 0
    torch.cuda.synchronize()
    return yd.cpu().numpy()


def _inputs(rng, n, lo, hi):
    mag = np.exp(rng.uniform(np.log(lo), np.log(hi), size=n))
    x = mag * rng.choice([-1.0, 1.0], size=n)
    # also mantissas near 1 and near 2 (worst cases of table-based estimates)
    x[:64] = 1.0 + np.arange(64) * 2.0 ** -52
    x[64:128] = 2.0 - np.arange(1, 65) * 2.0 ** -52
    return x


def test_rcp_fp64_within_two_ulp(cuda_ok):
    lib = fd.load_library(build_if_missing=True)
    rng = np.random.default_rng(17)
    x = _inputs(rng, 1 << 20, 1e-300, 1e300)
    y = _run(lib, x, True)
    ref = 1.0 / x
    ulp = np.spacing(np.abs(ref))
    err = np.abs(y - ref) / ulp
    assert np.all(np.isfinite(y))
    assert err.max() <= 2.0, err.max()


def test_rcp_fp64_pair_relative_error(cuda_ok):
    """The pair reciprocal of the FP64 volume kernel (an estimate from the FP32
    reciprocal of the mantissa, then one second-order Newton step): its
    relative error is the square of the estimate's plus the step's own
    rounding.  Required: the estimate within 2^-21.5 relative and the pair
    reciprocal within 2^-43 (about 1.1e-13), far below the 1e-11 parity
    tolerance on the term scale; over magnitudes 1e-300 .. 1e300 of both
    signs and mantissas next to 1 and 2."""
    lib = fd.load_library(build_if_missing=True)
    rng = np.random.default_rng(19)
    x = _inputs(rng, 1 << 20, 1e-300, 1e300)
    ref = 1.0 / x
    est = _run(lib, x, True, mode=3)
    rel_est = np.abs(est - ref) / np.abs(ref)
    y = _run(lib, x, True, mode=2)
    rel = np.abs(y - ref) / np.abs(ref)
    print(f"estimate: max rel {rel_est.max():.3e} = 2^{np.log2(rel_est.max()):.2f}; "
          f"pair reciprocal: max rel {rel.max():.3e} = 2^{np.log2(rel.max()):.2f}")
    assert np.all(np.isfinite(y))
    assert rel_est.max() <= 2.0 ** -21.5, rel_est.max()
    assert rel.max() <= 2.0 ** -43, rel.max()


def test_rsqrt_fp64_pair_relative_error(cuda_ok):
    """The reciprocal square root of the FP64 surface flux (|n| and the sound
    speed): FP32 estimate of the mantissa (times 2 for odd exponents), then one
    second-order Newton step.  Required: the estimate within 2^-21.5 relative
    and the result within 2^-42 (about 2.3e-13) over 1e-300 .. 1e300, odd and
    even exponents, mantissas next to 1 and 2."""
    lib = fd.load_library(build_if_missing=True)
    rng = np.random.default_rng(20)
    x = np.abs(_inputs(rng, 1 << 20, 1e-300, 1e300))
    x[128:192] = np.ldexp(1.0, np.arange(-32, 32))  # exact powers of two, both parities
    ref = 1.0 / np.sqrt(x)
    est = _run(lib, x, True, mode=5)
    y = _run(lib, x, True, mode=4)
    rel_est = np.abs(est - ref) / ref
    rel = np.abs(y - ref) / ref
    print(f"rsqrt estimate: max rel {rel_est.max():.3e} = 2^{np.log2(rel_est.max()):.2f}; "
          f"rsqrt: max rel {rel.max():.3e} = 2^{np.log2(rel.max()):.2f}")
    assert np.all(np.isfinite(y))
    assert rel_est.max() <= 2.0 ** -21.5, rel_est.max()
    assert rel.max() <= 2.0 ** -42, rel.max()


def test_rcp_fp32_relative_error(cuda_ok):
    lib = fd.load_library(build_if_missing=True)
    rng = np.random.default_rng(18)
    x = _inputs(rng, 1 << 20, 1e-30, 1e30).astype(np.float32)
    y = _run(lib, x, False).astype(np.float64)
    ref = 1.0 / x.astype(np.float64)
    rel = np.abs(y - ref) / np.abs(ref)
    assert rel.max() < 2.0 ** -22, rel.max()


def _ff(lib, op, x, y):
    xd = torch.from_numpy(x).to("cuda")
    yd = torch.from_numpy(y).to("cuda")
    od = torch.empty_like(xd)
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.esdg_selftest_ff(op, xd.numel(), ctypes.c_void_p(xd.data_ptr()), ctypes.c_void_p(yd.data_ptr()),
                                ctypes.c_void_p(od.data_ptr()), s) == 0
    torch.cuda.synchronize()
    return od.cpu().numpy()


@pytest.mark.parametrize("op", [0, 1, 2, 3, 4])
def test_float_float_arithmetic_error_bounds(cuda_ok, op):
    """Float-float add, sub, mul, fma and reciprocal against FP64.

    Each input is first split into hi + lo (about 2^-48 relative), so the
    bounds are relative to the operands: |err| <= 2^-44 (|x| + |y|) for sums,
    2^-44 |x y| for products and 2^-43 |1/x| for the Newton reciprocal."""
    lib = fd.load_library(build_if_missing=True)
    rng = np.random.default_rng(30 + op)
    n = 1 << 18
    x = np.exp(rng.uniform(np.log(1e-25), np.log(1e25), n)) * rng.choice([-1.0, 1.0], n)
    y = np.exp(rng.uniform(np.log(1e-25), np.log(1e25), n)) * rng.choice([-1.0, 1.0], n)
    # nearly equal operands exercise cancellation in sums and differences
    y[: n // 4] = -x[: n // 4] * (1 + rng.uniform(-1e-9, 1e-9, n // 4))
    got = _ff(lib, op, x, y)
    with np.errstate(over="ignore"):
        if op == 0:
            ref, scale = x + y, np.abs(x) + np.abs(y)
        elif op == 1:
            ref, scale = x - y, np.abs(x) + np.abs(y)
        elif op == 2:
            ref, scale = x * y, np.abs(x * y)
        elif op == 3:
            ref, scale = x * y + x, np.abs(x * y) + np.abs(x)
        else:
            ref, scale = 1.0 / x, np.abs(1.0 / x)
    ok = np.isfinite(ref) & (scale < 1e37) & (scale > 1e-28)
    rel = np.abs(got[ok] - ref[ok]) / scale[ok]
    bound = 2.0 ** -43 if op == 4 else 2.0 ** -44
    assert rel.max() < bound, (op, rel.max())
    # and the pair arithmetic really carries more than FP32 precision
    assert np.median(rel) < 2.0 ** -40


def test_float_float_log(cuda_ok):
    """Float-float logarithm (no FP64 instruction) against FP64 log: absolute error
    <= 2^-46 max(1, |ln x|) on positive inputs across 1e-20 .. 1e20."""
    lib = fd.load_library(build_if_missing=True)
    rng = np.random.default_rng(41)
    n = 1 << 18
    x = np.exp(rng.uniform(np.log(1e-20), np.log(1e20), n))
    x[:1000] = 1.0 + rng.uniform(-1e-6, 1e-6, 1000)   # near 1: ln x tiny
    x[1000:2000] = np.sqrt(2.0) * (1.0 + rng.uniform(-1e-7, 1e-7, 1000))  # reduction boundary
    got = _ff(lib, 5, x, x)
    ref = np.log(x)
    err = np.abs(got - ref) / np.maximum(1.0, np.abs(ref))
    assert err.max() < 2.0 ** -46, err.max()


def test_fp64_table_log(cuda_ok):
    """The FP64 kernel's per-node logarithm (10 FP64 operations, table-driven
    reduction to [0.75, 1.5), ln 2 rounded once) on the GPU:
    * bit for bit the steps of the method as run on the host with exactly
      rounded operations (tests/test_log_table.py), on a sample;
    * against numpy's log over the whole normal range, around 1, at the
      reduction boundaries 0.75, 1.5 and powers of two, and over the ranges of
      rho and 2b = rho/p of the workloads: within 1.5 ulp of the result plus
      |k| 2^-55 (the rounding of ln 2 times the binary exponent, which cancels
      in the differences the kernel takes)."""
    from tests.test_log_table import _table, log_steps
    lib = fd.load_library(build_if_missing=True)
    rng = np.random.default_rng(43)
    n = 1 << 20
    parts = [
        np.exp(rng.uniform(np.log(1e-300), np.log(1e300), n // 2)),
        1.0 + rng.uniform(-2.0 ** -8, 2.0 ** -8, n // 16),
        1.0 + rng.uniform(-1e-9, 1e-9, n // 16),
        1.0 + np.arange(-512, 512) * 2.0 ** -52,
        np.ldexp(1.0, rng.integers(-1000, 1000, n // 32)) * (1.0 + rng.uniform(-1e-6, 1e-6, n // 32)),
        0.75 * (1.0 + rng.uniform(-1e-5, 1e-5, n // 32)),
        1.5 * (1.0 + rng.uniform(-1e-5, 1e-5, n // 32)),
        rng.uniform(0.01, 2.0, n // 8),           # densities
        rng.uniform(1e-6, 1e-4, n // 8),          # 2b = rho / p
    ]
    x = np.concatenate(parts)
    x = x[(x > 0) & np.isfinite(x)]
    xd = torch.from_numpy(x).to("cuda")
    yd = torch.empty_like(xd)
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.esdg_selftest_log(xd.numel(), ctypes.c_void_p(xd.data_ptr()), ctypes.c_void_p(yd.data_ptr()), s) == 0
    torch.cuda.synchronize()
    y = yd.cpu().numpy()
    assert np.all(np.isfinite(y))
    assert np.all(y[x == 1.0] == 0.0)
    pairs, ln2 = _table()
    for idx in rng.choice(x.size, 4000, replace=False):
        assert y[idx] == log_steps(float(x[idx]), pairs, ln2)[0], x[idx]
    k = np.frexp(x)[1].astype(np.float64)  # binary exponent, within one of the method's k
    bound = 1.5 * np.spacing(np.abs(y)) + (np.abs(k) + 1.0) * 2.0 ** -55 + 2.0 ** -54
    err = np.abs(y - np.log(x))
    assert np.all(err <= bound), (np.max(err / bound), x[np.argmax(err / bound)])


