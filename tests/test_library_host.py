"""Host-side checks of the CUDA library: no GPU needed.

The library is built (nvcc cross-compiles here) and loaded; only host entry
points are called.  Compute calls need a device and live in the -m gpu tests.
"""
import ctypes
import os
import re

import numpy as np
import pytest

import flux_differencing_gb300 as fd
import oracle
from flux_differencing_gb300 import build as fbuild

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
HEADERS = [os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", h)
           for h in ("esdg.h", "esdg_bench.h")]


@pytest.fixture(scope="module")
def lib():
    fbuild.build()
    return fd.load_library()


def _declared_symbols(path):
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(esdg_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    syms = sorted(set(sum((_declared_symbols(h) for h in HEADERS), [])))
    assert "esdg_volume_rhs" in syms and "esdg_create" in syms and "esdg_bench_fma" in syms
    for s in syms:
        assert hasattr(lib, s), s
    # and the binding knows every one of them (signatures declared)
    assert set(syms) <= set(fd._SIGS), set(syms) - set(fd._SIGS)


def test_version(lib):
    assert lib.esdg_version() >= 100


@pytest.mark.parametrize("N", range(1, 9))
def test_library_operators_match_oracle(lib, N):
    """The library's host LGL/D setup (Newton on P_N', barycentric D) agrees with the
    oracle's independent construction (Newton on x P_N - P_{N-1}, classical D formula)."""
    x, w, D = fd.operators(N)
    xo, wo = oracle.lgl(N)
    Do = oracle.dmatrix(N)
    assert np.max(np.abs(x - xo)) < 4e-16
    assert np.max(np.abs(w - wo)) < 4e-16
    assert np.max(np.abs(D - Do)) < 8e-15 * max(1, N * N)


def test_operator_argument_errors(lib):
    x = np.zeros(10)
    assert lib.esdg_get_operators(0, x.ctypes.data, x.ctypes.data, x.ctypes.data) == fd.ESDG_ERR_UNSUPPORTED
    assert lib.esdg_get_operators(9, x.ctypes.data, x.ctypes.data, x.ctypes.data) == fd.ESDG_ERR_UNSUPPORTED
    assert lib.esdg_get_operators(3, None, x.ctypes.data, x.ctypes.data) == fd.ESDG_ERR_ARG
    assert b"N must be" in lib.esdg_last_error(None) or lib.esdg_last_error(None)


def _golden(name):
    rows = {}
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        k, *v = line.split()
        rows[k] = v
    return rows


def _eq6_pairs(N, i):
    """Pairs of 1-based thread i under Eq. 6: F_{i, 1+(i+l-2) mod Nq}, l = 2..N_l."""
    Nq = N + 1
    if N % 2 == 0:
        Nl = Nq // 2 + 1
    else:
        Nl = Nq // 2 + 1 if i <= Nq // 2 else Nq // 2
    return [(i, 1 + (i + l - 2) % Nq) for l in range(2, Nl + 1)]


def test_eq6_loop_bounds_golden():
    for line in open(os.path.join(GOLDEN, "eq6_loop_bounds.txt")):
        if line.startswith("#") or not line.strip():
            continue
        N, *nl = map(int, line.split())
        Nq = N + 1
        assert len(nl) == Nq
        pairs = []
        for i in range(1, Nq + 1):
            got = _eq6_pairs(N, i)
            assert len(got) == nl[i - 1] - 1
            pairs += got
        # every unordered off-diagonal pair exactly once
        unordered = sorted(tuple(sorted(p)) for p in pairs)
        assert unordered == sorted((a, b) for a in range(1, Nq + 1) for b in range(a + 1, Nq + 1))


def test_fig1_counts_and_library_schedule_N3(lib):
    g = _golden("fig1_schedule_N3.txt")
    # (a) upper triangular: thread i computes j > i
    ut = [sum(1 for j in range(1, 5) if j > i) for i in range(1, 5)]
    assert ut == [int(v) for v in g["upper_triangular_counts"]]
    # (b) the weighted cyclic assignment runs Nq/2 offsets on every thread; the
    # library runs the same offsets, but its antipodal offset -- the pairs
    # Fig. 1(b) evaluates twice with weight 1/2 -- once per pair
    # FP32: exactly Fig. 1(b) -- two evaluations per thread, antipodal pairs in both
    # orientations, each keeping its own share (weight 1/2 per evaluation, summed)
    H, partner, sides = fd.pair_schedule(3, "fp32")
    assert [H] * 4 == [int(v) for v in g["weighted_cyclic_counts"]]
    antipodal = sorted({tuple(sorted((p + 1, int(partner[p, H - 1]) + 1))) for p in range(4)})
    assert all(sides[p, H - 1] == 1 for p in range(4))
    assert antipodal == sorted(tuple(map(int, s.split(","))) for s in g["antipodal_pairs"])
    # FP64: the same antipodal pairs, each evaluated once in a pass of its own
    H, partner, sides = fd.pair_schedule(3, "fp64")
    antipodal = sorted(tuple(sorted((p + 1, int(partner[p, H - 1]) + 1))) for p in range(4) if sides[p, H - 1])
    assert antipodal == sorted(tuple(map(int, s.split(","))) for s in g["antipodal_pairs"])


@pytest.mark.parametrize("precision", ["fp64", "fp32", "fp64ff"])
@pytest.mark.parametrize("N", range(1, 9))
def test_library_schedule_covers_each_ordered_pair_once(lib, N, precision):
    """Each node receives exactly one contribution from every other node of its line.
    FP64 evaluations per line position are Eq. 6's loop counts N_l - 1; FP32 runs
    floor(Nq/2) evaluations on every position (Fig. 1(b))."""
    H, partner, sides = fd.pair_schedule(N, precision)
    Nq = N + 1
    assert H == Nq // 2
    got = np.zeros((Nq, Nq), dtype=int)
    evals = np.zeros(Nq, dtype=int)
    for p in range(Nq):
        for d in range(H):
            antipodal = Nq % 2 == 0 and d + 1 == H
            if sides[p, d] == 0:
                assert partner[p, d] == -1 and antipodal and p >= H and precision != "fp32"
                continue
            m = int(partner[p, d])
            assert m == (p + d + 1) % Nq
            got[p, m] += 1               # own share
            if sides[p, d] == 2:
                got[m, p] += 1           # partner's share
            else:
                assert sides[p, d] == 1 and antipodal and precision == "fp32"
            evals[p] += 1
    assert np.array_equal(got, 1 - np.eye(Nq, dtype=int))
    if precision != "fp32":
        assert list(evals) == [len(_eq6_pairs(N, i)) for i in range(1, Nq + 1)]
    else:
        assert list(evals) == [H] * Nq


def test_create_rejects_bad_arguments_before_touching_the_gpu(lib):
    h = ctypes.c_void_p()
    assert lib.esdg_create(None, 1, 1, 1, 3, 0, 0) == fd.ESDG_ERR_ARG
    assert lib.esdg_create(ctypes.byref(h), 1, 1, 1, 0, 0, 0) == fd.ESDG_ERR_UNSUPPORTED
    assert lib.esdg_create(ctypes.byref(h), 1, 1, 1, 9, 0, 0) == fd.ESDG_ERR_UNSUPPORTED
    assert lib.esdg_create(ctypes.byref(h), 1, 1, 1, 3, 3, 0) == fd.ESDG_ERR_UNSUPPORTED
    assert lib.esdg_create(ctypes.byref(h), 1, 1, 1, 3, 0, 5) == fd.ESDG_ERR_UNSUPPORTED
    assert lib.esdg_create(ctypes.byref(h), 0, 1, 1, 3, 0, 0) == fd.ESDG_ERR_ARG
    assert lib.esdg_create(ctypes.byref(h), 1 << 20, 1 << 20, 1, 3, 0, 0) == fd.ESDG_ERR_ARG
    assert not h.value
    # null handles are rejected by every call that takes one
    assert lib.esdg_volume_rhs(None, None, None, None, None, None) == fd.ESDG_ERR_ARG
    assert lib.esdg_set_params(None, 1.4) == fd.ESDG_ERR_ARG
    assert lib.esdg_destroy(None) == fd.ESDG_OK
    assert lib.esdg_last_error(None)


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """No CPU fallback: without libesdg.so every call raises."""
    monkeypatch.setattr(fd, "_lib", None)
    monkeypatch.setattr(fd, "library_path", lambda debug=False: str(tmp_path / "absent.so"))
    with pytest.raises(RuntimeError, match="missing"):
        fd.operators(3)


def test_library_lsrk_coefficients_are_fourth_order(lib):
    """The library's own table (C++), checked against the fourth-order conditions
    in exact arithmetic after reading its doubles back as rationals, and against
    the oracle's independent transcription of the published rationals."""
    from fractions import Fraction

    from oracle import lsrk
    A, B, C = fd.lsrk_coefficients()
    assert len(A) == len(B) == len(C) == 5
    for got, want in zip(A + B + C, lsrk.LSRK_A + lsrk.LSRK_B + lsrk.LSRK_C):
        assert abs(got - float(want)) <= 1e-16 * max(1.0, abs(float(want)))
    a, b, c = lsrk.butcher_tableau([Fraction(x) for x in A], [Fraction(x) for x in B])
    S = 5
    conds = [(sum(b), 1), (sum(b[i] * c[i] for i in range(S)), Fraction(1, 2)),
             (sum(b[i] * a[i][j] * c[j] for i in range(S) for j in range(S)), Fraction(1, 6)),
             (sum(b[i] * a[i][j] * a[j][k] * c[k] for i in range(S) for j in range(S) for k in range(S)),
              Fraction(1, 24))]
    for got, want in conds:
        assert abs(float(got - want)) < 1e-12
    for got, want in zip(c, C):
        assert abs(float(got) - want) < 1e-12


def test_reference_state_is_the_bubble_background():
    """Outside the bubble the generated state is exactly the hydrostatic background
    that reference_state() returns (the perturbation variables vanish there)."""
    import workloads as wl
    cfg = wl.get_config("bubble_N4")
    g = wl.generate(cfg)
    ref = wl.reference_state(cfg)
    r = np.sqrt((g["x"].numpy() - 500.0) ** 2 + (g["y"].numpy() - 500.0) ** 2 + (g["z"].numpy() - 350.0) ** 2)
    outside = r > 260.0
    assert outside.sum() > cfg.n // 2
    assert np.array_equal(g["q"][0].numpy()[outside], ref["rho_ref"].numpy()[outside])
