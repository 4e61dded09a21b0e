"""CPU oracle for the flux-differencing volume term (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never loads it and the
two share no code: the oracle is plain C (``esdg_oracle.c``), written from
"GPU Performance of an Entropy-Stable Discontinuous Galerkin Euler Solver with
Non-Conservative Terms" (Sec. 3 Eq. 2, Sec. 4.1 Eqs. 3-5), compiled with gcc
-O2 and no fast-math.  It covers the volume term and the surface term (the
entropy-conserving flux plus matrix dissipation at element faces).

Functions take and return numpy arrays.  ``real='d'`` uses the double build,
``real='ld'`` the long-double build (80-bit on x86-64, binary128 on aarch64).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = [os.path.join(_HERE, "esdg_oracle.c"), os.path.join(_HERE, "oracle_impl.inc")]
_LIB_PATH = os.path.join(_HERE, "_build", "libesdg_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle shared library (gcc, OpenMP, -O2, no fast-math)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or any(
        os.path.getmtime(s) > os.path.getmtime(_LIB_PATH) for s in _SRC)
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
               "-std=c11", "-o", tmp, _SRC[0], "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            for sfx in ("_d", "_ld"):
                real = ctypes.c_double if sfx == "_d" else ctypes.c_longdouble
                getattr(lib, "ora_lgl" + sfx).argtypes = [ctypes.c_int, P, P]
                getattr(lib, "ora_dmatrix" + sfx).argtypes = [ctypes.c_int, P, P]
                getattr(lib, "ora_metrics" + sfx).argtypes = [ctypes.c_int, ctypes.c_long, P, P, P, P, P]
                getattr(lib, "ora_flux" + sfx).argtypes = [P, real, P, real, P, real, P]
                getattr(lib, "ora_volume" + sfx).argtypes = [
                    ctypes.c_int, ctypes.c_long, P, P, P, real, ctypes.c_int, P, P, ctypes.c_int]
                getattr(lib, "ora_roe_matrices" + sfx).argtypes = [P, real, P, real, P, real, P, P, P]
                getattr(lib, "ora_dissipation" + sfx).argtypes = [P, real, P, real, P, real, P]
                getattr(lib, "ora_surface_flux" + sfx).argtypes = [P, real, P, real, P, real, ctypes.c_int, P]
                getattr(lib, "ora_surface" + sfx).argtypes = [
                    ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P, P, P, real,
                    ctypes.c_int, ctypes.c_int, P, P, ctypes.c_int]
            lib.ora_max_threads.restype = ctypes.c_int
            lib.ora_sizeof_long_double.restype = ctypes.c_int
            _lib = lib
    return _lib


def _dt(real: str):
    return np.float64 if real == "d" else np.longdouble


def _arr(a, real):
    return np.ascontiguousarray(np.asarray(a), dtype=_dt(real))


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def max_threads() -> int:
    return _load().ora_max_threads()


def lgl(N: int, real: str = "d"):
    """LGL nodes (ascending) and weights."""
    lib = _load()
    x = np.zeros(N + 1, dtype=_dt(real))
    w = np.zeros(N + 1, dtype=_dt(real))
    getattr(lib, "ora_lgl_" + real)(N, _ptr(x), _ptr(w))
    return x, w


def dmatrix(N: int, real: str = "d"):
    """LGL differentiation matrix, D[i, j] = l_j'(x_i)."""
    lib = _load()
    x, _ = lgl(N, real)
    D = np.zeros((N + 1, N + 1), dtype=_dt(real))
    getattr(lib, "ora_dmatrix_" + real)(N, _ptr(x), _ptr(D))
    return D


def metrics(N: int, K: int, x, y, z, real: str = "d"):
    """Curl-form metric terms (9, n) with plane 3*r + j = Ja^r_j, and J (n,)."""
    lib = _load()
    x, y, z = (_arr(v, real) for v in (x, y, z))
    n = K * (N + 1) ** 3
    assert x.size == y.size == z.size == n
    Ja = np.zeros((9, n), dtype=_dt(real))
    J = np.zeros(n, dtype=_dt(real))
    getattr(lib, "ora_metrics_" + real)(N, K, _ptr(x), _ptr(y), _ptr(z), _ptr(Ja), _ptr(J))
    return Ja, J


def flux(qi, phii, qm, phim, nvec, gamma=1.4, real: str = "d"):
    """Two-point flux F(q_i, q_m) . n including the gravity term (i is the '-' side)."""
    lib = _load()
    qi, qm, nvec = _arr(qi, real), _arr(qm, real), _arr(nvec, real)
    F = np.zeros(5, dtype=_dt(real))
    getattr(lib, "ora_flux_" + real)(_ptr(qi), phii, _ptr(qm), phim, _ptr(nvec), gamma, _ptr(F))
    return F


def volume(N: int, K: int, q, Ja, phi, gamma=1.4, form: int = 0, real: str = "d",
           with_scale: bool = False, nthreads: int | None = None):
    """Volume term (5, n); with_scale also returns sum |2 D F| per node and variable."""
    lib = _load()
    n = K * (N + 1) ** 3
    q = _arr(q, real).reshape(5, n)
    Ja = _arr(Ja, real).reshape(9, n)
    phi = _arr(phi, real).reshape(n)
    out = np.zeros((5, n), dtype=_dt(real))
    scale = np.zeros((5, n), dtype=_dt(real)) if with_scale else None
    nt = nthreads if nthreads is not None else max_threads()
    getattr(lib, "ora_volume_" + real)(N, K, _ptr(q), _ptr(Ja), _ptr(phi), gamma, form,
                                       _ptr(out), _ptr(scale) if with_scale else None, nt)
    return (out, scale) if with_scale else out


def roe_matrices(qm, phim, qp, phip, nvec, gamma=1.4, real: str = "d"):
    """Right eigenvectors R (columns), eigenvalues (unit normal) and scaling T at the averaged state."""
    lib = _load()
    qm, qp, nvec = _arr(qm, real), _arr(qp, real), _arr(nvec, real)
    R = np.zeros((5, 5), dtype=_dt(real))
    lam = np.zeros(5, dtype=_dt(real))
    T = np.zeros(5, dtype=_dt(real))
    getattr(lib, "ora_roe_matrices_" + real)(_ptr(qm), phim, _ptr(qp), phip, _ptr(nvec), gamma,
                                             _ptr(R), _ptr(lam), _ptr(T))
    return R, lam, T


def dissipation(qm, phim, qp, phip, nvec, gamma=1.4, real: str = "d"):
    """Matrix dissipation 1/2 |n| R |Lambda| T R^T [[w]] of the surface flux."""
    lib = _load()
    qm, qp, nvec = _arr(qm, real), _arr(qp, real), _arr(nvec, real)
    D = np.zeros(5, dtype=_dt(real))
    getattr(lib, "ora_dissipation_" + real)(_ptr(qm), phim, _ptr(qp), phip, _ptr(nvec), gamma, _ptr(D))
    return D


def surface_flux(qm, phim, qp, phip, nvec, gamma=1.4, dissipation: bool = True, real: str = "d"):
    """Surface flux F*(q-, q+; n): entropy-conserving flux with gravity, minus the dissipation."""
    lib = _load()
    qm, qp, nvec = _arr(qm, real), _arr(qp, real), _arr(nvec, real)
    F = np.zeros(5, dtype=_dt(real))
    getattr(lib, "ora_surface_flux_" + real)(_ptr(qm), phim, _ptr(qp), phip, _ptr(nvec), gamma,
                                             int(bool(dissipation)), _ptr(F))
    return F


def surface(N: int, K, q, Ja, phi, bc=(0, 0, 0), gamma=1.4, form: int = 0, dissipation: bool = True,
            real: str = "d", with_scale: bool = False, nthreads: int | None = None):
    """Surface term (5, n) on a Kx x Ky x Kz brick; bc[r] = 0 periodic, 1 slip wall.

    form 0 pairs with the strong (2D) volume form and subtracts the physical
    flux at the face nodes; form 1 (skew) adds F* alone.  with_scale also
    returns sum (|F*| + |f.n| + M)/w_0 per node and variable, M the magnitude
    bound 1/2 |n| |R| |Lambda| T |R|^T (|w-| + |w+|) of the dissipation's
    terms (its rounding scale: [[w]] is a difference of O(|w|) numbers).
    """
    lib = _load()
    Kx, Ky, Kz = (int(k) for k in K)
    n = Kx * Ky * Kz * (N + 1) ** 3
    q = _arr(q, real).reshape(5, n)
    Ja = _arr(Ja, real).reshape(9, n)
    phi = _arr(phi, real).reshape(n)
    bcs = np.ascontiguousarray(np.asarray(bc, dtype=np.int32).reshape(3))
    out = np.zeros((5, n), dtype=_dt(real))
    scale = np.zeros((5, n), dtype=_dt(real)) if with_scale else None
    nt = nthreads if nthreads is not None else max_threads()
    getattr(lib, "ora_surface_" + real)(N, Kx, Ky, Kz, _ptr(bcs), _ptr(q), _ptr(Ja), _ptr(phi), gamma,
                                        form, int(bool(dissipation)), _ptr(out),
                                        _ptr(scale) if with_scale else None, nt)
    return (out, scale) if with_scale else out
