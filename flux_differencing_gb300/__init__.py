"""GB300 flux-differencing volume term: Python binding of libesdg.so.

The binding only marshals arguments: every step of the volume term runs in
the library's CUDA kernels (see include/esdg.h for the C-ABI).  PyTorch
provides device memory and streams.  If the compiled library is missing the
import of this package still works, but every call raises: there is no CPU
fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

__all__ = [
    "ESDG_OK", "ESDG_FP64", "ESDG_FP32", "ESDG_FP64_FF", "ESDG_FORM_2D", "ESDG_FORM_SKEW", "ESDG_STATUS_NONPHYSICAL", "ESDG_STATUS_INDEX",
    "EsdgError", "library_path", "load_library", "operators", "pair_schedule", "VolumeOperator",
]

ESDG_OK = 0
ESDG_ERR_ARG, ESDG_ERR_UNSUPPORTED, ESDG_ERR_ALIGN, ESDG_ERR_CUDA, ESDG_ERR_STATE = 1, 2, 3, 4, 5
ESDG_FP64, ESDG_FP32, ESDG_FP64_FF = 0, 1, 2
_PRECISIONS = {"fp64": ESDG_FP64, "fp32": ESDG_FP32, "fp64ff": ESDG_FP64_FF}
ESDG_FORM_2D, ESDG_FORM_SKEW = 0, 1
ESDG_STATUS_NONPHYSICAL = 1
ESDG_STATUS_INDEX = 4  # debug library only: a kernel index was out of range

_ERRNAMES = {1: "ESDG_ERR_ARG", 2: "ESDG_ERR_UNSUPPORTED", 3: "ESDG_ERR_ALIGN", 4: "ESDG_ERR_CUDA",
             5: "ESDG_ERR_STATE"}

_HERE = os.path.dirname(os.path.abspath(__file__))
_lib = None
_lib_debug = None
_lock = threading.Lock()

# every symbol include/esdg.h declares, with its ctypes signature
_P = ctypes.c_void_p
_SIGS = {
    "esdg_create": (ctypes.c_int, [ctypes.POINTER(_P), ctypes.c_long, ctypes.c_long, ctypes.c_long,
                                   ctypes.c_int, ctypes.c_int, ctypes.c_int]),
    "esdg_destroy": (ctypes.c_int, [_P]),
    "esdg_set_params": (ctypes.c_int, [_P, ctypes.c_double]),
    "esdg_set_geometry": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P]),
    "esdg_volume_rhs": (ctypes.c_int, [_P, _P, _P, _P, _P, _P]),
    "esdg_volume_rhs_range": (ctypes.c_int, [_P, ctypes.c_long, ctypes.c_long, _P, _P, _P, _P, _P]),
    "esdg_set_boundary": (ctypes.c_int, [_P, ctypes.c_int, ctypes.c_int, ctypes.c_int]),
    "esdg_set_dissipation": (ctypes.c_int, [_P, ctypes.c_int]),
    "esdg_surface_rhs": (ctypes.c_int, [_P, _P, _P, _P, _P, _P]),
    "esdg_lsrk_coefficients": (ctypes.c_int, [ctypes.POINTER(ctypes.c_int), _P, _P, _P]),
    "esdg_set_coriolis": (ctypes.c_int, [_P, ctypes.c_double]),
    "esdg_set_reference": (ctypes.c_int, [_P, _P, _P]),
    "esdg_rk_stage": (ctypes.c_int, [_P, _P, _P, _P, _P, ctypes.c_double, ctypes.c_double, ctypes.c_double, _P]),
    "esdg_lsrk_step": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, ctypes.c_double, _P]),
    "esdg_diagnostics": (ctypes.c_int, [_P, _P, _P, _P, _P, _P]),
    "esdg_describe": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int),
                                     ctypes.POINTER(ctypes.c_longlong)]),
    "esdg_pipeline_create": (ctypes.c_int, [_P, ctypes.c_int, ctypes.POINTER(_P)]),
    "esdg_pipeline_submit": (ctypes.c_int, [_P, _P, _P, _P, _P]),
    "esdg_pipeline_wait": (ctypes.c_int, [_P]),
    "esdg_pipeline_last_error": (ctypes.c_char_p, [_P]),
    "esdg_pipeline_destroy": (ctypes.c_int, [_P]),
    "esdg_rhs": (ctypes.c_int, [_P, _P, _P, _P, _P, _P]),
    "esdg_get_status": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_uint), _P]),
    "esdg_last_error": (ctypes.c_char_p, [_P]),
    "esdg_get_operators": (ctypes.c_int, [ctypes.c_int, _P, _P, _P]),
    "esdg_pair_schedule": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_int), _P, _P]),
    "esdg_version": (ctypes.c_int, []),
    "esdg_volume_rhs_noalloc": (ctypes.c_int, [ctypes.c_long, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_double, _P, _P, _P, _P, ctypes.POINTER(ctypes.c_uint),
                                               _P]),
    # measurement kernels, include/esdg_bench.h
    "esdg_bench_fma": (ctypes.c_int, [ctypes.c_int, ctypes.c_long, ctypes.c_int, ctypes.c_int, _P, _P]),
    "esdg_selftest_rcp": (ctypes.c_int, [ctypes.c_int, ctypes.c_long, _P, _P, _P]),
    "esdg_selftest_ff": (ctypes.c_int, [ctypes.c_int, ctypes.c_long, _P, _P, _P, _P]),
    "esdg_selftest_log": (ctypes.c_int, [ctypes.c_long, _P, _P, _P]),
    "esdg_selftest_index_maps": (ctypes.c_int, [ctypes.c_int, ctypes.c_long, ctypes.c_long, ctypes.c_long,
                                                ctypes.POINTER(ctypes.c_int), ctypes.c_char_p, ctypes.c_int]),
}


class EsdgError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{_ERRNAMES.get(code, code)}: {msg}")
        self.code = code


def library_path(debug: bool = False) -> str:
    if debug:
        return os.path.join(_HERE, "_build_debug", "libesdg_debug.so")
    return os.path.join(_HERE, "_build", "libesdg.so")


def load_library(build_if_missing: bool = False, debug: bool = False):
    """Load libesdg.so (debug=True: libesdg_debug.so, the kernels with their index
    checks compiled in).  Raises if it is missing (no CPU fallback exists)."""
    global _lib, _lib_debug
    with _lock:
        if (_lib_debug if debug else _lib) is not None:
            return _lib_debug if debug else _lib
        path = library_path(debug)
        if not os.path.exists(path) or (debug and build_if_missing):
            if build_if_missing:
                from . import build as _build
                _build.build(debug=debug)
            else:
                raise RuntimeError(
                    f"{path} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'` "
                    "or `python flux_differencing_gb300/build.py`")
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if debug:
            _lib_debug = lib
        else:
            _lib = lib
        return lib


def _chk(op, rc: int, h=None):
    _check(rc, h, op.lib)


def _check(rc: int, h=None, lib=None):
    if rc != ESDG_OK:
        lib = lib or load_library()
        msg = lib.esdg_last_error(h).decode()
        raise EsdgError(rc, msg)


def operators(N: int):
    """LGL nodes, weights and D exactly as the kernels use them (host call)."""
    lib = load_library()
    x = np.zeros(N + 1)
    w = np.zeros(N + 1)
    D = np.zeros((N + 1, N + 1))
    _check(lib.esdg_get_operators(N, x.ctypes.data, w.ctypes.data, D.ctypes.data))
    return x, w, D


def pair_schedule(N: int, precision: str = "fp64"):
    """(H, partner[p, d-1], sides[p, d-1]) of the kernel's per-line pair schedule."""
    lib = load_library()
    H = ctypes.c_int(0)
    partner = np.zeros((N + 1) * ((N + 1) // 2), dtype=np.int32)
    sides = np.zeros_like(partner)
    prec = _PRECISIONS[precision]
    _check(lib.esdg_pair_schedule(N, prec, ctypes.byref(H), partner.ctypes.data, sides.ctypes.data))
    return H.value, partner.reshape(N + 1, -1), sides.reshape(N + 1, -1)


class Pipeline:
    """Pipelined volume-term evaluation from host buffers (esdg_pipeline_*).

    submit() enqueues the copies in, the kernel and the copy out on the next of
    `depth` slots and returns at once; wait() blocks until every submission
    has completed.  Host tensors should be pinned; keep them unchanged until
    their submission completes."""

    def __init__(self, op: "VolumeOperator", depth: int = 2):
        self.op = op
        self.lib = op.lib
        p = ctypes.c_void_p()
        _chk(self, self.lib.esdg_pipeline_create(op.h, int(depth), ctypes.byref(p)))
        self.p = p
        self.depth = int(depth)

    def _err(self, rc):
        if rc != 0:
            raise EsdgError(rc, self.lib.esdg_pipeline_last_error(self.p).decode())

    def submit(self, q, metrics, phi, out):
        for t, nm, k in ((q, "q", 5), (metrics, "metrics", 9), (phi, "phi", 1), (out, "out", 5)):
            if t.is_cuda or t.dtype != self.op.dtype or not t.is_contiguous() or t.numel() != k * self.op.n:
                raise ValueError(f"{nm}: need a contiguous host {self.op.dtype} tensor with {k * self.op.n} values")
        self._err(self.lib.esdg_pipeline_submit(self.p, ctypes.c_void_p(q.data_ptr()),
                                                ctypes.c_void_p(metrics.data_ptr()),
                                                ctypes.c_void_p(phi.data_ptr()), ctypes.c_void_p(out.data_ptr())))

    def wait(self):
        self._err(self.lib.esdg_pipeline_wait(self.p))

    def close(self):
        if getattr(self, "p", None):
            self.lib.esdg_pipeline_destroy(self.p)
            self.p = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def lsrk_coefficients():
    """(A, B, C) of the library's five-stage low-storage Runge-Kutta scheme (host call)."""
    lib = load_library()
    st = ctypes.c_int(0)
    A = (ctypes.c_double * 5)()
    B = (ctypes.c_double * 5)()
    C = (ctypes.c_double * 5)()
    _check(lib.esdg_lsrk_coefficients(ctypes.byref(st), A, B, C))
    return list(A)[:st.value], list(B)[:st.value], list(C)[:st.value]


def _stream_ptr(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dptr(t):
    return ctypes.c_void_p(t.data_ptr())


class VolumeOperator:
    """A handle for one mesh shape, order and precision.

    precision: "fp64", "fp32" or "fp64ff" (FP64 buffers, float-float pair
    arithmetic); form: "2d" (diagonal kept) or "skew"; bc: surface-term
    boundary kind per reference direction (0 periodic, 1 slip wall);
    dissipation: matrix dissipation in the surface flux.
    Tensors passed in must be contiguous CUDA tensors of the handle's dtype
    (node coordinates are always float64), laid out as described in esdg.h.
    """

    def __init__(self, Kx: int, Ky: int, Kz: int, N: int, precision: str = "fp64", form: str = "2d",
                 gamma: float = 1.4, bc=(0, 0, 0), dissipation: bool = True, debug: bool = False):
        import torch
        self.lib = load_library(build_if_missing=debug, debug=debug)
        self.Kx, self.Ky, self.Kz, self.N = int(Kx), int(Ky), int(Kz), int(N)
        self.K = self.Kx * self.Ky * self.Kz
        self.n = self.K * (self.N + 1) ** 3
        self.precision = precision
        self.dtype = {"fp64": torch.float64, "fp32": torch.float32, "fp64ff": torch.float64}[precision]
        prec = _PRECISIONS[precision]
        frm = {"2d": ESDG_FORM_2D, "skew": ESDG_FORM_SKEW}[form]
        h = ctypes.c_void_p()
        _chk(self, self.lib.esdg_create(ctypes.byref(h), self.Kx, self.Ky, self.Kz, self.N, prec, frm))
        self.h = h
        if gamma != 1.4:
            _chk(self, self.lib.esdg_set_params(self.h, float(gamma)), self.h)
        self.set_boundary(*bc)
        self.set_dissipation(dissipation)

    def set_boundary(self, bc_xi: int = 0, bc_eta: int = 0, bc_zeta: int = 0):
        """Surface-term boundary kind per reference direction: 0 periodic, 1 slip wall."""
        _chk(self, self.lib.esdg_set_boundary(self.h, int(bc_xi), int(bc_eta), int(bc_zeta)), self.h)
        self.bc = (int(bc_xi), int(bc_eta), int(bc_zeta))

    def set_dissipation(self, on: bool = True):
        """Surface flux with (default) or without the matrix dissipation."""
        _chk(self, self.lib.esdg_set_dissipation(self.h, int(bool(on))), self.h)
        self.dissipation = bool(on)

    def close(self):
        if getattr(self, "h", None):
            self.lib.esdg_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _req(self, t, numel, dtype=None, name="tensor"):
        dt = dtype or self.dtype
        if not t.is_cuda or t.dtype != dt or not t.is_contiguous() or t.numel() != numel:
            raise ValueError(f"{name}: need a contiguous CUDA {dt} tensor with {numel} elements, got "
                             f"{t.dtype} {tuple(t.shape)} on {t.device}")

    def set_geometry(self, x, y, z, metrics_out=None, J_out=None, stream=None):
        """Curl-form metric terms (9, n) (and J (n,) if J_out is given) from node coordinates."""
        import torch
        for t, nm in ((x, "x"), (y, "y"), (z, "z")):
            self._req(t, self.n, torch.float64, nm)
        if metrics_out is None:
            metrics_out = torch.empty((9, self.n), dtype=self.dtype, device=x.device)
        self._req(metrics_out, 9 * self.n, name="metrics_out")
        if J_out is not None:
            self._req(J_out, self.n, name="J_out")
        _chk(self, self.lib.esdg_set_geometry(self.h, _dptr(x), _dptr(y), _dptr(z), _dptr(metrics_out),
                                          _dptr(J_out) if J_out is not None else None, _stream_ptr(stream)),
               self.h)
        return metrics_out

    def volume_rhs(self, q, metrics, phi, out=None, stream=None, e_begin: int | None = None,
                   e_count: int | None = None):
        """Volume term (5, n); optionally only elements [e_begin, e_begin + e_count)."""
        import torch
        self._req(q, 5 * self.n, name="q")
        self._req(metrics, 9 * self.n, name="metrics")
        self._req(phi, self.n, name="phi")
        if out is None:
            out = torch.empty((5, self.n), dtype=self.dtype, device=q.device)
        self._req(out, 5 * self.n, name="out")
        sp = _stream_ptr(stream)
        if e_begin is None and e_count is None:
            rc = self.lib.esdg_volume_rhs(self.h, _dptr(q), _dptr(metrics), _dptr(phi), _dptr(out), sp)
        else:
            eb = 0 if e_begin is None else int(e_begin)
            ec = self.K - eb if e_count is None else int(e_count)
            rc = self.lib.esdg_volume_rhs_range(self.h, eb, ec, _dptr(q), _dptr(metrics), _dptr(phi),
                                                _dptr(out), sp)
        _check(rc, self.h)
        return out

    def surface_rhs(self, q, metrics, phi, out, stream=None):
        """Add the surface term into out (5, n): out = volume + surface after volume_rhs."""
        self._req(q, 5 * self.n, name="q")
        self._req(metrics, 9 * self.n, name="metrics")
        self._req(phi, self.n, name="phi")
        self._req(out, 5 * self.n, name="out")
        _chk(self, self.lib.esdg_surface_rhs(self.h, _dptr(q), _dptr(metrics), _dptr(phi), _dptr(out),
                                         _stream_ptr(stream)), self.h)
        return out

    def set_reference(self, rho_ref=None, p_ref=None):
        """Switch to perturbation variables about (rho_ref, p_ref) (both (n,) CUDA tensors of
        the handle's dtype), or back to full-state variables with no arguments.  The handle
        keeps references to the tensors so they stay alive."""
        if (rho_ref is None) != (p_ref is None):
            raise ValueError("rho_ref and p_ref must both be given or both be None")
        if rho_ref is not None:
            self._req(rho_ref, self.n, name="rho_ref")
            self._req(p_ref, self.n, name="p_ref")
        _chk(self, self.lib.esdg_set_reference(self.h, _dptr(rho_ref) if rho_ref is not None else None,
                                           _dptr(p_ref) if p_ref is not None else None), self.h)
        self._reference = (rho_ref, p_ref)

    def set_coriolis(self, f: float = 0.0):
        """f-plane Coriolis parameter (s^-1) of the time-stepping source h."""
        _chk(self, self.lib.esdg_set_coriolis(self.h, float(f)), self.h)
        self.coriolis = float(f)

    def rk_stage(self, q, dq, rhs, J, a: float, b: float, dt: float, stream=None):
        """dq <- a dq + dt (h - rhs/J); q <- q + b dq (in place)."""
        for t, nm, k in ((q, "q", 5), (dq, "dq", 5), (rhs, "rhs", 5), (J, "J", 1)):
            self._req(t, k * self.n, name=nm)
        _chk(self, self.lib.esdg_rk_stage(self.h, _dptr(q), _dptr(dq), _dptr(rhs), _dptr(J), float(a), float(b),
                                      float(dt), _stream_ptr(stream)), self.h)

    def lsrk_step(self, q, dq, rhs, metrics, phi, J, dt: float, stream=None):
        """One five-stage step of size dt, in place on q (dq and rhs are scratch)."""
        for t, nm, k in ((q, "q", 5), (dq, "dq", 5), (rhs, "rhs", 5), (metrics, "metrics", 9),
                         (phi, "phi", 1), (J, "J", 1)):
            self._req(t, k * self.n, name=nm)
        _chk(self, self.lib.esdg_lsrk_step(self.h, _dptr(q), _dptr(dq), _dptr(rhs), _dptr(metrics), _dptr(phi),
                                       _dptr(J), float(dt), _stream_ptr(stream)), self.h)

    def diagnostics(self, q, J, phi, out=None, stream=None):
        """(mass, energy, entropy) integrals as a CUDA float64 tensor of 3 values."""
        import torch
        self._req(q, 5 * self.n, name="q")
        self._req(J, self.n, name="J")
        self._req(phi, self.n, name="phi")
        if out is None:
            out = torch.empty(3, dtype=torch.float64, device=q.device)
        if not (out.is_cuda and out.dtype == torch.float64 and out.numel() >= 3):
            raise ValueError("out: need a CUDA float64 tensor of at least 3 values")
        _chk(self, self.lib.esdg_diagnostics(self.h, _dptr(q), _dptr(J), _dptr(phi), _dptr(out),
                                         _stream_ptr(stream)), self.h)
        return out

    def rhs(self, q, metrics, phi, out=None, stream=None):
        """Volume + surface term (5, n) through esdg_rhs: dq/dt = h - rhs/J."""
        import torch
        self._req(q, 5 * self.n, name="q")
        self._req(metrics, 9 * self.n, name="metrics")
        self._req(phi, self.n, name="phi")
        if out is None:
            out = torch.empty((5, self.n), dtype=self.dtype, device=q.device)
        self._req(out, 5 * self.n, name="out")
        _chk(self, self.lib.esdg_rhs(self.h, _dptr(q), _dptr(metrics), _dptr(phi), _dptr(out), _stream_ptr(stream)),
               self.h)
        return out

    def status(self, stream=None) -> int:
        """Read and clear the status word (synchronises the stream)."""
        v = ctypes.c_uint(0)
        _chk(self, self.lib.esdg_get_status(self.h, ctypes.byref(v), _stream_ptr(stream)), self.h)
        return v.value
