"""esdg_volume_rhs_noalloc: the entry point for callers that cannot allocate device memory.

Applications that own all device memory through their own pool, or that must
not call cudaMalloc while other streams are busy, cannot use esdg_create (it
allocates a device status word).  esdg_volume_rhs_noalloc takes no handle and
keeps its status word in a static device array of the library.  These tests
call it through the C-ABI and check it against the handle-based
esdg_volume_rhs, on two calls in a row (the second sees the array as the
first left it).  The file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import flux_differencing_gb300 as fd
import workloads as wl
from tests import harness as hz

pytestmark = pytest.mark.gpu


def _noalloc(lib, cfg, precision, q, Ja, phi, out, form=fd.ESDG_FORM_2D):
    status = ctypes.c_uint(12345)
    prec = fd.ESDG_FP64 if precision == "fp64" else fd.ESDG_FP32
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.esdg_volume_rhs_noalloc(cfg.K, cfg.N, prec, form, 1.4, ctypes.c_void_p(q.data_ptr()),
                                     ctypes.c_void_p(Ja.data_ptr()), ctypes.c_void_p(phi.data_ptr()),
                                     ctypes.c_void_p(out.data_ptr()), ctypes.byref(status), stream)
    assert rc == fd.ESDG_OK, lib.esdg_last_error(None)
    return status.value


@pytest.mark.parametrize("precision,N,form", [("fp64", 4, "2d"), ("fp64", 7, "2d"), ("fp32", 3, "2d"),
                                              ("fp32", 7, "2d"), ("fp64", 5, "skew"), ("fp32", 7, "skew")])
def test_noalloc_matches_handle_path_on_two_calls(cuda_ok, precision, N, form):
    lib = fd.load_library(build_if_missing=True)
    cfg = wl.small_config(N, K=(3, 2, 2), warp=True, precision=precision)
    g = wl.generate(cfg)
    ref, op, Ja = hz.run_gpu(cfg, g, form=form)             # handle path, same form
    _, scale = hz.run_oracle(cfg, g, form=0 if form == "2d" else 1)  # term scale for the tolerance
    dg = hz.to_device(g)
    q = dg["q"].to(op.dtype).contiguous()
    phi = dg["phi"].to(op.dtype).contiguous()
    abi_form = fd.ESDG_FORM_2D if form == "2d" else fd.ESDG_FORM_SKEW
    for call in range(2):
        out = torch.full((5, cfg.n), float("nan"), dtype=op.dtype, device="cuda")
        status = _noalloc(lib, cfg, precision, q, Ja, phi, out, form=abi_form)
        assert status == 0
        got = out.double().cpu().numpy()
        e, _ = hz.errors(got, ref, scale)
        assert e.max() < hz.TOL[precision], (call, e)


def test_noalloc_status_word_is_cleared_between_calls(cuda_ok):
    lib = fd.load_library(build_if_missing=True)
    cfg = wl.small_config(2, K=(2, 1, 1), warp=False)
    g = hz.to_device(wl.generate(cfg))
    op = fd.VolumeOperator(cfg.Kx, cfg.Ky, cfg.Kz, cfg.N, "fp64")
    Ja = op.set_geometry(g["x"], g["y"], g["z"])
    out = torch.empty((5, cfg.n), dtype=torch.float64, device="cuda")
    bad = g["q"].clone()
    bad[0, 3] = -1.0
    assert _noalloc(lib, cfg, "fp64", bad, Ja, g["phi"], out) & fd.ESDG_STATUS_NONPHYSICAL
    assert _noalloc(lib, cfg, "fp64", g["q"], Ja, g["phi"], out) == 0


def test_noalloc_rejects_bad_arguments(cuda_ok):
    lib = fd.load_library(build_if_missing=True)
    cfg = wl.small_config(3, K=(1, 1, 1), warp=False)
    g = hz.to_device(wl.generate(cfg))
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    out = torch.empty((5, cfg.n), dtype=torch.float64, device="cuda")
    Ja = torch.zeros((9, cfg.n), dtype=torch.float64, device="cuda")
    args = (P(g["q"]), P(Ja), P(g["phi"]), P(out), None, s)
    assert lib.esdg_volume_rhs_noalloc(1, 9, 0, 0, 1.4, *args) == fd.ESDG_ERR_UNSUPPORTED
    assert lib.esdg_volume_rhs_noalloc(0, 3, 0, 0, 1.4, *args) == fd.ESDG_ERR_ARG
    assert lib.esdg_volume_rhs_noalloc(1 << 31, 3, 0, 0, 1.4, *args) == fd.ESDG_ERR_ARG
    assert b"too large" in lib.esdg_last_error(None)
    assert lib.esdg_volume_rhs_noalloc(1, 3, 0, 0, 1.4, P(g["q"]), P(Ja), P(g["phi"]), P(g["q"]), None,
                                       s) == fd.ESDG_ERR_ARG
