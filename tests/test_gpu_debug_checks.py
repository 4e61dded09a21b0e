"""The kernels with their debug checks compiled in (libesdg_debug.so).

In the debug library every computed shared-memory, face-slot and global index
of the volume kernel (all modes: plain, volume + faces in one launch, fused
Runge-Kutta stage), the antipodal pass and the face-centric surface kernel is
range-checked: an index out of range sets ESDG_STATUS_INDEX and is redirected
in bounds, never trapping.  Shared memory is filled with NaN before each CTA
writes it, so that any read of a slot no phase wrote comes out as NaN.  These
tests run every order, ragged element counts (CTAs holding fewer elements
than they can) and every boundary pattern, and require: no index bit, finite
results, and the volume term within the parity tolerance of the oracle.
"""
import numpy as np
import pytest
import torch

import flux_differencing_gb300 as fd
import workloads as wl
from tests import harness as hz

pytestmark = pytest.mark.gpu

MESHES = {1: (5, 3, 2), 2: (3, 3, 2), 3: (3, 2, 3), 4: (2, 2, 3), 5: (3, 1, 3), 6: (2, 1, 3), 7: (3, 1, 2),
          8: (1, 2, 2)}
BCS = [(0, 0, 0), (1, 1, 1), (0, 1, 1)]


def _op(cfg, precision, bc, form="2d"):
    return fd.VolumeOperator(cfg.Kx, cfg.Ky, cfg.Kz, cfg.N, precision, form, bc=bc, debug=True)


def _inputs(op, g):
    Ja = op.set_geometry(g["x"].contiguous(), g["y"].contiguous(), g["z"].contiguous())
    q = g["q"].to(op.dtype).contiguous()
    phi = g["phi"].to(op.dtype).contiguous()
    return q, Ja, phi


@pytest.mark.parametrize("N", range(1, 9))
@pytest.mark.parametrize("precision", ["fp64", "fp32", "fp64ff"])
def test_debug_volume_and_surface(cuda_ok, N, precision):
    cfg = wl.small_config(N, K=MESHES[N], warp=True, state="noisy", precision=precision)
    g = hz.to_device(wl.generate(cfg))
    ref, scale = hz.run_oracle(cfg, wl.generate(cfg))
    for bc in BCS:
        op = _op(cfg, precision, bc)
        q, Ja, phi = _inputs(op, g)
        out = torch.full((5, cfg.n), float("nan"), dtype=op.dtype, device="cuda")
        op.volume_rhs(q, Ja, phi, out=out)
        st = op.status()
        assert not (st & fd.ESDG_STATUS_INDEX), (bc, st)
        got = out.double().cpu().numpy()
        assert np.all(np.isfinite(got))
        e, _ = hz.errors(got, ref, scale)
        assert e.max() < hz.TOL[precision], (bc, e)
        # surface term and volume + surface (FP32: one launch with the faces
        # evaluated by the volume kernel)
        op.surface_rhs(q, Ja, phi, out)
        r = op.rhs(q, Ja, phi)
        st = op.status()
        assert not (st & fd.ESDG_STATUS_INDEX), (bc, st)
        assert torch.isfinite(out).all() and torch.isfinite(r).all()
        op.close()


@pytest.mark.parametrize("N", [1, 2, 3, 4, 7, 8])
@pytest.mark.parametrize("precision", ["fp32", "fp64ff"])
def test_debug_fused_stages(cuda_ok, N, precision):
    """FP32: one launch per stage (faces and update in the volume kernel);
    float-float: the volume kernel applying the stage update in its store."""
    cfg = wl.small_config(N, K=MESHES[N], warp=True, state="noisy", precision=precision)
    g = hz.to_device(wl.generate(cfg))
    for bc in BCS:
        op = _op(cfg, precision, bc)
        J = torch.empty(cfg.n, dtype=op.dtype, device="cuda")
        Ja = op.set_geometry(g["x"].contiguous(), g["y"].contiguous(), g["z"].contiguous(), J_out=J)
        q = g["q"].to(op.dtype).contiguous()
        phi = g["phi"].to(op.dtype).contiguous()
        dq = torch.zeros_like(q)
        rhs = torch.zeros_like(q)
        for _ in range(2):
            op.lsrk_step(q, dq, rhs, Ja, phi, J, 1e-4)
        st = op.status()
        assert not (st & fd.ESDG_STATUS_INDEX), (bc, st)
        assert torch.isfinite(q).all()
        op.close()


@pytest.mark.parametrize("N", [1, 3, 4, 7])
def test_debug_fp32_both_log_mean_paths(cuda_ok, N):
    """FP32 CTAs on both sides of the log-mean switch (elements stretched by
    factors from 1.9 to 2.7), so the out-of-line wide phases run with the
    index checks too; plain volume, volume + faces and the fused stage."""
    from tests.test_gpu_parity import _element_ratio_state
    cfg = wl.small_config(N, K=(4, 3, 2), warp=True, precision="fp32")
    gh = _element_ratio_state(cfg, wl.generate(cfg), 1.9, 2.7)
    g = hz.to_device(gh)
    ref, scale = hz.run_oracle(cfg, gh)
    op = _op(cfg, "fp32", (0, 1, 1))
    J = torch.empty(cfg.n, dtype=op.dtype, device="cuda")
    Ja = op.set_geometry(g["x"].contiguous(), g["y"].contiguous(), g["z"].contiguous(), J_out=J)
    q = g["q"].to(op.dtype).contiguous()
    phi = g["phi"].to(op.dtype).contiguous()
    out = torch.full((5, cfg.n), float("nan"), dtype=op.dtype, device="cuda")
    op.volume_rhs(q, Ja, phi, out=out)
    assert not (op.status() & fd.ESDG_STATUS_INDEX), op.status()
    e, _ = hz.errors(out.double().cpu().numpy(), ref, scale)
    assert e.max() < hz.TOL["fp32"], e
    r = op.rhs(q, Ja, phi)
    dq = torch.zeros_like(q)
    rhs = torch.zeros_like(q)
    op.lsrk_step(q, dq, rhs, Ja, phi, J, 1e-4)
    assert not (op.status() & fd.ESDG_STATUS_INDEX), op.status()
    assert torch.isfinite(r).all() and torch.isfinite(q).all()
    op.close()
