"""Shared helpers for the parity tests: run the CUDA path and the oracle on the
same seeded inputs and measure the normalised error.

Error measure (per conserved variable c):
    e_c = max_i |gpu_c,i - oracle_c,i| / S_c,   S_c = max_i sum_r sum_m |2 D_im F^r_c(i, m)|
S_c is the magnitude of the terms the volume sum adds up (for the surface
term: sum over the node's faces of (|F*_c| + |f_c.n| + M_c)/w_0, M the
magnitude of the dissipation's terms, which carry rounding relative to |w|
because [[w]] is a difference of O(|w|) numbers); the plain relative
error max|diff| / max|oracle| is also returned because for nearly hydrostatic
states the momentum sum is a near-cancellation of pressure terms and its
plain relative error reflects that conditioning, not the kernel.
"""
import numpy as np
import torch

import flux_differencing_gb300 as fd
import oracle

TOL = {"fp64": 1e-11, "fp32": 1e-4, "fp64ff": 1e-11}


def to_device(g, device="cuda"):
    return {k: v.to(device) for k, v in g.items()}


def run_gpu(cfg, g, form="2d", precision=None, out=None, op=None):
    """Volume term on the GPU through the C-ABI; returns (out (5,n) float64 numpy, op, Ja)."""
    prec = precision or cfg.precision
    if op is None:
        op = fd.VolumeOperator(cfg.Kx, cfg.Ky, cfg.Kz, cfg.N, prec, form)
    dg = g if g["q"].is_cuda else to_device(g)
    Ja = op.set_geometry(dg["x"].contiguous(), dg["y"].contiguous(), dg["z"].contiguous())
    q = dg["q"].to(op.dtype).contiguous()
    phi = dg["phi"].to(op.dtype).contiguous()
    res = op.volume_rhs(q, Ja, phi, out=out)
    torch.cuda.synchronize()
    return res.double().cpu().numpy(), op, Ja


def run_oracle(cfg, g, form=0, K=None, nthreads=None):
    gc = {k: v.cpu().numpy() for k, v in g.items()}
    K = cfg.K if K is None else K
    Ja, _ = oracle.metrics(cfg.N, K, gc["x"], gc["y"], gc["z"])
    out, scale = oracle.volume(cfg.N, K, gc["q"], Ja, gc["phi"], form=form, with_scale=True,
                               nthreads=nthreads)
    return out, scale


def errors(got, ref, scale):
    """(normalised e_c per variable, plain relative error per variable)."""
    e = np.array([np.max(np.abs(got[c] - ref[c])) / np.max(scale[c]) for c in range(5)])
    plain = np.array([np.max(np.abs(got[c] - ref[c])) / max(np.max(np.abs(ref[c])), 1e-300) for c in range(5)])
    return e, plain


def run_gpu_surface(cfg, g, form="2d", precision=None, dissipation=True, bc=None, with_volume=False):
    """Surface term alone (or volume + surface) on the GPU; returns (out float64 numpy, op)."""
    prec = precision or cfg.precision
    bc = cfg.bc if bc is None else bc
    op = fd.VolumeOperator(cfg.Kx, cfg.Ky, cfg.Kz, cfg.N, prec, form, bc=bc, dissipation=dissipation)
    dg = g if g["q"].is_cuda else to_device(g)
    Ja = op.set_geometry(dg["x"].contiguous(), dg["y"].contiguous(), dg["z"].contiguous())
    q = dg["q"].to(op.dtype).contiguous()
    phi = dg["phi"].to(op.dtype).contiguous()
    if with_volume:
        res = op.rhs(q, Ja, phi)
    else:
        res = torch.zeros((5, cfg.n), dtype=op.dtype, device=q.device)
        op.surface_rhs(q, Ja, phi, res)
    torch.cuda.synchronize()
    return res.double().cpu().numpy(), op


def run_oracle_surface(cfg, g, form=0, dissipation=True, bc=None, nthreads=None):
    gc = {k: v.cpu().numpy() for k, v in g.items()}
    bc = cfg.bc if bc is None else bc
    Ja, _ = oracle.metrics(cfg.N, cfg.K, gc["x"], gc["y"], gc["z"])
    return oracle.surface(cfg.N, (cfg.Kx, cfg.Ky, cfg.Kz), gc["q"], Ja, gc["phi"], bc, form=form,
                          dissipation=dissipation, with_scale=True, nthreads=nthreads)
