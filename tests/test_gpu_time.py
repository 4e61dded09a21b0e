"""Time stepping and diagnostics on the GPU against the oracle (GPU required).

One five-stage step through esdg_lsrk_step is compared with oracle/lsrk.py on
the same inputs; the error of q after the step is normalised per conserved
variable by dt * max_i (S_vol + S_surf)_i / J_i (the magnitude of the summed
terms of the increment) plus the storage rounding 8 eps |q|.  Multi-step runs
check conservation and the entropy decrease on the GPU result alone.
"""
import math

import numpy as np
import pytest
import torch

import flux_differencing_gb300 as fd
import oracle
import workloads as wl
from oracle import lsrk
from tests import harness as hz
from tests import physics as ph

pytestmark = pytest.mark.gpu

EPS = {"fp64": 2.0 ** -52, "fp32": 2.0 ** -23, "fp64ff": 2.0 ** -52}


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_ok):
    fd.load_library(build_if_missing=True)


def _setup(cfg, form="2d", dissipation=True, coriolis=0.0):
    g = wl.generate(cfg)
    op = fd.VolumeOperator(cfg.Kx, cfg.Ky, cfg.Kz, cfg.N, cfg.precision, form, bc=cfg.bc,
                           dissipation=dissipation)
    if coriolis:
        op.set_coriolis(coriolis)
    dg = hz.to_device(g)
    J = torch.empty(cfg.n, dtype=op.dtype, device="cuda")
    Ja = op.set_geometry(dg["x"], dg["y"], dg["z"], J_out=J)
    q = dg["q"].to(op.dtype).contiguous()
    phi = dg["phi"].to(op.dtype).contiguous()
    return g, op, Ja, J, q, phi


def _stable_dt(cfg, q, phi, cfl=0.3):
    rho, u, p = ph.primitives(q, phi)
    speed = np.max(np.sqrt(np.sum(u * u, axis=0)) + np.sqrt(1.4 * p / rho))
    h = min(cfg.domain[0] / cfg.Kx, cfg.domain[1] / cfg.Ky, cfg.domain[2] / cfg.Kz)
    return cfl * h / speed / (cfg.N + 1) ** 2


@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("precision", ["fp64", "fp32", "fp64ff"])
def test_lsrk_step_parity(N, precision):
    cfg = wl.small_config(N, K=(2, 2, 2), warp=True, state="noisy", precision=precision, bc=(0, 1, 1))
    g, op, Ja, J, q, phi = _setup(cfg, coriolis=1e-3)
    qn, phin = g["q"].numpy(), g["phi"].numpy()
    dt = _stable_dt(cfg, qn, phin)
    dq = torch.zeros_like(q)
    rhs = torch.empty_like(q)
    op.lsrk_step(q, dq, rhs, Ja, phi, J, dt)
    torch.cuda.synchronize()
    assert op.status() == 0
    got = q.double().cpu().numpy()
    Jao, Jo = oracle.metrics(N, cfg.K, g["x"].numpy(), g["y"].numpy(), g["z"].numpy())
    K3 = (cfg.Kx, cfg.Ky, cfg.Kz)
    ref, _ = lsrk.lsrk_step(N, K3, qn, np.zeros_like(qn), Jao, phin, Jo, dt, bc=cfg.bc, coriolis=1e-3)
    _, vs = oracle.volume(N, cfg.K, qn, Jao, phin, with_scale=True)
    _, ss = oracle.surface(N, K3, qn, Jao, phin, cfg.bc, with_scale=True)
    scale = dt * np.max((vs + ss) / Jo, axis=1) + 8 * EPS[precision] * np.max(np.abs(qn), axis=1)
    err = np.max(np.abs(got - ref), axis=1) / scale
    assert err.max() < hz.TOL[precision], err


@pytest.mark.parametrize("N,K,bc,dissipation", [
    (1, (5, 3, 2), (0, 1, 0), True),   # 30 elements: two 16-element CTAs, neighbours inside one CTA
    (3, (3, 1, 2), (0, 0, 1), True),   # one element along eta, periodic: the face's neighbour is itself
    (4, (2, 3, 2), (1, 1, 1), True),   # walls on every side
    (7, (2, 2, 3), (0, 0, 0), True),   # fully periodic
    (5, (3, 2, 2), (0, 1, 1), False),  # entropy-conserving interface flux (no dissipation)
])
def test_lsrk_fp32_fused_stage_two_steps(N, K, bc, dissipation):
    """The FP32 step (one launch per stage, faces evaluated inside the volume
    kernel, q and rhs alternating as state buffers) against two oracle steps,
    on meshes that exercise the face-slot and neighbour indexing: several
    elements per CTA, a single element along a periodic direction, walls on
    every side, full periodicity, and the flux without dissipation."""
    cfg = wl.small_config(N, K=K, warp=True, state="noisy", precision="fp32", bc=bc)
    g, op, Ja, J, q, phi = _setup(cfg, dissipation=dissipation)
    qn, phin = g["q"].numpy(), g["phi"].numpy()
    dt = _stable_dt(cfg, qn, phin)
    dq = torch.zeros_like(q)
    rhs = torch.empty_like(q)
    for _ in range(2):
        op.lsrk_step(q, dq, rhs, Ja, phi, J, dt)
    torch.cuda.synchronize()
    assert op.status() == 0
    got = q.double().cpu().numpy()
    Jao, Jo = oracle.metrics(N, cfg.K, g["x"].numpy(), g["y"].numpy(), g["z"].numpy())
    K3 = (cfg.Kx, cfg.Ky, cfg.Kz)
    ref, dqo = lsrk.lsrk_step(N, K3, qn, np.zeros_like(qn), Jao, phin, Jo, dt, bc=cfg.bc, dissipation=dissipation)
    ref, _ = lsrk.lsrk_step(N, K3, ref, dqo, Jao, phin, Jo, dt, bc=cfg.bc, dissipation=dissipation)
    _, vs = oracle.volume(N, cfg.K, qn, Jao, phin, with_scale=True)
    _, ss = oracle.surface(N, K3, qn, Jao, phin, cfg.bc, dissipation=dissipation, with_scale=True)
    scale = 2 * dt * np.max((vs + ss) / Jo, axis=1) + 16 * EPS["fp32"] * np.max(np.abs(qn), axis=1)
    err = np.max(np.abs(got - ref), axis=1) / scale
    assert err.max() < hz.TOL["fp32"], err


def test_lsrk_fp32_fused_stage_perturbation_variables():
    """The fused FP32 step on perturbation variables (neighbour traces include
    rho_ref and p_ref) against the oracle step on the full FP64 state."""
    cfg = wl.small_config(4, K=(3, 2, 2), warp=True, state="noisy", precision="fp32", bc=(0, 1, 1))
    g, op, Ja, J, q, phi = _setup(cfg)
    ref_state = wl.reference_state(cfg)
    rr, pr = ref_state["rho_ref"], ref_state["p_ref"]
    op.set_reference(rr.to("cuda", torch.float32).contiguous(), pr.to("cuda", torch.float32).contiguous())
    qn, phin = g["q"].numpy(), g["phi"].numpy()
    qp = g["q"].clone()
    qp[0] -= rr
    qp[4] -= pr / 0.4 + rr * g["phi"]
    q = qp.to("cuda", torch.float32).contiguous()
    dt = _stable_dt(cfg, qn, phin)
    dq = torch.zeros_like(q)
    rhs = torch.empty_like(q)
    op.lsrk_step(q, dq, rhs, Ja, phi, J, dt)
    torch.cuda.synchronize()
    assert op.status() == 0
    got = q.double().cpu()
    got[0] += rr
    got[4] += pr / 0.4 + rr * g["phi"]
    got = got.numpy()
    Jao, Jo = oracle.metrics(4, cfg.K, g["x"].numpy(), g["y"].numpy(), g["z"].numpy())
    K3 = (cfg.Kx, cfg.Ky, cfg.Kz)
    ref, _ = lsrk.lsrk_step(4, K3, qn, np.zeros_like(qn), Jao, phin, Jo, dt, bc=cfg.bc)
    _, vs = oracle.volume(4, cfg.K, qn, Jao, phin, with_scale=True)
    _, ss = oracle.surface(4, K3, qn, Jao, phin, cfg.bc, with_scale=True)
    # the change q(t+dt) - q(t) in FP32 perturbation storage: rounding of the
    # small stored values instead of the full state
    scale = dt * np.max((vs + ss) / Jo, axis=1) + 8 * EPS["fp32"] * np.max(np.abs(qp.numpy()), axis=1)
    err = np.max(np.abs(got - ref), axis=1) / scale
    assert err.max() < hz.TOL["fp32"], err


@pytest.mark.parametrize("precision", ["fp64", "fp32"])
def test_diagnostics_parity(precision):
    cfg = wl.small_config(4, K=(3, 2, 2), warp=True, state="noisy", precision=precision)
    g, op, Ja, J, q, phi = _setup(cfg)
    d = op.diagnostics(q, J, phi).cpu().numpy()
    # oracle on exactly the values the GPU holds (rounded inputs, GPU Jacobian)
    ref = lsrk.diagnostics(cfg.N, cfg.K, q.double().cpu().numpy(), phi.double().cpu().numpy(),
                           J.double().cpu().numpy())
    for k in range(3):
        assert abs(d[k] - ref[k]) <= 1e-13 * abs(ref[k]), (k, d[k], ref[k])


def test_diagnostics_reproducible():
    cfg = wl.small_config(3, K=(4, 3, 2), warp=True, state="noisy")
    _, op, _, J, q, phi = _setup(cfg)
    a = op.diagnostics(q, J, phi).cpu().numpy()
    b = op.diagnostics(q, J, phi).cpu().numpy()
    assert np.array_equal(a, b)


@pytest.mark.parametrize("bc", [(0, 0, 0), (0, 1, 1), (1, 1, 1)])
def test_gpu_conservation_and_entropy_over_steps(bc):
    cfg = wl.small_config(3, K=(3, 3, 2), warp=True, state="noisy", bc=bc)
    g, op, Ja, J, q, phi = _setup(cfg)
    dt = _stable_dt(cfg, g["q"].numpy(), g["phi"].numpy())
    dq = torch.zeros_like(q)
    rhs = torch.empty_like(q)
    m0, e0, s0 = op.diagnostics(q, J, phi).cpu().numpy()
    prev = s0
    for _ in range(10):
        op.lsrk_step(q, dq, rhs, Ja, phi, J, dt)
        m, e, s = op.diagnostics(q, J, phi).cpu().numpy()
        assert abs(m - m0) <= 2e-14 * abs(m0)
        assert abs(e - e0) <= 2e-14 * abs(e0)
        assert s < prev
        prev = s
    assert op.status() == 0


@pytest.mark.parametrize("bc", [(0, 0, 0), (1, 1, 1)])
def test_fp32_global_conservation_over_steps(bc):
    """FP32 steps (the fused stage, each interface evaluated once from each
    side): integrated mass and total energy stay within the FP32 level the
    paper reports for its 32-bit runs (relative variations ~1e-6, Sec. 5.2)
    over 20 steps; the one-sided face evaluations cancel to rounding."""
    cfg = wl.small_config(3, K=(3, 3, 2), warp=True, state="noisy", precision="fp32", bc=bc)
    g, op, Ja, J, q, phi = _setup(cfg)
    dt = _stable_dt(cfg, g["q"].numpy(), g["phi"].numpy())
    dq = torch.zeros_like(q)
    rhs = torch.empty_like(q)
    m0, e0, _ = op.diagnostics(q, J, phi).cpu().numpy()
    worst = [0.0, 0.0]
    for _ in range(20):
        op.lsrk_step(q, dq, rhs, Ja, phi, J, dt)
        m, e, _ = op.diagnostics(q, J, phi).cpu().numpy()
        worst = [max(worst[0], abs(m - m0) / abs(m0)), max(worst[1], abs(e - e0) / abs(e0))]
    assert op.status() == 0
    assert worst[0] < 1e-6 and worst[1] < 1e-6, worst


def test_gpu_coriolis_rotation():
    cfg = wl.small_config(3, K=(2, 2, 2), warp=True, state="random", bc=(0, 0, 0))
    g, op, Ja, J, _, _ = _setup(cfg, coriolis=1e-2)
    n = cfg.n
    q = torch.from_numpy(ph.conserved(np.full(n, 1.0), np.tile(np.array([[10.0], [0.0], [0.0]]), (1, n)),
                                      np.full(n, 1.0e5), 0.0)).cuda().contiguous()
    phi = torch.zeros(n, dtype=torch.float64, device="cuda")
    dq = torch.zeros_like(q)
    rhs = torch.empty_like(q)
    for _ in range(20):
        op.lsrk_step(q, dq, rhs, Ja, phi, J, 0.5)
    got = q.cpu().numpy()
    ang = 1e-2 * 0.5 * 20
    assert np.allclose(got[1], 10.0 * math.cos(ang), rtol=0, atol=1e-9)
    assert np.allclose(got[2], -10.0 * math.sin(ang), rtol=0, atol=1e-9)


def test_lsrk_step_in_a_cuda_graph():
    """The step enqueues only launches on the given stream: captured once and
    replayed, it gives the same bits as the eager calls."""
    cfg = wl.small_config(3, K=(3, 2, 2), warp=True, state="noisy", bc=(0, 1, 1))
    g, op, Ja, J, q0, phi = _setup(cfg)
    dt = _stable_dt(cfg, g["q"].numpy(), g["phi"].numpy())
    q_e = q0.clone()
    dq_e = torch.zeros_like(q0)
    rhs_e = torch.empty_like(q0)
    for _ in range(3):
        op.lsrk_step(q_e, dq_e, rhs_e, Ja, phi, J, dt)
    q_g = q0.clone()
    dq_g = torch.zeros_like(q0)
    rhs_g = torch.empty_like(q0)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            op.lsrk_step(q_g, dq_g, rhs_g, Ja, phi, J, dt, stream=s)
    torch.cuda.synchronize()
    q_g.copy_(q0)  # capture does not execute; start from the same state
    dq_g.zero_()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(q_e, q_g)


@pytest.mark.parametrize("precision", ["fp64", "fp32", "fp64ff"])
def test_pipeline_from_host_buffers(precision):
    """esdg_pipeline_*: several submissions from pinned host buffers, overlapping,
    each giving the same bits as esdg_volume_rhs on device buffers."""
    cfg = wl.small_config(5, K=(3, 2, 2), warp=True, state="noisy", precision=precision)
    g, op, Ja, J, q, phi = _setup(cfg)
    ref = op.volume_rhs(q, Ja, phi).cpu()
    hq, hJ, hp = q.cpu().pin_memory(), Ja.cpu().pin_memory(), phi.cpu().pin_memory()
    outs = [torch.zeros(q.shape, dtype=q.dtype).pin_memory() for _ in range(5)]
    pipe = fd.Pipeline(op, depth=3)
    for o in outs:
        pipe.submit(hq, hJ, hp, o)
    pipe.wait()
    pipe.close()
    for o in outs:
        assert torch.equal(o, ref)
    with pytest.raises(ValueError):
        fd.Pipeline(op, 2).submit(q, Ja, phi, outs[0])  # device tensors are refused
