"""Parity of the CUDA volume term with the CPU oracle (GPU required).

Tolerances (normalised max-norm per conserved variable, see tests/harness.py):
1e-11 for the FP64 kernel and 1e-4 for the FP32 kernel, the FP32 kernel being
compared with the FP64 oracle on the original FP64 inputs.
"""
import numpy as np
import pytest
import torch

import flux_differencing_gb300 as fd
import oracle
import workloads as wl
from tests import harness as hz

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_ok):
    fd.load_library(build_if_missing=True)


# ----------------------------------------------------------------------------
# small meshes: every order, both forms, both precisions, ragged element counts

SMALL = [(N, K) for N in range(1, 9) for K in [(2, 2, 1), (3, 2, 3)]] + [(1, (17, 1, 2)), (2, (11, 1, 1)),
                                                                          (3, (5, 1, 1)), (4, (7, 1, 1)),
                                                                          (5, (3, 1, 1))]


PRECISIONS = ["fp64", "fp32", "fp64ff"]


@pytest.mark.parametrize("N,K", SMALL)
@pytest.mark.parametrize("precision", PRECISIONS)
def test_small_meshes(N, K, precision):
    cfg = wl.small_config(N, K=K, warp=True, precision=precision)
    g = wl.generate(cfg)
    got, op, _ = hz.run_gpu(cfg, g)
    assert op.status() == 0
    ref, scale = hz.run_oracle(cfg, g)
    e, _ = hz.errors(got, ref, scale)
    assert e.max() < hz.TOL[precision], e


def _wide_ratio_state(cfg, g, amp):
    """The generated state with the density stretched by exp(amp * smooth
    field) node by node (velocity and pressure kept, so 2b = rho/p stretches
    alike): pairs on one line then differ by factors up to about 50, beside
    close pairs, which drives every precision's far log-mean branch."""
    g = {k: v.clone() for k, v in g.items()}
    q = g["q"].double()
    rho = q[0]
    u = q[1:4] / rho
    phi = g["phi"].double()
    p = 0.4 * (q[4] - 0.5 * rho * (u * u).sum(0) - rho * phi)
    s = torch.exp(amp * torch.sin(g["x"] * 7.3e-3 + 0.4) * torch.cos(g["y"] * 5.1e-3)
                  * torch.sin(g["z"] * 3.3e-3 + 1.1))
    rho2 = rho * s
    g["q"] = torch.stack([rho2, rho2 * u[0], rho2 * u[1], rho2 * u[2],
                          p / 0.4 + 0.5 * rho2 * (u * u).sum(0) + rho2 * phi])
    return g


@pytest.mark.parametrize("N", [1, 3, 4, 7])
@pytest.mark.parametrize("precision", PRECISIONS)
def test_wide_density_ratios(N, precision):
    cfg = wl.small_config(N, K=(3, 2, 2), warp=True, precision=precision)
    g = _wide_ratio_state(cfg, wl.generate(cfg), 2.0)
    got, op, _ = hz.run_gpu(cfg, g)
    assert op.status() == 0
    ref, scale = hz.run_oracle(cfg, g)
    e, _ = hz.errors(got, ref, scale)
    assert e.max() < hz.TOL[precision], e


def _element_ratio_state(cfg, g, lo, hi):
    """The generated state with each element's density multiplied by
    r_e^(cos(pi a/N)/2), a the node's xi index and r_e running from lo to hi
    over the elements (velocity and pressure kept, so 2b = rho/p stretches
    alike): within element e the stretch spans a factor r_e."""
    g = {k: v.clone() for k, v in g.items()}
    q = g["q"].double()
    rho = q[0]
    u = q[1:4] / rho
    phi = g["phi"].double()
    p = 0.4 * (q[4] - 0.5 * rho * (u * u).sum(0) - rho * phi)
    nq = cfg.N + 1
    node = torch.arange(cfg.n)
    e = node // nq ** 3
    a = (node % nq).double()
    r = lo + (hi - lo) * e.double() / max(1, cfg.K - 1)
    s = torch.exp(0.5 * torch.log(r) * torch.cos(np.pi * a / cfg.N))
    rho2 = rho * s
    g["q"] = torch.stack([rho2, rho2 * u[0], rho2 * u[1], rho2 * u[2],
                          p / 0.4 + 0.5 * rho2 * (u * u).sum(0) + rho2 * phi])
    return g


@pytest.mark.parametrize("N", [1, 3, 4, 7])
def test_fp32_log_mean_forms_at_the_switch(N):
    """FP32 CTAs whose densities and values of b lie within a factor 2.25 use
    the polynomial log means for every pair; wider ones select per pair
    between the polynomials and the logarithm of the pair's ratio.  Elements
    stretched by factors from 1.9 to 2.7 put CTAs on both sides of the
    switch, and pairs on both sides of the polynomials' range."""
    cfg = wl.small_config(N, K=(4, 3, 2), warp=True, precision="fp32")
    g = _element_ratio_state(cfg, wl.generate(cfg), 1.9, 2.7)
    got, op, _ = hz.run_gpu(cfg, g)
    assert op.status() == 0
    ref, scale = hz.run_oracle(cfg, g)
    e, _ = hz.errors(got, ref, scale)
    assert e.max() < hz.TOL["fp32"], e


@pytest.mark.parametrize("N", [1, 2, 3, 4, 7, 8])
@pytest.mark.parametrize("precision", PRECISIONS)
def test_skew_form(N, precision):
    cfg = wl.small_config(N, K=(2, 3, 1), warp=True, precision=precision)
    g = wl.generate(cfg)
    got, _, _ = hz.run_gpu(cfg, g, form="skew")
    ref, scale = hz.run_oracle(cfg, g, form=1)
    e, _ = hz.errors(got, ref, scale)
    assert e.max() < hz.TOL[precision], e


@pytest.mark.parametrize("N", [2, 3, 7, 8])
def test_metrics_parity(N):
    """GPU curl-form metrics against the long-double oracle.

    The curl form applies D twice to products of coordinates, so double
    rounding contributes about eps * (max row sum |D|)^2 * h^2 with h the
    element size (the GPU works relative to an element-local origin)."""
    cfg = wl.small_config(N, K=(3, 2, 2), warp=True)
    g = wl.generate(cfg)
    op = fd.VolumeOperator(cfg.Kx, cfg.Ky, cfg.Kz, cfg.N, "fp64")
    dg = hz.to_device(g)
    J = torch.empty(cfg.n, dtype=torch.float64, device="cuda")
    Ja = op.set_geometry(dg["x"], dg["y"], dg["z"], J_out=J)
    Jo_a, Jo = oracle.metrics(N, cfg.K, g["x"].numpy(), g["y"].numpy(), g["z"].numpy(), real="ld")
    Jo_a, Jo = Jo_a.astype(np.float64), Jo.astype(np.float64)
    Ja = Ja.cpu().numpy()
    _, _, D = fd.operators(N)
    h = max(d / k for d, k in zip(cfg.domain, (cfg.Kx, cfg.Ky, cfg.Kz)))
    bound = 16 * 2.2e-16 * np.abs(D).sum(axis=1).max() ** 2 * h * h
    assert np.max(np.abs(Ja - Jo_a)) < bound, (np.max(np.abs(Ja - Jo_a)), bound)
    assert np.max(np.abs(Ja - Jo_a)) < 1e-12 * np.abs(Jo_a).max()
    assert np.max(np.abs(J.cpu().numpy() - Jo)) < 1e-13 * np.abs(Jo).max()
    # discrete metric identities hold for the GPU's metrics too
    Nq = N + 1
    np3 = Nq ** 3
    F = Ja.reshape(9, cfg.K, Nq, Nq, Nq)  # [plane, e, c, b, a]
    for j in range(3):
        div = (np.einsum("ik,ecbk->ecbi", D, F[0 * 3 + j])     # d/dxi of Ja^1_j
               + np.einsum("ik,ecka->ecia", D, F[1 * 3 + j])   # d/deta of Ja^2_j
               + np.einsum("ik,ekba->eiba", D, F[2 * 3 + j]))  # d/dzeta of Ja^3_j
        assert np.max(np.abs(div)) < 1e-12 * np.abs(Ja).max() * np.abs(D).max()


# ----------------------------------------------------------------------------
# the named workloads at full size

@pytest.mark.parametrize("name", ["tiny_box_N3", "bubble_N4", "channel_N7", "channel_N7_fp32", "channel_N7_ff"])
def test_named_workload_full(name):
    cfg = wl.get_config(name)
    g = wl.generate(cfg, device="cuda")
    got, op, _ = hz.run_gpu(cfg, g)
    assert op.status() == 0
    ref, scale = hz.run_oracle(cfg, g)
    e, plain = hz.errors(got, ref, scale)
    print(f"{name}: normalised {e.max():.2e} {np.array2string(e, precision=2)}; plain relative "
          f"{np.array2string(plain, precision=2)}")
    assert e.max() < hz.TOL[cfg.precision], e


@pytest.mark.parametrize("N", range(2, 9))
@pytest.mark.parametrize("precision", PRECISIONS)
def test_order_sweep_sampled(N, precision):
    """About 6.4e7 nodes per order; the oracle checks a sample of whole elements."""
    name = f"sweep_N{N}" + {"fp64": "", "fp32": "_fp32", "fp64ff": "_ff"}[precision]
    cfg = wl.get_config(name)
    g = wl.generate(cfg, device="cuda")
    got_full, op, _ = hz.run_gpu(cfg, g)
    assert op.status() == 0
    elems = wl.element_subset(cfg, 48)
    np3 = cfg.Nq ** 3
    idx = (elems[:, None] * np3 + np.arange(np3)[None, :]).reshape(-1)
    sub = {k: (v[:, idx] if v.dim() == 2 else v[idx]).cpu() for k, v in g.items()}
    ref, scale = hz.run_oracle(cfg, sub, K=len(elems))
    got = got_full[:, idx]
    e, _ = hz.errors(got, ref, scale)
    assert e.max() < hz.TOL[precision], e
    assert np.all(np.isfinite(got_full))
    del g


# ----------------------------------------------------------------------------
# properties: determinism, element-range split, status flag, errors

@pytest.mark.parametrize("precision", PRECISIONS)
def test_bitwise_deterministic_and_range_split(precision):
    cfg = wl.small_config(5, K=(5, 3, 2), warp=True, precision=precision)
    g = hz.to_device(wl.generate(cfg))
    op = fd.VolumeOperator(cfg.Kx, cfg.Ky, cfg.Kz, cfg.N, precision)
    Ja = op.set_geometry(g["x"], g["y"], g["z"])
    q = g["q"].to(op.dtype).contiguous()
    phi = g["phi"].to(op.dtype).contiguous()
    a = op.volume_rhs(q, Ja, phi).clone()
    b = op.volume_rhs(q, Ja, phi).clone()
    assert torch.equal(a, b)
    # two calls on disjoint element ranges compose into the full call, bitwise
    c = torch.full_like(a, float("nan"))
    half = cfg.K // 2 + 1
    op.volume_rhs(q, Ja, phi, out=c, e_begin=0, e_count=half)
    op.volume_rhs(q, Ja, phi, out=c, e_begin=half, e_count=cfg.K - half)
    torch.cuda.synchronize()
    assert torch.equal(a, c)


def test_nonphysical_state_sets_status_without_trapping():
    cfg = wl.small_config(3, K=(2, 1, 1), warp=False)
    g = hz.to_device(wl.generate(cfg))
    op = fd.VolumeOperator(cfg.Kx, cfg.Ky, cfg.Kz, cfg.N, "fp64")
    Ja = op.set_geometry(g["x"], g["y"], g["z"])
    q = g["q"].clone()
    q[0, 5] = -1.0  # negative density at one node
    out = op.volume_rhs(q, Ja, g["phi"])
    assert op.status() & fd.ESDG_STATUS_NONPHYSICAL
    assert op.status() == 0  # reading clears it
    # the other element is untouched by the bad node
    ok = op.volume_rhs(g["q"], Ja, g["phi"]).clone()
    np3 = cfg.Nq ** 3
    assert torch.equal(out[:, np3:], ok[:, np3:])


def test_call_errors_on_device():
    cfg = wl.small_config(2, K=(2, 1, 1), warp=False)
    g = hz.to_device(wl.generate(cfg))
    op = fd.VolumeOperator(cfg.Kx, cfg.Ky, cfg.Kz, cfg.N, "fp64")
    Ja = op.set_geometry(g["x"], g["y"], g["z"])
    q = g["q"].contiguous()
    # out aliasing an input
    with pytest.raises(fd.EsdgError, match="ESDG_ERR_ARG"):
        op.volume_rhs(q, Ja, g["phi"], out=q)
    # misaligned pointer
    buf = torch.zeros(5 * cfg.n + 1, dtype=torch.float64, device="cuda")
    with pytest.raises(fd.EsdgError, match="ESDG_ERR_ALIGN"):
        op.volume_rhs(q, Ja, g["phi"], out=buf[1:])
    # empty and out-of-range element ranges
    with pytest.raises(fd.EsdgError, match="ESDG_ERR_ARG"):
        op.volume_rhs(q, Ja, g["phi"], e_begin=0, e_count=0)
    with pytest.raises(fd.EsdgError, match="ESDG_ERR_ARG"):
        op.volume_rhs(q, Ja, g["phi"], e_begin=1, e_count=2)


def test_single_element_and_gamma():
    cfg = wl.small_config(4, K=(1, 1, 1), warp=True)
    g = wl.generate(cfg)
    op = fd.VolumeOperator(1, 1, 1, 4, "fp64", gamma=1.3)
    got, _, _ = hz.run_gpu(cfg, g, op=op)
    gc = {k: v.numpy() for k, v in g.items()}
    Ja, _ = oracle.metrics(4, 1, gc["x"], gc["y"], gc["z"])
    # the state generator used gamma = 1.4 for E; the volume term takes gamma as a parameter
    ref, scale = oracle.volume(4, 1, gc["q"], Ja, gc["phi"], gamma=1.3, with_scale=True)
    e, _ = hz.errors(got, ref, scale)
    assert e.max() < 1e-11
