"""Parity of the CUDA surface term with the CPU oracle (GPU required).

The surface term alone (added into a zeroed output) is compared with the
oracle's, normalised per conserved variable by the magnitude of the summed
face terms, sum (|F*| + |f.n|)/w_0 (tests/harness.py): 1e-11 for FP64 and
1e-4 for FP32 against the FP64 oracle on the original FP64 inputs.
"""
import numpy as np
import pytest
import torch

import flux_differencing_gb300 as fd
import oracle
import workloads as wl
from tests import harness as hz
from tests import physics as ph

pytestmark = pytest.mark.gpu

BCS = [(0, 0, 0), (1, 1, 1), (0, 1, 1), (1, 0, 0)]


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_ok):
    fd.load_library(build_if_missing=True)


@pytest.mark.parametrize("N", list(range(1, 9)))
@pytest.mark.parametrize("bc", BCS)
@pytest.mark.parametrize("precision", ["fp64", "fp32"])
def test_surface_small_meshes(N, bc, precision):
    """States with jumps across faces, so that the dissipation is exercised."""
    cfg = wl.small_config(N, K=(3, 2, 2), warp=True, precision=precision, bc=bc, state="noisy")
    g = wl.generate(cfg)
    got, op = hz.run_gpu_surface(cfg, g)
    assert op.status() == 0
    ref, scale = hz.run_oracle_surface(cfg, g)
    e, _ = hz.errors(got, ref, scale)
    assert e.max() < hz.TOL[precision], e


def test_noisy_state_makes_the_dissipation_count():
    """The dissipation must be a sizeable part of the surface term for the parity
    tests above to check it: with jumps of a few percent across faces it is."""
    cfg = wl.small_config(3, K=(2, 2, 2), warp=True, bc=(0, 1, 1), state="noisy")
    g = wl.generate(cfg)
    with_d, scale = hz.run_oracle_surface(cfg, g, dissipation=True)
    without, _ = hz.run_oracle_surface(cfg, g, dissipation=False)
    rel = np.abs(with_d - without).max(axis=1) / scale.max(axis=1)
    assert rel.min() > 1e-4, rel


@pytest.mark.parametrize("N", [1, 2, 3, 4, 7, 8])
@pytest.mark.parametrize("form,dissipation", [("skew", True), ("2d", False), ("skew", False)])
@pytest.mark.parametrize("precision", ["fp64", "fp32"])
def test_surface_forms_and_dissipation(N, form, dissipation, precision):
    cfg = wl.small_config(N, K=(2, 3, 2), warp=True, precision=precision, bc=(0, 1, 1), state="noisy")
    g = wl.generate(cfg)
    got, _ = hz.run_gpu_surface(cfg, g, form=form, dissipation=dissipation)
    ref, scale = hz.run_oracle_surface(cfg, g, form=1 if form == "skew" else 0, dissipation=dissipation)
    e, _ = hz.errors(got, ref, scale)
    assert e.max() < hz.TOL[precision], e


@pytest.mark.parametrize("K", [(1, 1, 1), (1, 4, 1), (5, 1, 2), (1, 1, 3)])
@pytest.mark.parametrize("bc", [(0, 0, 0), (1, 1, 1)])
def test_surface_degenerate_meshes(K, bc):
    """One element along a direction: periodic faces meet the same element."""
    cfg = wl.small_config(3, K=K, warp=True, bc=bc, state="noisy")
    g = wl.generate(cfg)
    got, _ = hz.run_gpu_surface(cfg, g)
    ref, scale = hz.run_oracle_surface(cfg, g)
    e, _ = hz.errors(got, ref, scale)
    assert e.max() < hz.TOL["fp64"], e


def test_surface_fp64ff_handle_runs_fp64_surface():
    cfg = wl.small_config(4, K=(2, 2, 2), warp=True, precision="fp64ff", bc=(0, 1, 1), state="noisy")
    g = wl.generate(cfg)
    got, _ = hz.run_gpu_surface(cfg, g)
    ref, scale = hz.run_oracle_surface(cfg, g)
    e, _ = hz.errors(got, ref, scale)
    assert e.max() < hz.TOL["fp64"], e


@pytest.mark.parametrize("name", ["tiny_box_N3", "bubble_N4", "channel_N7", "channel_N7_fp32"])
def test_surface_named_workloads(name):
    """The surface term of each workload at full size, with its boundary kinds."""
    cfg = wl.get_config(name)
    g = wl.generate(cfg)
    got, op = hz.run_gpu_surface(cfg, g)
    assert op.status() == 0
    ref, scale = hz.run_oracle_surface(cfg, g)
    e, plain = hz.errors(got, ref, scale)
    assert e.max() < hz.TOL[cfg.precision], (e, plain)


@pytest.mark.parametrize("precision", ["fp64", "fp32"])
def test_rhs_is_volume_plus_surface(precision):
    cfg = wl.small_config(5, K=(2, 2, 3), warp=True, precision=precision, bc=(0, 1, 1), state="noisy")
    g = wl.generate(cfg)
    got, _ = hz.run_gpu_surface(cfg, g, with_volume=True)
    vref, vscale = hz.run_oracle(cfg, g)
    sref, sscale = hz.run_oracle_surface(cfg, g)
    e, _ = hz.errors(got, vref + sref, vscale + sscale)
    assert e.max() < hz.TOL[precision], e


@pytest.mark.parametrize("N", list(range(1, 9)))
@pytest.mark.parametrize("bc", [(0, 1, 1), (1, 0, 1)])
@pytest.mark.parametrize("dissipation", [True, False])
def test_fp32_rhs_one_launch_parity(N, bc, dissipation):
    """esdg_rhs in FP32 is one launch of the volume kernel with the faces
    evaluated inside it (one-sided, as in the fused stage); against the
    oracle's volume + surface at every order, with walls and periodic
    directions and with the entropy-conserving interface flux alone.  K
    gives several elements per CTA at low N and one element along a
    periodic direction."""
    cfg = wl.small_config(N, K=(3, 1, 2), warp=True, precision="fp32", bc=bc, state="noisy")
    g = wl.generate(cfg)
    op = fd.VolumeOperator(cfg.Kx, cfg.Ky, cfg.Kz, N, "fp32", "2d", bc=bc, dissipation=dissipation)
    dg = hz.to_device(g)
    Ja = op.set_geometry(dg["x"], dg["y"], dg["z"])
    q = dg["q"].to(op.dtype).contiguous()
    phi = dg["phi"].to(op.dtype).contiguous()
    got = op.rhs(q, Ja, phi).double().cpu().numpy()
    torch.cuda.synchronize()
    assert op.status() == 0
    vref, vscale = hz.run_oracle(cfg, g)
    sref, sscale = hz.run_oracle_surface(cfg, g, dissipation=dissipation)
    e, _ = hz.errors(got, vref + sref, vscale + sscale)
    assert e.max() < hz.TOL["fp32"], e


@pytest.mark.parametrize("K", [(1, 1, 1), (1, 3, 1), (2, 1, 1)])
@pytest.mark.parametrize("bc", [(0, 0, 0), (1, 1, 1), (0, 1, 0)])
def test_fp32_rhs_one_launch_degenerate_meshes(K, bc):
    """The one-launch FP32 right-hand side on meshes of one or two elements
    per direction: periodic faces whose neighbour is the element itself, and
    walls on every side; against the oracle."""
    cfg = wl.small_config(3, K=K, warp=True, precision="fp32", bc=bc, state="noisy")
    g = wl.generate(cfg)
    op = fd.VolumeOperator(cfg.Kx, cfg.Ky, cfg.Kz, 3, "fp32", "2d", bc=bc)
    dg = hz.to_device(g)
    Ja = op.set_geometry(dg["x"], dg["y"], dg["z"])
    q = dg["q"].to(op.dtype).contiguous()
    phi = dg["phi"].to(op.dtype).contiguous()
    got = op.rhs(q, Ja, phi).double().cpu().numpy()
    torch.cuda.synchronize()
    assert op.status() == 0
    vref, vscale = hz.run_oracle(cfg, g)
    sref, sscale = hz.run_oracle_surface(cfg, g)
    e, _ = hz.errors(got, vref + sref, vscale + sscale)
    assert e.max() < hz.TOL["fp32"], e


def test_surface_is_deterministic():
    cfg = wl.small_config(7, K=(3, 3, 2), warp=True, bc=(0, 1, 1), state="noisy")
    g = wl.generate(cfg)
    a, _ = hz.run_gpu_surface(cfg, g)
    b, _ = hz.run_gpu_surface(cfg, g)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("N", [2, 4, 7])
def test_gpu_rhs_free_stream_and_conservation(N):
    """Properties of the GPU result alone: a constant state is steady on a warped
    periodic mesh, and the global integrals of mass and energy do not change."""
    cfg = wl.small_config(N, K=(3, 2, 2), warp=True, bc=(0, 0, 0))
    g = wl.generate(cfg)
    n = cfg.n
    _, w = oracle.lgl(N)
    idx = np.arange((N + 1) ** 3)
    om = np.tile(w[idx % (N + 1)] * w[(idx // (N + 1)) % (N + 1)] * w[idx // (N + 1) ** 2], cfg.K)
    qc = ph.conserved(np.full(n, 1.1), np.tile(np.array([[12.0], [-7.0], [4.0]]), (1, n)),
                      np.full(n, 9.0e4), 0.0)
    gc = dict(g)
    gc["q"] = torch.from_numpy(qc)
    gc["phi"] = torch.zeros(n, dtype=torch.float64)
    tot, _ = hz.run_gpu_surface(cfg, gc, with_volume=True)
    _, fvs = hz.run_oracle(cfg, gc)
    _, fss = hz.run_oracle_surface(cfg, gc)
    free_scale = (fvs + fss).max(axis=1)
    assert np.max(np.abs(tot).max(axis=1) / free_scale) < 1e3 * np.finfo(float).eps
    got, _ = hz.run_gpu_surface(cfg, g, with_volume=True)
    _, vscale = hz.run_oracle(cfg, g)
    _, sscale = hz.run_oracle_surface(cfg, g)
    mag = (vscale + sscale) @ om
    sums = got @ om
    for c in (0, 4):
        assert abs(sums[c]) < 1e-12 * mag[c]


def test_surface_status_flags_nonphysical_state():
    cfg = wl.small_config(3, K=(2, 2, 2), warp=False, bc=(0, 0, 0))
    g = wl.generate(cfg)
    g["q"][4, 0] = -1.0  # p < 0 at a corner node of element 0
    _, op = hz.run_gpu_surface(cfg, g)
    assert op.status() & 1


def test_surface_argument_errors():
    op = fd.VolumeOperator(2, 2, 2, 3)
    with pytest.raises(fd.EsdgError):
        op.set_boundary(0, 2, 0)
    n = op.n
    q = torch.ones((5, n), dtype=torch.float64, device="cuda")
    Ja = torch.ones((9, n), dtype=torch.float64, device="cuda")
    phi = torch.zeros(n, dtype=torch.float64, device="cuda")
    with pytest.raises(fd.EsdgError):
        op.surface_rhs(q, Ja, phi, q)  # out aliases q


@pytest.mark.parametrize("precision", ["fp64", "fp32", "fp64ff"])
@pytest.mark.parametrize("bc", [(0, 0, 0), (0, 1, 1)])
def test_rhs_entry_equals_volume_then_surface(precision, bc):
    """esdg_rhs runs both kernels in their skew forms (the 2D form's volume
    diagonal and the strong surface correction cancel); it must agree with
    esdg_volume_rhs followed by esdg_surface_rhs to rounding."""
    cfg = wl.small_config(4, K=(3, 2, 2), warp=True, state="noisy", precision=precision, bc=bc)
    g = wl.generate(cfg)
    op = fd.VolumeOperator(cfg.Kx, cfg.Ky, cfg.Kz, cfg.N, precision, "2d", bc=bc)
    dg = hz.to_device(g)
    Ja = op.set_geometry(dg["x"], dg["y"], dg["z"])
    q = dg["q"].to(op.dtype).contiguous()
    phi = dg["phi"].to(op.dtype).contiguous()
    a = op.volume_rhs(q, Ja, phi)
    op.surface_rhs(q, Ja, phi, a)
    b = op.rhs(q, Ja, phi)
    _, vs = hz.run_oracle(cfg, g)
    _, ss = hz.run_oracle_surface(cfg, g)
    e, _ = hz.errors(b.double().cpu().numpy(), a.double().cpu().numpy(), vs + ss)
    eps = 2.0 ** -23 if precision == "fp32" else 2.0 ** -52
    assert e.max() < 64 * eps, e
