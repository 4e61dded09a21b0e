"""The mixed-pipe volume kernel of ESDG_FP64_FF handles (GPU required).

Two persistent CTAs per SM, one in float-float arithmetic (FP32 pipes), one
in native FP64 (FP64 pipe); an element takes native FP64 when e mod 16 < k.
Each element's path is fixed by its index, so:
  * the elements of the FP64 class equal the native FP64 handle's result bit
    for bit, the others the float-float kernel's (k = 0);
  * k = 16 reproduces the native FP64 handle and k = 0 the float-float kernel;
  * two runs agree bit for bit, and element ranges compose;
  * every k meets the FP64 parity tolerance against the oracle.
The mesh has more elements than resident CTAs, so both roles take elements
of both classes (a class exhausted early helps with the other).
"""
import numpy as np
import pytest
import torch

import flux_differencing_gb300 as fd
import workloads as wl
from tests import harness as hz

pytestmark = pytest.mark.gpu


def _run(cfg, g, precision, k=None, e_range=None):
    op = fd.VolumeOperator(cfg.Kx, cfg.Ky, cfg.Kz, cfg.N, precision)
    if k is not None:
        op.set_mixed_pipes(k)
    Ja = op.set_geometry(g["x"], g["y"], g["z"])
    out = torch.full((5, cfg.n), float("nan"), dtype=torch.float64, device="cuda")
    if e_range is None:
        op.volume_rhs(g["q"], Ja, g["phi"], out=out)
    else:
        for e0, ec in e_range:
            op.volume_rhs(g["q"], Ja, g["phi"], out=out, e_begin=e0, e_count=ec)
    assert op.status() == 0
    res = out.cpu().numpy()
    op.close()
    return res


@pytest.fixture(scope="module")
def case():
    cfg = wl.small_config(7, K=(9, 8, 7), warp=True)  # 504 elements, N = 7
    g = wl.generate(cfg)
    ref, scale = hz.run_oracle(cfg, g)
    return cfg, hz.to_device(g), ref, scale


def test_classes_follow_their_paths(cuda_ok, case):
    cfg, g, _, _ = case
    fp64 = _run(cfg, g, "fp64")
    ff_only = _run(cfg, g, "fp64ff", k=0)
    np3 = cfg.Nq ** 3
    for k in (3, 8):
        mixed = _run(cfg, g, "fp64ff", k=k)
        e = np.arange(cfg.K)
        cls64 = np.repeat(e % 16 < k, np3)
        assert np.array_equal(mixed[:, cls64], fp64[:, cls64]), k
        assert np.array_equal(mixed[:, ~cls64], ff_only[:, ~cls64]), k
    assert np.array_equal(_run(cfg, g, "fp64ff", k=16), fp64)


def test_reproducible_and_ranges_compose(cuda_ok, case):
    cfg, g, _, _ = case
    a = _run(cfg, g, "fp64ff")
    b = _run(cfg, g, "fp64ff")
    assert np.array_equal(a, b)
    # ranges starting off a multiple of 16 and with ragged lengths
    c = _run(cfg, g, "fp64ff", e_range=[(0, 37), (37, 200), (237, cfg.K - 237)])
    assert np.array_equal(a, c)


@pytest.mark.parametrize("k", [0, 1, 3, 8, 15, 16])
def test_mixed_parity(cuda_ok, case, k):
    cfg, g, ref, scale = case
    got = _run(cfg, g, "fp64ff", k=k)
    e, _ = hz.errors(got, ref, scale)
    assert e.max() < hz.TOL["fp64ff"], (k, e)


def test_mixed_pipes_rejects_bad_arguments(cuda_ok):
    op = fd.VolumeOperator(2, 1, 1, 7, "fp64")
    with pytest.raises(fd.EsdgError):
        op.set_mixed_pipes(3)  # only float-float handles mix pipes
    op.close()
    op = fd.VolumeOperator(2, 1, 1, 7, "fp64ff")
    for bad in (-1, 17):
        with pytest.raises(fd.EsdgError):
            op.set_mixed_pipes(bad)
    op.close()
