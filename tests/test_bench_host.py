"""Host-side logic of bench.py (no GPU): face-node counts of the surface
roofline, the guard that drops a committed ncu traffic record once the kernel
source changes, and the operation-count formula."""
import itertools
import os
from types import SimpleNamespace

import numpy as np
import pytest

import bench


def _brute_surface_counts(N, Kx, Ky, Kz, bc):
    """Interior interface nodes (each interface once) and wall face nodes, by
    walking all six faces of every element: a face on a wall boundary is a
    wall face, every other face is one of the two sides of an interface (a
    single element along a periodic direction meets itself)."""
    Nq2 = (N + 1) ** 2
    Kd = (Kx, Ky, Kz)
    walls = sides = 0
    for idx in itertools.product(range(Kx), range(Ky), range(Kz)):
        for r in range(3):
            for step in (-1, 1):
                if bc[r] and not 0 <= idx[r] + step < Kd[r]:
                    walls += 1
                else:
                    sides += 1
    assert sides % 2 == 0
    return sides // 2 * Nq2, walls * Nq2


@pytest.mark.parametrize("N", [1, 3, 7])
@pytest.mark.parametrize("K", [(3, 2, 2), (1, 4, 2), (2, 1, 1), (4, 3, 5)])
@pytest.mark.parametrize("bc", [(0, 0, 0), (1, 1, 1), (0, 1, 1), (1, 0, 1)])
def test_surface_counts_match_brute_force(N, K, bc):
    cfg = SimpleNamespace(N=N, Kx=K[0], Ky=K[1], Kz=K[2], K=K[0] * K[1] * K[2], bc=bc)
    assert bench.surface_counts(cfg) == _brute_surface_counts(N, *K, bc)


def test_channel_face_counts():
    # the N = 7 channel: periodic in x, walls in y and z
    cfg = SimpleNamespace(N=7, Kx=64, Ky=16, Kz=8, K=8192, bc=(0, 1, 1))
    assert bench.surface_counts(cfg) == (1474560, 196608)


def test_traffic_record_only_for_the_committed_source(monkeypatch):
    """A committed ncu record is used only while the kernel source hash equals
    the one it was captured with (the guard itself, independent of whether the
    working tree's kernel has been re-profiled yet)."""
    import glob
    import json
    recs = []
    for path in glob.glob(os.path.join(bench.ROOT, "profiles", "*.md")):
        with open(path) as f:
            recs += [json.loads(line.split(":", 1)[1]) for line in f if line.startswith("traffic_record:")]
    rec = [r for r in recs if r["kernel"] == "volume_kernel<double, 7>" and r["workload"] == "channel_N7"]
    assert rec, "no committed traffic record for the FP64 N = 7 channel kernel"
    monkeypatch.setattr(bench, "kernel_source_sha", lambda kind="volume": rec[0]["source_sha"])
    got = bench.recorded_traffic("volume_kernel<double, 7>", "channel_N7")
    assert isinstance(got, int) and got > 0
    # the algorithmic bytes are 15 planes in and 5 out of 4,194,304 doubles; ncu
    # sees a little less written (part of the output still in L2)
    assert 0.9 * 20 * 8 * 4194304 < got < 1.05 * 20 * 8 * 4194304
    monkeypatch.setattr(bench, "kernel_source_sha", lambda kind="volume": "0" * 16)
    assert bench.recorded_traffic("volume_kernel<double, 7>", "channel_N7") is None


def test_operation_counts():
    # each unordered pair once per direction: 3 (Nq - 1)/2 pairs per node
    for N in range(1, 9):
        Nq = N + 1
        expect = bench.PAIR_OPS * 3 * (Nq - 1) / 2 + bench.NODE_OPS + bench.DIAG_OPS * 6 / Nq
        assert bench.flops_per_dof(N) == pytest.approx(expect)
        assert bench.flops_per_dof(N, form2d=False) == pytest.approx(expect - bench.DIAG_OPS * 6 / Nq)
    assert bench.flops_per_dof(7) == pytest.approx(935.0)


def test_launch_counts():
    assert [bench.step_launches(p) for p in ("fp64", "fp64ff", "fp32")] == [25, 20, 5]
    assert [bench.rhs_launches(p) for p in ("fp64", "fp64ff", "fp32")] == [4, 4, 1]


def test_parity_numbers_measures():
    """e_c is the difference over the term scale S_c, plain the difference over
    max|oracle|, kappa their ratio; pass/fail follows the precision's bar."""
    ref = np.zeros((5, 6))
    ref[:, 2] = [2.0, -4.0, 1.0, 0.5, 8.0]
    scale = np.ones((5, 6)) * 10.0
    got = ref.copy()
    got[1, 4] += 1e-12  # only rho_u1 differs
    par = bench.parity_numbers(got, ref, scale, "fp64")
    r = par["per_variable"]["rho_u1"]
    assert r["e_c"] == pytest.approx(1e-13)
    assert r["plain"] == pytest.approx(1e-12 / 4.0)
    assert r["kappa"] == pytest.approx(10.0 / 4.0)
    assert par["per_variable"]["rho"]["e_c"] == 0.0
    assert par["max_e_c"] == pytest.approx(1e-13) and par["pass"]
    assert not bench.parity_numbers(got + 1e-9, ref, scale, "fp64")["pass"]
    assert bench.parity_numbers(got + 1e-9, ref, scale, "fp32")["pass"]


def test_gpu_rows_picks_element_columns():
    cfg = SimpleNamespace(Nq=3)  # 27 nodes per element
    out = np.arange(5 * 4 * 27, dtype=float).reshape(5, 4 * 27)
    rows = bench.gpu_rows(out, cfg, np.array([1, 3]))
    assert rows.shape == (5, 54)
    assert np.array_equal(rows[:, :27], out[:, 27:54])
    assert np.array_equal(rows[:, 27:], out[:, 81:108])


def test_same_mesh_ignores_precision_only():
    import dataclasses

    import workloads as wl
    base = wl.get_config("channel_N7")
    assert bench._same_mesh(base, wl.get_config("channel_N7_fp32"))
    assert bench._same_mesh(base, dataclasses.replace(base, precision="fp64ff"))
    assert not bench._same_mesh(base, wl.get_config("sweep_N7"))


def test_issue_roofline_from_record(monkeypatch):
    cfg = SimpleNamespace(name="channel_N7_ff", n=4194304)
    monkeypatch.setattr(bench, "recorded_field", lambda kernel, workload, field, kind="volume": 3200.0)
    r = bench.issue_roofline("volume_kernel<double, 7, ff>", cfg, 1e-3)
    expect = 3200.0 / 32 * 4194304 / 1e-3
    assert r["bound"] == "issue" and r["achieved"] == pytest.approx(expect / 1e9)
    assert r["frac"] == pytest.approx(expect / bench.ISSUE_PEAK_WARP_INST_PER_S)
    monkeypatch.setattr(bench, "recorded_field", lambda *a, **k: None)
    assert bench.issue_roofline("volume_kernel<double, 7, ff>", cfg, 1e-3) is None
