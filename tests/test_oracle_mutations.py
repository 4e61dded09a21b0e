"""Planted mistakes in a copy of the oracle must each fail at least one pin.

Every mutant is a textual edit of oracle/oracle_impl.inc compiled into a
temporary library on the CPU; the real oracle is never modified.  The pin
functions of test_oracle_pins.py run against the mutant by swapping the
oracle module's loaded library for the duration of the check.
"""
import ctypes
import os
import shutil
import subprocess

import pytest

import oracle
from tests import test_oracle_pins as pins
from tests import test_oracle_surface_pins as spins

MUTANTS = [
    ("gravity sign", "REAL grav = rho_hat * (phim - phii) / 2;", "REAL grav = rho_hat * (phii - phim) / 2;"),
    ("gravity one-sided b from the + side", "REAL rho_hat = b_avg * rho_ln / bi;", "REAL rho_hat = b_avg * rho_ln / bm;"),
    ("energy flux drops {{phi}}", "- uu_avg / 2 + phi_avg", "- uu_avg / 2"),
    ("energy flux drops |{{u}}|^2", "+ ua[0] * ua[0] + ua[1] * ua[1] + ua[2] * ua[2])", ")"),
    ("pressure mean without the 2", "REAL p_hat = rho_avg / (2 * b_avg);", "REAL p_hat = rho_avg / b_avg;"),
    ("arithmetic instead of log mean", "return d / log1p(d / a);", "return (a + c) / 2;"),
    ("transposed D in the volume sum", "REAL coef = 2 * D[ai[r] * Nq + k];", "REAL coef = 2 * D[k * Nq + ai[r]];"),
    ("D instead of 2D", "REAL coef = 2 * D[ai[r] * Nq + k];", "REAL coef = D[ai[r] * Nq + k];"),
    ("metric not averaged", "nvec[s] = (Ja[(3 * r + s) * npts + gi] + Ja[(3 * r + s) * npts + gm]) / 2;",
     "nvec[s] = Ja[(3 * r + s) * npts + gi];"),
    ("metric planes transposed", "Ja[(3 * r + n) * npts + e * np3 + i] = -acc[i];",
     "Ja[(3 * n + r) * npts + e * np3 + i] = -acc[i];"),
    ("metric sign", "Ja[(3 * r + n) * npts + e * np3 + i] = -acc[i];", "Ja[(3 * r + n) * npts + e * np3 + i] = acc[i];"),
    ("mass flux with arithmetic mean density", "REAL Frho = rho_ln * un;", "REAL Frho = rho_avg * un;"),
    # surface term
    ("dissipation added instead of subtracted", "for (int v = 0; v < 5; ++v) F[v] -= D[v];",
     "for (int v = 0; v < 5; ++v) F[v] += D[v];"),
    ("dissipation without the 1/2", "D[r] = nn * s / 2;", "D[r] = nn * s;"),
    ("dissipation without |n|", "D[r] = nn * s / 2;", "D[r] = s / 2;"),
    ("shear scaling rho instead of p", "T[2] = p;", "T[2] = rho;"),
    ("entropy-wave scaling without gamma-1", "T[1] = rho * (gamma - 1) / gamma;", "T[1] = rho / gamma;"),
    ("enthalpy without phi", "REAL H = a * a / (gamma - 1) + uu / 2 + phi;", "REAL H = a * a / (gamma - 1) + uu / 2;"),
    ("entropy wave without phi", "{1, u[0], u[1], u[2], uu / 2 + phi},", "{1, u[0], u[1], u[2], uu / 2},"),
    ("shear eigenvalue", "lam[2] = un;", "lam[2] = un + a;"),
    ("sound speed without gamma", "REAL a = sqrt(gamma * p / rho);", "REAL a = sqrt(p / rho);"),
    ("wall keeps the normal momentum", "for (int s = 0; s < 3; ++s) qp[1 + s] = qi[1 + s] - 2 * mn * nh[s];",
     "for (int s = 0; s < 3; ++s) qp[1 + s] = qi[1 + s];"),
    ("face normal not outward", "for (int s = 0; s < 3; ++s) own[s] = side * Ja[(3 * r + s) * npts + gi];",
     "for (int s = 0; s < 3; ++s) own[s] = Ja[(3 * r + s) * npts + gi];"),
    ("neighbour node not across the face", "aj[r] = N - ai[r];", "aj[r] = ai[r];"),
    ("lifting by w_0 instead of 1/w_0", "REAL inv_w0 = 1 / wn[0];", "REAL inv_w0 = wn[0];"),
    ("strong form keeps the physical flux", "if (form == 0) FN(phys_flux)(qi, phi[gi], own, gamma, f);", ""),
]


def _checks():
    """(name, callable) pairs: each raises AssertionError when its pin fails."""
    return [
        ("affine metrics", lambda: pins.test_metrics_affine_closed_form(4)),
        ("trilinear metrics", lambda: pins.test_metrics_trilinear_closed_form(3)),
        ("metric identities", lambda: pins.test_metric_identities_warped(3)),
        ("consistency", pins.test_flux_consistency_with_physical_flux),
        ("symmetry/gravity scaling", pins.test_flux_symmetry_and_gravity_partner_scaling),
        ("pair entropy", lambda: pins.test_flux_pair_entropy_conservation("d", 5e-12)),
        ("conservation", lambda: pins.test_volume_conservation_per_element(3)),
        ("entropy identity", lambda: pins.test_volume_sbp_entropy_identity(3, 0)),
        ("free stream", lambda: pins.test_free_stream_preservation_curved(3, 1.0e4)),
        ("hydrostatic", lambda: pins.test_hydrostatic_gravity_closed_form(4)),
        ("surface consistency", spins.test_surface_flux_consistency),
        ("eigenvectors", lambda: spins.test_eigenvectors_of_the_flux_jacobian(True)),
        ("entropy Jacobian", lambda: spins.test_scaled_eigenvectors_give_the_entropy_jacobian(True)),
        ("Roe limit", lambda: spins.test_small_jump_limit_is_roe_dissipation(True)),
        ("entropy stability", spins.test_surface_flux_is_entropy_stable),
        ("surface free stream", lambda: spins.test_free_stream_volume_plus_surface(2, 1, 0.0)),
        ("global conservation", lambda: spins.test_global_conservation(1, (0, 1, 1))),
        ("entropy production", lambda: spins.test_entropy_production_equals_face_dissipation(2, (0, 1, 1))),
    ]


def _build_mutant(tmp_path, old, new):
    src_dir = os.path.dirname(oracle._SRC[0])
    for f in ("esdg_oracle.c", "oracle_impl.inc"):
        shutil.copy(os.path.join(src_dir, f), tmp_path / f)
    inc = (tmp_path / "oracle_impl.inc").read_text()
    assert inc.count(old) == 1, old
    (tmp_path / "oracle_impl.inc").write_text(inc.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", str(so),
                    str(tmp_path / "esdg_oracle.c"), "-lm"], check=True)
    return str(so)


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, name, old, new):
    so = _build_mutant(tmp_path, old, new)
    real = oracle._load()
    mutant = ctypes.CDLL(so)
    for sfx in ("_d", "_ld"):
        for fn in ("ora_lgl", "ora_dmatrix", "ora_metrics", "ora_flux", "ora_volume", "ora_roe_matrices",
                   "ora_dissipation", "ora_surface_flux", "ora_surface"):
            getattr(mutant, fn + sfx).argtypes = getattr(real, fn + sfx).argtypes
    mutant.ora_max_threads.restype = ctypes.c_int
    caught = []
    oracle._lib = mutant
    try:
        for cname, check in _checks():
            try:
                check()
            except (AssertionError, FloatingPointError, ValueError):
                caught.append(cname)
    finally:
        oracle._lib = real
    assert caught, f"planted mistake '{name}' passed every pin"
