"""Pins of the oracle's time stepping (oracle/lsrk.py) to facts other than itself.

* The 2N-storage coefficients, expanded to the classical Butcher tableau in
  exact rational arithmetic, satisfy the eight conditions for order four, and
  the tableau's abscissae equal the scheme's published c values.
* On a scalar linear ODE the global error falls by 2^4 per halving of dt.
* With the semi-discrete ESDG operator (volume + surface), mass and total
  energy integrals stay constant to round-off over several steps (periodic
  and walled meshes), the entropy integral decreases with dissipation and
  changes only at the time-discretisation level without it.
* A uniform state under the f-plane Coriolis source rotates its momentum at
  angular speed f (closed form).
"""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle
import workloads as wl
from oracle import lsrk
from tests import physics as ph


def test_order_four_conditions():
    a, b, c = lsrk.butcher_tableau()
    S = len(b)
    F = Fraction
    conds = {
        "sum b = 1": (sum(b), F(1)),
        "b.c = 1/2": (sum(b[i] * c[i] for i in range(S)), F(1, 2)),
        "b.c^2 = 1/3": (sum(b[i] * c[i] ** 2 for i in range(S)), F(1, 3)),
        "b.A.c = 1/6": (sum(b[i] * a[i][j] * c[j] for i in range(S) for j in range(S)), F(1, 6)),
        "b.c^3 = 1/4": (sum(b[i] * c[i] ** 3 for i in range(S)), F(1, 4)),
        "b.(c A c) = 1/8": (sum(b[i] * c[i] * a[i][j] * c[j] for i in range(S) for j in range(S)), F(1, 8)),
        "b.A.c^2 = 1/12": (sum(b[i] * a[i][j] * c[j] ** 2 for i in range(S) for j in range(S)), F(1, 12)),
        "b.A.A.c = 1/24": (sum(b[i] * a[i][j] * a[j][k] * c[k] for i in range(S) for j in range(S)
                              for k in range(S)), F(1, 24)),
    }
    for name, (got, want) in conds.items():
        assert abs(float(got - want)) < 1e-12, (name, float(got - want))
    # not fifth order: the scheme is a genuine fourth-order one
    five = sum(b[i] * c[i] ** 4 for i in range(S))
    assert abs(float(five - F(1, 5))) > 1e-6


def _order_defects(A, B):
    a, b, c = lsrk.butcher_tableau(A, B)
    S = len(b)
    return [float(sum(b) - 1),
            float(sum(b[i] * c[i] for i in range(S)) - Fraction(1, 2)),
            float(sum(b[i] * c[i] ** 2 for i in range(S)) - Fraction(1, 3)),
            float(sum(b[i] * a[i][j] * c[j] for i in range(S) for j in range(S)) - Fraction(1, 6)),
            float(sum(b[i] * c[i] ** 3 for i in range(S)) - Fraction(1, 4))]


@pytest.mark.parametrize("which", [("A", k) for k in range(1, 5)] + [("B", k) for k in range(5)])
def test_a_wrong_digit_breaks_the_order_conditions(which):
    """Each coefficient is pinned: a relative change of 1e-9 in any one of them
    violates an order condition by far more than the 1e-12 the test allows."""
    A, B = list(lsrk.LSRK_A), list(lsrk.LSRK_B)
    tab, k = which
    coeffs = A if tab == "A" else B
    coeffs[k] = coeffs[k] * (1 + Fraction(1, 10 ** 9))
    assert max(abs(d) for d in _order_defects(A, B)) > 1e-11


def test_abscissae_match_published_c():
    _, _, c = lsrk.butcher_tableau()
    for got, want in zip(c, lsrk.LSRK_C):
        assert abs(float(got - want)) < 1e-12


def test_scalar_convergence_order():
    """y' = -y + cos(t), y(0) = 1, exact y = (e^-t + cos t + sin t)/2: error ratio 16."""
    def solve(nsteps, T=2.0):
        dt = T / nsteps
        y, dy, t = 1.0, 0.0, 0.0
        for _ in range(nsteps):
            for s in range(5):
                ts = t + float(lsrk.LSRK_C[s]) * dt
                dy = float(lsrk.LSRK_A[s]) * dy + dt * (-y + math.cos(ts))
                y += float(lsrk.LSRK_B[s]) * dy
            t += dt
        return y
    exact = 0.5 * (math.exp(-2.0) + math.cos(2.0) + math.sin(2.0))
    errs = [abs(solve(n) - exact) for n in (8, 16, 32)]
    for e1, e2 in zip(errs, errs[1:]):
        assert 13.0 < e1 / e2 < 19.0, errs


def _mesh(N, K3, bc, state="noisy"):
    cfg = wl.small_config(N, K=K3, warp=True, state=state, bc=bc)
    g = wl.generate(cfg)
    Ja, J = oracle.metrics(N, cfg.K, g["x"].numpy(), g["y"].numpy(), g["z"].numpy())
    return cfg, g["q"].numpy(), g["phi"].numpy(), Ja, J


def _dt(cfg, q, phi, Ja, J, cfl=0.3):
    """A stable step: cfl * min element size / (max |u| + c) / (N+1)^2."""
    rho, u, p = ph.primitives(q, phi)
    speed = np.max(np.sqrt(np.sum(u * u, axis=0)) + np.sqrt(1.4 * p / rho))
    h = min(cfg.domain[0] / cfg.Kx, cfg.domain[1] / cfg.Ky, cfg.domain[2] / cfg.Kz)
    return cfl * h / speed / (cfg.N + 1) ** 2


@pytest.mark.parametrize("bc", [(0, 0, 0), (0, 1, 1)])
def test_conservation_and_entropy_over_steps(bc):
    N = 2
    cfg, q, phi, Ja, J = _mesh(N, (2, 2, 2), bc)
    K3 = (cfg.Kx, cfg.Ky, cfg.Kz)
    dt = _dt(cfg, q, phi, Ja, J)
    m0, e0, s0 = lsrk.diagnostics(N, cfg.K, q, phi, J)
    dq = np.zeros_like(q)
    ents = [s0]
    for _ in range(4):
        q, dq = lsrk.lsrk_step(N, K3, q, dq, Ja, phi, J, dt, bc=bc)
        m, e, s = lsrk.diagnostics(N, cfg.K, q, phi, J)
        assert abs(m - m0) <= 1e-14 * abs(m0)
        assert abs(e - e0) <= 1e-14 * abs(e0)
        ents.append(s)
    # entropy eta = -rho s/(gamma-1) decreases with the dissipative surface flux
    assert all(b < a for a, b in zip(ents, ents[1:])), ents


def test_entropy_conserved_without_dissipation_up_to_time_error():
    N = 2
    cfg, q, phi, Ja, J = _mesh(N, (2, 2, 2), (0, 0, 0))
    K3 = (cfg.Kx, cfg.Ky, cfg.Kz)
    dt = _dt(cfg, q, phi, Ja, J, cfl=0.1)
    _, _, s0 = lsrk.diagnostics(N, cfg.K, q, phi, J)
    q1, _ = lsrk.lsrk_step(N, K3, q, np.zeros_like(q), Ja, phi, J, dt, dissipation=False)
    _, _, s1 = lsrk.diagnostics(N, cfg.K, q1, phi, J)
    q2, _ = lsrk.lsrk_step(N, K3, q, np.zeros_like(q), Ja, phi, J, dt, dissipation=True)
    _, _, s2 = lsrk.diagnostics(N, cfg.K, q2, phi, J)
    # the entropy change without dissipation is far below the dissipative one
    assert abs(s1 - s0) < 1e-3 * abs(s2 - s0)
    assert s2 < s0


def test_coriolis_rotation_closed_form():
    """A uniform state on a periodic mesh: (rho u1, rho u2) rotates by -f t."""
    N = 2
    cfg, _, _, Ja, J = _mesh(N, (2, 2, 1), (0, 0, 0), state="random")
    n = cfg.n
    q = ph.conserved(np.full(n, 1.0), np.tile(np.array([[10.0], [0.0], [0.0]]), (1, n)),
                     np.full(n, 1.0e5), 0.0)
    phi = np.zeros(n)
    f = 1.0e-2
    dt = 0.5  # acoustically stable on these 5 km elements
    K3 = (cfg.Kx, cfg.Ky, cfg.Kz)
    q1, dq = q, np.zeros_like(q)
    for _ in range(20):
        q1, dq = lsrk.lsrk_step(N, K3, q1, dq, Ja, phi, J, dt, coriolis=f)
    ang = f * dt * 20
    assert np.allclose(q1[1], 10.0 * math.cos(ang), rtol=0, atol=1e-9)
    assert np.allclose(q1[2], -10.0 * math.sin(ang), rtol=0, atol=1e-9)
    assert np.allclose(q1[0], 1.0, rtol=0, atol=1e-12)
