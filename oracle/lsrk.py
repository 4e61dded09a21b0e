"""Time stepping of the semi-discrete system (test infrastructure, CPU).

Only the test suite may import this module.  It advances
    dq/dt = h(q) - (volume + surface)(q) / J
with a low-storage explicit Runge-Kutta scheme in the 2N-storage form of
Williamson (1980): for stages s = 1..5,
    dq <- A_s dq + dt L(q),   q <- q + B_s dq.

"GPU Performance of an Entropy-Stable Discontinuous Galerkin Euler Solver with
Non-Conservative Terms" (Sec. 3) uses a fourteen-stage fourth-order scheme
whose coefficients it does not print, and says the code previously used the
five-stage fourth-order scheme of Carpenter and Kennedy (1994).  That scheme
is the one here: its coefficients are the published rationals, checked by
tests/test_oracle_lsrk.py against the eight fourth-order conditions of the
equivalent Butcher tableau.

h is the f-plane Coriolis source of Eq. 2's h term: (0, f rho u2, -f rho u1,
0, 0) for rotation about z (zero by default).  Global diagnostics: mass and
total energy integrals sum_i omega_i J_i q_i, and the entropy integral
sum_i omega_i J_i eta_i with eta = -rho s/(gamma - 1), s = ln(p rho^-gamma).
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np

import oracle

# Carpenter & Kennedy (1994), five-stage fourth-order 2N-storage scheme
LSRK_A = [Fraction(0),
          Fraction(-567301805773, 1357537059087),
          Fraction(-2404267990393, 2016746695238),
          Fraction(-3550918686646, 2091501179385),
          Fraction(-1275806237668, 842570457699)]
LSRK_B = [Fraction(1432997174477, 9575080441755),
          Fraction(5161836677717, 13612068292357),
          Fraction(1720146321549, 2090206949498),
          Fraction(3134564353537, 4481467310338),
          Fraction(2277821191437, 14882151754819)]
LSRK_C = [Fraction(0),
          Fraction(1432997174477, 9575080441755),
          Fraction(2526269341429, 6820363962896),
          Fraction(2006345519317, 3224310063776),
          Fraction(2802321613138, 2924317926251)]


def butcher_tableau(A=LSRK_A, B=LSRK_B):
    """The classical tableau (a_ij, b_i, c_i) of a 2N-storage scheme, in exact rationals.

    With k_s = L(q_s): dq_s = sum_{j<=s} (prod_{m=j+1..s} A_m) dt k_j and
    q_{s+1} = q_1 + sum_{m<=s} B_m dq_m, so a_{s+1,j} = sum_{m=j..s} B_m prod A.
    """
    S = len(A)
    # coefficient of k_j in dq_m: prod_{l=j+1..m} A_l for j <= m
    def dq_coef(m, j):
        if j > m:
            return Fraction(0)
        c = Fraction(1)
        for l in range(j + 1, m + 1):
            c *= A[l]
        return c
    a = [[Fraction(0)] * S for _ in range(S)]
    for s in range(1, S):
        for j in range(s):
            a[s][j] = sum((B[m] * dq_coef(m, j) for m in range(j, s)), Fraction(0))
    b = [sum((B[m] * dq_coef(m, j) for m in range(j, S)), Fraction(0)) for j in range(S)]
    c = [sum(a[s], Fraction(0)) for s in range(S)]
    return a, b, c


def rhs(N, K3, q, Ja, phi, J, gamma=1.4, form=0, bc=(0, 0, 0), dissipation=True, coriolis=0.0,
        nthreads=None):
    """L(q) = h(q) - (volume + surface)(q) / J, shape (5, n)."""
    K = K3[0] * K3[1] * K3[2]
    vol = oracle.volume(N, K, q, Ja, phi, gamma, form=form, nthreads=nthreads)
    srf = oracle.surface(N, K3, q, Ja, phi, bc, gamma, form=form, dissipation=dissipation, nthreads=nthreads)
    L = -(vol + srf) / J
    if coriolis:
        L[1] += coriolis * q[2]
        L[2] -= coriolis * q[1]
    return L


def lsrk_step(N, K3, q, dq, Ja, phi, J, dt, **kw):
    """One step of the five-stage scheme; returns (q, dq) (new arrays)."""
    q = np.array(q, dtype=np.float64)
    dq = np.array(dq, dtype=np.float64)
    for s in range(5):
        L = rhs(N, K3, q, Ja, phi, J, **kw)
        dq = float(LSRK_A[s]) * dq + dt * L
        q = q + float(LSRK_B[s]) * dq
    return q, dq


def omega(N, K):
    """Quadrature weight w_a w_b w_c of every node of K elements."""
    _, w = oracle.lgl(N)
    Nq = N + 1
    idx = np.arange(Nq ** 3)
    return np.tile(w[idx % Nq] * w[(idx // Nq) % Nq] * w[idx // (Nq * Nq)], K)


def diagnostics(N, K, q, phi, J, gamma=1.4):
    """(mass, total energy, entropy) integrals, each summed exactly (math.fsum)."""
    om = omega(N, K) * J
    rho = q[0]
    uu = (q[1] ** 2 + q[2] ** 2 + q[3] ** 2) / rho ** 2
    p = (gamma - 1.0) * (q[4] - 0.5 * rho * uu - rho * phi)
    s = np.log(p) - gamma * np.log(rho)
    eta = -rho * s / (gamma - 1.0)
    return (math.fsum(om * rho), math.fsum(om * q[4]), math.fsum(om * eta))
