"""Closed-form quantities used by the pins, written from the governing equations.

These formulas are not the two-point flux: they are the physical flux of the
Euler equations with buoyancy (Eq. 1a-1c of "GPU Performance of an
Entropy-Stable Discontinuous Galerkin Euler Solver with Non-Conservative
Terms", with E including rho*phi) and the entropy pair of that system
(s = ln(p rho^-gamma), eta = -rho s/(gamma-1)).  The pins check the oracle's
two-point flux against them.
"""
import numpy as np


def primitives(q, phi, gamma=1.4):
    q = np.asarray(q)
    rho = q[0]
    u = q[1:4] / rho
    p = (gamma - 1.0) * (q[4] - 0.5 * rho * np.sum(u * u, axis=0) - rho * phi)
    return rho, u, p


def conserved(rho, u, p, phi, gamma=1.4):
    """q = (rho, rho u, E) with E = p/(gamma-1) + rho|u|^2/2 + rho phi (Sec. 2)."""
    rho = np.asarray(rho, dtype=np.float64)
    u = np.asarray(u, dtype=np.float64)
    E = p / (gamma - 1.0) + 0.5 * rho * np.sum(u * u, axis=0) + rho * phi
    return np.stack([rho, rho * u[0], rho * u[1], rho * u[2], E])


def physical_flux(q, phi, n, gamma=1.4):
    """n . f(q): mass rho u.n, momentum rho u (u.n) + p n, energy (E + p) u.n (Eq. 1).

    q has shape (5, ...), n has shape (3, ...) matching q's trailing shape.
    """
    q = np.asarray(q)
    n = np.asarray(n)
    rho, u, p = primitives(q, phi, gamma)
    un = np.sum(u * n, axis=0)
    return np.stack([rho * un,
                     rho * u[0] * un + p * n[0],
                     rho * u[1] * un + p * n[1],
                     rho * u[2] * un + p * n[2],
                     (q[4] + p) * un])


def entropy_vars(q, phi, gamma=1.4):
    """w = d eta / d q for eta = -rho s/(gamma-1), s = ln(p rho^-gamma), E containing rho phi.

    w = ((gamma - s)/(gamma-1) - b|u|^2 + 2 b phi, 2 b u, -2 b), b = rho/(2p).
    """
    rho, u, p = primitives(q, phi, gamma)
    s = np.log(p) - gamma * np.log(rho)
    b = rho / (2.0 * p)
    uu = np.sum(u * u, axis=0)
    w0 = (gamma - s) / (gamma - 1.0) - b * uu + 2.0 * b * phi
    return np.stack([w0, 2.0 * b * u[0], 2.0 * b * u[1], 2.0 * b * u[2], -2.0 * b])


def entropy_potential(q, n, gamma=1.4):
    """psi . n = rho u . n."""
    return float(q[1] * n[0] + q[2] * n[1] + q[3] * n[2])


def bary_dmatrix(x):
    """Differentiation matrix on nodes x by barycentric weights (textbook form)."""
    x = np.asarray(x, dtype=np.float64)
    n = x.size
    lam = np.array([1.0 / np.prod([x[j] - x[k] for k in range(n) if k != j]) for j in range(n)])
    D = np.zeros((n, n))
    for i in range(n):
        for j in range(n):
            if i != j:
                D[i, j] = (lam[j] / lam[i]) / (x[i] - x[j])
        D[i, i] = -np.sum(D[i, :])
    return D
