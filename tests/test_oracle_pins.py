"""Pins of the CPU oracle to facts other than its own formulas.

Each test names what it checks in "GPU Performance of an Entropy-Stable
Discontinuous Galerkin Euler Solver with Non-Conservative Terms" (the ESDG GPU
paper) or in textbook mathematics.  A plausible slip in the oracle (a dropped
term, a wrong sign or side, a transposed D or metric index, a wrong factor of
two) fails at least one of them; test_planted_mistakes checks a few.
"""
import math

import numpy as np
import pytest

import oracle
import workloads as wl
from tests import physics as ph

GAMMA = 1.4
NS = list(range(1, 9))


# ----------------------------------------------------------------------------
# operators: LGL nodes, weights, D (Sec. 3)

@pytest.mark.parametrize("N", NS)
def test_lgl_nodes_match_library_roots(N):
    """Interior LGL nodes are the roots of P_N' (numpy's Legendre routine)."""
    x, w = oracle.lgl(N)
    ref = wl.node_positions(N)
    assert np.max(np.abs(x - ref)) < 4e-15
    # end weight closed form 2/(N(N+1)) and total weight 2
    assert abs(w[0] - 2.0 / (N * (N + 1))) < 1e-15
    assert abs(w[-1] - 2.0 / (N * (N + 1))) < 1e-15
    assert abs(np.sum(w) - 2.0) < 4e-15


@pytest.mark.parametrize("N", NS)
def test_lgl_quadrature_exact_to_2N_minus_1(N):
    x, w = oracle.lgl(N)
    for k in range(0, 2 * N):
        exact = 0.0 if k % 2 else 2.0 / (k + 1)
        assert abs(np.sum(w * x ** k) - exact) < 1e-14, k
    # and not exact at degree 2N (Lobatto rule), which pins the node set
    assert abs(np.sum(w * x ** (2 * N)) - 2.0 / (2 * N + 1)) > 1e-6


@pytest.mark.parametrize("N", NS)
def test_dmatrix_sbp_identities(N):
    x, w = oracle.lgl(N)
    D = oracle.dmatrix(N)
    # exact on polynomials of degree <= N
    for k in range(0, N + 1):
        d = k * x ** (k - 1) if k else np.zeros_like(x)
        assert np.max(np.abs(D @ x ** k - d)) < 2e-13 * max(1, N * N), k
    Q = np.diag(w) @ D
    B = np.zeros_like(Q)
    B[0, 0], B[-1, -1] = -1.0, 1.0
    assert np.max(np.abs(Q + Q.T - B)) < 2e-14
    assert np.max(np.abs(D.sum(axis=1))) < 2e-13
    assert abs(D[0, 0] + N * (N + 1) / 4) < 1e-14
    # textbook barycentric construction agrees
    assert np.max(np.abs(D - ph.bary_dmatrix(x))) < 1e-12 * (N + 1) ** 2


def test_dmatrix_N1_closed_form():
    D = oracle.dmatrix(1)
    assert np.allclose(D, [[-0.5, 0.5], [-0.5, 0.5]], atol=0, rtol=0)


# ----------------------------------------------------------------------------
# metric terms (Sec. 3, G_jk), curl form

def _affine_element(N, A, x0):
    """Node coordinates of x = x0 + A xi on one element."""
    xi = wl.node_positions(N)
    Nq = N + 1
    a, b, c = np.meshgrid(np.arange(Nq), np.arange(Nq), np.arange(Nq), indexing="ij")
    # node index a + Nq(b + Nq c): build in that order
    idx = np.arange(Nq ** 3)
    a, b, c = idx % Nq, (idx // Nq) % Nq, idx // (Nq * Nq)
    R = np.stack([xi[a], xi[b], xi[c]])
    X = x0[:, None] + A @ R
    return X[0], X[1], X[2]


@pytest.mark.parametrize("N", [1, 2, 4, 7])
def test_metrics_affine_closed_form(N):
    rng = np.random.default_rng(11 + N)
    A = np.diag([300.0, 200.0, 50.0]) + 20.0 * rng.standard_normal((3, 3))
    x, y, z = _affine_element(N, A, np.array([1.0, 2.0, 3.0]))
    Ja, J = oracle.metrics(N, 1, x, y, z)
    detA = np.linalg.det(A)
    cof = detA * np.linalg.inv(A)  # row r = J d xi_r / d x
    for r in range(3):
        for j in range(3):
            assert np.max(np.abs(Ja[3 * r + j] - cof[r, j])) < 1e-11 * np.abs(cof).max()
    assert np.max(np.abs(J - detA)) < 1e-12 * abs(detA)


def _trilinear_element(N, corners):
    xi = wl.node_positions(N)
    Nq = N + 1
    idx = np.arange(Nq ** 3)
    s, t, u = xi[idx % Nq], xi[(idx // Nq) % Nq], xi[idx // (Nq * Nq)]

    def shape(s, t, u):
        out = []
        for k in range(8):
            cs, ct, cu = (1 if k & 1 else -1), (1 if k & 2 else -1), (1 if k & 4 else -1)
            out.append((1 + cs * s) * (1 + ct * t) * (1 + cu * u) / 8.0)
        return np.array(out)

    def dshape(s, t, u, d):
        out = []
        for k in range(8):
            cs, ct, cu = (1 if k & 1 else -1), (1 if k & 2 else -1), (1 if k & 4 else -1)
            f = [(1 + cs * s), (1 + ct * t), (1 + cu * u)]
            f[d] = [cs, ct, cu][d] * np.ones_like(s)
            out.append(f[0] * f[1] * f[2] / 8.0)
        return np.array(out)

    X = corners.T @ shape(s, t, u)  # (3, npts)
    dX = [corners.T @ dshape(s, t, u, d) for d in range(3)]  # dX[d][n] = d X_n / d xi_d
    return X, dX


@pytest.mark.parametrize("N", [2, 3, 5, 8])
def test_metrics_trilinear_closed_form(N):
    """For a trilinear hexahedron the curl form is exact once N >= 2.

    Each product X_l d X_m has degree <= 2 per reference direction, so its
    degree-N interpolant is exact and Ja^r equals the analytic cofactors
    x_eta x x_zeta, x_zeta x x_xi, x_xi x x_eta.
    """
    rng = np.random.default_rng(5 + N)
    base = np.array([[(k & 1), (k >> 1) & 1, (k >> 2) & 1] for k in range(8)], dtype=float)
    corners = base * np.array([100.0, 80.0, 60.0]) + 12.0 * rng.standard_normal((8, 3))
    X, dX = _trilinear_element(N, corners)
    Ja, J = oracle.metrics(N, 1, X[0], X[1], X[2])
    cof = [np.cross(dX[1].T, dX[2].T).T, np.cross(dX[2].T, dX[0].T).T, np.cross(dX[0].T, dX[1].T).T]
    scale = max(np.abs(c).max() for c in cof)
    for r in range(3):
        for j in range(3):
            assert np.max(np.abs(Ja[3 * r + j] - cof[r][j])) < 1e-12 * scale, (r, j)
    Jex = np.einsum("ij,ij->j", dX[0], np.cross(dX[1].T, dX[2].T).T)
    assert np.max(np.abs(J - Jex)) < 1e-12 * np.abs(Jex).max()


def _ref_derivative(f, D, Nq, r):
    F = f.reshape(Nq, Nq, Nq)  # [c, b, a]
    axis = 2 - r
    return np.moveaxis(np.tensordot(D, np.moveaxis(F, axis, 0), axes=(1, 0)), 0, axis).reshape(-1)


@pytest.mark.parametrize("N", [1, 3, 4, 7])
def test_metric_identities_warped(N):
    """sum_r D^r Ja^r_j = 0 at every node (discrete divergence of a discrete curl)."""
    cfg = wl.small_config(N, K=(2, 2, 1), warp=True)
    g = wl.generate(cfg)
    Ja, J = oracle.metrics(N, cfg.K, g["x"].numpy(), g["y"].numpy(), g["z"].numpy())
    Nq = N + 1
    D = ph.bary_dmatrix(wl.node_positions(N))
    np3 = Nq ** 3
    for e in range(cfg.K):
        sl = slice(e * np3, (e + 1) * np3)
        for j in range(3):
            div = sum(_ref_derivative(Ja[3 * r + j, sl], D, Nq, r) for r in range(3))
            scale = np.abs(Ja[:, sl]).max() * np.abs(D).max()
            assert np.max(np.abs(div)) < 1e-12 * scale
    assert J.min() > 0


# ----------------------------------------------------------------------------
# two-point flux (Sec. 4.1, Eqs. 3-5)

def _random_pair(rng, phi_scale=3e4):
    rho = rng.uniform(0.2, 1.5, size=2)
    u = rng.uniform(-40, 40, size=(3, 2))
    p = rng.uniform(2e3, 1.2e5, size=2)
    phi = rng.uniform(0.0, phi_scale, size=2)
    q = ph.conserved(rho, u, p, phi, GAMMA)
    nvec = rng.standard_normal(3) * rng.uniform(0.1, 1e3)
    return q[:, 0], q[:, 1], phi, nvec, (rho, u, p)


def test_flux_consistency_with_physical_flux():
    """F(q, q) . n equals the physical flux n . f(q) of Eq. 1 and G(q, q) = 0."""
    rng = np.random.default_rng(1)
    for _ in range(200):
        qi, _, phi, nvec, _ = _random_pair(rng)
        F = oracle.flux(qi, phi[0], qi, phi[0], nvec)
        f = ph.physical_flux(qi, phi[0], nvec)
        assert np.max(np.abs(F - f) / (np.abs(f) + 1e-300 + np.abs(f).max() * 1e-3)) < 1e-12


def test_flux_symmetry_and_gravity_partner_scaling():
    """Sec. 4.1: the flux splits into a symmetric part S and a gravity part G(i,m) that
    is linear in [[phi]], acts on momentum only, and maps to -G(i,m) b_i/b_m under the
    swap; mass and energy components are fully symmetric."""
    rng = np.random.default_rng(2)
    for _ in range(200):
        _, _, phi, nvec, (rho, u, p) = _random_pair(rng)
        b = rho / (2 * p)
        # same primitive states, geopotential zero on both sides: G vanishes
        q0 = ph.conserved(rho, u, p, np.zeros(2), GAMMA)
        S_im = oracle.flux(q0[:, 0], 0.0, q0[:, 1], 0.0, nvec)
        S_mi = oracle.flux(q0[:, 1], 0.0, q0[:, 0], 0.0, nvec)
        assert np.max(np.abs(S_im - S_mi) / (np.abs(S_im) + 1e-9)) < 1e-13
        q = ph.conserved(rho, u, p, phi, GAMMA)
        F_im = oracle.flux(q[:, 0], phi[0], q[:, 1], phi[1], nvec)
        F_mi = oracle.flux(q[:, 1], phi[1], q[:, 0], phi[0], nvec)
        # mass and energy symmetric
        assert abs(F_im[0] - F_mi[0]) <= 1e-13 * abs(F_im[0]) + 1e-300
        assert abs(F_im[4] - F_mi[4]) <= 1e-12 * abs(F_im[4])
        # momentum: G = F - S is parallel to n, and the partner's G is -G b_i/b_m
        G_im = F_im[1:4] - S_im[1:4]
        G_mi = F_mi[1:4] - S_mi[1:4]
        scale = np.abs(F_im[1:4]).max()
        gi = G_im @ nvec / (nvec @ nvec)
        assert np.max(np.abs(G_im - gi * nvec)) < 1e-11 * scale
        assert np.max(np.abs(G_mi + G_im * b[0] / b[1])) < 1e-11 * scale
        # linear in the jump [[phi]] and independent of the mean {{phi}}
        q2 = ph.conserved(rho, u, p, phi + 1234.5, GAMMA)
        F2 = oracle.flux(q2[:, 0], phi[0] + 1234.5, q2[:, 1], phi[1] + 1234.5, nvec)
        assert np.max(np.abs(F2[1:4] - F_im[1:4])) < 1e-11 * scale
        q3 = ph.conserved(rho, u, p, np.array([phi[0], phi[0] + 2 * (phi[1] - phi[0])]), GAMMA)
        F3 = oracle.flux(q3[:, 0], phi[0], q3[:, 1], phi[0] + 2 * (phi[1] - phi[0]), nvec)
        assert np.max(np.abs((F3[1:4] - S_im[1:4]) - 2 * G_im)) < 1e-11 * scale


@pytest.mark.parametrize("real,tol", [("d", 5e-12), ("ld", 5e-15)])
def test_flux_pair_entropy_conservation(real, tol):
    """Sec. 3 asks the volume flux to conserve entropy.  For a non-symmetric pair flux
    this is w_i . F(i,m) - w_m . F(m,i) = psi_i . n - psi_m . n with psi = rho u.
    The entropy variables come from eta = -rho s/(gamma-1) (tests/physics.py)."""
    rng = np.random.default_rng(3)
    worst = 0.0
    for trial in range(300):
        qi, qm, phi, nvec, (rho, u, p) = _random_pair(rng)
        if trial % 3 == 0:  # nearly equal states exercise the log-mean limit
            qm = ph.conserved(rho[0] * (1 + 1e-7), u[:, 0] + 1e-6, p[0] * (1 - 3e-7), phi[1], GAMMA)
        Fi = oracle.flux(qi, phi[0], qm, phi[1], nvec, real=real).astype(np.float64)
        Fm = oracle.flux(qm, phi[1], qi, phi[0], nvec, real=real).astype(np.float64)
        # evaluate the identity in long double to see the flux's own error
        wi = ph.entropy_vars(qi.astype(np.longdouble), np.longdouble(phi[0]))
        wm = ph.entropy_vars(qm.astype(np.longdouble), np.longdouble(phi[1]))
        lhs = wi @ Fi.astype(np.longdouble) - wm @ Fm.astype(np.longdouble)
        rhs = np.longdouble(ph.entropy_potential(qi, nvec)) - np.longdouble(ph.entropy_potential(qm, nvec))
        mag = np.abs(wi) @ np.abs(Fi) + np.abs(wm) @ np.abs(Fm)
        worst = max(worst, float(abs(lhs - rhs) / mag))
    assert worst < tol, worst


# ----------------------------------------------------------------------------
# whole-element invariants of the volume term (Eq. 2 volume part)

def _case(N, K=(2, 1, 1), warp=True, state="random", seed=None):
    cfg = wl.small_config(N, K=K, warp=warp, state=state, seed=seed)
    g = wl.generate(cfg)
    x, y, z = g["x"].numpy(), g["y"].numpy(), g["z"].numpy()
    Ja, J = oracle.metrics(N, cfg.K, x, y, z)
    return cfg, g["q"].numpy(), g["phi"].numpy(), Ja, J


def _face_sums(N, K, q, phi, Ja, fn):
    """sum over r and the two r-faces of omega_face * (fn at xi_r=+1 - fn at xi_r=-1).

    fn(q_nodes, phi_nodes, n_nodes) -> (ncomp, nodes)."""
    Nq = N + 1
    np3 = Nq ** 3
    _, w = oracle.lgl(N)
    idx = np.arange(np3)
    ai = [idx % Nq, (idx // Nq) % Nq, idx // (Nq * Nq)]
    res = []
    for e in range(K):
        sl = slice(e * np3, (e + 1) * np3)
        tot = 0.0
        for r in range(3):
            o = [s for s in range(3) if s != r]
            wf = w[ai[o[0]]] * w[ai[o[1]]]
            n = Ja[3 * r:3 * r + 3, sl]
            val = fn(q[:, sl], phi[sl], n)
            plus = ai[r] == N
            minus = ai[r] == 0
            tot = tot + (val[:, plus] * wf[plus]).sum(axis=1) - (val[:, minus] * wf[minus]).sum(axis=1)
        res.append(tot)
    return np.array(res)


def _omega(N):
    _, w = oracle.lgl(N)
    Nq = N + 1
    idx = np.arange(Nq ** 3)
    return w[idx % Nq] * w[(idx // Nq) % Nq] * w[idx // (Nq * Nq)]


@pytest.mark.parametrize("N", [1, 2, 3, 4, 7])
def test_volume_conservation_per_element(N):
    """Mass and energy: sum_i omega_i out_i equals the boundary sum of the physical
    flux, because Q = W D is skew up to B and F is symmetric in those components."""
    cfg, q, phi, Ja, J = _case(N)
    out, scale = oracle.volume(N, cfg.K, q, Ja, phi, with_scale=True)
    om = _omega(N)
    faces = _face_sums(N, cfg.K, q, phi, Ja, lambda qq, pp, nn: ph.physical_flux(qq, pp, nn))
    np3 = (N + 1) ** 3
    for e in range(cfg.K):
        sl = slice(e * np3, (e + 1) * np3)
        lhs = (out[:, sl] * om).sum(axis=1)
        mag = (scale[:, sl] * om).sum(axis=1)
        for c in (0, 4):
            assert abs(lhs[c] - faces[e][c]) < 1e-13 * mag[c], (e, c)


@pytest.mark.parametrize("N", [1, 2, 3, 4, 7])
def test_volume_conservation_momentum_without_gravity(N):
    cfg, q, phi, Ja, J = _case(N)
    phi0 = np.full_like(phi, 777.0)
    rho, u, p = ph.primitives(q, phi)
    q0 = ph.conserved(rho, u, p, phi0)
    out, scale = oracle.volume(N, cfg.K, q0, Ja, phi0, with_scale=True)
    om = _omega(N)
    faces = _face_sums(N, cfg.K, q0, phi0, Ja, lambda qq, pp, nn: ph.physical_flux(qq, pp, nn))
    np3 = (N + 1) ** 3
    for e in range(cfg.K):
        sl = slice(e * np3, (e + 1) * np3)
        lhs = (out[:, sl] * om).sum(axis=1)
        mag = (scale[:, sl] * om).sum(axis=1)
        assert np.all(np.abs(lhs - faces[e]) < 1e-13 * mag), e


@pytest.mark.parametrize("N", [1, 2, 3, 4, 6, 7])
@pytest.mark.parametrize("form", [0, 1])
def test_volume_sbp_entropy_identity(N, form):
    """sum_i omega_i w_i . out_i = sum_r faces omega_f [(w.f~ - psi~)|+ - (.)|-]
    + sum_i omega_i psi_i . sum_r (D^r Ja^r)_i   (2D form); the skew form has
    -psi~ in place of w.f~ - psi~.  Follows from Q + Q^T = B and the pair
    entropy condition; holds to round-off on curved meshes with gravity."""
    cfg, q, phi, Ja, J = _case(N, K=(2, 2, 1))
    out, scale = oracle.volume(N, cfg.K, q, Ja, phi, form=form, with_scale=True)
    w = ph.entropy_vars(q, phi)
    om = _omega(N)

    def bterm(qq, pp, nn):
        psi = qq[1] * nn[0] + qq[2] * nn[1] + qq[3] * nn[2]
        if form == 0:
            wf = np.sum(ph.entropy_vars(qq, pp) * ph.physical_flux(qq, pp, nn), axis=0)
            return (wf - psi)[None, :]
        return (-psi)[None, :]

    faces = _face_sums(N, cfg.K, q, phi, Ja, bterm)
    Nq = N + 1
    np3 = Nq ** 3
    D = ph.bary_dmatrix(wl.node_positions(N))
    for e in range(cfg.K):
        sl = slice(e * np3, (e + 1) * np3)
        lhs = np.sum(om * np.sum(w[:, sl] * out[:, sl], axis=0))
        mag = np.sum(om * np.sum(np.abs(w[:, sl]) * scale[:, sl], axis=0))
        divJa = np.stack([sum(_ref_derivative(Ja[3 * r + j, sl], D, Nq, r) for r in range(3)) for j in range(3)])
        metric_term = np.sum(om * np.sum(q[1:4, sl] * divJa, axis=0))
        rhs = faces[e][0] + metric_term
        assert abs(lhs - rhs) < 2e-13 * mag, (e, lhs, rhs, mag)


@pytest.mark.parametrize("N", [2, 3, 5, 7, 8])
@pytest.mark.parametrize("phi_const", [0.0, 1.0e4])
def test_free_stream_preservation_curved(N, phi_const):
    """Constant rho, u, p and constant geopotential on a warped mesh give zero."""
    cfg = wl.small_config(N, K=(2, 2, 2), warp=True)
    g = wl.generate(cfg)
    Ja, J = oracle.metrics(N, cfg.K, g["x"].numpy(), g["y"].numpy(), g["z"].numpy())
    n = cfg.n
    phi = np.full(n, phi_const)
    q = ph.conserved(np.full(n, 1.1), np.tile(np.array([[12.0], [-7.0], [3.0]]), (1, n)),
                     np.full(n, 9.0e4), phi)
    out, scale = oracle.volume(N, cfg.K, q, Ja, phi, with_scale=True)
    for c in range(5):
        assert np.max(np.abs(out[c])) < 1e3 * 2.2e-16 * np.max(scale[c]), c


@pytest.mark.parametrize("N", [1, 2, 4, 7])
def test_hydrostatic_gravity_closed_form(N):
    """u = 0, rho and p constant, phi = g z on an axis-aligned affine element: the pressure
    parts cancel and the gravity term gives out_mz = rho g J exactly (Eqs. 4-5 with
    rho_hat = rho when b is uniform), all other components zero."""
    hx, hy, hz = 400.0, 300.0, 120.0
    x, y, z = _affine_element(N, np.diag([hx / 2, hy / 2, hz / 2]), np.array([0.0, 0.0, 500.0]))
    Ja, J = oracle.metrics(N, 1, x, y, z)
    n = x.size
    rho0, p0 = 1.1, 9.0e4
    phi = 9.81 * z
    q = ph.conserved(np.full(n, rho0), np.zeros((3, n)), np.full(n, p0), phi)
    out, scale = oracle.volume(N, 1, q, Ja, phi, with_scale=True)
    Jc = hx * hy * hz / 8
    S = scale.max()
    assert np.max(np.abs(out[0])) < 1e-13 * S
    assert np.max(np.abs(out[1])) < 1e-12 * S
    assert np.max(np.abs(out[2])) < 1e-12 * S
    assert np.max(np.abs(out[4])) < 1e-13 * S
    # relative to the closed-form value itself, not to the (much larger) pressure scale
    assert np.max(np.abs(out[3] - rho0 * 9.81 * Jc)) < 1e-10 * rho0 * 9.81 * Jc


@pytest.mark.parametrize("N", [1, 2, 3, 5, 8])
def test_2d_minus_skew_is_end_node_flux(N):
    """out_2D - out_skew = sum_r 2 D_ii Ja^r(i) . f(q_i); D_00 = -N(N+1)/4, D_NN = +N(N+1)/4."""
    cfg, q, phi, Ja, J = _case(N)
    o2 = oracle.volume(N, cfg.K, q, Ja, phi, form=0)
    o1, scale = oracle.volume(N, cfg.K, q, Ja, phi, form=1, with_scale=True)
    Nq = N + 1
    idx = np.arange(cfg.n) % Nq ** 3
    ai = [idx % Nq, (idx // Nq) % Nq, idx // (Nq * Nq)]
    expect = np.zeros_like(o2)
    for r in range(3):
        f = ph.physical_flux(q, phi, Ja[3 * r:3 * r + 3])
        dii = np.where(ai[r] == 0, -N * (N + 1) / 4.0, np.where(ai[r] == N, N * (N + 1) / 4.0, 0.0))
        expect += 2 * dii * f
    for c in range(5):
        assert np.max(np.abs((o2[c] - o1[c]) - expect[c])) < 1e-12 * np.max(scale[c] + np.abs(expect[c]))


# ----------------------------------------------------------------------------
# the double oracle against its long-double twin (rounding floor)

@pytest.mark.parametrize("N", [1, 3])
def test_double_matches_long_double(N):
    cfg, q, phi, Ja, J = _case(N, K=(2, 1, 1), state="box" if N == 3 else "random")
    Jal, _ = oracle.metrics(N, cfg.K, *(wl.generate(cfg)[k].numpy() for k in ("x", "y", "z")), real="ld")
    od, scale = oracle.volume(N, cfg.K, q, Ja, phi, with_scale=True)
    ol = oracle.volume(N, cfg.K, q, Jal, phi, real="ld")
    for c in range(5):
        err = np.max(np.abs(od[c] - ol[c].astype(np.float64))) / np.max(scale[c])
        assert err < 1e-14, (c, err)


def test_tiny_box_config_runs_quickly():
    """The tiny periodic box (4x4x4 elements, N=3) finishes in well under a second."""
    import time
    cfg = wl.get_config("tiny_box_N3")
    g = wl.generate(cfg)
    Ja, J = oracle.metrics(cfg.N, cfg.K, g["x"].numpy(), g["y"].numpy(), g["z"].numpy())
    t0 = time.time()
    out = oracle.volume(cfg.N, cfg.K, g["q"].numpy(), Ja, g["phi"].numpy())
    assert time.time() - t0 < 5.0
    assert np.all(np.isfinite(out))
