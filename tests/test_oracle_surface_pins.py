"""Pins of the oracle's surface term to facts other than its own formulas.

The ESDG GPU paper ("GPU Performance of an Entropy-Stable Discontinuous
Galerkin Euler Solver with Non-Conservative Terms", Sec. 3 after Eq. 2) builds
the surface flux from the entropy-conserving flux plus a matrix dissipation
"akin to a Roe Riemann solver" and leaves the formula to its reference.  What
pins the reading here:

* flux level: consistency, the eigen-structure of the flux Jacobian (the
  Jacobian by complex-step differentiation of the physical flux in
  tests/physics.py), the entropy Jacobian R T R^T = dq/dw (dw/dq by complex
  step of the entropy variables), the small-jump limit 1/2 |A_n| [[q]] of a
  Roe-type dissipation (|A_n| from numpy's eigendecomposition), conservation
  and entropy stability;
* mesh level: free-stream preservation of volume + surface, global
  conservation, exact entropy conservation without dissipation and an entropy
  production equal to the sum of the face dissipation terms with it.
"""
import numpy as np
import pytest

import oracle
import workloads as wl
from tests import physics as ph

GAMMA = 1.4


def _random_state(rng, phi_scale=3e4):
    rho = rng.uniform(0.2, 1.5)
    u = rng.uniform(-60, 60, size=3)
    p = rng.uniform(2e3, 1.2e5)
    phi = rng.uniform(0.0, phi_scale)
    q = ph.conserved(np.array([rho]), u.reshape(3, 1), np.array([p]), phi, GAMMA)[:, 0]
    return q, phi


def _random_normal(rng):
    return rng.standard_normal(3) * rng.uniform(0.1, 1e3)


def _complex_step_jacobian(fun, x, h=1e-30):
    """d fun / d x by complex-step differentiation (exact to rounding for analytic fun)."""
    x = np.asarray(x, dtype=np.float64)
    cols = []
    for k in range(x.size):
        xc = x.astype(np.complex128)
        step = h * max(1.0, abs(x[k]))
        xc[k] += 1j * step
        cols.append(np.imag(fun(xc)) / step)
    return np.stack(cols, axis=1)


def _flux_jacobian(q, phi, n):
    return _complex_step_jacobian(lambda qq: ph.physical_flux(qq, phi, n, GAMMA), q)


def _abs_matrix(A):
    lam, V = np.linalg.eig(A)
    return np.real(V @ np.diag(np.abs(lam)) @ np.linalg.inv(V))


# ----------------------------------------------------------------------------
# flux level

def test_surface_flux_consistency():
    """F*(q, q; n) is the physical flux n . f(q) of Eq. 1; the dissipation vanishes."""
    rng = np.random.default_rng(11)
    for _ in range(200):
        q, phi = _random_state(rng)
        n = _random_normal(rng)
        F = oracle.surface_flux(q, phi, q, phi, n)
        f = ph.physical_flux(q, phi, n)
        assert np.max(np.abs(F - f)) <= 1e-12 * np.abs(f).max()
        assert np.all(oracle.dissipation(q, phi, q, phi, n) == 0.0)


@pytest.mark.parametrize("with_phi", [False, True])
def test_eigenvectors_of_the_flux_jacobian(with_phi):
    """A_n R = R Lambda for the Jacobian of n^ . f (Eq. 1, E containing rho phi)."""
    rng = np.random.default_rng(12)
    for _ in range(50):
        q, phi = _random_state(rng, 3e4 if with_phi else 0.0)
        n = _random_normal(rng)
        R, lam, _ = oracle.roe_matrices(q, phi, q, phi, n)
        A = _flux_jacobian(q, phi, n / np.linalg.norm(n))
        res = A @ R - R @ np.diag(lam)
        assert np.max(np.abs(res)) <= 1e-10 * np.abs(A).max() * np.abs(R).max()
        # the eigenvalues are those of the Jacobian
        ev = np.sort(np.real(np.linalg.eigvals(A)))
        assert np.max(np.abs(np.sort(lam) - ev)) <= 1e-8 * np.abs(ev).max()


@pytest.mark.parametrize("with_phi", [False, True])
def test_scaled_eigenvectors_give_the_entropy_jacobian(with_phi):
    """R T R^T = dq/dw (the inverse Hessian of eta = -rho s/(gamma-1)): the scaling that
    makes R |Lambda| T R^T [[w]] a dissipation in entropy variables."""
    rng = np.random.default_rng(13)
    for _ in range(50):
        q, phi = _random_state(rng, 3e4 if with_phi else 0.0)
        n = _random_normal(rng)
        R, _, T = oracle.roe_matrices(q, phi, q, phi, n)
        dwdq = _complex_step_jacobian(lambda qq: ph.entropy_vars(qq, phi, GAMMA), q)
        M = R @ np.diag(T) @ R.T
        Minv = np.linalg.inv(dwdq)
        # M is symmetric positive definite: |M_ij| <= sqrt(M_ii M_jj) sets each entry's scale
        d = np.sqrt(np.abs(np.diag(Minv)))
        assert np.max(np.abs(M - Minv) / np.outer(d, d)) < 1e-10


@pytest.mark.parametrize("with_phi", [False, True])
def test_small_jump_limit_is_roe_dissipation(with_phi):
    """For q+- = q +- eps d/2 the dissipation tends to 1/2 |A_n| (q+ - q-), the upwind
    (Roe) dissipation, with |A_n| = V |Lambda| V^-1 of the Jacobian of n . f."""
    rng = np.random.default_rng(14)
    for _ in range(40):
        q, phi = _random_state(rng, 3e4 if with_phi else 0.0)
        n = _random_normal(rng)
        d = rng.standard_normal(5) * np.abs(q) * np.array([1, 1, 1, 1, 0.1])
        eps = 1e-6
        qm = q - eps * d / 2
        qp = q + eps * d / 2
        D = oracle.dissipation(qm.astype(np.longdouble), phi, qp.astype(np.longdouble), phi, n,
                               real="ld").astype(np.float64)
        ref = 0.5 * _abs_matrix(_flux_jacobian(q, phi, n)) @ (qp - qm)
        assert np.max(np.abs(D - ref)) <= 1e-8 * np.abs(ref).max()


def test_surface_flux_conservation():
    """F*(a, b; n) = -F*(b, a; -n) when both sides carry the same phi (no gravity
    fluctuation); mass and energy stay antisymmetric for any phi."""
    rng = np.random.default_rng(15)
    for _ in range(200):
        qa, phi = _random_state(rng)
        qb, phib = _random_state(rng)
        qb_same = ph.conserved(*[np.array([v]) if np.ndim(v) == 0 else v.reshape(3, 1)
                                 for v in ph.primitives(qb, phib)], phi, GAMMA)[:, 0]
        n = _random_normal(rng)
        F1 = oracle.surface_flux(qa, phi, qb_same, phi, n)
        F2 = oracle.surface_flux(qb_same, phi, qa, phi, -n)
        assert np.max(np.abs(F1 + F2)) <= 1e-12 * np.abs(F1).max()
        G1 = oracle.surface_flux(qa, phi, qb, phib, n)
        G2 = oracle.surface_flux(qb, phib, qa, phi, -n)
        for c in (0, 4):
            assert abs(G1[c] + G2[c]) <= 1e-12 * np.abs(G1).max()


def test_surface_flux_is_entropy_stable():
    """[[w]] . D >= 0 for arbitrary pairs (large jumps included), i.e. the surface
    flux dissipates entropy relative to the entropy-conserving flux."""
    rng = np.random.default_rng(16)
    for trial in range(400):
        qa, pa = _random_state(rng)
        qb, pb = _random_state(rng)
        if trial % 4 == 0:
            qb, pb = qa * (1 + 1e-4 * rng.standard_normal(5)), pa
        n = _random_normal(rng)
        D = oracle.dissipation(qa, pa, qb, pb, n)
        dw = ph.entropy_vars(qb, pb) - ph.entropy_vars(qa, pa)
        prod = float(dw @ D)
        assert prod >= -1e-12 * np.abs(dw) @ np.abs(D)
        Fs = oracle.surface_flux(qa, pa, qb, pb, n)
        Fe = oracle.flux(qa, pa, qb, pb, n)
        assert np.max(np.abs((Fe - Fs) - D)) <= 1e-12 * (np.abs(Fe).max() + np.abs(D).max())


# ----------------------------------------------------------------------------
# mesh level

def _mesh(N, K, bc, state="random", warp=True, seed=None):
    cfg = wl.small_config(N, K=K, warp=warp, state=state, seed=seed, bc=bc)
    g = wl.generate(cfg)
    Ja, J = oracle.metrics(N, cfg.K, g["x"].numpy(), g["y"].numpy(), g["z"].numpy())
    return cfg, g["q"].numpy(), g["phi"].numpy(), Ja, J


def _omega(N):
    _, w = oracle.lgl(N)
    Nq = N + 1
    idx = np.arange(Nq ** 3)
    return w[idx % Nq] * w[(idx // Nq) % Nq] * w[idx // (Nq * Nq)]


@pytest.mark.parametrize("N", [2, 3, 5])
@pytest.mark.parametrize("form", [0, 1])
@pytest.mark.parametrize("phi_const", [0.0, 1.0e4])
def test_free_stream_volume_plus_surface(N, form, phi_const):
    """A constant state with constant phi on a warped periodic mesh is steady:
    volume + surface vanishes to round-off (needs the metric identities, the
    lifting 1/w_0, outward normals and the face pairing)."""
    cfg, q, _, Ja, _ = _mesh(N, (2, 3, 2), (0, 0, 0))
    n = cfg.n
    qc = ph.conserved(np.full(n, 1.1), np.tile(np.array([[12.0], [-7.0], [4.0]]), (1, n)),
                      np.full(n, 9.0e4), phi_const, GAMMA)
    phi = np.full(n, phi_const)
    vol, vs = oracle.volume(N, cfg.K, qc, Ja, phi, GAMMA, form=form, with_scale=True)
    srf, ss = oracle.surface(N, (cfg.Kx, cfg.Ky, cfg.Kz), qc, Ja, phi, (0, 0, 0), GAMMA, form=form,
                             with_scale=True)
    tot = vol + srf
    scale = (vs + ss).max(axis=1)
    assert np.max(np.abs(tot).max(axis=1) / scale) < 1e3 * np.finfo(float).eps


@pytest.mark.parametrize("N", [1, 2, 4])
@pytest.mark.parametrize("bc", [(0, 0, 0), (1, 1, 1), (0, 1, 1)])
def test_global_conservation(N, bc):
    """sum_i omega_i (volume + surface)_c = 0 for mass and energy (out is the
    J-weighted divergence, so this is d/dt of the integral); momentum too on a
    periodic mesh without gravity.  Slip walls carry no mass or energy."""
    cfg, q, phi, Ja, _ = _mesh(N, (2, 2, 3), bc)
    om = np.tile(_omega(N), cfg.K)
    K3 = (cfg.Kx, cfg.Ky, cfg.Kz)
    for dissipation in (False, True):
        vol, vs = oracle.volume(N, cfg.K, q, Ja, phi, GAMMA, with_scale=True)
        srf, ss = oracle.surface(N, K3, q, Ja, phi, bc, GAMMA, dissipation=dissipation, with_scale=True)
        tot = (vol + srf) @ om
        mag = (vs + ss) @ om
        for c in (0, 4):
            assert abs(tot[c]) <= 1e-12 * mag[c], (c, tot[c], mag[c])
    if bc == (0, 0, 0):
        phi0 = np.zeros_like(phi)
        rho, u, p = ph.primitives(q, phi)
        q0 = ph.conserved(rho, u, p, phi0, GAMMA)
        vol, vs = oracle.volume(N, cfg.K, q0, Ja, phi0, GAMMA, with_scale=True)
        srf, ss = oracle.surface(N, K3, q0, Ja, phi0, bc, GAMMA, with_scale=True)
        tot = (vol + srf) @ om
        mag = (vs + ss) @ om
        for c in (1, 2, 3):
            assert abs(tot[c]) <= 1e-12 * mag[c]


def _entropy_sum(N, cfg, q, phi, out, scale):
    w = ph.entropy_vars(q, phi)
    om = np.tile(_omega(N), cfg.K)
    return float(np.sum(om * np.sum(w * out, axis=0))), float(np.sum(om * np.sum(np.abs(w) * scale, axis=0)))


@pytest.mark.parametrize("N", [1, 2, 3, 5])
@pytest.mark.parametrize("bc", [(0, 0, 0), (0, 1, 1), (1, 1, 1)])
def test_entropy_conservation_without_dissipation(N, bc):
    """With the entropy-conserving flux alone at the faces, sum_i omega_i w_i . out_i
    vanishes (strong volume form plus surface): the semi-discrete scheme conserves
    entropy on periodic meshes and at slip walls (Sec. 3)."""
    cfg, q, phi, Ja, _ = _mesh(N, (2, 2, 2), bc)
    K3 = (cfg.Kx, cfg.Ky, cfg.Kz)
    vol, vs = oracle.volume(N, cfg.K, q, Ja, phi, GAMMA, with_scale=True)
    srf, ss = oracle.surface(N, K3, q, Ja, phi, bc, GAMMA, dissipation=False, with_scale=True)
    tot, mag = _entropy_sum(N, cfg, q, phi, vol + srf, vs + ss)
    assert abs(tot) <= 1e-11 * mag, (tot, mag)


def _face_dissipation_sum(N, cfg, q, phi, Ja, bc):
    """sum over faces of omega_face [[w]] . D (interior, once per face) and of
    omega_face (-w_i . D(i, ghost)) at slip walls, from the pair dissipation."""
    Nq = N + 1
    np3 = Nq ** 3
    _, w1 = oracle.lgl(N)
    Kd = (cfg.Kx, cfg.Ky, cfg.Kz)
    n = cfg.n
    total = 0.0
    for e in range(cfg.K):
        ec = (e % cfg.Kx, (e // cfg.Kx) % cfg.Ky, e // (cfg.Kx * cfg.Ky))
        for r in range(3):
            for i in range(np3):
                ai = [i % Nq, (i // Nq) % Nq, i // (Nq * Nq)]
                if ai[r] != N and not (ai[r] == 0 and ec[r] == 0 and bc[r] == 1):
                    continue
                o = [s for s in range(3) if s != r]
                wf = w1[ai[o[0]]] * w1[ai[o[1]]]
                gi = e * np3 + i
                side = 1 if ai[r] == N else -1
                en = list(ec)
                en[r] += side
                qi, pi_ = q[:, gi], phi[gi]
                if 0 <= en[r] < Kd[r] or bc[r] == 0:
                    if ai[r] != N:
                        continue
                    en[r] %= Kd[r]
                    aj = list(ai)
                    aj[r] = 0
                    gj = (en[0] + cfg.Kx * (en[1] + cfg.Ky * en[2])) * np3 + aj[0] + Nq * (aj[1] + Nq * aj[2])
                    nv = (Ja[3 * r:3 * r + 3, gi] + Ja[3 * r:3 * r + 3, gj]) / 2
                    D = oracle.dissipation(qi, pi_, q[:, gj], phi[gj], nv)
                    dw = ph.entropy_vars(q[:, gj], phi[gj]) - ph.entropy_vars(qi, pi_)
                    total += wf * float(dw @ D)
                else:
                    nv = side * Ja[3 * r:3 * r + 3, gi]
                    nh = nv / np.linalg.norm(nv)
                    g = qi.copy()
                    g[1:4] = qi[1:4] - 2 * (qi[1:4] @ nh) * nh
                    D = oracle.dissipation(qi, pi_, g, pi_, nv)
                    total += wf * float(-ph.entropy_vars(qi, pi_) @ D)
    return total


@pytest.mark.parametrize("N,bc", [(1, (0, 0, 0)), (2, (0, 1, 1)), (3, (1, 1, 1))])
def test_entropy_production_equals_face_dissipation(N, bc):
    """With dissipation, sum_i omega_i w_i . out_i equals the face sum of the pair
    dissipation's entropy production and is positive (d eta/dt <= 0)."""
    cfg, q, phi, Ja, _ = _mesh(N, (2, 2, 2), bc)
    K3 = (cfg.Kx, cfg.Ky, cfg.Kz)
    vol, vs = oracle.volume(N, cfg.K, q, Ja, phi, GAMMA, with_scale=True)
    srf, ss = oracle.surface(N, K3, q, Ja, phi, bc, GAMMA, dissipation=True, with_scale=True)
    tot, mag = _entropy_sum(N, cfg, q, phi, vol + srf, vs + ss)
    ref = _face_dissipation_sum(N, cfg, q, phi, Ja, bc)
    assert ref > 0
    assert abs(tot - ref) <= 1e-11 * mag, (tot, ref, mag)


def test_surface_double_matches_long_double():
    """The double oracle's own rounding on the surface term, against long double."""
    cfg, q, phi, Ja, _ = _mesh(3, (2, 2, 2), (0, 1, 1))
    K3 = (cfg.Kx, cfg.Ky, cfg.Kz)
    d, sc = oracle.surface(3, K3, q, Ja, phi, (0, 1, 1), GAMMA, with_scale=True)
    ld = oracle.surface(3, K3, q, Ja, phi, (0, 1, 1), GAMMA, real="ld")
    err = np.abs(d - ld.astype(np.float64)).max(axis=1) / sc.max(axis=1)
    assert err.max() < 1e-14
