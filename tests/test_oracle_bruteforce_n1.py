"""Brute-force pin of the oracle at N = 1, in 40-digit arithmetic.

An independent restatement of the whole volume term for one element of
polynomial order 1, written from the formulas of "GPU Performance of an
Entropy-Stable Discontinuous Galerkin Euler Solver with Non-Conservative
Terms" (the ESDG GPU paper) and not from the oracle's code:

* Sec. 3, Eq. 2: the volume term of node i is
  sum_r sum_m 2 D_{a_r(i) a_r(m)} (F + G)^r(q_i, q_m), m running over the
  r-line through i, the diagonal m = i included (2D form) or left out (skew
  form);
* at N = 1 the LGL nodes are -1, +1 and the Lagrange basis is (1 -+ s)/2, so
  every derivative below is the derivative of that basis (D = [[-1/2, 1/2],
  [-1/2, 1/2]]), taken here from the basis functions themselves;
* metric terms in the conservative curl form: Ja^i_n = -e_i . curl(X_l grad X_m)
  with (n, m, l) cyclic, the product interpolated at the nodes and the curl
  taken of that interpolant; J = dX/dxi . (dX/deta x dX/dzeta);
* Eq. 4: momentum flux {{rho}}_log {{u_k}} {{u}}.n + n_k ({{rho}}/(2{{b}}) +
  rho_hat [[phi]]/2), b = rho/(2p), rho_hat = {{b}} {{rho}}_log / b_i (Eq. 5,
  node i the "-" side); mass flux {{rho}}_log {{u}}.n; energy flux the
  entropy-conserving completion F_rho (1/(2 (gamma-1) {{b}}_log) - {{|u|^2}}/2
  + {{phi}} + |{{u}}|^2) + {{u}}.n {{rho}}/(2{{b}}); n the averaged metric
  (Ja^r(i) + Ja^r(m))/2;
* the logarithmic mean (c - a)/(ln c - ln a) evaluated literally (40 digits
  leave more than 25 after the cancellation for the closest pairs used here),
  and a for c = a.

The double oracle must agree with it to 1e-14, relative to the term scale and
relative to the result itself; the long double oracle to 1e-17 of the term
scale.  Inputs are random single
elements, affine and warped (trilinear), with a non-constant geopotential.
"""
import numpy as np
import pytest

import oracle

mp = pytest.importorskip("mpmath")
mp.mp.dps = 40

GAMMA = 1.4
NODE = (-1, 1)  # LGL nodes at N = 1


def _nid(a, b, c):
    return a + 2 * (b + 2 * c)


def _dbasis(k):
    """Derivative of the N = 1 Lagrange basis function of node k (constant)."""
    return mp.mpf(-1) / 2 if k == 0 else mp.mpf(1) / 2


def _deriv(f, r, a, b, c):
    """d/dxi_r of the nodal interpolant of f (8 values) at node (a, b, c)."""
    s = mp.mpf(0)
    for k in (0, 1):
        idx = [a, b, c]
        idx[r] = k
        s += _dbasis(k) * f[_nid(*idx)]
    return s


def _nodes():
    return [(a, b, c) for c in (0, 1) for b in (0, 1) for a in (0, 1)]


def metrics_mp(X):
    """Curl-form metric terms Ja[r][j] (lists of 8 nodal values) and J."""
    Ja = [[None] * 3 for _ in range(3)]
    for n in range(3):
        m, l = (n + 1) % 3, (n + 2) % 3
        # W_k = X_l d_k X_m at the nodes (their interpolant is W)
        W = [[X[l][_nid(*t)] * _deriv(X[m], k, *t) for t in _nodes()] for k in range(3)]
        # curl W, component i = d_j W_k - d_k W_j with (i, j, k) cyclic
        for i in range(3):
            j, k = (i + 1) % 3, (i + 2) % 3
            Ja[i][n] = [-(_deriv(W[k], j, *t) - _deriv(W[j], k, *t)) for t in _nodes()]
    J = []
    for t in _nodes():
        d = [[_deriv(X[s], r, *t) for s in range(3)] for r in range(3)]  # d[r] = dX/dxi_r
        cr = [d[1][1] * d[2][2] - d[1][2] * d[2][1], d[1][2] * d[2][0] - d[1][0] * d[2][2],
              d[1][0] * d[2][1] - d[1][1] * d[2][0]]
        J.append(sum(d[0][s] * cr[s] for s in range(3)))
    return Ja, J


def _logmean(a, c):
    return a if a == c else (c - a) / (mp.log(c) - mp.log(a))


def _prim(q, phi):
    rho = q[0]
    u = [q[1] / rho, q[2] / rho, q[3] / rho]
    uu = sum(x * x for x in u)
    p = (GAMMA - 1) * (q[4] - rho * uu / 2 - rho * phi)
    return rho, u, p, rho / (2 * p), uu


def two_point(qi, phii, qm, phim, n, gravity_side="i"):
    """(F + G)(q_i, q_m) . n, node i the '-' side; five components.
    gravity_side="m" plants a mistake (b_m in rho_hat) for the last test."""
    ri, ui, pi, bi, uui = _prim(qi, phii)
    rm, um, pm, bm, uum = _prim(qm, phim)
    g = mp.mpf(GAMMA)
    rln = _logmean(ri, rm)
    bln = _logmean(bi, bm)
    ra, ba = (ri + rm) / 2, (bi + bm) / 2
    ua = [(ui[k] + um[k]) / 2 for k in range(3)]
    Un = sum(ua[k] * n[k] for k in range(3))
    phat = ra / (2 * ba)
    rho_hat = ba * rln / (bi if gravity_side == "i" else bm)
    jump_phi = phim - phii
    Frho = rln * Un
    Fm = [Frho * ua[k] + n[k] * (phat + rho_hat * jump_phi / 2) for k in range(3)]
    FE = Frho * (1 / (2 * (g - 1) * bln) - (uui + uum) / 4 + (phii + phim) / 2
                 + sum(x * x for x in ua)) + Un * phat
    return [Frho, Fm[0], Fm[1], Fm[2], FE]


def volume_mp(q, phi, Ja, form2d=True, gravity_side="i"):
    """Volume term (5 x 8) and its term scale S_c = max_i sum |2 D (F + G)_c|."""
    out = [[mp.mpf(0)] * 8 for _ in range(5)]
    mag = [[mp.mpf(0)] * 8 for _ in range(5)]
    for t in _nodes():
        i = _nid(*t)
        qi = [q[v][i] for v in range(5)]
        for r in range(3):
            for k in (0, 1):
                s = list(t)
                s[r] = k
                m = _nid(*s)
                if m == i and not form2d:
                    continue
                qm = [q[v][m] for v in range(5)]
                n = [(Ja[r][j][i] + Ja[r][j][m]) / 2 for j in range(3)]
                f = two_point(qi, phi[i], qm, phi[m], n, gravity_side)
                w = 2 * _dbasis(k)  # 2 D_{a_r(i) k}: the same in both rows at N = 1
                for v in range(5):
                    out[v][i] += w * f[v]
                    mag[v][i] += abs(w * f[v])
    return out, [max(mag[v]) for v in range(5)]


def _element(rng, warped):
    """Node coordinates (3 x 8, double) of one element: a random affine map,
    optionally with each vertex moved (a trilinear element)."""
    A = np.eye(3) * rng.uniform(200.0, 800.0, 3) + rng.uniform(-60.0, 60.0, (3, 3))
    x0 = rng.uniform(-1e3, 1e3, 3)
    X = np.empty((3, 8))
    for (a, b, c) in _nodes():
        xi = np.array([NODE[a], NODE[b], NODE[c]], dtype=float)
        X[:, _nid(a, b, c)] = x0 + A @ xi
    if warped:
        X += rng.uniform(-40.0, 40.0, X.shape)
    return X


def _state(rng, X, equal_rho_lines=False):
    rho = rng.uniform(0.8, 1.5, 8)
    if equal_rho_lines:
        rho[1::2] = rho[0::2]  # equal density on every xi-line: L(a, a) = a
    u = rng.uniform(-30.0, 30.0, (3, 8))
    p = rng.uniform(0.7e5, 1.3e5, 8)
    phi = 9.81 * X[2] + rng.uniform(-50.0, 50.0, 8)
    E = p / (GAMMA - 1) + 0.5 * rho * (u * u).sum(axis=0) + rho * phi
    q = np.stack([rho, rho * u[0], rho * u[1], rho * u[2], E])
    return q, phi


CASES = [(seed, warped, eq) for seed, warped, eq in
         [(11, False, False), (12, False, True), (13, True, False), (14, True, False), (15, True, True),
          (16, False, False)]]


@pytest.mark.parametrize("seed,warped,equal_rho", CASES)
def test_oracle_matches_bruteforce_at_n1(seed, warped, equal_rho):
    rng = np.random.default_rng(seed)
    X = _element(rng, warped)
    q, phi = _state(rng, X, equal_rho)

    Xm = [[mp.mpf(float(v)) for v in X[d]] for d in range(3)]
    Jam, Jm = metrics_mp(Xm)
    # metric terms and J: oracle (double) against the brute force
    Jo_a, Jo = oracle.metrics(1, 1, X[0].copy(), X[1].copy(), X[2].copy())
    ja_ref = np.array([[float(Jam[r][j][i]) for i in range(8)] for r in range(3) for j in range(3)])
    assert np.max(np.abs(Jo_a - ja_ref)) <= 1e-14 * np.max(np.abs(ja_ref))
    assert np.max(np.abs(Jo - np.array([float(v) for v in Jm]))) <= 1e-14 * max(abs(float(v)) for v in Jm)

    qm = [[mp.mpf(float(v)) for v in q[c]] for c in range(5)]
    phim = [mp.mpf(float(v)) for v in phi]
    for form in (0, 1):
        ref, S = volume_mp(qm, phim, Jam, form2d=(form == 0))
        ref_d = np.array([[float(v) for v in ref[c]] for c in range(5)])
        S_d = np.array([float(v) for v in S])
        got = oracle.volume(1, 1, q.copy(), Jo_a, phi.copy(), gamma=GAMMA, form=form)
        e = np.max(np.abs(got - ref_d), axis=1) / S_d
        assert e.max() <= 1e-14, (form, e)
        # and plainly relative per variable (these random states are far from
        # the near-cancellations of a hydrostatic balance: S_c/max|out_c| < 50)
        plain = np.max(np.abs(got - ref_d), axis=1) / np.max(np.abs(ref_d), axis=1)
        assert plain.max() <= 1e-14, (form, plain)
        # the long double oracle on the same inputs: tighter still
        Jl_a, _ = oracle.metrics(1, 1, X[0].copy(), X[1].copy(), X[2].copy(), real="ld")
        got_ld = oracle.volume(1, 1, q.copy(), Jl_a, phi.copy(), gamma=GAMMA, form=form, real="ld")
        diff = np.array([[float(mp.mpf(str(got_ld[c, i])) - ref[c][i]) for i in range(8)] for c in range(5)])
        e_ld = np.max(np.abs(diff), axis=1) / S_d
        assert e_ld.max() <= 1e-17, (form, e_ld)


def test_bruteforce_is_not_trivially_satisfied():
    """The comparison above can fail: a flux with the gravity term on the
    wrong side (b_m in place of b_i, Eq. 5) moves the brute force away from
    the oracle by far more than the tolerance."""
    rng = np.random.default_rng(13)
    X = _element(rng, True)
    q, phi = _state(rng, X)
    Xm = [[mp.mpf(float(v)) for v in X[d]] for d in range(3)]
    Jam, _ = metrics_mp(Xm)
    qm = [[mp.mpf(float(v)) for v in q[c]] for c in range(5)]
    phim = [mp.mpf(float(v)) for v in phi]
    ref, S = volume_mp(qm, phim, Jam)
    bad, _ = volume_mp(qm, phim, Jam, gravity_side="m")
    e = max(abs(float(bad[c][i] - ref[c][i])) / float(S[c]) for c in range(5) for i in range(8))
    assert e > 1e-8
