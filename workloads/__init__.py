"""Seeded synthetic inputs for the flux-differencing volume term.

This module is shared by the CUDA path's tests and bench and by the CPU
oracle's tests.  It holds none of the volume term's arithmetic: it only places
mesh nodes and evaluates analytic initial states at those nodes.  Everything is
a deterministic function of a config and its seed.

Layout produced (the library's layout):
  * element e = ex + Kx*(ey + Ky*ez)
  * node      = a + Nq*(b + Nq*c), a runs along the first reference direction
  * a field of n = K*Nq^3 nodes is a flat array indexed e*Nq^3 + node
  * q is (5, n) in the order (rho, rho*u1, rho*u2, rho*u3, E)

Node positions on the reference interval come from numpy's Legendre routines
(the roots of P_N' plus the end points); they only decide where the mesh is
sampled.  The method's own LGL nodes, weights and derivative matrix are built
independently by the library and by the oracle.

State recipes follow the test problems of "GPU Performance of an
Entropy-Stable Discontinuous Galerkin Euler Solver with Non-Conservative
Terms": the rising thermal bubble (Sec. 5.1, Eq. 9 cosine bubble) and the
baroclinic channel (Sec. 5.2).  The channel's published initial condition is
not printed on that page, so the channel state here is a balanced-jet stand-in
with the stated domain and jet speed.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

GAMMA = 1.4
GRAV = 9.81
R_D = 287.0
C_P = GAMMA * R_D / (GAMMA - 1.0)  # 1004.5
P0 = 1.0e5

__all__ = [
    "GAMMA", "GRAV", "R_D", "C_P", "P0",
    "Config", "CONFIGS", "get_config", "small_config", "node_positions",
    "generate", "generate_elements", "element_subset", "reference_state",
]


def node_positions(N: int) -> np.ndarray:
    """Positions of the N+1 Gauss-Lobatto points on [-1, 1] (numpy library routine)."""
    from numpy.polynomial import legendre as leg

    c = np.zeros(N + 1)
    c[N] = 1.0
    inner = np.sort(leg.legroots(leg.legder(c)).real) if N >= 2 else np.zeros(0)
    return np.concatenate([[-1.0], inner, [1.0]])


@dataclasses.dataclass(frozen=True)
class Config:
    name: str
    N: int
    Kx: int
    Ky: int
    Kz: int
    precision: str          # "fp64" or "fp32"
    state: str              # "box", "bubble", "channel", "random", "noisy" (random + per-node jumps)
    domain: tuple           # (Lx, Ly, Lz), origin at 0
    warp: bool
    seed: int
    description: str = ""
    # surface term only: per reference direction 0 = periodic, 1 = slip wall
    bc: tuple = (0, 0, 0)

    @property
    def Nq(self) -> int:
        return self.N + 1

    @property
    def K(self) -> int:
        return self.Kx * self.Ky * self.Kz

    @property
    def n(self) -> int:
        return self.K * self.Nq ** 3


def _seed(cfg_index: int, N: int) -> int:
    return 20261202 + 10 * cfg_index + N


def _sweep_K(N: int) -> int:
    # elements per dimension so that K*(N+1)^3 is about 6.4e7 nodes
    return {1: 200, 2: 133, 3: 100, 4: 80, 5: 67, 6: 57, 7: 50, 8: 44}[N]


def _make_configs() -> dict:
    cfgs = {}
    cfgs["tiny_box_N3"] = Config(
        "tiny_box_N3", 3, 4, 4, 4, "fp64", "box", (1000.0, 1000.0, 1000.0), False, _seed(1, 3),
        "4x4x4 affine periodic box, N=3, constant state plus 1% smooth perturbations")
    cfgs["bubble_N4"] = Config(
        "bubble_N4", 4, 16, 16, 16, "fp64", "bubble", (1000.0, 1000.0, 1000.0), False, _seed(2, 4),
        "1000 m box, 16^3 affine elements, N=4, hydrostatic background + 0.5 K cosine bubble",
        (1, 1, 1))
    cfgs["channel_N7"] = Config(
        "channel_N7", 7, 64, 16, 8, "fp64", "channel", (4.0e7, 6.0e6, 3.0e4), True, _seed(3, 7),
        "40000x6000x30 km channel, 64x16x8 warped elements, N=7, balanced jet + 1 K bump",
        (0, 1, 1))
    cfgs["channel_N7_fp32"] = dataclasses.replace(
        cfgs["channel_N7"], name="channel_N7_fp32", precision="fp32",
        description="channel_N7 with FP32 state, metrics and geopotential")
    cfgs["channel_N7_ff"] = dataclasses.replace(
        cfgs["channel_N7"], name="channel_N7_ff", precision="fp64ff",
        description="channel_N7 with FP64 buffers and float-float pair arithmetic")
    for N in range(2, 9):
        k = _sweep_K(N)
        for prec in ("fp64", "fp32", "fp64ff"):
            nm = f"sweep_N{N}" + {"fp64": "", "fp32": "_fp32", "fp64ff": "_ff"}[prec]
            cfgs[nm] = Config(
                nm, N, k, k, k, prec, "random", (1.0e4, 1.0e4, 1.0e4), True, _seed(5, N),
                f"warped periodic 10 km cube, {k}^3 elements, N={N}, about 6.4e7 nodes")
    return cfgs


CONFIGS = _make_configs()


def get_config(name: str) -> Config:
    return CONFIGS[name]


def small_config(N: int, K=(2, 2, 2), warp=True, state="random", seed=None,
                 precision="fp64", domain=(1.0e4, 1.0e4, 1.0e4), bc=(0, 0, 0)) -> Config:
    """A small mesh of any order for parity sweeps (several tiles, ragged counts)."""
    Kx, Ky, Kz = K
    s = seed if seed is not None else _seed(9, N) + 1000 * (Kx + 7 * Ky + 49 * Kz)
    return Config(f"small_N{N}_{Kx}x{Ky}x{Kz}_{state}{'_warp' if warp else ''}",
                  N, Kx, Ky, Kz, precision, state, tuple(domain), warp, s, "", tuple(bc))


# ----------------------------------------------------------------------------
# mesh

def _reference_coords(cfg: Config, elems: torch.Tensor, device) -> tuple:
    """Undeformed node coordinates, each of shape (len(elems), Nq^3)."""
    Nq = cfg.Nq
    xi = torch.tensor(node_positions(cfg.N), dtype=torch.float64, device=device)
    ex = elems % cfg.Kx
    ey = (elems // cfg.Kx) % cfg.Ky
    ez = elems // (cfg.Kx * cfg.Ky)
    hx = cfg.domain[0] / cfg.Kx
    hy = cfg.domain[1] / cfg.Ky
    hz = cfg.domain[2] / cfg.Kz
    node = torch.arange(Nq ** 3, device=device)
    a = node % Nq
    b = (node // Nq) % Nq
    c = node // (Nq * Nq)
    # position inside the element in units of elements: index + (xi+1)/2
    fx = ex[:, None].to(torch.float64) + 0.5 * (xi[a][None, :] + 1.0)
    fy = ey[:, None].to(torch.float64) + 0.5 * (xi[b][None, :] + 1.0)
    fz = ez[:, None].to(torch.float64) + 0.5 * (xi[c][None, :] + 1.0)
    return fx, fy, fz, (hx, hy, hz)


def _warp_params(cfg: Config, rng: np.random.Generator) -> dict:
    # wavelength about 4 elements, rounded so it divides the mesh (periodic)
    lam = []
    for K in (cfg.Kx, cfg.Ky, cfg.Kz):
        waves = max(1, int(round(K / 4.0)))
        lam.append(K / waves)
    phases = rng.uniform(0.0, 2.0 * math.pi, size=(3, 3))
    return {"lam": lam, "phases": phases, "amp": 0.05}


def _mesh(cfg: Config, elems: torch.Tensor, device, rng_draws: dict) -> tuple:
    fx, fy, fz, (hx, hy, hz) = _reference_coords(cfg, elems, device)
    if cfg.warp:
        wp = rng_draws["warp"]
        lam = wp["lam"]
        ph = wp["phases"]
        amp = wp["amp"]
        disp = []
        for j in range(3):
            s = (torch.sin(2 * math.pi * fx / lam[0] + ph[j, 0])
                 * torch.sin(2 * math.pi * fy / lam[1] + ph[j, 1])
                 * torch.sin(2 * math.pi * fz / lam[2] + ph[j, 2]))
            disp.append(amp * s)
        fx = fx + disp[0]
        fy = fy + disp[1]
        fz = fz + disp[2]
    return fx * hx, fy * hy, fz * hz


# ----------------------------------------------------------------------------
# states

def _smooth_field_params(rng: np.random.Generator, nmodes: int = 6) -> dict:
    return {
        "amp": rng.uniform(0.5, 1.0, size=nmodes),
        "k": rng.integers(1, 4, size=(nmodes, 3)),
        "phase": rng.uniform(0.0, 2.0 * math.pi, size=nmodes),
    }


def _smooth_field(p: dict, X, Y, Z, domain) -> torch.Tensor:
    """Sum of periodic sine modes scaled so that |s| <= 1 everywhere."""
    s = torch.zeros_like(X)
    for a, k, th in zip(p["amp"], p["k"], p["phase"]):
        arg = 2 * math.pi * (k[0] * X / domain[0] + k[1] * Y / domain[1] + k[2] * Z / domain[2]) + th
        s = s + float(a) * torch.sin(arg)
    return s / float(np.sum(np.abs(p["amp"])))


def _draws(cfg: Config) -> dict:
    """Every random number a config uses, drawn once in a fixed order."""
    rng = np.random.default_rng(cfg.seed)
    d = {"warp": _warp_params(cfg, rng)}
    d["fields"] = [_smooth_field_params(rng) for _ in range(5)]
    d["bump"] = {
        "xc": rng.uniform(0.2, 0.8), "yc": rng.uniform(0.3, 0.7), "zc": rng.uniform(0.2, 0.5),
    }
    d["noise_seed"] = int(rng.integers(0, 2 ** 31 - 1))
    return d


def _energy(rho, u1, u2, u3, p, phi):
    return p / (GAMMA - 1.0) + 0.5 * rho * (u1 * u1 + u2 * u2 + u3 * u3) + rho * phi


def _state(cfg: Config, X, Y, Z, draws: dict, elems: torch.Tensor):
    dom = cfg.domain
    f = draws["fields"]
    if cfg.state == "box":
        u0 = (10.0, 5.0, -3.0)
        umag = math.sqrt(sum(v * v for v in u0))
        rho = 1.2 * (1.0 + 0.01 * _smooth_field(f[0], X, Y, Z, dom))
        u1 = u0[0] + 0.01 * umag * _smooth_field(f[1], X, Y, Z, dom)
        u2 = u0[1] + 0.01 * umag * _smooth_field(f[2], X, Y, Z, dom)
        u3 = u0[2] + 0.01 * umag * _smooth_field(f[3], X, Y, Z, dom)
        p = 1.0e5 * (1.0 + 0.01 * _smooth_field(f[4], X, Y, Z, dom))
    elif cfg.state in ("random", "noisy"):
        rho = 1.0 + 0.05 * _smooth_field(f[0], X, Y, Z, dom)
        p = 1.0e5 * (1.0 + 0.05 * _smooth_field(f[1], X, Y, Z, dom))
        u1 = 20.0 * _smooth_field(f[2], X, Y, Z, dom)
        u2 = 20.0 * _smooth_field(f[3], X, Y, Z, dom)
        u3 = 20.0 * _smooth_field(f[4], X, Y, Z, dom)
        if cfg.state == "noisy":
            # independent per-node perturbations: states jump across element faces
            g = torch.Generator(device="cpu")
            g.manual_seed(draws["noise_seed"])
            full = 2.0 * torch.rand((5, cfg.K, cfg.Nq ** 3), generator=g, dtype=torch.float64) - 1.0
            xi = full[:, elems.cpu(), :].to(X.device)
            rho = rho * (1.0 + 0.02 * xi[0])
            p = p * (1.0 + 0.02 * xi[1])
            u1 = u1 + 2.0 * xi[2]
            u2 = u2 + 2.0 * xi[3]
            u3 = u3 + 2.0 * xi[4]
    elif cfg.state == "bubble":
        theta0 = 300.0
        exner = 1.0 - GRAV * Z / (C_P * theta0)
        p = P0 * exner ** (C_P / R_D)
        xc, yc, zc, rc = 0.5 * dom[0], 0.5 * dom[1], 350.0, 250.0
        r = torch.sqrt((X - xc) ** 2 + (Y - yc) ** 2 + (Z - zc) ** 2)
        dtheta = torch.where(r <= rc, 0.25 * (1.0 + torch.cos(math.pi * r / rc)), torch.zeros_like(r))
        theta = theta0 + dtheta
        rho = p / (R_D * theta * exner)
        # velocity: zero plus 1e-6 uniform noise per node and component
        g = torch.Generator(device="cpu")
        g.manual_seed(draws["noise_seed"])
        full = 1e-6 * (2.0 * torch.rand((3, cfg.K, cfg.Nq ** 3), generator=g, dtype=torch.float64) - 1.0)
        sel = full[:, elems.cpu(), :].to(X.device)
        u1, u2, u3 = sel[0], sel[1], sel[2]
    elif cfg.state == "channel":
        theta0, nbv, f0, ujet = 300.0, 0.01, 1.0e-4, 35.0
        Ly, zt = dom[1], dom[2]
        ez = torch.exp(-nbv * nbv * Z / GRAV)
        exner = 1.0 + GRAV * GRAV / (C_P * theta0 * nbv * nbv) * (ez - 1.0)
        theta_b = theta0 / ez
        # jet and its thermal-wind temperature gradient: f0 du/dz = -(g/theta0) dtheta/dy
        sz = torch.sin(math.pi * Z / (2.0 * zt))
        cz = torch.cos(math.pi * Z / (2.0 * zt))
        sy = torch.sin(math.pi * Y / Ly)
        u1 = ujet * sy * sy * sz
        int_sy2 = 0.5 * Y - Ly * torch.sin(2.0 * math.pi * Y / Ly) / (4.0 * math.pi)
        theta_tw = -(f0 * theta0 / GRAV) * ujet * (math.pi / (2.0 * zt)) * cz * int_sy2
        bp = draws["bump"]
        xc, yc, zcb = bp["xc"] * dom[0], bp["yc"] * dom[1], bp["zc"] * dom[2]
        bump = torch.exp(-((X - xc) ** 2 + (Y - yc) ** 2) / (5.0e5 ** 2) - (Z - zcb) ** 2 / (5.0e3 ** 2))
        theta = theta_b + theta_tw + bump
        p = P0 * exner ** (C_P / R_D)
        rho = p / (R_D * theta * exner)
        u2 = torch.zeros_like(u1)
        u3 = torch.zeros_like(u1)
    else:
        raise ValueError(cfg.state)
    phi = GRAV * Z
    E = _energy(rho, u1, u2, u3, p, phi)
    q = torch.stack([rho, rho * u1, rho * u2, rho * u3, E])
    return q, phi


def generate_elements(cfg: Config, elems, device="cpu") -> dict:
    """Inputs for the listed elements only (bit-identical to the same slice of generate())."""
    elems = torch.as_tensor(elems, dtype=torch.int64, device=device)
    draws = _draws(cfg)
    X, Y, Z = _mesh(cfg, elems, device, draws)
    q, phi = _state(cfg, X, Y, Z, draws, elems)
    return {
        "x": X.reshape(-1), "y": Y.reshape(-1), "z": Z.reshape(-1),
        "q": q.reshape(5, -1), "phi": phi.reshape(-1),
    }


def generate(cfg: Config, device="cpu", chunk_elems: int = 1 << 16) -> dict:
    """All inputs of a config in float64 on `device` (chunked to bound temporaries)."""
    n_per = cfg.Nq ** 3
    out = {
        "x": torch.empty(cfg.n, dtype=torch.float64, device=device),
        "y": torch.empty(cfg.n, dtype=torch.float64, device=device),
        "z": torch.empty(cfg.n, dtype=torch.float64, device=device),
        "q": torch.empty((5, cfg.n), dtype=torch.float64, device=device),
        "phi": torch.empty(cfg.n, dtype=torch.float64, device=device),
    }
    for e0 in range(0, cfg.K, chunk_elems):
        e1 = min(cfg.K, e0 + chunk_elems)
        part = generate_elements(cfg, torch.arange(e0, e1), device=device)
        sl = slice(e0 * n_per, e1 * n_per)
        for key in ("x", "y", "z", "phi"):
            out[key][sl] = part[key]
        out["q"][:, sl] = part["q"]
    return out


def reference_state(cfg: Config, device="cpu", chunk_elems: int = 1 << 16) -> dict:
    """The hydrostatic background of a workload at its nodes, float64:
    {"rho_ref": (n,), "p_ref": (n,)}.

    bubble: the theta0 = 300 K neutral atmosphere the bubble sits in;
    channel: the stratified background theta_b(z) with its Exner function
    (no jet, no thermal-wind correction, no bump).  Other states have no
    hydrostatic background and get rho_ref = 1, p_ref = 1e5."""
    out = {"rho_ref": torch.empty(cfg.n, dtype=torch.float64, device=device),
           "p_ref": torch.empty(cfg.n, dtype=torch.float64, device=device)}
    n_per = cfg.Nq ** 3
    draws = _draws(cfg)
    for e0 in range(0, cfg.K, chunk_elems):
        e1 = min(cfg.K, e0 + chunk_elems)
        elems = torch.arange(e0, e1, device=device)
        _, _, Z = _mesh(cfg, elems, device, draws)
        if cfg.state == "bubble":
            theta0 = 300.0
            exner = 1.0 - GRAV * Z / (C_P * theta0)
            p = P0 * exner ** (C_P / R_D)
            rho = p / (R_D * theta0 * exner)
        elif cfg.state == "channel":
            theta0, nbv = 300.0, 0.01
            ez = torch.exp(-nbv * nbv * Z / GRAV)
            exner = 1.0 + GRAV * GRAV / (C_P * theta0 * nbv * nbv) * (ez - 1.0)
            p = P0 * exner ** (C_P / R_D)
            rho = p / (R_D * (theta0 / ez) * exner)
        else:
            rho = torch.ones_like(Z)
            p = torch.full_like(Z, 1.0e5)
        sl = slice(e0 * n_per, e1 * n_per)
        out["rho_ref"][sl] = rho.reshape(-1)
        out["p_ref"][sl] = p.reshape(-1)
    return out


def element_subset(cfg: Config, count: int, seed: int = 7) -> np.ndarray:
    """A reproducible sample of element indices, always including the first and last."""
    rng = np.random.default_rng(seed + cfg.seed)
    pick = rng.choice(cfg.K, size=min(count, cfg.K), replace=False)
    return np.unique(np.concatenate([[0, cfg.K - 1], pick]))
