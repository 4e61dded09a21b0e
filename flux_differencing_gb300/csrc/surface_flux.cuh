// Interface flux of the surface term, shared by the face-centric surface
// kernel (surface_kernel.cu) and the FP32 Runge-Kutta stage, which evaluates
// each element's faces from its own side inside the volume kernel.
//
// F* = F_ec(q_i, q_j) . n + G(i, j) . n - D: the entropy-conserving two-point
// flux with the gravity term (Eqs. 3-5 of "GPU Performance of an
// Entropy-Stable Discontinuous Galerkin Euler Solver with Non-Conservative
// Terms") minus the matrix dissipation 1/2 |n| R |Lambda| T R^T [[w]]
// (Sec. 3), evaluated at the averaged state.  Because F_ec is symmetric and
// R |Lambda| R^-1 = |A(n^)| is even in n^, the flux of node j with the normal
// -n is -F_ec . n + D + G(i,j) b_i/b_j: evaluating the face from either side
// gives the same two contributions up to rounding.
#pragma once

#include <cuda_runtime.h>

#include <type_traits>

#include "esdg_internal.h"
#include "numeric.cuh"

namespace esdg {

__device__ __forceinline__ double sqrt_(double x) { return sqrt(x); }
__device__ __forceinline__ float sqrt_(float x) { return sqrtf(x); }
__device__ __forceinline__ ff sqrt_(ff x) { return ff_sqrt(x); }
// logarithms of the (rare) far-pair path: CUDA's log in FP64, whose compact
// code keeps the surface kernel's registers (the volume kernel's inlined
// table log, four copies here, raised them from 122 to 138 and halved the
// occupancy)
__device__ __forceinline__ double far_log(double x) { return log(x); }
__device__ __forceinline__ float far_log(float x) { return Num<float>::log_(x); }
__device__ __forceinline__ ff far_log(ff x) { return Num<ff>::log_(x); }


template <typename C>
struct FaceNode {
    C rho, u1, u2, u3, uu, E, p, b, ib, phi;
};

// Node state from the conserved variables; with a reference state (perturbed),
// rho and E are perturbations from (rho_ref, E_ref = p_ref/(gamma-1) +
// rho_ref phi) and p = p_ref + (gamma-1)(E' - rho|u|^2/2 - rho' phi).
template <typename C>
__device__ __forceinline__ FaceNode<C> node_state(C rho_in, C m1, C m2, C m3, C E_in, C phi, C gm1, bool perturbed,
                                                  C rho_ref, C p_ref) {
    FaceNode<C> s;
    const C rho = perturbed ? rho_ref + rho_in : rho_in;
    const C irho = Num<C>::rcp_pair(rho);
    s.rho = rho;
    s.u1 = m1 * irho;
    s.u2 = m2 * irho;
    s.u3 = m3 * irho;
    s.uu = fma(s.u3, s.u3, fma(s.u2, s.u2, s.u1 * s.u1));
    if (perturbed) {
        s.p = fma(gm1, E_in - fma(C(0.5) * rho, s.uu, rho_in * phi), p_ref);
        s.E = fma(s.p, Num<C>::rcp(gm1), rho * fma(C(0.5), s.uu, phi));
    } else {
        s.E = E_in;
        s.p = gm1 * (E_in - rho * fma(C(0.5), s.uu, phi));
    }
    s.b = C(0.5) * rho * Num<C>::rcp_pair(s.p);
    s.ib = C(2.0) * s.p * irho;  // 1/b
    s.phi = phi;
    return s;
}

// physical flux f(q) . n of Eq. 1, accumulated with sign c (+-1) into o
template <typename C>
__device__ __forceinline__ void add_phys_flux(const FaceNode<C>& s, C n0, C n1, C n2, C c, C (&o)[5]) {
    const C un = c * fma(s.u3, n2, fma(s.u2, n1, s.u1 * n0));
    const C ru = s.rho * un;
    const C cp = c * s.p;
    o[0] = o[0] + ru;
    o[1] = fma(ru, s.u1, fma(cp, n0, o[1]));
    o[2] = fma(ru, s.u2, fma(cp, n1, o[2]));
    o[3] = fma(ru, s.u3, fma(cp, n2, o[3]));
    o[4] = fma(un, s.E + s.p, o[4]);
}

template <typename C>
struct Consts {
    C gm1, igm1, c_g, gamma, c_ac, c_en;
};

// 2 atanh(f)/f = 2 (1 + u/3 + u^2/5 + u^3/7) + O(u^4), u = f^2
template <typename C>
__device__ __forceinline__ C atanh_ratio(C u) {
    return fma(u, fma(u, fma(u, C(2.0 / 7.0), C(2.0 / 5.0)), C(2.0 / 3.0)), C(2.0));
}

// The interface flux between node i ("-", owning the normal n) and node j
// ("+").  Returns F_ec + G(i,j) - D for node i in fi and the far node's
// -F_ec + D + G(i,j) b_i/b_j in fj (its flux with the normal -n).
template <typename C>
__device__ __forceinline__ void interface_flux(const FaceNode<C>& I, const FaceNode<C>& J, C n0, C n1, C n2,
                                               const Consts<C>& k, bool dissipation, C (&fi)[5], C (&fj)[5]) {
    const C a1 = C(0.5) * (I.u1 + J.u1), a2 = C(0.5) * (I.u2 + J.u2), a3 = C(0.5) * (I.u3 + J.u3);
    const C U = fma(a3, n2, fma(a2, n1, a1 * n0));
    const C phib = C(0.5) * (I.phi + J.phi);

    // log means and log jumps of rho and b, with f = (a+ - a-)/(a+ + a-), u = f^2:
    //   {{a}}_log = {{a}} (1 - u/3 - 4u^2/45 - 44u^3/945) + O(u^4),
    //   [[ln a]] = 2 atanh(f),  1/{{a}}_log = [[ln a]]/[[a]] = atanh_ratio(u)/(a+ + a-)
    const C rsum = I.rho + J.rho, drho = J.rho - I.rho;
    const C irs = Num<C>::rcp_pair(rsum);
    const C fr = drho * irs;
    const C ur = fr * fr;
    const C bsum = I.b + J.b, db = J.b - I.b;
    const C ibs = Num<C>::rcp_pair(bsum);
    const C fb = db * ibs;
    const C ub = fb * fb;
    const bool cr = Num<C>::close_ratio(fr), cb = Num<C>::close_ratio(fb);
    const C polr = fma(ur, fma(ur, fma(ur, C(-22.0 / 945.0), C(-2.0 / 45.0)), C(-1.0 / 6.0)), C(0.5));
    const C polb = atanh_ratio(ub);
    C rho_ln = rsum * polr;
    C inv_bln = ibs * polb;
    C dlr = fr * atanh_ratio(ur);
    C dlb = fb * polb;
    if (!__all_sync(__activemask(), cr && cb)) {
        // a far pair in this warp: logarithms for all its lanes, selected per lane
        const C lr = far_log(J.rho) - far_log(I.rho);
        const C lb = far_log(J.b) - far_log(I.b);
        rho_ln = sel(cr, rho_ln, drho * Num<C>::rcp_pair(sel(cr, C(1.0), lr)));
        inv_bln = sel(cb, inv_bln, lb * Num<C>::rcp_pair(sel(cb, C(1.0), db)));
        dlr = sel(cr, dlr, lr);
        dlb = sel(cb, dlb, lb);
    }

    // entropy-conserving flux (Eqs. 3-4) and the gravity term (Eq. 5)
    const C p_hat = C(0.5) * rsum * ibs;  // {{rho}}/(2{{b}})
    const C Fr = rho_ln * U;
    const C aa = fma(a3, a3, fma(a2, a2, a1 * a1));
    const C uu_avg = C(0.5) * (I.uu + J.uu);
    const C FE = fma(Fr, fma(k.c_g, inv_bln, fma(C(-0.5), uu_avg, phib + aa)), U * p_hat);
    // G(i,j) = 1/2 rho_ln {{b}} (phi_j - phi_i)/b_i n;  the far side's is G(i,j) b_i/b_j
    const C gq = C(0.25) * rho_ln * bsum * (J.phi - I.phi);
    const C gi = gq * I.ib;
    const C gj = gq * J.ib;

    C D0 = C(0.0), D1 = C(0.0), D2 = C(0.0), D3 = C(0.0), D4 = C(0.0);
    if (dissipation) {
        // averaged state: sound speed and total enthalpy; |n| and 1/|n|.  FP64
        // takes both square roots from reciprocal square roots (an FP32
        // estimate and one Newton step, Num<double>::rsqrt_pair).
        const C a_sq = k.gamma * p_hat * Num<C>::rcp_pair(rho_ln);
        const C nsq = fma(n2, n2, fma(n1, n1, n0 * n0));
        C a, nn, inn;
        if constexpr (std::is_same<C, double>::value) {
            a = a_sq * Num<C>::rsqrt_pair(a_sq);
            inn = Num<C>::rsqrt_pair(nsq);
            nn = nsq * inn;
        } else {
            a = sqrt_(a_sq);
            nn = sqrt_(nsq);
            inn = Num<C>::rcp(nn);
        }
        const C a_sq_g = a_sq * k.igm1;  // a^2/(gamma-1)
        const C ke = fma(C(0.5), aa, phib);  // |u|^2/2 + phi
        const C H = a_sq_g + ke;
        // [[w]] for w = ((gamma-s)/(gamma-1) - b|u|^2 + 2 b phi, 2 b u, -2 b),
        // [[s]] = (1 - gamma)[[ln rho]] - [[ln b]]
        const C d1 = fma(dlb, k.igm1, dlr) - (J.b * fma(C(-2.0), J.phi, J.uu) - I.b * fma(C(-2.0), I.phi, I.uu));
        const C dm1 = C(2.0) * (J.b * J.u1 - I.b * I.u1);
        const C dm2 = C(2.0) * (J.b * J.u2 - I.b * I.u2);
        const C dm3 = C(2.0) * (J.b * J.u3 - I.b * I.u3);
        const C d5 = C(-2.0) * db;
        // shear input v = [[w_m]] + u [[w_5]] and its normal part
        const C v1 = fma(a1, d5, dm1), v2 = fma(a2, d5, dm2), v3 = fma(a3, d5, dm3);
        const C vn = fma(v3, n2, fma(v2, n1, v1 * n0));  // n . v (n unnormalised)
        const C inn2 = inn * inn;
        // wave strengths
        const C beta = fma(H, d5, fma(a3, dm3, fma(a2, dm2, fma(a1, dm1, d1))));
        const C alpha_e = fma(-a_sq_g, d5, beta);
        // the dissipation's factor 1/2 is carried by c_ac, c_en (halved
        // constants) and ls, so the wave strengths below are already halved
        const C anu = a * vn * inn;
        const C rc = rho_ln * k.c_ac;
        const C lam_p = fabs(fma(a, nn, U)) * rc;
        const C lam_m = fabs(fma(-a, nn, U)) * rc;
        const C aU = fabs(U);
        const C cp_ = lam_p * (beta + anu);
        const C cm_ = lam_m * (beta - anu);
        const C ce = aU * rho_ln * k.c_en * alpha_e;
        const C ls = aU * (C(0.5) * p_hat);
        const C csum = cp_ + cm_;
        const C cdif = (cp_ - cm_) * a * inn;
        const C c0 = csum + ce;
        const C svn = ls * vn * inn2;
        D0 = c0;
        D1 = fma(c0, a1, fma(cdif, n0, ls * v1)) - svn * n0;
        D2 = fma(c0, a2, fma(cdif, n1, ls * v2)) - svn * n1;
        D3 = fma(c0, a3, fma(cdif, n2, ls * v3)) - svn * n2;
        const C uv = fma(a3, v3, fma(a2, v2, a1 * v1));
        D4 = fma(csum, H, fma(cdif, U, fma(ce, ke, ls * uv))) - svn * U;
    }

    // momentum: F_rho {{u}} + p_hat n (+ gravity, scaled per side)
    const C m1 = fma(Fr, a1, p_hat * n0), m2 = fma(Fr, a2, p_hat * n1), m3 = fma(Fr, a3, p_hat * n2);
    fi[0] = Fr - D0;
    fi[1] = fma(gi, n0, m1) - D1;
    fi[2] = fma(gi, n1, m2) - D2;
    fi[3] = fma(gi, n2, m3) - D3;
    fi[4] = FE - D4;
    fj[0] = D0 - Fr;
    fj[1] = fma(gj, n0, D1 - m1);
    fj[2] = fma(gj, n1, D2 - m2);
    fj[3] = fma(gj, n2, D3 - m3);
    fj[4] = D4 - FE;
}

}  // namespace esdg
