// Surface-flux kernel for sm_103a: the surface term of Eq. 2 of "GPU
// Performance of an Entropy-Stable Discontinuous Galerkin Euler Solver with
// Non-Conservative Terms" (Sec. 3), added into the volume term's output.
//
// What it computes: at every face node i of every element, with j the node
// across the face (or a mirror ghost at a slip wall),
//     out_i += (1/w_0) [ F*(q_i, q_j; n) - delta_2D f(q_i) . n_own ]
// where n = +-(Ja^r(i) + Ja^r(j))/2 is the outward averaged normal, n_own =
// +-Ja^r(i), and F* is the entropy-conserving two-point flux with the gravity
// term (Eqs. 3-5) minus the matrix dissipation 1/2 |n| R |Lambda| T R^T [[w]]
// (Sec. 3: a Roe-type diagonalisation evaluated at the averaged state rho_ln,
// {{u}}, p_hat = {{rho}}/(2{{b}}), {{phi}}; [[w]] the jump of the entropy
// variables).  The 2D (strong) volume form keeps the physical flux on its
// diagonal, so the surface subtracts it; the skew form adds F* alone.
//
// How (GB300 design):
//  * Face-centric: one thread per interface node evaluates F* once and feeds
//    both elements -- the far side receives -F_ec + D plus the gravity term
//    scaled by b_i/b_j (the partner rule of the volume term, Sec. 4.1).  One
//    launch per reference direction: within a direction every node lies on
//    at most one face, so the read-modify-write of `out` never races and the
//    summation order is fixed (bitwise deterministic).
//  * Consecutive threads take consecutive face nodes of one element face, so
//    zeta faces read contiguous runs of (N+1)^2 nodes and eta faces runs of
//    N+1; xi faces gather with stride N+1.
//  * The dissipation is formed without tangent vectors: the two shear waves
//    share the eigenvalue u.n, so together they are the projection
//    (I - n^ n^T) onto the face, and the acoustic pair enters through the
//    sum and difference of its two wave strengths.
//  * Reciprocals, logarithms and log means use the volume kernel's numerics.
#include <cuda_runtime.h>

#include "esdg_internal.h"
#include "volume_kernel.cuh"

namespace esdg {

__device__ __forceinline__ double sqrt_(double x) { return sqrt(x); }
__device__ __forceinline__ float sqrt_(float x) { return sqrtf(x); }

namespace {

template <typename T>
struct FaceNode {
    T rho, u1, u2, u3, uu, E, p, b, lr, lb, phi;
};

template <typename T>
__device__ __forceinline__ FaceNode<T> node_state(T rho, T m1, T m2, T m3, T E, T phi, T gm1) {
    FaceNode<T> s;
    const T irho = Num<T>::rcp(rho);
    s.rho = rho;
    s.u1 = m1 * irho;
    s.u2 = m2 * irho;
    s.u3 = m3 * irho;
    s.uu = fma(s.u3, s.u3, fma(s.u2, s.u2, s.u1 * s.u1));
    s.E = E;
    s.p = gm1 * (E - rho * fma(T(0.5), s.uu, phi));
    s.b = T(0.5) * rho * Num<T>::rcp(s.p);
    s.lr = Num<T>::log_(rho);
    s.lb = Num<T>::log_(s.b);
    s.phi = phi;
    return s;
}

// physical flux f(q) . n of Eq. 1, accumulated with weight c into o
template <typename T>
__device__ __forceinline__ void add_phys_flux(const FaceNode<T>& s, T n0, T n1, T n2, T c, T (&o)[5]) {
    const T un = fma(s.u3, n2, fma(s.u2, n1, s.u1 * n0));
    const T ru = c * s.rho * un;
    const T cp = c * s.p;
    o[0] = fma(c, s.rho * un, o[0]);
    o[1] = fma(ru, s.u1, fma(cp, n0, o[1]));
    o[2] = fma(ru, s.u2, fma(cp, n1, o[2]));
    o[3] = fma(ru, s.u3, fma(cp, n2, o[3]));
    o[4] = fma(c * un, s.E + s.p, o[4]);
}

// The interface flux between node i ("-", owning the normal n) and node j
// ("+").  Returns F_ec + G(i,j) - D for node i in fi and the far node's
// -F_ec + D + G(i,j) b_i/b_j in fj (its flux with the normal -n).
template <typename T>
__device__ __forceinline__ void interface_flux(const FaceNode<T>& I, const FaceNode<T>& J, T n0, T n1, T n2,
                                               const SurfaceConsts<T>& k, bool dissipation,
                                               T (&fi)[5], T (&fj)[5]) {
    // averages
    const T a1 = T(0.5) * (I.u1 + J.u1), a2 = T(0.5) * (I.u2 + J.u2), a3 = T(0.5) * (I.u3 + J.u3);
    const T U = fma(a3, n2, fma(a2, n1, a1 * n0));
    const T rsum = I.rho + J.rho;
    const T bsum = I.b + J.b;
    const T phib = T(0.5) * (I.phi + J.phi);

    // {{rho}}_log: (rho+ - rho-)/(ln rho+ - ln rho-), or the series when close
    const T dlr = J.lr - I.lr;
    const bool cr = Num<T>::close(dlr);
    const T rr = Num<T>::rcp(sel(cr, rsum, dlr));
    const T tr = (J.rho - I.rho) * rr;
    const T ur = tr * tr;
    const T polr = fma(ur, fma(ur, fma(ur, T(-22.0 / 945.0), T(-2.0 / 45.0)), T(-1.0 / 6.0)), T(0.5));
    const T rho_ln = sel(cr, rsum * polr, tr);

    // 1/{{b}}_log and 1/(b+ + b-) from one reciprocal
    const T db = J.b - I.b;
    const T dlb = J.lb - I.lb;
    const bool cb = Num<T>::close(dlb);
    const T rb = Num<T>::rcp(sel(cb, bsum, db * bsum));
    const T inv_bsum = sel(cb, rb, db * rb);
    const T fb = db * inv_bsum;
    const T ub = fb * fb;
    const T polb = fma(ub, fma(ub, fma(ub, T(2.0 / 7.0), T(2.0 / 5.0)), T(2.0 / 3.0)), T(2.0));
    const T inv_bln = sel(cb, inv_bsum * polb, dlb * (bsum * rb));

    // entropy-conserving flux (Eqs. 3-4) and the gravity term (Eq. 5)
    const T p_hat = T(0.5) * rsum * inv_bsum;  // {{rho}}/(2{{b}})
    const T Fr = rho_ln * U;
    const T aa = fma(a3, a3, fma(a2, a2, a1 * a1));
    const T uu_avg = T(0.5) * (I.uu + J.uu);
    const T FE = fma(Fr, fma(k.c_g, inv_bln, fma(T(-0.5), uu_avg, phib + aa)), U * p_hat);
    // G(i,j) = 1/2 rho_ln {{b}} (phi_j - phi_i)/b_i n
    const T gq = T(0.25) * rho_ln * bsum * (J.phi - I.phi);
    const T gi = gq * Num<T>::rcp(I.b);
    const T gj = gq * Num<T>::rcp(J.b);

    T D0 = T(0), D1 = T(0), D2 = T(0), D3 = T(0), D4 = T(0);
    if (dissipation) {
        // averaged state and its sound speed and total enthalpy
        const T a_sq = k.gamma * p_hat * Num<T>::rcp(rho_ln);
        const T a = sqrt_(a_sq);
        const T a_sq_g = a_sq * k.igm1;                  // a^2/(gamma-1)
        const T ke = fma(T(0.5), aa, phib);              // |u|^2/2 + phi
        const T H = a_sq_g + ke;
        // jump of the entropy variables w = ((gamma-s)/(gamma-1) - b|u|^2 + 2 b phi, 2 b u, -2 b),
        // with [[s]] = (1 - gamma)[[ln rho]] - [[ln b]]
        const T d1 = fma(dlb, k.igm1, dlr) - (J.b * fma(T(-2.0), J.phi, J.uu) - I.b * fma(T(-2.0), I.phi, I.uu));
        const T dm1 = T(2.0) * (J.b * J.u1 - I.b * I.u1);
        const T dm2 = T(2.0) * (J.b * J.u2 - I.b * I.u2);
        const T dm3 = T(2.0) * (J.b * J.u3 - I.b * I.u3);
        const T d5 = T(-2.0) * db;
        // shear input v = [[w_m]] + u [[w_5]] and its normal part
        const T v1 = fma(a1, d5, dm1), v2 = fma(a2, d5, dm2), v3 = fma(a3, d5, dm3);
        const T vn = fma(v3, n2, fma(v2, n1, v1 * n0));  // n . v (n unnormalised)
        const T nsq = fma(n2, n2, fma(n1, n1, n0 * n0));
        const T inn = Num<T>::rcp(sqrt_(nsq));
        const T nn = nsq * inn;
        const T inn2 = inn * inn;
        // wave strengths: beta = r_acoustic-common . [[w]]
        const T beta = fma(H, d5, fma(a3, dm3, fma(a2, dm2, fma(a1, dm1, d1))));
        const T alpha_e = fma(-a_sq_g, d5, beta);
        const T anu = a * vn * inn;
        const T lam_p = fabs(fma(a, nn, U)) * rho_ln * k.c_ac;
        const T lam_m = fabs(fma(-a, nn, U)) * rho_ln * k.c_ac;
        const T aU = fabs(U);
        const T cp_ = lam_p * (beta + anu);
        const T cm_ = lam_m * (beta - anu);
        const T ce = aU * rho_ln * k.c_en * alpha_e;
        const T ls = aU * p_hat;
        const T csum = cp_ + cm_;
        const T cdif = (cp_ - cm_) * a * inn;
        const T c0 = csum + ce;
        const T svn = ls * vn * inn2;
        D0 = T(0.5) * c0;
        D1 = T(0.5) * (fma(c0, a1, fma(cdif, n0, ls * v1)) - svn * n0);
        D2 = T(0.5) * (fma(c0, a2, fma(cdif, n1, ls * v2)) - svn * n1);
        D3 = T(0.5) * (fma(c0, a3, fma(cdif, n2, ls * v3)) - svn * n2);
        const T uv = fma(a3, v3, fma(a2, v2, a1 * v1));
        D4 = T(0.5) * (fma(csum, H, fma(cdif, U, fma(ce, ke, ls * uv))) - svn * U);
    }

    // momentum: F_rho {{u}} + p_hat n (+ gravity, scaled per side)
    const T m1 = fma(Fr, a1, p_hat * n0), m2 = fma(Fr, a2, p_hat * n1), m3 = fma(Fr, a3, p_hat * n2);
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

// Node index of face node (s1, s2) on the face a_DIR = A of a (N+1)^3 element.
template <int N, int DIR>
__device__ __forceinline__ int face_node(int A, int s1, int s2) {
    constexpr int NQ = N + 1;
    if constexpr (DIR == 0) return A + NQ * (s1 + NQ * s2);
    else if constexpr (DIR == 1) return s1 + NQ * (A + NQ * s2);
    else return s1 + NQ * (s2 + NQ * A);
}

template <typename T>
__device__ __forceinline__ void load_node(const SurfaceArgs<T>& a, long long g, int dir, T (&q)[5], T& phi, T (&n)[3]) {
    const long long st = a.n;
#pragma unroll
    for (int v = 0; v < 5; ++v) q[v] = __ldg(a.q + v * st + g);
    phi = __ldg(a.phi + g);
#pragma unroll
    for (int s = 0; s < 3; ++s) n[s] = __ldg(a.Ja + (3 * dir + s) * st + g);
}

template <typename T>
__device__ __forceinline__ void add_out(const SurfaceArgs<T>& a, long long g, const T (&f)[5]) {
    const long long st = a.n;
#pragma unroll
    for (int v = 0; v < 5; ++v) a.out[v * st + g] = fma(a.inv_w0, f[v], a.out[v * st + g]);
}

// One thread per slot.  Slots [0, K (N+1)^2): the +xi_DIR face of element e
// (an interface with the next element, wrapped when periodic, or a wall).
// Slots beyond: the -xi_DIR faces of the first layer of elements when the
// direction has walls.
template <typename T, int N, int DIR>
__global__ void __launch_bounds__(256) surface_kernel(const __grid_constant__ SurfaceArgs<T> a) {
    constexpr int NQ = N + 1;
    constexpr int NF = NQ * NQ;
    const long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long K = a.Kx * a.Ky * a.Kz;
    const long long Kd[3] = {a.Kx, a.Ky, a.Kz};
    const long long stride = (DIR == 0) ? 1 : (DIR == 1) ? a.Kx : a.Kx * a.Ky;
    const bool wall_dir = a.bc[DIR] != 0;
    const long long n_plus = K * NF;
    const long long n_minus = wall_dir ? (K / Kd[DIR]) * NF : 0;
    if (t >= n_plus + n_minus) return;

    long long e;
    int f;
    bool plus_face;
    if (t < n_plus) {
        e = t / NF;
        f = (int)(t - e * NF);
        plus_face = true;
    } else {
        const long long u = t - n_plus;
        const long long k = u / NF;
        f = (int)(u - k * NF);
        // element with index 0 along DIR, k enumerating the other two indices
        if (DIR == 0) e = k * a.Kx;
        else if (DIR == 1) e = (k % a.Kx) + (k / a.Kx) * a.Kx * a.Ky;
        else e = k;
        plus_face = false;
    }
    const int s1 = f % NQ, s2 = f / NQ;
    const long long er = (DIR == 0) ? e % a.Kx : (DIR == 1) ? (e / a.Kx) % a.Ky : e / (a.Kx * a.Ky);
    const SurfaceConsts<T> k = a.k;
    const long long NP3 = (long long)NQ * NQ * NQ;

    T qi[5], phii, ni[3];
    const long long gi = e * NP3 + face_node<N, DIR>(plus_face ? N : 0, s1, s2);
    load_node(a, gi, DIR, qi, phii, ni);
    const FaceNode<T> I = node_state(qi[0], qi[1], qi[2], qi[3], qi[4], phii, k.gm1);
    bool bad = !positive(I.rho) || !positive(I.p);

    const bool interior = plus_face && (er + 1 < Kd[DIR] || !wall_dir);
    if (interior) {
        const long long ej = (er + 1 < Kd[DIR]) ? e + stride : e - (Kd[DIR] - 1) * stride;
        const long long gj = ej * NP3 + face_node<N, DIR>(0, s1, s2);
        T qj[5], phij, nj[3];
        load_node(a, gj, DIR, qj, phij, nj);
        const FaceNode<T> J = node_state(qj[0], qj[1], qj[2], qj[3], qj[4], phij, k.gm1);
        bad |= !positive(J.rho) || !positive(J.p);
        const T n0 = T(0.5) * (ni[0] + nj[0]), n1 = T(0.5) * (ni[1] + nj[1]), n2 = T(0.5) * (ni[2] + nj[2]);
        T fi[5], fj[5];
        interface_flux(I, J, n0, n1, n2, k, a.dissipation != 0, fi, fj);
        if (a.form == 0) {
            add_phys_flux(I, ni[0], ni[1], ni[2], T(-1), fi);
            add_phys_flux(J, nj[0], nj[1], nj[2], T(1), fj);
        }
        add_out(a, gi, fi);
        add_out(a, gj, fj);
    } else {
        // slip wall: mirror ghost (rho, m - 2 (m.n^) n^, E), same phi, outward normal
        const T sg = plus_face ? T(1) : T(-1);
        const T n0 = sg * ni[0], n1 = sg * ni[1], n2 = sg * ni[2];
        const T inn = Num<T>::rcp(sqrt_(fma(n2, n2, fma(n1, n1, n0 * n0))));
        const T h0 = n0 * inn, h1 = n1 * inn, h2 = n2 * inn;
        const T mn = T(2.0) * fma(qi[3], h2, fma(qi[2], h1, qi[1] * h0));
        FaceNode<T> G = I;
        const T un2 = mn * Num<T>::rcp(qi[0]);
        G.u1 = fma(-un2, h0, I.u1);
        G.u2 = fma(-un2, h1, I.u2);
        G.u3 = fma(-un2, h2, I.u3);
        T fi[5], fg[5];
        interface_flux(I, G, n0, n1, n2, k, a.dissipation != 0, fi, fg);
        if (a.form == 0) add_phys_flux(I, n0, n1, n2, T(-1), fi);
        add_out(a, gi, fi);
    }
    if (bad) atomicOr(a.status, 1u);
}

template <typename T, int N>
cudaError_t launch_surface_n(const SurfaceArgs<T>& a, cudaStream_t s) {
    constexpr int NF = (N + 1) * (N + 1);
    const long long K = a.Kx * a.Ky * a.Kz;
    const long long Kd[3] = {a.Kx, a.Ky, a.Kz};
    for (int dir = 0; dir < 3; ++dir) {
        const long long slots = K * NF + (a.bc[dir] ? (K / Kd[dir]) * NF : 0);
        const long long blocks = (slots + 255) / 256;
        if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
        if (dir == 0) surface_kernel<T, N, 0><<<(unsigned)blocks, 256, 0, s>>>(a);
        else if (dir == 1) surface_kernel<T, N, 1><<<(unsigned)blocks, 256, 0, s>>>(a);
        else surface_kernel<T, N, 2><<<(unsigned)blocks, 256, 0, s>>>(a);
        const cudaError_t err = cudaGetLastError();
        if (err != cudaSuccess) return err;
    }
    return cudaSuccess;
}

template <typename T>
cudaError_t launch_surface_any(const SurfaceArgs<T>& a, int N, cudaStream_t s) {
    switch (N) {
        case 1: return launch_surface_n<T, 1>(a, s);
        case 2: return launch_surface_n<T, 2>(a, s);
        case 3: return launch_surface_n<T, 3>(a, s);
        case 4: return launch_surface_n<T, 4>(a, s);
        case 5: return launch_surface_n<T, 5>(a, s);
        case 6: return launch_surface_n<T, 6>(a, s);
        case 7: return launch_surface_n<T, 7>(a, s);
        case 8: return launch_surface_n<T, 8>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

#if ESDG_SURF_PREC == 0
cudaError_t launch_surface_fp64(const SurfaceArgs<double>& a, int N, cudaStream_t s) {
    return launch_surface_any<double>(a, N, s);
}
#else
cudaError_t launch_surface_fp32(const SurfaceArgs<float>& a, int N, cudaStream_t s) {
    return launch_surface_any<float>(a, N, s);
}
#endif

}  // namespace esdg
