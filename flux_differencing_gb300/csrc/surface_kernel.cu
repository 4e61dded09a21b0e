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
//  * No logarithm in the common case: closeness of the two states is tested
//    on f = (a+ - a-)/(a+ + a-), and when every lane of a warp is close the
//    log means and the log jumps [[ln a]] = 2 atanh(f) of the entropy
//    variables come from their series in f^2.  Only warps holding a far pair
//    take the four logarithms.
//  * The dissipation is formed without tangent vectors: the two shear waves
//    share the eigenvalue u.n, so together they are the projection
//    (I - n^ n^T) onto the face, and the acoustic pair enters through the
//    sum and difference of its two wave strengths.
//  * Arithmetic type C: the I/O type, or float-float for FP64 buffers
//    (ESDG_FP64_FF), which moves the arithmetic from GB300's narrow FP64 pipe
//    to the FP32 pipes.
#include <cuda_runtime.h>

#include "esdg_internal.h"
#include "numeric.cuh"
#include "surface_flux.cuh"
#include "surface_index.cuh"

namespace esdg {

namespace {

template <typename T>
__device__ __forceinline__ void load_node(const SurfaceArgs<T>& a, long long g, int dir, T (&q)[5], T& phi,
                                          T (&n)[3], T (&ref)[2]) {
    const long long st = a.n;
#pragma unroll
    for (int v = 0; v < 5; ++v) q[v] = __ldg(a.q + v * st + g);
    phi = __ldg(a.phi + g);
#pragma unroll
    for (int s = 0; s < 3; ++s) n[s] = __ldg(a.Ja + (3 * dir + s) * st + g);
    ref[0] = a.rho_ref ? __ldg(a.rho_ref + g) : T(0);
    ref[1] = a.rho_ref ? __ldg(a.p_ref + g) : T(0);
}

template <typename T, typename C>
__device__ __forceinline__ FaceNode<C> node_from(const T (&q)[5], T phi, const T (&ref)[2], C gm1, bool perturbed) {
    using CV = Conv<T, C>;
    return node_state<C>(CV::in(q[0]), CV::in(q[1]), CV::in(q[2]), CV::in(q[3]), CV::in(q[4]), CV::in(phi), gm1,
                         perturbed, CV::in(ref[0]), CV::in(ref[1]));
}

template <typename T, typename C>
__device__ __forceinline__ void add_out(const SurfaceArgs<T>& a, long long g, const C (&f)[5]) {
    const long long st = a.n;
#pragma unroll
    for (int v = 0; v < 5; ++v)
        a.out[v * st + g] = fma(a.inv_w0, Conv<T, C>::out(f[v]), a.out[v * st + g]);
}

// One thread per slot.  Slots [0, K (N+1)^2): the +xi_DIR face of element e
// (an interface with the next element, wrapped when periodic, or a wall).
// Slots beyond: the -xi_DIR faces of the first layer of elements when the
// direction has walls.
// Float-float needs ~127 registers unbounded (two CTAs per SM) and is bound by
// latency there; a bound of three CTAs per SM (80 registers, a 228-byte
// spill) measured 0.44 -> 0.405 ms per call on the N = 7 channel, four CTAs
// (64 registers) no better.  FP32, bound by DRAM line traffic: four CTAs per
// SM (64 registers, no spill; unbounded it takes 69-72 and runs three) keep
// more loads in flight, 0.155 -> 0.142 ms per call; five (48 registers)
// spill.
template <typename C>
struct SurfaceOccupancy {
    static constexpr int value = std::is_same<C, ff>::value ? 3 : std::is_same<C, float>::value ? 4 : 1;
};

template <typename T, typename C, int N, int DIR>
__global__ void __launch_bounds__(256, SurfaceOccupancy<C>::value) surface_kernel(const __grid_constant__ SurfaceArgs<T> a) {
    constexpr int NQ = N + 1;
    using CV = Conv<T, C>;
    const long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long Kd[3] = {a.Kx, a.Ky, a.Kz};
    const long long stride = (DIR == 0) ? 1 : (DIR == 1) ? a.Kx : a.Kx * a.Ky;
    const bool wall_dir = a.bc[DIR] != 0;
    long long e, er;
    int f;
    bool plus_face;
    if (!surface_slot<N>(DIR, t, a.Kx, a.Ky, a.Kz, wall_dir, e, f, plus_face, er)) return;
    const int s1 = f % NQ, s2 = f / NQ;
    const long long NP3 = (long long)NQ * NQ * NQ;
    Consts<C> k;
    k.gm1 = CV::in(a.k.gm1);
    k.igm1 = CV::in(a.k.igm1);
    k.c_g = CV::in(a.k.c_g);
    k.gamma = CV::in(a.k.gamma);
    k.c_ac = CV::in(a.k.c_ac);
    k.c_en = CV::in(a.k.c_en);

    const bool perturbed = a.rho_ref != nullptr;
    T qi[5], phii, ni[3], ri[2];
    const long long gi = checked(e * NP3 + face_node<N, DIR>(plus_face ? N : 0, s1, s2), a.n, a.status);
    load_node(a, gi, DIR, qi, phii, ni, ri);
    const FaceNode<C> I = node_from<T, C>(qi, phii, ri, k.gm1, perturbed);
    bool bad = !positive(I.rho) || !positive(I.p);

    const bool interior = plus_face && (er + 1 < Kd[DIR] || !wall_dir);
    if (interior) {
        const long long ej = (er + 1 < Kd[DIR]) ? e + stride : e - (Kd[DIR] - 1) * stride;
        const long long gj = checked(ej * NP3 + face_node<N, DIR>(0, s1, s2), a.n, a.status);
        T qj[5], phij, nj[3], rj[2];
        load_node(a, gj, DIR, qj, phij, nj, rj);
        const FaceNode<C> J = node_from<T, C>(qj, phij, rj, k.gm1, perturbed);
        bad |= !positive(J.rho) || !positive(J.p);
        const C n0 = CV::in(T(0.5) * (ni[0] + nj[0]));
        const C n1 = CV::in(T(0.5) * (ni[1] + nj[1]));
        const C n2 = CV::in(T(0.5) * (ni[2] + nj[2]));
        C fi[5], fj[5];
        interface_flux(I, J, n0, n1, n2, k, a.dissipation != 0, fi, fj);
        if (a.form == 0) {
            add_phys_flux(I, CV::in(ni[0]), CV::in(ni[1]), CV::in(ni[2]), C(-1.0), fi);
            add_phys_flux(J, CV::in(nj[0]), CV::in(nj[1]), CV::in(nj[2]), C(1.0), fj);
        }
        add_out<T, C>(a, gi, fi);
        add_out<T, C>(a, gj, fj);
    } else {
        // slip wall: mirror ghost (rho, m - 2 (m.n^) n^, E), same phi, outward normal
        const T sg = plus_face ? T(1) : T(-1);
        const C n0 = CV::in(sg * ni[0]), n1 = CV::in(sg * ni[1]), n2 = CV::in(sg * ni[2]);
        const C inn = Num<C>::rcp(sqrt_(fma(n2, n2, fma(n1, n1, n0 * n0))));
        const C h0 = n0 * inn, h1 = n1 * inn, h2 = n2 * inn;
        const C un2 = C(2.0) * fma(I.u3, h2, fma(I.u2, h1, I.u1 * h0));
        FaceNode<C> G = I;
        G.u1 = fma(-un2, h0, I.u1);
        G.u2 = fma(-un2, h1, I.u2);
        G.u3 = fma(-un2, h2, I.u3);
        C fi[5], fg[5];
        interface_flux(I, G, n0, n1, n2, k, a.dissipation != 0, fi, fg);
        if (a.form == 0) add_phys_flux(I, n0, n1, n2, C(-1.0), fi);
        add_out<T, C>(a, gi, fi);
    }
    if (bad) atomicOr(a.status, 1u);
}

template <typename T, typename C, int N>
cudaError_t launch_surface_n(const SurfaceArgs<T>& a, cudaStream_t s) {
    constexpr int NF = (N + 1) * (N + 1);
    const long long K = a.Kx * a.Ky * a.Kz;
    const long long Kd[3] = {a.Kx, a.Ky, a.Kz};
    for (int dir = 0; dir < 3; ++dir) {
        const long long slots = K * NF + (a.bc[dir] ? (K / Kd[dir]) * NF : 0);
        const long long blocks = (slots + 255) / 256;
        if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
        if (dir == 0) surface_kernel<T, C, N, 0><<<(unsigned)blocks, 256, 0, s>>>(a);
        else if (dir == 1) surface_kernel<T, C, N, 1><<<(unsigned)blocks, 256, 0, s>>>(a);
        else surface_kernel<T, C, N, 2><<<(unsigned)blocks, 256, 0, s>>>(a);
        const cudaError_t err = cudaGetLastError();
        if (err != cudaSuccess) return err;
    }
    return cudaSuccess;
}

template <typename T, typename C>
cudaError_t launch_surface_any(const SurfaceArgs<T>& a, int N, cudaStream_t s) {
    switch (N) {
        case 1: return launch_surface_n<T, C, 1>(a, s);
        case 2: return launch_surface_n<T, C, 2>(a, s);
        case 3: return launch_surface_n<T, C, 3>(a, s);
        case 4: return launch_surface_n<T, C, 4>(a, s);
        case 5: return launch_surface_n<T, C, 5>(a, s);
        case 6: return launch_surface_n<T, C, 6>(a, s);
        case 7: return launch_surface_n<T, C, 7>(a, s);
        case 8: return launch_surface_n<T, C, 8>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

#if ESDG_SURF_PREC == 0
cudaError_t launch_surface_fp64(const SurfaceArgs<double>& a, int N, cudaStream_t s) {
    return launch_surface_any<double, double>(a, N, s);
}
#elif ESDG_SURF_PREC == 1
cudaError_t launch_surface_fp32(const SurfaceArgs<float>& a, int N, cudaStream_t s) {
    return launch_surface_any<float, float>(a, N, s);
}
#else
cudaError_t launch_surface_fp64ff(const SurfaceArgs<double>& a, int N, cudaStream_t s) {
    return launch_surface_any<double, ff>(a, N, s);
}
#endif

}  // namespace esdg
