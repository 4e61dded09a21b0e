// Flux-differencing volume kernel for sm_103a, templated on the element type
// and the polynomial order.
//
// What it computes (the volume part of Eq. 2 of "GPU Performance of an
// Entropy-Stable Discontinuous Galerkin Euler Solver with Non-Conservative
// Terms", Sec. 3): for every node i and reference direction r,
//     out_i += (1/w_{p}) sum_m 2 Q_{p p'} (F + G)^r(i, m)
// over the nodes m of the r-line through i (p, p' their positions on the
// line, Q = W D so that 2 Q_{pp'}/w_p = 2 D_{pp'}).  F is the
// entropy-conservative two-point flux (Eqs. 3-4), G the gravity term (Eqs.
// 4-5), both contracted with the averaged metric (Ja^r(i) + Ja^r(m))/2.
//
// How (GB300 design):
//  * One CTA handles EPB whole elements.  A load phase reads the 15 input
//    planes with coalesced loads straight into registers and writes per-node
//    derived quantities to shared memory: u = m/rho, b = rho/(2p), 1/b,
//    log rho, log b, h = phi/2 - |u|^2/4 (Sec. 4.1: primitives and logarithms
//    once per node, not per pair), plus phi and the metric terms.
//  * Three direction phases (eta, zeta, then xi).  In each, every line's Nq
//    nodes occupy Nq consecutive lanes of one warp.  The lane at line
//    position p evaluates the pairs (p, p+d mod Nq), d = 1..floor(Nq/2) --
//    the weighted cyclic assignment of Sec. 4.1 Eq. 6 / Fig. 1(b): every lane
//    does the same number of evaluations.  For d < Nq/2 the pair's result
//    feeds both nodes ("half-sweep"): the partner's share is formed with
//    2 Q_{p'p} = -2 Q_{pp'} and the gravity partner scaling G -> -G b_i/b_m
//    (Sec. 4.1) and moved to the partner lane by a warp shuffle, so no
//    atomics and a fixed summation order (bitwise deterministic).  For the
//    antipodal offset d = Nq/2 (Nq even) both nodes evaluate the pair and
//    keep their own side, which is Fig. 1(b)'s two weight-1/2 evaluations.
//  * The mass flux is {{rho}}_log {{u}}.n, the energy flux the entropy-
//    conserving completion (see the oracle); both are formed directly from
//    the contravariant direction vector, never as a 3x5 flux matrix (Sec.
//    4.1).  Log means use the per-node logarithms, switching to a series in
//    ((a+ - a-)/(a+ + a-))^2 when the two logarithms are close, and 1/{{b}}_log
//    is computed directly (Sec. 4.1).  The choice between the two is a select,
//    not a branch, so lanes of a warp never diverge on it.
//  * Per-direction sums are scaled by 1/w once per node and combined in
//    shared memory; the xi phase writes the result with coalesced stores.
//  * No tensor cores: the flux is a nonlinear function of each pair.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "esdg_internal.h"

namespace esdg {

template <int N>
struct Shape {
    static constexpr int NQ = N + 1;
    static constexpr int NP3 = NQ * NQ * NQ;
    static constexpr int NL = NQ * NQ;       // lines per element and direction
    static constexpr int LPW = 32 / NQ;      // whole lines per warp
    static constexpr int H = NQ / 2;         // pair offsets per lane
    static constexpr bool EVEN = (NQ % 2) == 0;
    // elements per CTA: keeps lanes busy and the CTA at <= 512 threads
    // (<= 864 for N = 8, where a single element already needs 27 warps)
    static constexpr int EPB = (N == 1) ? 16 : (N == 2) ? 10 : (N == 3) ? 4 : (N == 4) ? 3
                             : (N == 5) ? 2 : 1;
    static constexpr int LINES = EPB * NL;
    static constexpr int WARPS = (LINES + LPW - 1) / LPW;
    static constexpr int THREADS = WARPS * 32;
    static constexpr int NODES = EPB * NP3;
};

// shared-memory field indices (each field is an array of Shape::NODES values)
enum SmemField {
    F_RHO = 0, F_U1, F_U2, F_U3, F_B, F_INVB, F_LNRHO, F_LNB, F_PHI, F_H,
    F_JA0,              // 9 metric planes F_JA0 .. F_JA0 + 8
    F_ACC0 = F_JA0 + 9, // 5 accumulators
    F_COUNT = F_ACC0 + 5
};

template <typename T>
struct Num;
template <>
struct Num<double> {
    // |log a+ - log a-| below which the series form of the log mean is used:
    // (a+ - a-)/(a+ + a-) < ~1e-2, series truncation error < 1e-17
    static __device__ __forceinline__ double tau() { return 2.0e-2; }
    static __device__ __forceinline__ double log_(double x) { return log(x); }
    static __device__ __forceinline__ double rcp(double x) { return 1.0 / x; }
};
template <>
struct Num<float> {
    // (a+ - a-)/(a+ + a-) < ~0.1, series truncation error < 1e-9
    static __device__ __forceinline__ float tau() { return 0.2f; }
    static __device__ __forceinline__ float log_(float x) { return logf(x); }
    static __device__ __forceinline__ float rcp(float x) { return 1.0f / x; }
};

// Log mean {{a}}_log = (a+ - a-)/(log a+ - log a-) (Eq. 3) from per-node
// logarithms.  With f = (a+ - a-)/(a+ + a-) and u = f^2,
//   {{a}}_log = {{a}} * f / atanh(f) = {{a}} (1 - u/3 - 4u^2/45 - 44u^3/945 - ...),
// which is used when the logarithms are close.  One reciprocal either way.
template <typename T>
__device__ __forceinline__ T log_mean(T ai, T am, T lai, T lam) {
    const T d = am - ai;
    const T s = am + ai;
    const T dl = lam - lai;
    const bool close = fabs(dl) < Num<T>::tau();
    const T r = Num<T>::rcp(close ? s : dl);
    const T t = d * r;          // close: f ; far: the log mean itself
    const T u = t * t;
    const T poly = T(1) - u * (T(1.0 / 3.0) + u * (T(4.0 / 45.0) + u * T(44.0 / 945.0)));
    const T ser = T(0.5) * s * poly;
    return close ? ser : t;
}

// 1/{{b}}_log (computed directly, Sec. 4.1) and 1/(b+ + b-).  With f and u as
// above, 1/{{b}}_log = (2/(b+ + b-)) atanh(f)/f = (2/(b+ + b-)) (1 + u/3 + u^2/5 + u^3/7 + ...).
// Far apart: 1/{{b}}_log = (log b+ - log b-)/(b+ - b-); both reciprocals then
// come from the single reciprocal of (b+ - b-)(b+ + b-).
template <typename T>
__device__ __forceinline__ void inv_log_mean(T bi, T bm, T lbi, T lbm, T& inv_ln, T& inv_sum) {
    const T d = bm - bi;
    const T s = bm + bi;
    const T dl = lbm - lbi;
    const bool close = fabs(dl) < Num<T>::tau();
    const T ds = d * s;
    const T r = Num<T>::rcp(close ? s : ds);
    inv_sum = close ? r : d * r;
    const T f = d * inv_sum;
    const T u = f * f;
    const T P = T(1) + u * (T(1.0 / 3.0) + u * (T(1.0 / 5.0) + u * T(1.0 / 7.0)));
    const T ser = T(2) * inv_sum * P;
    const T far = dl * (s * r);
    inv_ln = close ? ser : far;
}

template <typename T>
__device__ __forceinline__ T shfl(T v, int src) {
    return __shfl_sync(0xffffffffu, v, src);
}

// One direction phase.  R = 0 (xi), 1 (eta), 2 (zeta).  MODE = 0: write the
// scaled sum to the shared accumulators; 1: add to them; 2: add the shared
// accumulators and store to global memory.
template <typename T, int N, int R, int MODE>
__device__ __forceinline__ void direction_phase(const VolumeArgs<T>& a, T* __restrict__ sm,
                                                int e_count, long long node0) {
    using S = Shape<N>;
    constexpr int NQ = S::NQ;
    constexpr int NP3 = S::NP3;
    constexpr int NODES = S::NODES;
    constexpr int STR = (R == 0) ? 1 : (R == 1) ? NQ : NQ * NQ;

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int slot = lane / NQ;
    const int p = lane - slot * NQ;
    int L = warp * S::LPW + slot;
    const bool valid = (slot < S::LPW) && (L < S::LINES) && (L / S::NL < e_count);
    if (!valid) L = 0;  // compute on element 0's first line, discard
    const int el = L / S::NL;
    const int ell = L - el * S::NL;
    int base;
    if (R == 0) base = el * NP3 + NQ * ell;
    else if (R == 1) base = el * NP3 + (ell % NQ) + NQ * NQ * (ell / NQ);
    else base = el * NP3 + ell;
    const int i = base + p * STR;

    const T* __restrict__ s_rho = sm + F_RHO * NODES;
    const T* __restrict__ s_u1 = sm + F_U1 * NODES;
    const T* __restrict__ s_u2 = sm + F_U2 * NODES;
    const T* __restrict__ s_u3 = sm + F_U3 * NODES;
    const T* __restrict__ s_b = sm + F_B * NODES;
    const T* __restrict__ s_ib = sm + F_INVB * NODES;
    const T* __restrict__ s_lr = sm + F_LNRHO * NODES;
    const T* __restrict__ s_lb = sm + F_LNB * NODES;
    const T* __restrict__ s_phi = sm + F_PHI * NODES;
    const T* __restrict__ s_h = sm + F_H * NODES;
    const T* __restrict__ s_A0 = sm + (F_JA0 + 3 * R + 0) * NODES;
    const T* __restrict__ s_A1 = sm + (F_JA0 + 3 * R + 1) * NODES;
    const T* __restrict__ s_A2 = sm + (F_JA0 + 3 * R + 2) * NODES;

    const T rho_i = s_rho[i], u1_i = s_u1[i], u2_i = s_u2[i], u3_i = s_u3[i];
    const T b_i = s_b[i], ib_i = s_ib[i], lr_i = s_lr[i], lb_i = s_lb[i];
    const T phi_i = s_phi[i], h_i = s_h[i];
    const T A0_i = s_A0[i], A1_i = s_A1[i], A2_i = s_A2[i];

    T acc0 = T(0), acc1 = T(0), acc2 = T(0), acc3 = T(0), acc4 = T(0);

#pragma unroll
    for (int d = 1; d <= S::H; ++d) {
        const bool both = !(S::EVEN && d == S::H);  // antipodal: own side only
        int pm = p + d;
        if (pm >= NQ) pm -= NQ;
        const T c2q = a.ops.Q2[p * NQ + pm];
        const int m = base + pm * STR;

        const T rho_m = s_rho[m], u1_m = s_u1[m], u2_m = s_u2[m], u3_m = s_u3[m];
        const T b_m = s_b[m], ib_m = s_ib[m];

        const T A0 = A0_i + s_A0[m], A1 = A1_i + s_A1[m], A2 = A2_i + s_A2[m];  // 2 x avg metric
        const T s1 = u1_i + u1_m, s2 = u2_i + u2_m, s3 = u3_i + u3_m;          // 2 x avg velocity
        const T Un = s1 * A0 + s2 * A1 + s3 * A2;                               // 4 x {{u}}.n

        const T rho_ln = log_mean<T>(rho_i, rho_m, lr_i, s_lr[m]);
        T inv_bln, inv_bsum;
        inv_log_mean<T>(b_i, b_m, lb_i, s_lb[m], inv_bln, inv_bsum);
        const T bsum = b_i + b_m;
        const T ph = T(0.25) * (rho_i + rho_m) * inv_bsum;       // {{rho}}/(2{{b}}) / 2
        const T g = T(0.125) * rho_ln * bsum * (s_phi[m] - phi_i);  // gravity, Eqs. 4-5
        const T frh = (T(0.125) * c2q) * rho_ln * Un;             // 2Q F_rho / 2
        const T fr = frh + frh;                                     // 2Q F_rho
        const T ss = s1 * s1 + s2 * s2 + s3 * s3;
        const T Kf = a.c_g * inv_bln + (h_i + s_h[m]) + T(0.25) * ss;
        const T fE = fr * Kf + (T(0.5) * c2q) * Un * ph;          // 2Q F_E
        const T gq = c2q * g;
        const T phq = c2q * ph;
        const T Pi = gq * ib_i + phq;   // own:     2Q (p_hat/2 + G scale at b_i)
        acc0 += fr;
        acc1 += frh * s1 + A0 * Pi;
        acc2 += frh * s2 + A1 * Pi;
        acc3 += frh * s3 + A2 * Pi;
        acc4 += fE;
        if (both) {
            // partner's share: 2Q_{p'p} (F + G(m,i)) with 2Q_{p'p} = -2Q_{pp'} and
            // G(m,i) = -G(i,m) b_i/b_m
            const T Pm = gq * ib_m - phq;
            const T t1 = A0 * Pm - frh * s1;
            const T t2 = A1 * Pm - frh * s2;
            const T t3 = A2 * Pm - frh * s3;
            int src = p - d;
            if (src < 0) src += NQ;
            src += slot * NQ;
            acc0 -= shfl(fr, src);
            acc1 += shfl(t1, src);
            acc2 += shfl(t2, src);
            acc3 += shfl(t3, src);
            acc4 -= shfl(fE, src);
        }
    }

    if (a.form == 0 && (p == 0 || p == N)) {
        // diagonal pair m == i: 2 Q_pp Ja^r(i) . f(q_i), f the physical flux (Eq. 1)
        const T qd = a.ops.Q2[p * NQ + p];
        const T Uc = u1_i * A0_i + u2_i * A1_i + u3_i * A2_i;
        const T rU = qd * rho_i * Uc;
        const T pr = qd * T(0.5) * rho_i * ib_i;
        const T Hh = a.c_h * ib_i + T(2) * (phi_i - h_i);  // (E + p)/rho
        acc0 += rU;
        acc1 += rU * u1_i + pr * A0_i;
        acc2 += rU * u2_i + pr * A1_i;
        acc3 += rU * u3_i + pr * A2_i;
        acc4 += rU * Hh;
    }

    const T iw = a.ops.invw[p];
    T* s_acc = sm + F_ACC0 * NODES;
    if (MODE == 0 && valid) {
        s_acc[0 * NODES + i] = acc0 * iw;
        s_acc[1 * NODES + i] = acc1 * iw;
        s_acc[2 * NODES + i] = acc2 * iw;
        s_acc[3 * NODES + i] = acc3 * iw;
        s_acc[4 * NODES + i] = acc4 * iw;
    } else if (MODE == 1 && valid) {
        s_acc[0 * NODES + i] += acc0 * iw;
        s_acc[1 * NODES + i] += acc1 * iw;
        s_acc[2 * NODES + i] += acc2 * iw;
        s_acc[3 * NODES + i] += acc3 * iw;
        s_acc[4 * NODES + i] += acc4 * iw;
    } else if (MODE == 2 && valid) {
        // xi phase: i = L*NQ + p is the block-linear node, so lanes store contiguously
        const long long g = node0 + i;
        T* __restrict__ o = a.out;
        const long long n = a.n;
        o[0 * n + g] = s_acc[0 * NODES + i] + acc0 * iw;
        o[1 * n + g] = s_acc[1 * NODES + i] + acc1 * iw;
        o[2 * n + g] = s_acc[2 * NODES + i] + acc2 * iw;
        o[3 * n + g] = s_acc[3 * NODES + i] + acc3 * iw;
        o[4 * n + g] = s_acc[4 * NODES + i] + acc4 * iw;
    }
}

template <typename T, int N>
__global__ void __launch_bounds__(Shape<N>::THREADS, (sizeof(T) == 4 && Shape<N>::THREADS <= 512) ? 2 : 1)
volume_kernel(const __grid_constant__ VolumeArgs<T> a) {
    using S = Shape<N>;
    constexpr int NP3 = S::NP3;
    constexpr int NODES = S::NODES;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    T* sm = reinterpret_cast<T*>(smem_raw);

    const long long e0 = a.e_begin + (long long)blockIdx.x * S::EPB;
    const long long rem = a.e_end - e0;
    const int e_count = rem < S::EPB ? (int)rem : S::EPB;
    const long long node0 = e0 * NP3;

    // ---- load phase: one node per thread, coalesced plane reads -> derived values
    bool bad = false;
    for (int t = threadIdx.x; t < NODES; t += S::THREADS) {
        T rho = T(1), m1 = T(0), m2 = T(0), m3 = T(0), E = T(1), phi = T(0);
        T ja[9];
#pragma unroll
        for (int k = 0; k < 9; ++k) ja[k] = T(0);
        if (t < e_count * NP3) {
            const long long g = node0 + t;
            const long long n = a.n;
            rho = __ldg(a.q + g);
            m1 = __ldg(a.q + n + g);
            m2 = __ldg(a.q + 2 * n + g);
            m3 = __ldg(a.q + 3 * n + g);
            E = __ldg(a.q + 4 * n + g);
            phi = __ldg(a.phi + g);
#pragma unroll
            for (int k = 0; k < 9; ++k) ja[k] = __ldg(a.Ja + k * n + g);
        }
        const T irho = Num<T>::rcp(rho);
        const T u1 = m1 * irho, u2 = m2 * irho, u3 = m3 * irho;
        const T uu = u1 * u1 + u2 * u2 + u3 * u3;
        T pr = a.gm1 * (E - T(0.5) * rho * uu - rho * phi);
        if (t >= e_count * NP3) pr = T(0.5) * a.gm1;  // padding node: b = 1/gm1, finite
        bad |= !(rho > T(0)) || !(pr > T(0));
        const T ipr = Num<T>::rcp(pr);
        const T b = T(0.5) * rho * ipr;
        const T ib = T(2) * pr * irho;
        sm[F_RHO * NODES + t] = rho;
        sm[F_U1 * NODES + t] = u1;
        sm[F_U2 * NODES + t] = u2;
        sm[F_U3 * NODES + t] = u3;
        sm[F_B * NODES + t] = b;
        sm[F_INVB * NODES + t] = ib;
        sm[F_LNRHO * NODES + t] = Num<T>::log_(rho);
        sm[F_LNB * NODES + t] = Num<T>::log_(b);
        sm[F_PHI * NODES + t] = phi;
        sm[F_H * NODES + t] = T(0.5) * phi - T(0.25) * uu;
#pragma unroll
        for (int k = 0; k < 9; ++k) sm[(F_JA0 + k) * NODES + t] = ja[k];
    }
    if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) atomicOr(a.status, 1u);
    __syncthreads();

    direction_phase<T, N, 1, 0>(a, sm, e_count, node0);
    __syncthreads();
    direction_phase<T, N, 2, 1>(a, sm, e_count, node0);
    __syncthreads();
    direction_phase<T, N, 0, 2>(a, sm, e_count, node0);
}

template <typename T, int N>
cudaError_t launch_volume(const VolumeArgs<T>& a, cudaStream_t s) {
    using S = Shape<N>;
    const long long K = a.e_end - a.e_begin;
    if (K <= 0) return cudaSuccess;
    const size_t smem = sizeof(T) * (size_t)F_COUNT * S::NODES;
    static bool attr_done = false;  // per instantiation; set once per process
    if (!attr_done) {
        cudaError_t err = cudaFuncSetAttribute(volume_kernel<T, N>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
        attr_done = true;
    }
    const long long blocks = (K + S::EPB - 1) / S::EPB;
    volume_kernel<T, N><<<(unsigned)blocks, S::THREADS, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace esdg
