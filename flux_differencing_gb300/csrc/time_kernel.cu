// Time stepping and global diagnostics for sm_103a.
//
// The semi-discrete system of "GPU Performance of an Entropy-Stable
// Discontinuous Galerkin Euler Solver with Non-Conservative Terms" (Sec. 3,
// Eq. 2) is dq/dt = h - (volume + surface)/J.  One stage of a 2N-storage
// low-storage Runge-Kutta scheme (Williamson's form) updates every node with
//     dq <- A dq + dt (h - rhs/J),   q <- q + B dq,
// h being the f-plane Coriolis source (0, f rho u2, -f rho u1, 0, 0).  The
// stage is an HBM-bound stream over q, dq, rhs and J (26 values per node),
// one node per thread with coalesced plane accesses.
//
// Diagnostics: the mass, total-energy and entropy integrals
// sum_i w_a w_b w_c J_i (rho_i, E_i, eta_i), eta = -rho s/(gamma-1),
// s = ln(p rho^-gamma), accumulated in FP64 with a compensated (Neumaier)
// sum per thread, a fixed-order tree per block and a fixed-order final pass,
// so the result is bitwise reproducible for a given mesh size.
#include <cuda_runtime.h>

#include "esdg_internal.h"
#include "numeric.cuh"

namespace esdg {
namespace {

template <typename T>
__global__ void __launch_bounds__(256) rk_stage_kernel(const __grid_constant__ RkArgs<T> a) {
    const long long n = a.n;
    const T A = a.A, B = a.B, dt = a.dt, f = a.coriolis;
    T* __restrict__ qp = a.q;
    T* __restrict__ dqp = a.dq;
    const T* __restrict__ rp = a.rhs;
    const bool use_dq = A != T(0);
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x) {
        // dt L = dt h + sc rhs with sc = -dt/J; the reciprocal by estimate +
        // Newton (FP64: within 2 ulp).  About 20 FP64 operations per node, which
        // keeps the FP64 stage near the memory roofline on GB300's FP64 pipe.
        const T sc = -dt * Num<T>::rcp(a.J[i]);
        // all loads before any store (the pointers are restrict-qualified)
        T qv[5], dL[5], dqv[5];
#pragma unroll
        for (int v = 0; v < 5; ++v) {
            qv[v] = qp[v * n + i];
            dL[v] = rp[v * n + i] * sc;
            dqv[v] = use_dq ? dqp[v * n + i] : T(0);
        }
        if (f != T(0)) {
            const T fdt = f * dt;
            dL[1] = fma(fdt, qv[2], dL[1]);
            dL[2] = fma(-fdt, qv[1], dL[2]);
        }
        // a first stage (A == 0) neither reads dq nor lets its old contents through
#pragma unroll
        for (int v = 0; v < 5; ++v) {
            const T d = use_dq ? fma(A, dqv[v], dL[v]) : dL[v];
            dqp[v * n + i] = d;
            qp[v * n + i] = fma(B, d, qv[v]);
        }
    }
}

// a + b with the rounding error carried in c (Neumaier)
__device__ __forceinline__ void comp_add(double& s, double& c, double x) {
    const double t = s + x;
    c += (fabs(s) >= fabs(x)) ? ((s - t) + x) : ((x - t) + s);
    s = t;
}

template <typename T>
__global__ void __launch_bounds__(256) diag_partial_kernel(const __grid_constant__ DiagArgs<T> a) {
    __shared__ double red[3][256];
    const long long n = a.n;
    const int Nq = a.Nq;
    double s[3] = {0, 0, 0}, c[3] = {0, 0, 0};
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x) {
        const int nd = (int)(i % a.np3);
        const double w = a.w[nd % Nq] * a.w[(nd / Nq) % Nq] * a.w[nd / (Nq * Nq)];
        const double wJ = w * (double)a.J[i];
        const double m1 = a.q[n + i], m2 = a.q[2 * n + i], m3 = a.q[3 * n + i];
        const double phi = a.phi[i];
        double rho = a.q[i], E = a.q[4 * n + i], p;
        if (a.rho_ref) {
            // perturbation variables: rho = rho_ref + rho', E = E_ref + E',
            // E_ref = p_ref/(gamma-1) + rho_ref phi
            const double rr = a.rho_ref[i], pr = a.p_ref[i];
            const double rp = rho, Ep = E;
            rho = rr + rp;
            p = pr + a.gm1 * (Ep - 0.5 * (m1 * m1 + m2 * m2 + m3 * m3) / rho - rp * phi);
            E = Ep + pr / a.gm1 + rr * phi;
        } else {
            p = a.gm1 * (E - 0.5 * (m1 * m1 + m2 * m2 + m3 * m3) / rho - rho * phi);
        }
        const double ent = -rho * (log(p) - a.gamma * log(rho)) / a.gm1;
        comp_add(s[0], c[0], wJ * rho);
        comp_add(s[1], c[1], wJ * E);
        comp_add(s[2], c[2], wJ * ent);
    }
    for (int k = 0; k < 3; ++k) red[k][threadIdx.x] = s[k] + c[k];
    __syncthreads();
    for (int h = 128; h > 0; h >>= 1) {
        if ((int)threadIdx.x < h)
            for (int k = 0; k < 3; ++k) red[k][threadIdx.x] += red[k][threadIdx.x + h];
        __syncthreads();
    }
    if (threadIdx.x == 0)
        for (int k = 0; k < 3; ++k) a.partials[3 * blockIdx.x + k] = red[k][0];
}

__global__ void __launch_bounds__(256) diag_final_kernel(const double* __restrict__ partials, int blocks,
                                                         double* __restrict__ out) {
    __shared__ double red[3][256];
    double s[3] = {0, 0, 0}, c[3] = {0, 0, 0};
    for (int b = threadIdx.x; b < blocks; b += blockDim.x)
        for (int k = 0; k < 3; ++k) comp_add(s[k], c[k], partials[3 * b + k]);
    for (int k = 0; k < 3; ++k) red[k][threadIdx.x] = s[k] + c[k];
    __syncthreads();
    for (int h = 128; h > 0; h >>= 1) {
        if ((int)threadIdx.x < h)
            for (int k = 0; k < 3; ++k) red[k][threadIdx.x] += red[k][threadIdx.x + h];
        __syncthreads();
    }
    if (threadIdx.x == 0)
        for (int k = 0; k < 3; ++k) out[k] = red[k][0];
}

long long stream_blocks(long long n) {
    long long b = (n + 255) / 256;
    const long long cap = 152LL * 8;  // grid-stride beyond eight CTAs per SM
    return b < cap ? b : cap;
}

}  // namespace

template <typename T>
cudaError_t launch_rk_stage(const RkArgs<T>& a, cudaStream_t s) {
    if (a.n <= 0) return cudaSuccess;
    rk_stage_kernel<T><<<(unsigned)stream_blocks(a.n), 256, 0, s>>>(a);
    return cudaGetLastError();
}
template cudaError_t launch_rk_stage<double>(const RkArgs<double>&, cudaStream_t);
template cudaError_t launch_rk_stage<float>(const RkArgs<float>&, cudaStream_t);

template <typename T>
cudaError_t launch_diagnostics(const DiagArgs<T>& a, double* out, cudaStream_t s) {
    const int blocks = kDiagBlocks;
    diag_partial_kernel<T><<<blocks, 256, 0, s>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    diag_final_kernel<<<1, 256, 0, s>>>(a.partials, blocks, out);
    return cudaGetLastError();
}
template cudaError_t launch_diagnostics<double>(const DiagArgs<double>&, double*, cudaStream_t);
template cudaError_t launch_diagnostics<float>(const DiagArgs<float>&, double*, cudaStream_t);

}  // namespace esdg
