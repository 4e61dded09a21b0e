// Metric terms of curved hexahedral elements, computed on the GPU in FP64.
//
// The ESDG GPU paper (Sec. 3) uses diagonal matrices G_jk of metric terms,
// the derivatives of the k-th reference coordinate with respect to the j-th
// physical coordinate, scaled by the Jacobian; it does not print a discrete
// form.  This file uses the conservative curl form
//     Ja^r_j = -( curl_xi ( X_l grad_xi X_m ) )_r ,  (j, m, l) cyclic,
// in which the products X_l d_s X_m are formed at the nodes and every
// derivative is the LGL differentiation matrix.  Because the three 1-D
// derivative operators commute, the discrete divergence sum_r D^r Ja^r_j
// vanishes to round-off, which is what makes a constant state stay constant
// on a curved mesh.  J = x_xi . (x_eta x x_zeta) is returned on request.
//
// One CTA per element, one thread per node; the element's coordinates,
// their derivatives and the products stay in shared memory.  This runs once
// per mesh, so it is written for clarity rather than speed.
#include <cuda_runtime.h>

#include "esdg_internal.h"

namespace esdg {

namespace {

__device__ __forceinline__ double ref_deriv(const double* __restrict__ f, const double* D, int NQ,
                                            int a, int b, int c, int s) {
    double acc = 0.0;
    if (s == 0) {
        for (int k = 0; k < NQ; ++k) acc += D[a * NQ + k] * f[k + NQ * (b + NQ * c)];
    } else if (s == 1) {
        for (int k = 0; k < NQ; ++k) acc += D[b * NQ + k] * f[a + NQ * (k + NQ * c)];
    } else {
        for (int k = 0; k < NQ; ++k) acc += D[c * NQ + k] * f[a + NQ * (b + NQ * k)];
    }
    return acc;
}

__global__ void geometry_kernel(const __grid_constant__ GeometryArgs g) {
    const int NQ = g.N + 1;
    const int NP3 = NQ * NQ * NQ;
    const long long n = g.K * (long long)NP3;
    const long long e = blockIdx.x;
    extern __shared__ double sm[];
    double* X = sm;              // [3][NP3]
    double* dX = sm + 3 * NP3;   // [3 coords][3 dirs][NP3]
    double* W = sm + 12 * NP3;   // [3 j][3 s][NP3]: X_l d_s X_m

    const int t = threadIdx.x;
    const bool act = t < NP3;
    const int a = t % NQ, b = (t / NQ) % NQ, c = t / (NQ * NQ);
    // Coordinates relative to an element-local origin (midpoint of two
    // opposite corners).  The curl form is exactly invariant under a shift of
    // X_l (the shift multiplies curl(grad X_m), which vanishes because the 1-D
    // derivative matrices commute), while the rounding of D (X_l D X_m) grows
    // with |X|^2: the shift keeps the metric terms accurate far from the origin.
    const long long e0 = e * NP3, e1 = e * NP3 + NP3 - 1;
    const double ox = 0.5 * (g.x[e0] + g.x[e1]);
    const double oy = 0.5 * (g.y[e0] + g.y[e1]);
    const double oz = 0.5 * (g.z[e0] + g.z[e1]);
    if (act) {
        X[0 * NP3 + t] = g.x[e * NP3 + t] - ox;
        X[1 * NP3 + t] = g.y[e * NP3 + t] - oy;
        X[2 * NP3 + t] = g.z[e * NP3 + t] - oz;
    }
    __syncthreads();
    if (act) {
        for (int j = 0; j < 3; ++j)
            for (int s = 0; s < 3; ++s)
                dX[(3 * j + s) * NP3 + t] = ref_deriv(X + j * NP3, g.D, NQ, a, b, c, s);
    }
    __syncthreads();
    if (act) {
        for (int j = 0; j < 3; ++j) {
            const int m = (j + 1) % 3, l = (j + 2) % 3;
            for (int s = 0; s < 3; ++s) W[(3 * j + s) * NP3 + t] = X[l * NP3 + t] * dX[(3 * m + s) * NP3 + t];
        }
    }
    __syncthreads();
    if (!act) return;
    double Ja[9];
    for (int j = 0; j < 3; ++j) {
        for (int r = 0; r < 3; ++r) {
            const int s1 = (r + 1) % 3, s2 = (r + 2) % 3;
            const double curl = ref_deriv(W + (3 * j + s2) * NP3, g.D, NQ, a, b, c, s1) -
                                ref_deriv(W + (3 * j + s1) * NP3, g.D, NQ, a, b, c, s2);
            Ja[3 * r + j] = -curl;
        }
    }
    // J = x_xi . (x_eta x x_zeta); dX[(3 j + s)] = d X_j / d xi_s
    const double x0 = dX[0 * NP3 + t], y0 = dX[3 * NP3 + t], z0 = dX[6 * NP3 + t];
    const double x1 = dX[1 * NP3 + t], y1 = dX[4 * NP3 + t], z1 = dX[7 * NP3 + t];
    const double x2 = dX[2 * NP3 + t], y2 = dX[5 * NP3 + t], z2 = dX[8 * NP3 + t];
    const double J = x0 * (y1 * z2 - z1 * y2) - y0 * (x1 * z2 - z1 * x2) + z0 * (x1 * y2 - y1 * x2);
    const long long gi = e * NP3 + t;
    if (g.fp32) {
        float* o = static_cast<float*>(g.Ja);
        for (int k = 0; k < 9; ++k) o[k * n + gi] = (float)Ja[k];
        if (g.J) static_cast<float*>(g.J)[gi] = (float)J;
    } else {
        double* o = static_cast<double*>(g.Ja);
        for (int k = 0; k < 9; ++k) o[k * n + gi] = Ja[k];
        if (g.J) static_cast<double*>(g.J)[gi] = J;
    }
}

}  // namespace

cudaError_t launch_geometry(const GeometryArgs& a, cudaStream_t s) {
    const int NQ = a.N + 1;
    const int NP3 = NQ * NQ * NQ;
    const size_t smem = sizeof(double) * 21 * (size_t)NP3;
    cudaError_t err = cudaFuncSetAttribute(geometry_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)smem);
    if (err != cudaSuccess) return err;
    const int threads = ((NP3 + 31) / 32) * 32;
    geometry_kernel<<<(unsigned)a.K, threads, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace esdg
