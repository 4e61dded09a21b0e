// Host side of the C-ABI declared in include/esdg.h: handles, argument
// checks, operator tables and kernel dispatch.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <string>

#include "esdg.h"
#include "esdg_internal.h"

struct esdg_ctx {
    long long Kx = 0, Ky = 0, Kz = 0, K = 0, n = 0;
    int N = 0, Nq = 0, precision = 0, form = 0;
    double gamma = 1.4;
    int bc[3] = {ESDG_BC_PERIODIC, ESDG_BC_PERIODIC, ESDG_BC_PERIODIC};
    int dissipation = 1;
    double coriolis = 0.0;
    const void* ref_rho = nullptr;  // perturbation variables: reference density and pressure
    const void* ref_p = nullptr;
    int device = 0;
    unsigned* d_status = nullptr;
    double* d_partials = nullptr;  // diagnostics scratch, 3 * kDiagBlocks doubles
    double nodes[esdg::kMaxNq];
    double weights[esdg::kMaxNq];
    double D[esdg::kMaxNq * esdg::kMaxNq];
    esdg::OpTables<double> op64;
    esdg::OpTables<float> op32;
    std::string err;
};

namespace {

thread_local std::string g_create_error;

int fail(esdg_handle h, int code, const std::string& msg) {
    if (h) h->err = msg;
    else g_create_error = msg;
    return code;
}

int cuda_fail(esdg_handle h, cudaError_t e, const char* what) {
    return fail(h, ESDG_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void* a, size_t an, const void* b, size_t bn) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + bn && b0 < a0 + an;
}

// Legendre P_N and its derivative by the paired recurrences
//   (k+1) P_{k+1} = (2k+1) x P_k - k P_{k-1},   P'_{k+1} = P'_{k-1} + (2k+1) P_k.
void legendre(int N, long double x, long double& P, long double& dP) {
    long double p0 = 1, p1 = x, d0 = 0, d1 = 1;
    if (N == 0) { P = 1; dP = 0; return; }
    for (int k = 1; k < N; ++k) {
        long double p2 = ((2 * k + 1) * x * p1 - k * p0) / (k + 1);
        long double d2 = d0 + (2 * k + 1) * p1;
        p0 = p1; p1 = p2; d0 = d1; d1 = d2;
    }
    P = p1;
    dP = d1;
}

}  // namespace

namespace esdg {

// LGL nodes: +-1 and the roots of P_N', found by Newton's method on P_N' with
// P_N'' from Legendre's equation (1 - x^2) P'' = 2 x P' - N (N+1) P.
// Weights 2 / (N (N+1) P_N(x)^2).  D from barycentric weights
// lambda_j = 1 / prod_{k != j} (x_j - x_k):  D_ij = (lambda_j / lambda_i) / (x_i - x_j),
// D_ii = -sum_{j != i} D_ij (rows of D annihilate constants).
void lgl_operators(int N, double* nodes, double* weights, double* D) {
    const int Nq = N + 1;
    long double x[kMaxNq], w[kMaxNq], lam[kMaxNq];
    const long double pi = 3.141592653589793238462643383279502884L;
    for (int j = 0; j < Nq; ++j) {
        long double xj = -cosl(pi * j / N);
        if (j == 0) xj = -1;
        if (j == N) xj = 1;
        if (j > 0 && j < N) {
            for (int it = 0; it < 60; ++it) {
                long double P, dP;
                legendre(N, xj, P, dP);
                const long double d2P = (2 * xj * dP - (long double)N * (N + 1) * P) / (1 - xj * xj);
                const long double step = dP / d2P;
                xj -= step;
                if (fabsl(step) < 1e-21L) break;
            }
        }
        long double P, dP;
        legendre(N, xj, P, dP);
        x[j] = xj;
        w[j] = 2.0L / ((long double)N * (N + 1) * P * P);
    }
    for (int j = 0; j < Nq; ++j) {
        long double prod = 1;
        for (int k = 0; k < Nq; ++k)
            if (k != j) prod *= (x[j] - x[k]);
        lam[j] = 1 / prod;
    }
    for (int i = 0; i < Nq; ++i) {
        long double diag = 0;
        for (int j = 0; j < Nq; ++j) {
            if (j == i) continue;
            const long double dij = (lam[j] / lam[i]) / (x[i] - x[j]);
            D[i * Nq + j] = (double)dij;
            diag -= dij;
        }
        D[i * Nq + i] = (double)diag;
        nodes[i] = (double)x[i];
        weights[i] = (double)w[i];
    }
}

void set_unhandled_error(const char* msg) { g_create_error = msg; }

template <typename T>
void fill_op_tables(OpTables<T>& t, int N) {
    double x[kMaxNq], w[kMaxNq], D[kMaxNq * kMaxNq];
    lgl_operators(N, x, w, D);
    const int Nq = N + 1;
    std::memset(&t, 0, sizeof(t));
    for (int i = 0; i < Nq; ++i) {
        t.invw[i] = (T)(1.0L / (long double)w[i]);
        for (int j = 0; j < Nq; ++j) t.Q2[i * Nq + j] = (T)(2.0L * (long double)w[i] * (long double)D[i * Nq + j]);
    }
    t.diag[0] = (T)(2.0L * (long double)D[0]);
    t.diag[N] = (T)(2.0L * (long double)D[N * Nq + N]);
}
template void fill_op_tables<double>(OpTables<double>&, int);
template void fill_op_tables<float>(OpTables<float>&, int);

}  // namespace esdg

namespace {


template <typename T>
esdg::VolumeArgs<T> volume_args(const esdg_ctx* h, const void* q, const void* Ja, const void* phi, void* out,
                                long long e0, long long e1, const esdg::OpTables<T>& ops, int form) {
    esdg::VolumeArgs<T> a;
    std::memset(&a, 0, sizeof(a));  // rk_* null: the kernel writes out
    a.q = static_cast<const T*>(q);
    a.Ja = static_cast<const T*>(Ja);
    a.phi = static_cast<const T*>(phi);
    a.out = static_cast<T*>(out);
    a.n = h->n;
    a.e_begin = e0;
    a.e_end = e1;
    a.gm1 = (T)(h->gamma - 1.0);
    a.c_g = (T)(1.0 / (2.0 * (h->gamma - 1.0)));
    a.c_h = (T)(h->gamma / (2.0 * (h->gamma - 1.0)));
    a.form = form;
    a.status = h->d_status;
    a.rho_ref = static_cast<const T*>(h->ref_rho);
    a.p_ref = static_cast<const T*>(h->ref_p);
    a.ops = ops;
    return a;
}

template <typename T>
esdg::SurfaceConsts<T> surface_consts(const esdg_ctx* h) {
    const long double g = h->gamma;
    esdg::SurfaceConsts<T> k;
    k.gm1 = (T)(g - 1);
    k.igm1 = (T)(1 / (g - 1));
    k.c_g = (T)(1 / (2 * (g - 1)));
    k.gamma = (T)g;
    k.c_ac = (T)(1 / (4 * g));       // half the acoustic-wave scaling 1/(2 gamma)
    k.c_en = (T)((g - 1) / (2 * g));  // half the entropy-wave scaling (gamma - 1)/gamma
    return k;
}

// The surface fields of the FP32 volume kernel's face modes (the fused stage
// and volume + surface to out).
static void set_face_fields(const esdg_ctx* h, esdg::VolumeArgs<float>& a) {
    a.Kx = h->Kx;
    a.Ky = h->Ky;
    a.Kz = h->Kz;
    for (int r = 0; r < 3; ++r) a.bc[r] = h->bc[r];
    a.dissipation = h->dissipation;
    a.inv_w0 = (float)(1.0L / (long double)h->weights[0]);
    a.sk = surface_consts<float>(h);
}

template <typename T>
esdg::SurfaceArgs<T> surface_args(const esdg_ctx* h, const void* q, const void* Ja, const void* phi, void* out,
                                  int form) {
    esdg::SurfaceArgs<T> a;
    std::memset(&a, 0, sizeof(a));
    a.q = static_cast<const T*>(q);
    a.Ja = static_cast<const T*>(Ja);
    a.phi = static_cast<const T*>(phi);
    a.out = static_cast<T*>(out);
    a.n = h->n;
    a.Kx = h->Kx;
    a.Ky = h->Ky;
    a.Kz = h->Kz;
    for (int r = 0; r < 3; ++r) a.bc[r] = h->bc[r];
    a.form = form;
    a.dissipation = h->dissipation;
    a.inv_w0 = (T)(1.0L / (long double)h->weights[0]);
    a.k = surface_consts<T>(h);
    a.status = h->d_status;
    a.rho_ref = static_cast<const T*>(h->ref_rho);
    a.p_ref = static_cast<const T*>(h->ref_p);
    return a;
}

// Carpenter & Kennedy (1994), five-stage fourth-order 2N-storage Runge-Kutta
// scheme: numerator and denominator of A_k, B_k, c_k (exact integers).
const long double kLsrkA[5][2] = {{0.0L, 1.0L},
                                  {-567301805773.0L, 1357537059087.0L},
                                  {-2404267990393.0L, 2016746695238.0L},
                                  {-3550918686646.0L, 2091501179385.0L},
                                  {-1275806237668.0L, 842570457699.0L}};
const long double kLsrkB[5][2] = {{1432997174477.0L, 9575080441755.0L},
                                  {5161836677717.0L, 13612068292357.0L},
                                  {1720146321549.0L, 2090206949498.0L},
                                  {3134564353537.0L, 4481467310338.0L},
                                  {2277821191437.0L, 14882151754819.0L}};
const long double kLsrkC[5][2] = {{0.0L, 1.0L},
                                  {1432997174477.0L, 9575080441755.0L},
                                  {2526269341429.0L, 6820363962896.0L},
                                  {2006345519317.0L, 3224310063776.0L},
                                  {2802321613138.0L, 2924317926251.0L}};
double lsrk_coef(const long double (&r)[2]) { return (double)(r[0] / r[1]); }

template <typename T>
esdg::DiagArgs<T> diag_args(const esdg_ctx* h, const void* q, const void* J, const void* phi) {
    esdg::DiagArgs<T> a;
    std::memset(&a, 0, sizeof(a));
    a.q = static_cast<const T*>(q);
    a.J = static_cast<const T*>(J);
    a.phi = static_cast<const T*>(phi);
    a.rho_ref = static_cast<const T*>(h->ref_rho);
    a.p_ref = static_cast<const T*>(h->ref_p);
    a.n = h->n;
    a.Nq = h->Nq;
    a.np3 = h->Nq * h->Nq * h->Nq;
    a.gamma = h->gamma;
    a.gm1 = h->gamma - 1.0;
    for (int k = 0; k < h->Nq; ++k) a.w[k] = h->weights[k];
    a.partials = h->d_partials;
    return a;
}

cudaError_t dispatch_fp64(int N, const esdg::VolumeArgs<double>& a, cudaStream_t s) {
    switch (N) {
        case 1: return esdg::launch_volume_fp64_n1(a, s);
        case 2: return esdg::launch_volume_fp64_n2(a, s);
        case 3: return esdg::launch_volume_fp64_n3(a, s);
        case 4: return esdg::launch_volume_fp64_n4(a, s);
        case 5: return esdg::launch_volume_fp64_n5(a, s);
        case 6: return esdg::launch_volume_fp64_n6(a, s);
        case 7: return esdg::launch_volume_fp64_n7(a, s);
        case 8: return esdg::launch_volume_fp64_n8(a, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t dispatch_fp64ff(int N, const esdg::VolumeArgs<double>& a, cudaStream_t s) {
    switch (N) {
        case 1: return esdg::launch_volume_fp64ff_n1(a, s);
        case 2: return esdg::launch_volume_fp64ff_n2(a, s);
        case 3: return esdg::launch_volume_fp64ff_n3(a, s);
        case 4: return esdg::launch_volume_fp64ff_n4(a, s);
        case 5: return esdg::launch_volume_fp64ff_n5(a, s);
        case 6: return esdg::launch_volume_fp64ff_n6(a, s);
        case 7: return esdg::launch_volume_fp64ff_n7(a, s);
        case 8: return esdg::launch_volume_fp64ff_n8(a, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t dispatch_fp32(int N, const esdg::VolumeArgs<float>& a, cudaStream_t s) {
    switch (N) {
        case 1: return esdg::launch_volume_fp32_n1(a, s);
        case 2: return esdg::launch_volume_fp32_n2(a, s);
        case 3: return esdg::launch_volume_fp32_n3(a, s);
        case 4: return esdg::launch_volume_fp32_n4(a, s);
        case 5: return esdg::launch_volume_fp32_n5(a, s);
        case 6: return esdg::launch_volume_fp32_n6(a, s);
        case 7: return esdg::launch_volume_fp32_n7(a, s);
        case 8: return esdg::launch_volume_fp32_n8(a, s);
    }
    return cudaErrorInvalidValue;
}

int check_device(esdg_handle h) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(h, e, "cudaGetDevice");
    if (dev != h->device)
        return fail(h, ESDG_ERR_STATE, "handle was created on device " + std::to_string(h->device) +
                                           " but device " + std::to_string(dev) + " is current");
    return ESDG_OK;
}

}  // namespace

extern "C" {

int esdg_version(void) { return 100; }

int esdg_get_operators(int N, double* nodes, double* weights, double* D) {
    if (N < 1 || N > esdg::kMaxN) return fail(nullptr, ESDG_ERR_UNSUPPORTED, "N must be in 1..8");
    if (!nodes || !weights || !D) return fail(nullptr, ESDG_ERR_ARG, "null output pointer");
    esdg::lgl_operators(N, nodes, weights, D);
    return ESDG_OK;
}

int esdg_pair_schedule(int N, int precision, int* H_out, int* partner, int* sides) {
    if (N < 1 || N > esdg::kMaxN) return fail(nullptr, ESDG_ERR_UNSUPPORTED, "N must be in 1..8");
    if (precision != ESDG_FP64 && precision != ESDG_FP32 && precision != ESDG_FP64_FF)
        return fail(nullptr, ESDG_ERR_UNSUPPORTED, "precision must be ESDG_FP64, ESDG_FP32 or ESDG_FP64_FF");
    if (!H_out || !partner || !sides) return fail(nullptr, ESDG_ERR_ARG, "null output pointer");
    // Must match volume_kernel.cuh: direction_phase evaluates offsets
    // d < Nq/2 on every position.  For even Nq the antipodal offset d = Nq/2
    // is, in FP64 (SplitAntipodal), evaluated once by the lower position in
    // antipodal_phase; in FP32 both positions evaluate it and keep their own
    // share.
    const bool split = precision != ESDG_FP32;
    const int Nq = N + 1, H = Nq / 2;
    *H_out = H;
    for (int p = 0; p < Nq; ++p)
        for (int d = 1; d <= H; ++d) {
            const bool antipodal = (Nq % 2 == 0) && d == H;
            int pt = (p + d) % Nq, sd = 2;
            if (antipodal && split && p >= H) { pt = -1; sd = 0; }
            else if (antipodal && !split) sd = 1;
            partner[p * H + d - 1] = pt;
            sides[p * H + d - 1] = sd;
        }
    return ESDG_OK;
}

const char* esdg_last_error(esdg_handle h) {
    if (h) return h->err.c_str();
    return g_create_error.c_str();
}

int esdg_create(esdg_handle* out, long Kx, long Ky, long Kz, int N, int precision, int form) {
    if (!out) return fail(nullptr, ESDG_ERR_ARG, "out is NULL");
    *out = nullptr;
    if (N < 1 || N > esdg::kMaxN) return fail(nullptr, ESDG_ERR_UNSUPPORTED, "N must be in 1..8");
    if (precision != ESDG_FP64 && precision != ESDG_FP32 && precision != ESDG_FP64_FF)
        return fail(nullptr, ESDG_ERR_UNSUPPORTED, "precision must be ESDG_FP64, ESDG_FP32 or ESDG_FP64_FF");
    if (form != ESDG_FORM_2D && form != ESDG_FORM_SKEW)
        return fail(nullptr, ESDG_ERR_UNSUPPORTED, "form must be ESDG_FORM_2D or ESDG_FORM_SKEW");
    if (Kx < 1 || Ky < 1 || Kz < 1) return fail(nullptr, ESDG_ERR_ARG, "element counts must be >= 1");
    const long double Kld = (long double)Kx * Ky * Kz * (N + 1) * (N + 1) * (N + 1);
    if (Kld > (long double)(1LL << 40)) return fail(nullptr, ESDG_ERR_ARG, "mesh too large");

    esdg_ctx* h = new esdg_ctx();
    h->Kx = Kx; h->Ky = Ky; h->Kz = Kz;
    h->K = (long long)Kx * Ky * Kz;
    h->N = N;
    h->Nq = N + 1;
    h->n = h->K * h->Nq * h->Nq * h->Nq;
    h->precision = precision;
    h->form = form;
    esdg::lgl_operators(N, h->nodes, h->weights, h->D);
    esdg::fill_op_tables(h->op64, N);
    esdg::fill_op_tables(h->op32, N);
    cudaError_t e = cudaGetDevice(&h->device);
    if (e == cudaSuccess) e = cudaMalloc(&h->d_status, sizeof(unsigned));
    if (e == cudaSuccess) e = cudaMemset(h->d_status, 0, sizeof(unsigned));
    if (e == cudaSuccess) e = cudaMalloc(&h->d_partials, sizeof(double) * 3 * esdg::kDiagBlocks);
    if (e != cudaSuccess) {
        std::string msg = std::string("device status word: ") + cudaGetErrorString(e);
        if (h->d_status) cudaFree(h->d_status);
        if (h->d_partials) cudaFree(h->d_partials);
        delete h;
        return fail(nullptr, ESDG_ERR_CUDA, msg);
    }
    *out = h;
    return ESDG_OK;
}

int esdg_destroy(esdg_handle h) {
    if (!h) return ESDG_OK;
    if (h->d_status) cudaFree(h->d_status);
    if (h->d_partials) cudaFree(h->d_partials);
    delete h;
    return ESDG_OK;
}

int esdg_set_params(esdg_handle h, double gamma) {
    if (!h) return fail(nullptr, ESDG_ERR_ARG, "null handle");
    if (!(gamma > 1.0 && gamma < 10.0)) return fail(h, ESDG_ERR_ARG, "gamma must be in (1, 10)");
    h->gamma = gamma;
    return ESDG_OK;
}

int esdg_set_geometry(esdg_handle h, const double* x, const double* y, const double* z, void* metrics_out,
                      void* J_out, void* stream) {
    if (!h) return fail(nullptr, ESDG_ERR_ARG, "null handle");
    if (!x || !y || !z || !metrics_out) return fail(h, ESDG_ERR_ARG, "null coordinate or metrics pointer");
    if (!aligned16(x) || !aligned16(y) || !aligned16(z) || !aligned16(metrics_out) || (J_out && !aligned16(J_out)))
        return fail(h, ESDG_ERR_ALIGN, "device pointers must be 16-byte aligned");
    if (int rc = check_device(h)) return rc;
    esdg::GeometryArgs g;
    std::memset(&g, 0, sizeof(g));
    g.x = x; g.y = y; g.z = z;
    g.Ja = metrics_out;
    g.J = J_out;
    g.K = h->K;
    g.N = h->N;
    g.fp32 = h->precision == ESDG_FP32;
    std::memcpy(g.D, h->D, sizeof(double) * h->Nq * h->Nq);
    cudaError_t e = esdg::launch_geometry(g, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(h, e, "geometry kernel launch");
    return ESDG_OK;
}

static int volume_range(esdg_handle h, long e_begin, long e_count, const void* q, const void* metrics,
                        const void* phi, void* out, void* stream, int form) {
    if (!h) return fail(nullptr, ESDG_ERR_ARG, "null handle");
    if (!q || !metrics || !phi || !out) return fail(h, ESDG_ERR_ARG, "null device pointer");
    if (e_begin < 0 || e_count < 1 || e_begin + e_count > h->K)
        return fail(h, ESDG_ERR_ARG, "element range outside 0..K");
    if (!aligned16(q) || !aligned16(metrics) || !aligned16(phi) || !aligned16(out))
        return fail(h, ESDG_ERR_ALIGN, "device pointers must be 16-byte aligned");
    const size_t es = h->precision == ESDG_FP32 ? sizeof(float) : sizeof(double);
    const size_t nb = es * (size_t)h->n;
    if (overlaps(out, 5 * nb, q, 5 * nb) || overlaps(out, 5 * nb, metrics, 9 * nb) || overlaps(out, 5 * nb, phi, nb))
        return fail(h, ESDG_ERR_ARG, "out overlaps an input");
    if (int rc = check_device(h)) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (h->precision == ESDG_FP64)
        e = dispatch_fp64(h->N, volume_args<double>(h, q, metrics, phi, out, e_begin, e_begin + e_count, h->op64, form), s);
    else if (h->precision == ESDG_FP64_FF)
        e = dispatch_fp64ff(h->N, volume_args<double>(h, q, metrics, phi, out, e_begin, e_begin + e_count, h->op64, form), s);
    else
        e = dispatch_fp32(h->N, volume_args<float>(h, q, metrics, phi, out, e_begin, e_begin + e_count, h->op32, form), s);
    if (e != cudaSuccess) return cuda_fail(h, e, "volume kernel launch");
    return ESDG_OK;
}

int esdg_volume_rhs_range(esdg_handle h, long e_begin, long e_count, const void* q, const void* metrics,
                          const void* phi, void* out, void* stream) {
    if (!h) return fail(nullptr, ESDG_ERR_ARG, "null handle");
    return volume_range(h, e_begin, e_count, q, metrics, phi, out, stream, h->form);
}

int esdg_volume_rhs(esdg_handle h, const void* q, const void* metrics, const void* phi, void* out, void* stream) {
    if (!h) return fail(nullptr, ESDG_ERR_ARG, "null handle");
    return volume_range(h, 0, (long)h->K, q, metrics, phi, out, stream, h->form);
}

int esdg_set_boundary(esdg_handle h, int bc_xi, int bc_eta, int bc_zeta) {
    if (!h) return fail(nullptr, ESDG_ERR_ARG, "null handle");
    const int b[3] = {bc_xi, bc_eta, bc_zeta};
    for (int r = 0; r < 3; ++r)
        if (b[r] != ESDG_BC_PERIODIC && b[r] != ESDG_BC_WALL)
            return fail(h, ESDG_ERR_ARG, "boundary kind must be ESDG_BC_PERIODIC or ESDG_BC_WALL");
    for (int r = 0; r < 3; ++r) h->bc[r] = b[r];
    return ESDG_OK;
}

int esdg_set_dissipation(esdg_handle h, int on) {
    if (!h) return fail(nullptr, ESDG_ERR_ARG, "null handle");
    h->dissipation = on ? 1 : 0;
    return ESDG_OK;
}

static int surface_form(esdg_handle h, const void* q, const void* metrics, const void* phi, void* out, void* stream,
                        int form) {
    if (!h) return fail(nullptr, ESDG_ERR_ARG, "null handle");
    if (!q || !metrics || !phi || !out) return fail(h, ESDG_ERR_ARG, "null device pointer");
    if (!aligned16(q) || !aligned16(metrics) || !aligned16(phi) || !aligned16(out))
        return fail(h, ESDG_ERR_ALIGN, "device pointers must be 16-byte aligned");
    const size_t es = h->precision == ESDG_FP32 ? sizeof(float) : sizeof(double);
    const size_t nb = es * (size_t)h->n;
    if (overlaps(out, 5 * nb, q, 5 * nb) || overlaps(out, 5 * nb, metrics, 9 * nb) || overlaps(out, 5 * nb, phi, nb))
        return fail(h, ESDG_ERR_ARG, "out overlaps an input");
    if (int rc = check_device(h)) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (h->precision == ESDG_FP32)
        e = esdg::launch_surface_fp32(surface_args<float>(h, q, metrics, phi, out, form), h->N, s);
    else if (h->precision == ESDG_FP64_FF)
        e = esdg::launch_surface_fp64ff(surface_args<double>(h, q, metrics, phi, out, form), h->N, s);
    else
        e = esdg::launch_surface_fp64(surface_args<double>(h, q, metrics, phi, out, form), h->N, s);
    if (e != cudaSuccess) return cuda_fail(h, e, "surface kernel launch");
    return ESDG_OK;
}

int esdg_surface_rhs(esdg_handle h, const void* q, const void* metrics, const void* phi, void* out, void* stream) {
    if (!h) return fail(nullptr, ESDG_ERR_ARG, "null handle");
    return surface_form(h, q, metrics, phi, out, stream, h->form);
}

// Volume + surface.  The 2D volume form's diagonal f(q_i).Ja^r(i) at face
// nodes and the strong surface form's -f(q_i).n_own are equal and opposite,
// so the sum is the skew volume form plus F* alone: both kernels run in their
// skew forms, which skips that pair of terms (same result up to rounding).
int esdg_rhs(esdg_handle h, const void* q, const void* metrics, const void* phi, void* out, void* stream) {
    if (!h) return fail(nullptr, ESDG_ERR_ARG, "null handle");
    if (h->precision == ESDG_FP32) {
        // one launch: the volume kernel evaluates each element's faces itself
        // (one-sided, as in the fused stage) and writes volume + surface
        if (!q || !metrics || !phi || !out) return fail(h, ESDG_ERR_ARG, "null device pointer");
        if (!aligned16(q) || !aligned16(metrics) || !aligned16(phi) || !aligned16(out))
            return fail(h, ESDG_ERR_ALIGN, "device pointers must be 16-byte aligned");
        const size_t nb = sizeof(float) * (size_t)h->n;
        if (overlaps(out, 5 * nb, q, 5 * nb) || overlaps(out, 5 * nb, metrics, 9 * nb) ||
            overlaps(out, 5 * nb, phi, nb))
            return fail(h, ESDG_ERR_ARG, "out overlaps an input");
        if (int rc = check_device(h)) return rc;
        auto a = volume_args<float>(h, q, metrics, phi, out, 0, h->K, h->op32, ESDG_FORM_SKEW);
        a.with_faces = 1;
        set_face_fields(h, a);
        const cudaError_t e = dispatch_fp32(h->N, a, static_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return cuda_fail(h, e, "volume kernel launch (volume + faces)");
        return ESDG_OK;
    }
    if (int rc = volume_range(h, 0, (long)h->K, q, metrics, phi, out, stream, ESDG_FORM_SKEW)) return rc;
    return surface_form(h, q, metrics, phi, out, stream, ESDG_FORM_SKEW);
}

int esdg_lsrk_coefficients(int* stages, double* A, double* B, double* C) {
    if (!stages) return fail(nullptr, ESDG_ERR_ARG, "stages is NULL");
    *stages = 5;
    for (int k = 0; k < 5; ++k) {
        if (A) A[k] = lsrk_coef(kLsrkA[k]);
        if (B) B[k] = lsrk_coef(kLsrkB[k]);
        if (C) C[k] = lsrk_coef(kLsrkC[k]);
    }
    return ESDG_OK;
}

int esdg_set_reference(esdg_handle h, const void* rho_ref, const void* p_ref) {
    if (!h) return fail(nullptr, ESDG_ERR_ARG, "null handle");
    if ((rho_ref == nullptr) != (p_ref == nullptr))
        return fail(h, ESDG_ERR_ARG, "rho_ref and p_ref must both be set or both be NULL");
    if ((rho_ref && !aligned16(rho_ref)) || (p_ref && !aligned16(p_ref)))
        return fail(h, ESDG_ERR_ALIGN, "device pointers must be 16-byte aligned");
    h->ref_rho = rho_ref;
    h->ref_p = p_ref;
    return ESDG_OK;
}

int esdg_set_coriolis(esdg_handle h, double f) {
    if (!h) return fail(nullptr, ESDG_ERR_ARG, "null handle");
    if (!(f == f) || f > 1.0 || f < -1.0) return fail(h, ESDG_ERR_ARG, "|f| must be at most 1 s^-1");
    h->coriolis = f;
    return ESDG_OK;
}

int esdg_rk_stage(esdg_handle h, void* q, void* dq, const void* rhs, const void* J, double a, double b, double dt,
                  void* stream) {
    if (!h) return fail(nullptr, ESDG_ERR_ARG, "null handle");
    if (!q || !dq || !rhs || !J) return fail(h, ESDG_ERR_ARG, "null device pointer");
    if (!aligned16(q) || !aligned16(dq) || !aligned16(rhs) || !aligned16(J))
        return fail(h, ESDG_ERR_ALIGN, "device pointers must be 16-byte aligned");
    const size_t es = h->precision == ESDG_FP32 ? sizeof(float) : sizeof(double);
    const size_t nb = es * (size_t)h->n;
    if (overlaps(q, 5 * nb, dq, 5 * nb) || overlaps(q, 5 * nb, rhs, 5 * nb) || overlaps(dq, 5 * nb, rhs, 5 * nb) ||
        overlaps(q, 5 * nb, J, nb) || overlaps(dq, 5 * nb, J, nb))
        return fail(h, ESDG_ERR_ARG, "q, dq, rhs and J must not overlap");
    if (int rc = check_device(h)) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (h->precision == ESDG_FP32) {
        esdg::RkArgs<float> r{static_cast<float*>(q), static_cast<float*>(dq), static_cast<const float*>(rhs),
                              static_cast<const float*>(J), h->n, (float)a, (float)b, (float)dt,
                              (float)h->coriolis};
        e = esdg::launch_rk_stage(r, s);
    } else {
        esdg::RkArgs<double> r{static_cast<double*>(q), static_cast<double*>(dq), static_cast<const double*>(rhs),
                               static_cast<const double*>(J), h->n, a, b, dt, h->coriolis};
        e = esdg::launch_rk_stage(r, s);
    }
    if (e != cudaSuccess) return cuda_fail(h, e, "Runge-Kutta stage launch");
    return ESDG_OK;
}

// One fused stage: the surface term (skew form) accumulated into S at face
// nodes, then the volume kernel (skew form) adds it and applies the stage
// update to dq and q in its store, resetting S to zero where it read it.
// One fused stage.  FP32: volume and surface in one launch, reading q and
// writing the new state to q_out (!= q).  Float-float: the surface term into
// S, then the volume kernel consuming S and updating q in place (q_out == q).
static int fused_stage(esdg_handle h, void* q, void* q_out, void* dq, void* S, const void* metrics,
                       const void* phi, const void* J, double A, double B, double dt, void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (h->precision == ESDG_FP32) {
        auto a = volume_args<float>(h, q, metrics, phi, nullptr, 0, h->K, h->op32, ESDG_FORM_SKEW);
        a.rk_q = static_cast<float*>(q);
        a.rk_qout = static_cast<float*>(q_out);
        a.rk_dq = static_cast<float*>(dq);
        a.rk_J = static_cast<const float*>(J);
        a.rk_A = (float)A;
        a.rk_B = (float)B;
        a.rk_dt = (float)dt;
        a.rk_f = (float)h->coriolis;
        set_face_fields(h, a);
        e = dispatch_fp32(h->N, a, s);
    } else {
        if (int rc = surface_form(h, q, metrics, phi, S, stream, ESDG_FORM_SKEW)) return rc;
        auto a = volume_args<double>(h, q, metrics, phi, nullptr, 0, h->K, h->op64, ESDG_FORM_SKEW);
        a.rk_q = static_cast<double*>(q);
        a.rk_qout = static_cast<double*>(q);
        a.rk_dq = static_cast<double*>(dq);
        a.rk_S = static_cast<double*>(S);
        a.rk_J = static_cast<const double*>(J);
        a.rk_A = A;
        a.rk_B = B;
        a.rk_dt = dt;
        a.rk_f = h->coriolis;
        e = h->precision == ESDG_FP64_FF ? dispatch_fp64ff(h->N, a, s) : dispatch_fp64(h->N, a, s);
    }
    if (e != cudaSuccess) return cuda_fail(h, e, "volume kernel launch (fused stage)");
    return ESDG_OK;
}

int esdg_lsrk_step(esdg_handle h, void* q, void* dq, void* rhs, const void* metrics, const void* phi, const void* J,
                   double dt, void* stream) {
    if (!h) return fail(nullptr, ESDG_ERR_ARG, "null handle");
    if (!q || !dq || !rhs || !metrics || !phi || !J) return fail(h, ESDG_ERR_ARG, "null device pointer");
    if (!aligned16(q) || !aligned16(dq) || !aligned16(rhs) || !aligned16(metrics) || !aligned16(phi) ||
        !aligned16(J))
        return fail(h, ESDG_ERR_ALIGN, "device pointers must be 16-byte aligned");
    const size_t es = h->precision == ESDG_FP32 ? sizeof(float) : sizeof(double);
    const size_t nb = es * (size_t)h->n;
    const void* ins[4] = {q, dq, rhs, J};
    const size_t sz[4] = {5 * nb, 5 * nb, 5 * nb, nb};
    for (int x = 0; x < 4; ++x)
        for (int y = x + 1; y < 4; ++y)
            if (overlaps(ins[x], sz[x], ins[y], sz[y])) return fail(h, ESDG_ERR_ARG, "q, dq, rhs and J must not overlap");
    if (overlaps(q, 5 * nb, metrics, 9 * nb) || overlaps(q, 5 * nb, phi, nb) || overlaps(rhs, 5 * nb, metrics, 9 * nb) ||
        overlaps(rhs, 5 * nb, phi, nb) || overlaps(dq, 5 * nb, metrics, 9 * nb) || overlaps(dq, 5 * nb, phi, nb))
        return fail(h, ESDG_ERR_ARG, "q, dq and rhs must not overlap metrics or phi");
    if (int rc = check_device(h)) return rc;
    if (h->precision == ESDG_FP64) {
        // native FP64: the volume kernel is bound by the FP64 pipe, where the
        // fused update's extra FP64 work and tail loads cost more (0.23 ms per
        // stage on the N = 7 channel) than the separate stage kernel (0.16 ms)
        for (int k = 0; k < 5; ++k) {
            if (int rc = esdg_rhs(h, q, metrics, phi, rhs, stream)) return rc;
            if (int rc = esdg_rk_stage(h, q, dq, rhs, J, lsrk_coef(kLsrkA[k]), lsrk_coef(kLsrkB[k]), dt, stream))
                return rc;
        }
        return ESDG_OK;
    }
    if (h->precision == ESDG_FP32) {
        // state buffers alternate q -> rhs -> q ...; five stages end in rhs
        void* buf[2] = {q, rhs};
        for (int k = 0; k < 5; ++k)
            if (int rc = fused_stage(h, buf[k & 1], buf[(k + 1) & 1], dq, nullptr, metrics, phi, J,
                                     lsrk_coef(kLsrkA[k]), lsrk_coef(kLsrkB[k]), dt, stream))
                return rc;
        const cudaError_t e =
            cudaMemcpyAsync(q, rhs, 5 * nb, cudaMemcpyDeviceToDevice, static_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return cuda_fail(h, e, "copying the new state back to q");
        return ESDG_OK;
    }
    // float-float: rhs serves as the face accumulator S: zero at the start,
    // and every stage leaves it zero again
    cudaError_t e = cudaMemsetAsync(rhs, 0, 5 * nb, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(h, e, "clearing the surface accumulator");
    for (int k = 0; k < 5; ++k)
        if (int rc = fused_stage(h, q, q, dq, rhs, metrics, phi, J, lsrk_coef(kLsrkA[k]), lsrk_coef(kLsrkB[k]),
                                 dt, stream))
            return rc;
    return ESDG_OK;
}

int esdg_diagnostics(esdg_handle h, const void* q, const void* J, const void* phi, double* out3, void* stream) {
    if (!h) return fail(nullptr, ESDG_ERR_ARG, "null handle");
    if (!q || !J || !phi || !out3) return fail(h, ESDG_ERR_ARG, "null device pointer");
    if (!aligned16(q) || !aligned16(J) || !aligned16(phi))
        return fail(h, ESDG_ERR_ALIGN, "device pointers must be 16-byte aligned");
    if (int rc = check_device(h)) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (h->precision == ESDG_FP32)
        e = esdg::launch_diagnostics(diag_args<float>(h, q, J, phi), out3, s);
    else
        e = esdg::launch_diagnostics(diag_args<double>(h, q, J, phi), out3, s);
    if (e != cudaSuccess) return cuda_fail(h, e, "diagnostics launch");
    return ESDG_OK;
}

int esdg_describe(esdg_handle h, int* precision, int* N, long long* n) {
    if (!h) return fail(nullptr, ESDG_ERR_ARG, "null handle");
    if (precision) *precision = h->precision;
    if (N) *N = h->N;
    if (n) *n = h->n;
    return ESDG_OK;
}

int esdg_get_status(esdg_handle h, unsigned* flags, void* stream) {
    if (!h) return fail(nullptr, ESDG_ERR_ARG, "null handle");
    if (!flags) return fail(h, ESDG_ERR_ARG, "flags is NULL");
    if (int rc = check_device(h)) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, h->d_status, sizeof(unsigned), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(h->d_status, 0, sizeof(unsigned), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(h, e, "reading the status word");
    *flags = v;
    return ESDG_OK;
}

}  // extern "C"
