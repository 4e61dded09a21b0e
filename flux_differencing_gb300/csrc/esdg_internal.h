// Internal declarations shared by the host API and the kernel translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <string>

namespace esdg {

constexpr int kMaxN = 8;
constexpr int kMaxNq = kMaxN + 1;

// Operator tables passed by value to the volume kernel (they live in the
// kernel's parameter space, i.e. the constant bank).
//   Q2[i*Nq + j] = 2 w_i D_ij   (twice the SBP matrix Q = W D)
//   invw[i]      = 1 / w_i
//   diag[i]      = 2 D_ii at the end nodes i = 0, N (the 2D form's diagonal
//                  factor), 0 at interior nodes
template <typename T>
struct OpTables {
    T Q2[kMaxNq * kMaxNq];
    T invw[kMaxNq];
    T diag[kMaxNq];
};

// Fill the tables of order N from the library's LGL operators (host).
template <typename T>
void fill_op_tables(OpTables<T>& t, int N);

// Surface term: constants derived from gamma.
template <typename T>
struct SurfaceConsts {
    T gm1;     // gamma - 1
    T igm1;    // 1/(gamma - 1)
    T c_g;     // 1/(2 (gamma - 1))
    T gamma;
    T c_ac;    // 1/(4 gamma): half the acoustic-wave entry 1/(2 gamma) of the eigenvector scaling
    T c_en;    // (gamma - 1)/(2 gamma): half the entropy-wave entry (gamma - 1)/gamma
};

template <typename T>
struct VolumeArgs {
    const T* q;        // 5 planes
    const T* Ja;       // 9 planes
    const T* phi;      // 1 plane
    T* out;            // 5 planes
    long long n;       // plane stride (all nodes of the mesh)
    long long e_begin; // first element of this launch
    long long e_end;   // one past the last element
    T gm1;             // gamma - 1
    T c_g;             // 1 / (2 (gamma - 1))
    T c_h;             // gamma / (2 (gamma - 1))
    int form;          // 0: 2D form (diagonal kept), 1: skew form
    unsigned* status;  // device status word (atomicOr of ESDG_STATUS_* bits)
    const T* rho_ref;  // reference density (1 plane) or nullptr: q is then the full state
    const T* p_ref;    // reference pressure (1 plane), with rho_ref
    // Fused Runge-Kutta stage (rk_q != nullptr): instead of writing out, each
    // node takes rhs = volume + surface and applies
    // dq <- A dq + dt (h - rhs/J), q <- q + B dq to rk_dq and q.
    //  * float-float: the surface term comes accumulated in rk_S at face
    //    nodes (consumed and reset to zero there); q is updated in place
    //    (rk_q == q, rk_qout == rk_q).
    //  * FP32: the kernel evaluates each element's faces itself (one-sided,
    //    with the surface fields below) and writes the new state to rk_qout,
    //    a second buffer: neighbouring elements read their face traces from q
    //    during the launch.  rk_S is unused.
    T* rk_q;
    T* rk_qout;
    T* rk_dq;
    T* rk_S;
    const T* rk_J;
    T rk_A, rk_B, rk_dt, rk_f;
    // FP32, rk_q == nullptr: also evaluate the surface term (skew form, with
    // the surface fields below) in the kernel and write volume + surface to out
    int with_faces;
    // surface fields of the FP32 fused stage and of with_faces
    long long Kx, Ky, Kz;  // element e = ex + Kx (ey + Ky ez)
    int bc[3];             // per direction: 0 periodic, 1 slip wall
    int dissipation;       // 0: entropy-conserving interface flux only
    T inv_w0;              // 1 / (LGL end weight)
    SurfaceConsts<T> sk;
    OpTables<T> ops;
};

// Launchers, one per (precision, N); defined in the instantiation units.
// fp64ff: FP64 inputs and outputs, pair arithmetic in float-float.
#define ESDG_DECLARE_LAUNCH(N)                                                         \
    cudaError_t launch_volume_fp64_n##N(const VolumeArgs<double>& a, cudaStream_t s);   \
    cudaError_t launch_volume_fp32_n##N(const VolumeArgs<float>& a, cudaStream_t s);    \
    cudaError_t launch_volume_fp64ff_n##N(const VolumeArgs<double>& a, cudaStream_t s);
ESDG_DECLARE_LAUNCH(1)
ESDG_DECLARE_LAUNCH(2)
ESDG_DECLARE_LAUNCH(3)
ESDG_DECLARE_LAUNCH(4)
ESDG_DECLARE_LAUNCH(5)
ESDG_DECLARE_LAUNCH(6)
ESDG_DECLARE_LAUNCH(7)
ESDG_DECLARE_LAUNCH(8)
#undef ESDG_DECLARE_LAUNCH

template <typename T>
struct SurfaceArgs {
    const T* q;        // 5 planes
    const T* Ja;       // 9 planes
    const T* phi;      // 1 plane
    T* out;            // 5 planes, accumulated into
    long long n;       // plane stride
    long long Kx, Ky, Kz;
    int bc[3];         // per direction: 0 periodic, 1 slip wall
    int form;          // 0: 2D form (subtract the physical flux), 1: skew form
    int dissipation;   // 0: entropy-conserving flux only
    T inv_w0;          // 1 / (LGL end weight)
    SurfaceConsts<T> k;
    unsigned* status;
    const T* rho_ref;  // as in VolumeArgs
    const T* p_ref;
};

// Launch the three direction passes of the surface term (one per launch).
cudaError_t launch_surface_fp64(const SurfaceArgs<double>& a, int N, cudaStream_t s);
cudaError_t launch_surface_fp32(const SurfaceArgs<float>& a, int N, cudaStream_t s);
// FP64 buffers, float-float arithmetic
cudaError_t launch_surface_fp64ff(const SurfaceArgs<double>& a, int N, cudaStream_t s);

// One stage of the 2N-storage Runge-Kutta update (all pointers device, planes
// of stride n): dq <- A dq + dt (h - rhs/J), q <- q + B dq.
template <typename T>
struct RkArgs {
    T* q;              // 5 planes
    T* dq;             // 5 planes
    const T* rhs;      // 5 planes: volume + surface
    const T* J;        // 1 plane
    long long n;
    T A, B, dt;
    T coriolis;        // f of the f-plane source (0, f rho u2, -f rho u1, 0, 0)
};
template <typename T>
cudaError_t launch_rk_stage(const RkArgs<T>& a, cudaStream_t s);

// Global integrals (mass, total energy, entropy) with a fixed two-level
// reduction over kDiagBlocks CTAs.
constexpr int kDiagBlocks = 608;
template <typename T>
struct DiagArgs {
    const T* q;
    const T* J;
    const T* phi;
    const T* rho_ref;  // as in VolumeArgs
    const T* p_ref;
    long long n;
    int Nq, np3;
    double gamma, gm1;
    double w[kMaxNq];  // LGL weights
    double* partials;  // 3 * kDiagBlocks doubles
};
template <typename T>
cudaError_t launch_diagnostics(const DiagArgs<T>& a, double* out, cudaStream_t s);

// Geometry: curl-form metrics in FP64 from node coordinates.
struct GeometryArgs {
    const double* x;
    const double* y;
    const double* z;
    void* Ja;          // 9 planes, double or float
    void* J;           // 1 plane or nullptr
    long long K;
    int N;
    int fp32;          // output element type
    double D[kMaxNq * kMaxNq];
};
cudaError_t launch_geometry(const GeometryArgs& a, cudaStream_t s);

// Host-side operators (long double internally, rounded once to double).
void lgl_operators(int N, double* nodes, double* weights, double* D);

// Record the message that esdg_last_error(NULL) returns on this thread (for
// entry points that have no handle).
void set_unhandled_error(const char* msg);
inline void set_unhandled_error(const std::string& msg) { set_unhandled_error(msg.c_str()); }

}  // namespace esdg
