/*
 * esdg.h -- C-ABI of the GB300 flux-differencing volume-term library.
 *
 * The library evaluates the volume term of the entropy-stable discontinuous
 * Galerkin (ESDG) discretisation of the Euler equations with buoyancy in
 * "GPU Performance of an Entropy-Stable Discontinuous Galerkin Euler Solver
 * with Non-Conservative Terms" (Sec. 3 Eq. 2, volume part; Sec. 4.1 Eqs. 3-6
 * and Fig. 1).  For every hexahedral element of (N+1)^3 Legendre-Gauss-Lobatto
 * (LGL) nodes, every node i and every reference direction r it forms
 *
 *     out_i = sum_r sum_{m on the r-line through i} 2 D_{a_r(i) a_r(m)} F^r(q_i, q_m)
 *
 * where F^r is the two-point entropy-conservative flux of Eqs. 3-4 contracted
 * with the averaged metric terms (Ja^r(i) + Ja^r(m))/2, plus the
 * non-conservative two-point gravity term of Eqs. 4-5 (rho_hat [[phi]] / 2).
 * The output is NOT divided by the Jacobian J and NOT negated: the volume
 * contribution to dq/dt is -out / J.  The Coriolis source h of Eq. 2 is not
 * included.
 *
 * Conventions shared by every call:
 *   - element e = ex + Kx*(ey + Ky*ez); node = a + Nq*(b + Nq*c) with Nq = N+1,
 *     a along the first reference direction (xi), b along eta, c along zeta.
 *   - n = K * Nq^3 nodes, K = Kx*Ky*Kz.  Every field is stored as planes of n
 *     values: value (v, e, node) sits at offset v*n + e*Nq^3 + node.
 *   - q:       5 planes (rho, rho*u1, rho*u2, rho*u3, E), E = p/(gamma-1) +
 *              rho|u|^2/2 + rho*phi (Sec. 2).
 *   - metrics: 9 planes, plane 3*r + j holds Ja^r_j = J d(xi_r)/d(x_j).
 *   - phi:     1 plane, the geopotential g*z at the nodes.
 *   - out:     5 planes in the order of q.
 *   - "precision" selects the element type of q, metrics, phi, out and J:
 *     ESDG_FP64 -> double, ESDG_FP32 -> float.  Node coordinates are always
 *     double.
 *   - Device pointers must be 16-byte aligned.  The caller allocates and owns
 *     every buffer and stream; the library never frees caller memory.
 *   - Streams are passed as cudaStream_t cast to void* (NULL = legacy default).
 *   - Calls are asynchronous on the given stream unless stated otherwise.
 *   - Every call returns ESDG_OK or an ESDG_ERR_* code; on error nothing is
 *     launched and esdg_last_error() describes the cause.
 *   - A handle is not thread-safe: use one handle per host thread.
 */
#ifndef ESDG_H
#define ESDG_H

#ifdef __cplusplus
extern "C" {
#endif

typedef struct esdg_ctx* esdg_handle;
typedef struct esdg_pipeline_s* esdg_pipeline;

enum {
    ESDG_OK = 0,
    ESDG_ERR_ARG = 1,          /* null handle/pointer, bad size, aliasing */
    ESDG_ERR_UNSUPPORTED = 2,  /* N outside 1..8, unknown precision or form */
    ESDG_ERR_ALIGN = 3,        /* a device pointer is not 16-byte aligned */
    ESDG_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
    ESDG_ERR_STATE = 5         /* call not valid in the handle's state */
};

/* ESDG_FP64_FF: FP64 inputs, metrics and outputs (element type double, the
 * same buffers as ESDG_FP64); the per-node precompute runs in FP64 and the
 * pair arithmetic in float-float (each value the unevaluated sum of two
 * floats, about 48 significant bits) on the FP32 pipes, which on GB300 run at
 * 64 times the FP64 rate.  Results agree with the FP64 oracle within the same
 * 1e-11 tolerance as ESDG_FP64.  Values must stay inside the FP32 exponent
 * range (about 1e-30 .. 1e38 in magnitude for full accuracy). */
enum { ESDG_FP64 = 0, ESDG_FP32 = 1, ESDG_FP64_FF = 2 };

/* ESDG_FORM_2D keeps the diagonal pairs m == i (the strong form whose
 * diagonal contributes 2 D_ii Ja^r(i).f(q_i) at the two end nodes of a line);
 * ESDG_FORM_SKEW drops them (the skew-symmetric operator whose diagonal is
 * zero; Fig. 1 omits diagonal pairs).  The two differ only at element-face
 * nodes, by exactly that end-node flux. */
enum { ESDG_FORM_2D = 0, ESDG_FORM_SKEW = 1 };

/* Status bits set by kernels and read with esdg_get_status(). */
enum {
    ESDG_STATUS_NONPHYSICAL = 1u, /* some node had rho <= 0, p <= 0 or NaN */
    ESDG_STATUS_INDEX = 4u        /* debug library only (libesdg_debug.so): a kernel computed a
                                     shared-memory, face-slot or global index out of range (the
                                     access was redirected in bounds; results are then invalid) */
};

/* Create a handle for a mesh of Kx*Ky*Kz elements of order N (1..8).
 * Builds the LGL nodes, weights and differentiation matrix (Sec. 3) on the
 * host in long double.  Allocates host memory, one 4-byte device status
 * word and a 14.6 KB diagnostics scratch buffer on the current device; the
 * handle must be used on that device.
 * Errors: ESDG_ERR_ARG (out == NULL, K < 1 or K*Nq^3 > 2^40),
 * ESDG_ERR_UNSUPPORTED (N, precision or form), ESDG_ERR_CUDA. */
int esdg_create(esdg_handle* out, long Kx, long Ky, long Kz, int N, int precision, int form);

/* Release the handle and its status word.  Not stream-ordered: the caller
 * must make sure no launch that uses the handle is still running.
 * Accepts NULL. */
int esdg_destroy(esdg_handle h);

/* Ratio of specific heats (default 1.4).  Errors: ESDG_ERR_ARG unless
 * 1 < gamma < 10. */
int esdg_set_params(esdg_handle h, double gamma);

/* Metric terms of the element geometry (Sec. 3, G_jk) in the conservative
 * curl form Ja^r_j = -(curl_xi (X_l grad_xi X_m))_r, (j, m, l) cyclic, with
 * every derivative taken by the LGL differentiation matrix, computed in FP64
 * on the GPU and rounded to the handle's precision.  Also J = x_xi . (x_eta x
 * x_zeta) when J_out != NULL.
 *   x, y, z      device, double, n values each: node coordinates.
 *   metrics_out  device, 9*n values of the handle's precision (written).
 *   J_out        device, n values of the handle's precision, or NULL.
 * Errors: ESDG_ERR_ARG (null handle or pointers), ESDG_ERR_ALIGN,
 * ESDG_ERR_CUDA. */
int esdg_set_geometry(esdg_handle h, const double* x, const double* y, const double* z,
                      void* metrics_out, void* J_out, void* stream);

/* The volume term for all K elements (see the top of this file).
 *   q        device, 5*n values (read).
 *   metrics  device, 9*n values (read).
 *   phi      device, n values (read).
 *   out      device, 5*n values (written); must not overlap any input.
 * Enqueues one kernel launch on `stream`; no synchronisation and no
 * allocation.  Nodes with rho <= 0 or p <= 0 set ESDG_STATUS_NONPHYSICAL in
 * the handle's status word and produce non-finite values; nothing traps.
 * Errors: ESDG_ERR_ARG, ESDG_ERR_ALIGN, ESDG_ERR_CUDA (launch failure). */
int esdg_volume_rhs(esdg_handle h, const void* q, const void* metrics, const void* phi,
                    void* out, void* stream);

/* As esdg_volume_rhs, restricted to elements [e_begin, e_begin + e_count)
 * of the same full-size arrays (planes keep their stride n).  Elements are
 * independent, so disjoint ranges compose bitwise into the full result; this
 * is how the element range of a mesh is split across calls, streams or
 * devices.  Errors as esdg_volume_rhs, plus ESDG_ERR_ARG when the range is
 * empty or leaves 0..K. */
int esdg_volume_rhs_range(esdg_handle h, long e_begin, long e_count, const void* q,
                          const void* metrics, const void* phi, void* out, void* stream);

/* Boundary kinds of the surface term, per reference direction of the brick
 * of elements (element e = ex + Kx (ey + Ky ez)). */
enum { ESDG_BC_PERIODIC = 0, ESDG_BC_WALL = 1 };

/* Boundary kind of each reference direction for esdg_surface_rhs (default
 * periodic in all three).  ESDG_BC_WALL is a slip wall: the state outside
 * the face is the mirror image (rho, m - 2 (m.n^) n^, E) of the inside state
 * with the same phi, so no mass or energy crosses it.
 * Errors: ESDG_ERR_ARG (null handle or unknown kind). */
int esdg_set_boundary(esdg_handle h, int bc_xi, int bc_eta, int bc_zeta);

/* on != 0 (default): the surface flux is the entropy-conserving flux minus
 * the matrix dissipation; on == 0: the entropy-conserving flux alone (the
 * semi-discrete scheme then conserves entropy, which tests use). */
int esdg_set_dissipation(esdg_handle h, int on);

/* The surface term of Eq. 2 (Sec. 3 of the ESDG GPU paper: the surface flux
 * F* is the entropy-conserving flux plus matrix dissipation, "akin to a Roe
 * Riemann solver"; the paper leaves the formula to its reference), ADDED
 * into out.  At every face node i of every element, with j the node of the
 * neighbouring element at the same position (or the wall's mirror state):
 *     out_i += (1/w_0) [ F*(q_i, q_j; n) - f(q_i) . n_own ]     (ESDG_FORM_2D)
 *     out_i += (1/w_0) F*(q_i, q_j; n)                          (ESDG_FORM_SKEW)
 * with w_0 the LGL end weight, n = +-(Ja^r(i) + Ja^r(j))/2 the outward
 * averaged normal (n = n_own = +-Ja^r(i) at a wall), f the physical flux and
 *     F* = F_ec(q_i, q_j; n) + G(i, j; n) - 1/2 |n| R |Lambda| T R^T [[w]],
 * F_ec + G the volume term's two-point flux (Eqs. 3-5), [[w]] = w_j - w_i the
 * jump of the entropy variables, and R, Lambda, T the eigenvectors,
 * eigenvalues (unit normal) and entropy scaling (R T R^T = dq/dw) of the
 * flux Jacobian at the averaged state rho_ln, {{u}}, {{rho}}/(2{{b}}),
 * {{phi}}.  So out = volume + surface after esdg_volume_rhs then this call
 * on the same stream, and dq/dt = -out/J.
 *   q, metrics, phi  device, as esdg_volume_rhs (read).
 *   out              device, 5*n values (read and written); must not overlap
 *                    an input.
 * Enqueues three kernel launches (one per reference direction) on `stream`;
 * no synchronisation and no allocation.  ESDG_FP64_FF handles run the
 * surface arithmetic in float-float, like their volume term.  Non-physical
 * states set ESDG_STATUS_NONPHYSICAL.
 * Errors: ESDG_ERR_ARG, ESDG_ERR_ALIGN, ESDG_ERR_CUDA (launch failure). */
int esdg_surface_rhs(esdg_handle h, const void* q, const void* metrics, const void* phi,
                     void* out, void* stream);

/* Perturbation variables (Sec. 5.2 of the ESDG GPU paper attributes its FP32
 * pressure noise to carrying the full state and names perturbation variables
 * as the remedy).  After this call every q argument of the handle's
 * entry points (volume, surface, Runge-Kutta stage and step, diagnostics) is
 * the perturbation q' = q - (rho_ref, 0, 0, 0, E_ref) from a reference state
 * at rest, E_ref = p_ref/(gamma-1) + rho_ref phi; the kernels form
 * rho = rho_ref + rho' and p = p_ref + (gamma-1)(E' - rho|u|^2/2 - rho' phi),
 * which avoids the cancellation of E against rho phi and p/(gamma-1), and the
 * time step accumulates the small q' rather than the large q.  The output
 * (volume + surface) is unchanged in meaning: the divergence of the full
 * state's fluxes (so dq'/dt = dq/dt).  The reference is typically a
 * hydrostatic background, but any positive state works.
 *   rho_ref, p_ref  device, n values each of the handle's precision (read
 *                   by every later call; the caller keeps them alive), or
 *                   both NULL to return to full-state variables.
 * esdg_volume_rhs_noalloc always takes full-state variables.
 * Errors: ESDG_ERR_ARG (only one pointer NULL), ESDG_ERR_ALIGN. */
int esdg_set_reference(esdg_handle h, const void* rho_ref, const void* p_ref);

/* ---- time stepping (the semi-discrete system of Eq. 2) -------------------
 * dq/dt = h - (volume + surface)/J, advanced with the five-stage fourth-order
 * 2N-storage Runge-Kutta scheme of Carpenter and Kennedy (1994), which the
 * ESDG GPU paper (Sec. 3) names as the scheme it used before its fourteen-
 * stage one (whose coefficients it does not print).  h is the f-plane
 * Coriolis source of Eq. 2's h term: (0, f rho u2, -f rho u1, 0, 0). */

/* The scheme's coefficients: *stages = 5; A, B, C (5 doubles each, any may
 * be NULL) receive A_k, B_k and the stage times c_k of
 *     dq <- A_k dq + dt L(q),   q <- q + B_k dq.
 * Host only.  Errors: ESDG_ERR_ARG (stages NULL). */
int esdg_lsrk_coefficients(int* stages, double* A, double* B, double* C);

/* Coriolis parameter f in s^-1 (default 0).  Errors: ESDG_ERR_ARG (|f| > 1). */
int esdg_set_coriolis(esdg_handle h, double f);

/* One Runge-Kutta stage on every node:
 *     dq <- a dq + dt (h(q) - rhs/J),   q <- q + b dq.
 *   q    device, 5*n values (read and written).
 *   dq   device, 5*n values (written; also read unless a == 0, so a first
 *        stage needs no initialised dq).
 *   rhs  device, 5*n values (read): volume + surface at q.
 *   J    device, n values (read): the Jacobian from esdg_set_geometry.
 * All of the handle's precision (FP64 for ESDG_FP64_FF); none may overlap.
 * Enqueues one launch on `stream`.  Errors: ESDG_ERR_ARG, ESDG_ERR_ALIGN,
 * ESDG_ERR_CUDA. */
int esdg_rk_stage(esdg_handle h, void* q, void* dq, const void* rhs, const void* J, double a, double b,
                  double dt, void* stream);

/* One full time step of size dt: five stages of esdg_rhs (boundary kinds
 * and dissipation of the handle) and esdg_rk_stage, the same arithmetic
 * organised per precision:
 *  - ESDG_FP32: one launch per stage.  The volume kernel also evaluates each
 *    element's faces (from the element's own side, reading the neighbours'
 *    face traces) and applies the stage update in its store; since the
 *    neighbours read q during the launch, stages alternate between q and
 *    rhs as state buffers and a final device copy returns the state to q
 *    (5 launches and one copy per step).
 *  - ESDG_FP64_FF: per stage the surface term into an accumulator, then the
 *    volume kernel adding it and applying the update in place (20 launches
 *    and one memset per step).
 *  - ESDG_FP64, bound by its FP64 pipe: esdg_rhs and the separate stage
 *    kernel (25 launches).
 * Everything is on `stream`, with no synchronisation and no allocation (so
 * the call can be captured into a CUDA graph).  rhs is scratch (5*n values:
 * the second state buffer, the surface accumulator or the right-hand side).
 * q, dq, rhs and J must not overlap one another, metrics or phi.  Errors: as
 * the component calls. */
int esdg_lsrk_step(esdg_handle h, void* q, void* dq, void* rhs, const void* metrics, const void* phi,
                   const void* J, double dt, void* stream);

/* Global integrals of the state, written to out3 (device, 3 doubles):
 * mass sum_i w_i J_i rho_i, total energy sum_i w_i J_i E_i and entropy
 * sum_i w_i J_i eta_i with eta = -rho s/(gamma-1), s = ln(p rho^-gamma) and
 * w_i the product of the node's three LGL weights.  FP64 accumulation with a
 * fixed reduction order (bitwise reproducible); uses the handle's scratch
 * (so calls on one handle must not run concurrently).  Two launches on
 * `stream`.  Errors: ESDG_ERR_ARG, ESDG_ERR_ALIGN, ESDG_ERR_CUDA. */
int esdg_diagnostics(esdg_handle h, const void* q, const void* J, const void* phi, double* out3,
                     void* stream);

/* Shape of a handle: *precision (ESDG_FP64, ESDG_FP32, ESDG_FP64_FF), order N
 * and node count n = K (N+1)^3; any output pointer may be NULL.  Host only.
 * Errors: ESDG_ERR_ARG (null handle). */
int esdg_describe(esdg_handle h, int* precision, int* N, long long* n);

/* ---- pipelined evaluation from host buffers ------------------------------
 * For callers whose state lives in host memory.  A pipeline owns `depth`
 * slots, each with device buffers for q, metrics, phi and out (of the
 * handle's precision) and a stream; esdg_pipeline_submit enqueues, on the
 * next slot, the host-to-device copies of the inputs, esdg_volume_rhs and the
 * copy of the result to out_host, and returns without waiting, so that the
 * copies of one submission overlap the kernel of another.  Host buffers
 * should be pinned (cudaHostAlloc / cudaHostRegister) for the copies to be
 * asynchronous; the caller keeps them unchanged until the submission has
 * completed: after esdg_pipeline_wait, or once `depth` later submissions have
 * been made and waited for.  Submissions on one slot run in order; slots run
 * concurrently.  Not thread-safe. */
#define ESDG_PIPELINE_MAX_DEPTH 4

/* Allocate the slots (depth in 1..ESDG_PIPELINE_MAX_DEPTH; 29 * n values of
 * the handle's precision per slot) on the current device.  The handle must
 * outlive the pipeline.  Errors: ESDG_ERR_ARG, ESDG_ERR_CUDA. */
int esdg_pipeline_create(esdg_handle h, int depth, esdg_pipeline* out);

/* Enqueue one volume-term evaluation from host buffers (layouts as in
 * esdg_volume_rhs): q_host 5*n, metrics_host 9*n, phi_host n values (read),
 * out_host 5*n values (written when the submission completes).
 * Errors: ESDG_ERR_ARG, ESDG_ERR_CUDA, and the errors of esdg_volume_rhs. */
int esdg_pipeline_submit(esdg_pipeline p, const void* q_host, const void* metrics_host, const void* phi_host,
                         void* out_host);

/* Wait for every submission made so far.  Errors: ESDG_ERR_ARG, ESDG_ERR_CUDA. */
int esdg_pipeline_wait(esdg_pipeline p);

/* Description of the pipeline's last error (never NULL). */
const char* esdg_pipeline_last_error(esdg_pipeline p);

/* Wait for outstanding work and free the slots.  Accepts NULL. */
int esdg_pipeline_destroy(esdg_pipeline p);

/* The full right-hand side: out = volume + surface (boundary kinds and
 * dissipation of the handle), dq/dt = h - out/J.  For ESDG_FORM_2D the volume
 * diagonal f(q_i).Ja^r(i) at face nodes and the surface term's -f(q_i).n_own
 * cancel exactly, so both kernels run in their skew forms: the same result as
 * esdg_volume_rhs followed by esdg_surface_rhs up to rounding, with less
 * work.  Arguments as esdg_volume_rhs (out written).  ESDG_FP32: one launch,
 * the volume kernel evaluating each element's faces from its own side (each
 * interface once per side); ESDG_FP64 and ESDG_FP64_FF: the volume kernel and
 * the three face-centric surface launches (four launches).  Everything on
 * `stream`.  Errors: as esdg_volume_rhs. */
int esdg_rhs(esdg_handle h, const void* q, const void* metrics, const void* phi, void* out, void* stream);

/* Copy the status word to *flags and clear it.  Synchronises `stream`.
 * Errors: ESDG_ERR_ARG, ESDG_ERR_CUDA. */
int esdg_get_status(esdg_handle h, unsigned* flags, void* stream);

/* Human-readable description of the last error on this handle (or of the last
 * failed esdg_create when h == NULL).  Never NULL. */
const char* esdg_last_error(esdg_handle h);

/* LGL nodes (ascending), weights and differentiation matrix D (row-major,
 * D[i*(N+1) + j] = l_j'(x_i)) exactly as the kernels use them, in double.
 * Host only; no GPU needed.  Errors: ESDG_ERR_ARG, ESDG_ERR_UNSUPPORTED. */
int esdg_get_operators(int N, double* nodes, double* weights, double* D);

/* The pair schedule of one coordinate line, as the volume kernel of the given
 * precision runs it (Sec. 4.1 Eq. 6, cyclic assignment).  Line position p
 * evaluates the pairs (p, (p + d) mod Nq) for d = 1..H with H = floor(Nq/2),
 * each pair once, its result added to both nodes.  When Nq is even, d = Nq/2
 * joins antipodal nodes, the pairs Fig. 1(b) evaluates twice with weight 1/2.
 * ESDG_FP64: only the lower position p < Nq/2 evaluates such a pair, once, in
 * a separate pass of the kernel (sides 2; the upper position has partner -1,
 * sides 0).  ESDG_FP32: both positions evaluate it and keep their own share
 * (sides 1), which is Fig. 1(b)'s weighting summed per node.  Writes, for each
 * p and d, the partner index to partner[p*H + d-1] and the number of nodes
 * that receive the evaluation's result to sides[p*H + d-1].  Returns H
 * through *H_out.  Host only.  Errors: ESDG_ERR_ARG, ESDG_ERR_UNSUPPORTED. */
int esdg_pair_schedule(int N, int precision, int* H_out, int* partner, int* sides);

/* Library version as an integer (major*10000 + minor*100 + patch). */
int esdg_version(void);

/* The volume term of esdg_volume_rhs for callers that cannot allocate device
 * memory.  The paper has no counterpart: this is a library service.
 *
 * esdg_create allocates a 4-byte device status word per handle with
 * cudaMalloc.  Some callers cannot allow that: applications that give all of
 * the device memory to their own pool and forbid any other allocation, or
 * code that must not call cudaMalloc on a busy device because the call can
 * wait for work on other streams.  This entry point takes no handle and
 * allocates nothing (no cudaMalloc, cudaFree or allocating library routine).
 * Its only scratch is a file-scope __device__ array of 64 words (256 bytes)
 * in the library, of which the volume kernel uses one status word; every
 * device that loads the library holds that array until the process exits.
 *
 *   K          number of elements; n = K*(N+1)^3 nodes per plane.  At most
 *              2^31-1 elements and 2^40 nodes per call (ESDG_ERR_ARG beyond).
 *   N, precision, form, gamma   as for esdg_create / esdg_set_params.
 *   q, metrics, phi, out        device pointers exactly as for esdg_volume_rhs.
 *   status_out host pointer or NULL.  When non-NULL the call waits for the
 *              kernel (synchronises `stream`) and stores the status bits
 *              (ESDG_STATUS_*) of this call there.
 *   stream     cudaStream_t cast to void*.
 *
 * The first call on a device looks up the device address of the scratch
 * array with cudaGetSymbolAddress (with that device current) and keeps it
 * for that device's context; make that first call before any stream
 * capture.  If the context is destroyed and created again (cudaDeviceReset),
 * the next call sees a new context identifier and looks the address up
 * again.  Every call on a
 * device shares the one status word: the call clears it on `stream` before
 * its kernel, so calls whose work overlaps on the GPU (different streams)
 * race on it and may see each other's bits.
 * Errors: ESDG_ERR_ARG, ESDG_ERR_UNSUPPORTED, ESDG_ERR_ALIGN, ESDG_ERR_CUDA;
 * esdg_last_error(NULL) describes the cause. */
int esdg_volume_rhs_noalloc(long K, int N, int precision, int form, double gamma, const void* q,
                            const void* metrics, const void* phi, void* out, unsigned* status_out,
                            void* stream);

#ifdef __cplusplus
}
#endif

#endif /* ESDG_H */
