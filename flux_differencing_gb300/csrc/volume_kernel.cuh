// Flux-differencing volume kernel for sm_103a, templated on the element type
// and the polynomial order.
//
// What it computes (the volume part of Eq. 2 of "GPU Performance of an
// Entropy-Stable Discontinuous Galerkin Euler Solver with Non-Conservative
// Terms", Sec. 3): for every node i and reference direction r,
//     out_i += (1/w_p) sum_m 2 Q_{p p'} (F + G)^r(i, m)
// over the nodes m of the r-line through i (p, p' their positions on the
// line, Q = W D so that 2 Q_{pp'}/w_p = 2 D_{pp'}).  F is the
// entropy-conservative two-point flux (Eqs. 3-4), G the gravity term (Eqs.
// 4-5), both contracted with the averaged metric (Ja^r(i) + Ja^r(m))/2.
//
// How (GB300 design):
//  * One CTA handles EPB whole elements.  A load phase reads the 15 input
//    planes with coalesced loads straight into registers and writes per-node
//    derived quantities to shared memory: u = m/rho, b = rho/(2p), 1/b,
//    log rho, log b (FP64 and float-float), h = phi/2 - |u|^2/4 (Sec. 4.1:
//    primitives and logarithms once per node, not per pair), plus phi and the
//    metric terms.  The same
//    phase adds the diagonal pairs m == i of the 2D form, which only exist at
//    element-face nodes, for all three directions at once.
//  * Three direction phases (eta, zeta, then xi).  In each, every line's Nq
//    nodes occupy Nq consecutive lanes of one warp.  The lane at line
//    position p evaluates the pairs (p, p+d mod Nq) for d < Nq/2 -- the
//    cyclic assignment of Sec. 4.1 Eq. 6: every lane does the same number of
//    evaluations.  Each pair's result feeds both nodes ("half-sweep"): the
//    partner's share is formed with 2 Q_{p'p} = -2 Q_{pp'} and the gravity
//    partner scaling G -> -G b_i/b_m (Sec. 4.1) and moved to the partner lane
//    by a warp shuffle, so no atomics and a fixed summation order (bitwise
//    deterministic).
//  * For even Nq the antipodal pairs (p, p + Nq/2) are where Eq. 6 loses
//    balance and Fig. 1(b) evaluates each pair twice with weight 1/2.  In
//    FP64 and float-float they get a pass of their own per direction: within
//    one direction every node is in exactly one antipodal pair, so one thread
//    evaluates the pair once and adds both shares to shared memory without
//    races, and the threads left over are whole idle warps, which cost no
//    issue slots.  FP32 keeps the in-phase evaluation (cheaper there).
//  * Shared memory is laid out per order (padding or an XOR swizzle, and the
//    order in which lines are dealt to warps) so that the partner loads of
//    every direction phase are free of bank conflicts where possible.
//  * The mass flux is {{rho}}_log {{u}}.n, the energy flux the entropy-
//    conserving completion; both are formed directly from the contravariant
//    direction vector, never as a 3x5 flux matrix (Sec. 4.1).  FP64 and
//    float-float log means use the per-node logarithms, switching to a series
//    in the difference of the logarithms (no reciprocal) when the two are
//    close, and 1/{{b}}_log is computed directly (Sec. 4.1).  The closeness
//    test runs on the integer pipe; a warp vote skips the branch no lane
//    needs, a mixed warp evaluates both and selects per lane.  FP32 forms
//    the log means from polynomials in ((a+ - a-)/(a+ + a-))^2 where the
//    CTA's values lie within a factor kNarrowRatio, without logarithms
//    (NarrowCheck).  The per-node values are stored pre-scaled (u/2, 2b,
//    phi/8) so that no factor of two is applied per pair.
//  * FP32 at N = 3..8 evaluates two offsets per instruction in packed
//    float2 registers (issue-bound kernel; PackPairs).
//  * Further instantiations (MODE) change the final store: a Runge-Kutta
//    stage update fused into it (FP32 and float-float time steps), and in
//    FP32 the element's own faces evaluated in the kernel (neighbour traces
//    gathered while the element loads), so that a whole stage, or the full
//    right-hand side, is one launch.
//  * FP64 per-node logarithms by a table-driven reduction (log_fp64.cuh).
//  * FP64 on GB300 has 1/64 of the FP32 rate, so the FP64 kernel is bound by
//    its FP64 instruction count: reciprocals are a hardware estimate refined
//    by one third-order Newton-Raphson step rather than a correctly rounded
//    division, constants that depend only on the lane are hoisted, and sums
//    are written as FMA chains.
//  * Per-direction sums are scaled by 1/w once per node and combined in
//    shared memory; the xi phase writes the result with coalesced stores.
//  * No tensor cores: the flux is a nonlinear function of each pair.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "esdg_internal.h"
#include "floatfloat.cuh"
#include "numeric.cuh"
#include "packed.cuh"
#include "surface_flux.cuh"

namespace esdg {

// FP32 logarithmic-mean polynomials (kLogMeanRatio, kInvLogMeanRatio on
// u = f^2 <= kLogMeanPolyU), written by gen_logmean_poly.py
#include "logmean_poly.inc"

// A CTA whose node densities and values of b lie within this factor of one
// another (largest <= kNarrowRatio x smallest) takes the polynomial log means
// for all its pairs: |f| <= 1.25/3.25, u <= 0.148, inside the fitted range
// with room for the rounding of f.  Others select per pair between the
// polynomials and the logarithm of the pair's ratio.
constexpr float kNarrowRatio = 2.25f;
constexpr float kLog2E = 1.4426950408889634f;  // 1/ln 2
constexpr float kLn2F = 0.6931471805599453f;
static_assert((kNarrowRatio - 1.0f) * (kNarrowRatio - 1.0f) <
                  kLogMeanPolyU * (kNarrowRatio + 1.0f) * (kNarrowRatio + 1.0f),
              "narrow pairs must stay inside the polynomials' range");

template <int N>
struct Shape {
    static constexpr int NQ = N + 1;
    static constexpr int NP3 = NQ * NQ * NQ;
    static constexpr int NL = NQ * NQ;       // lines per element and direction
    static constexpr int LPW = 32 / NQ;      // whole lines per warp
    static constexpr int H = NQ / 2;         // pair offsets per lane
    static constexpr bool EVEN = (NQ % 2) == 0;
    // elements per CTA: keeps lanes busy and the CTA at <= 512 threads
    // (864 for N = 8, where one element already needs 27 warps)
    static constexpr int EPB = (N == 1) ? 16 : (N == 2) ? 10 : (N == 3) ? 4 : (N == 4) ? 3
                             : (N == 5) ? 2 : 1;
    static constexpr int LINES = EPB * NL;
    static constexpr int WARPS = (LINES + LPW - 1) / LPW;
    static constexpr int THREADS = WARPS * 32;
    static constexpr int NODES = EPB * NP3;
};

// Shared-memory layout of one node field.  SWZ: rows of Nq along xi with the
// column XOR-swizzled by (c ^ (b & MASK)); otherwise padded strides P1 (eta)
// and P2 (zeta).  ORDr = 1 deals the lines of direction r to warps with the
// second of the two other indices varying fastest.  The values come from a
// search over paddings, swizzles and line orders that minimises shared-memory
// wavefronts of the partner loads (32-bit words): conflict-free for N = 1, 3,
// 7, 8; about 1.3x of ideal for N = 4, 5, 6 and 1.7x for N = 2.
template <int N>
struct Layout;
template <> struct Layout<1> { static constexpr bool SWZ = false; static constexpr int P1 = 2, P2 = 4, MASK = 0, ORD0 = 0, ORD1 = 0, ORD2 = 0; };
template <> struct Layout<2> { static constexpr bool SWZ = false; static constexpr int P1 = 3, P2 = 9, MASK = 0, ORD0 = 0, ORD1 = 0, ORD2 = 0; };
template <> struct Layout<3> { static constexpr bool SWZ = true; static constexpr int P1 = 4, P2 = 16, MASK = 0, ORD0 = 0, ORD1 = 0, ORD2 = 1; };
template <> struct Layout<4> { static constexpr bool SWZ = false; static constexpr int P1 = 5, P2 = 26, MASK = 0, ORD0 = 0, ORD1 = 0, ORD2 = 0; };
template <> struct Layout<5> { static constexpr bool SWZ = false; static constexpr int P1 = 6, P2 = 37, MASK = 0, ORD0 = 0, ORD1 = 1, ORD2 = 0; };
template <> struct Layout<6> { static constexpr bool SWZ = false; static constexpr int P1 = 7, P2 = 50, MASK = 0, ORD0 = 0, ORD1 = 0, ORD2 = 0; };
template <> struct Layout<7> { static constexpr bool SWZ = true; static constexpr int P1 = 8, P2 = 64, MASK = 6, ORD0 = 0, ORD1 = 0, ORD2 = 1; };
template <> struct Layout<8> { static constexpr bool SWZ = false; static constexpr int P1 = 9, P2 = 93, MASK = 0, ORD0 = 0, ORD1 = 1, ORD2 = 0; };

template <int N>
struct Slots {
    using S = Shape<N>;
    using Lo = Layout<N>;
    static constexpr int NQ = S::NQ;
    static constexpr int ES = Lo::SWZ ? S::NP3 : Lo::P2 * NQ;  // element stride
    static constexpr int SIZE = S::EPB * ES;                    // values per field
    static __host__ __device__ __forceinline__ int at(int el, int a, int b, int c) {
        if constexpr (Lo::SWZ) return el * ES + NQ * (b + NQ * c) + (a ^ ((c ^ (b & Lo::MASK)) & (NQ - 1)));
        else return el * ES + a + Lo::P1 * b + Lo::P2 * c;
    }
};

// shared-memory fields (each an array of Slots<N>::SIZE values)
enum SmemField {
    F_RHO = 0, F_U1, F_U2, F_U3, F_B, F_INVB, F_LNRHO, F_LNB, F_PHI, F_H,
    F_JA0,              // 9 metric planes F_JA0 .. F_JA0 + 8
    F_ACC0 = F_JA0 + 9, // 5 accumulators
    F_COUNT = F_ACC0 + 5
};

// two FP32 pair evaluations in packed registers: per-half estimate and test
template <>
struct Num<p2> {
    static __device__ __forceinline__ p2 rcp(p2 x) { return p2(Num<float>::rcp(x.v.x), Num<float>::rcp(x.v.y)); }
    static __device__ __forceinline__ p2 lg2(p2 x) { return p2(Num<float>::lg2(x.v.x), Num<float>::lg2(x.v.y)); }
    static __device__ __forceinline__ m2 above(p2 u, float lim) {
        return m2{Num<float>::above(u.v.x, lim), Num<float>::above(u.v.y, lim)};
    }
};

// Node (a, b, c) of line `ell` of direction R at line position p.  R may be
// a compile-time constant (folded) or a runtime value.
template <int N>
__host__ __device__ __forceinline__ void line_node(int R, int ell, int p, int& a, int& b, int& c) {
    using Lo = Layout<N>;
    constexpr int NQ = N + 1;
    const int ord = (R == 0) ? Lo::ORD0 : (R == 1) ? Lo::ORD1 : Lo::ORD2;
    const int o1 = ord ? ell / NQ : ell % NQ;
    const int o2 = ord ? ell % NQ : ell / NQ;
    a = (R == 0) ? p : o1;
    b = (R == 1) ? p : (R == 0) ? o1 : o2;
    c = (R == 2) ? p : o2;
}

// Load-phase order of an element's nodes.  FP64 (FaceFirst) takes the face
// nodes first -- the slabs c = 0 and c = N, then for each inner slab the
// rows b = 0 and b = N and the ends a = 0, N of its other rows -- and the
// (N-1)^3 interior nodes after them, so that whole warps of interior nodes
// skip the 2D form's diagonal term (nonzero only at line ends), which a
// warp otherwise evaluates as soon as one of its lanes holds a face node
// (every warp does, in the natural order).  The same lines are read; only
// the order of the nodes within the element changes.  Other precisions keep
// the natural order (fully coalesced loads matter more there).
template <typename C>
struct FaceFirst {
    static constexpr bool value = std::is_same<C, double>::value;
};

template <int N>
__host__ __device__ __forceinline__ int face_first_node(int k) {
    constexpr int NQ = N + 1;
    constexpr int SLAB = NQ * NQ;
    constexpr int NI = N - 1;                    // interior nodes per line
    constexpr int RING = 4 * N;                  // face nodes of an inner slab
    constexpr int FACE = 2 * SLAB + NI * RING;   // = NQ^3 - NI^3
    int a, b, c;
    if (k < 2 * SLAB) {
        c = k < SLAB ? 0 : N;
        const int r = k < SLAB ? k : k - SLAB;
        a = r % NQ;
        b = r / NQ;
    } else if (k < FACE) {
        const int u = k - 2 * SLAB;
        c = 1 + u / RING;
        const int r = u % RING;
        if (r < 2 * NQ) {
            a = r % NQ;
            b = r < NQ ? 0 : N;
        } else {
            const int w = r - 2 * NQ;
            a = (w & 1) ? N : 0;
            b = 1 + (w >> 1);
        }
    } else if constexpr (NI > 0) {
        const int i = k - FACE;
        a = 1 + i % NI;
        b = 1 + (i / NI) % NI;
        c = 1 + i / (NI * NI);
    } else {
        a = b = c = 0;  // N = 1 has no interior node: not reached
    }
    return a + NQ * (b + NQ * c);
}

// Whether the antipodal pairs of even Nq get their own pass (evaluated once,
// both shares written to shared memory) or stay in the direction phases
// (evaluated by both nodes, own share kept).  The pass halves those
// evaluations, which pays in FP64, where the FP64 pipe is the bound; the FP32
// kernel is bound by instruction issue and shared-memory traffic, where the
// pass's extra loads, stores and barriers cost as much as they save.
template <typename T>
struct SplitAntipodal {
    static constexpr bool value = sizeof(T) == 8;
};

// Whether the kernel checks, per CTA, that its node values lie within
// kNarrowRatio of one another.  Such a CTA takes the polynomial log means for
// every pair, with no test; the others add, per pair, the logarithm of the
// pair's ratio and a select for the pairs beyond the polynomials' range.
// The FP32 kernel has no per-node logarithms.  FP64 and float-float keep
// theirs (series near equal values, logarithms of the node values beyond):
// polynomials accurate to their precision would need a far higher degree.
template <typename C>
struct NarrowCheck {
    static constexpr bool value = std::is_same<C, float>::value;
};

// Values of one node that a pair evaluation reads (metric terms of the
// current direction only).
template <typename T>
struct NodeVals {
    T rho, u1, u2, u3, b, ib, lr, lb, phi, h, A0, A1, A2;
};

template <int N, typename T>
__device__ __forceinline__ NodeVals<T> load_node(const T* __restrict__ sm, int i, int R) {
    constexpr int FS = Slots<N>::SIZE;
    NodeVals<T> v;
    v.rho = sm[F_RHO * FS + i];
    v.u1 = sm[F_U1 * FS + i];
    v.u2 = sm[F_U2 * FS + i];
    v.u3 = sm[F_U3 * FS + i];
    v.b = sm[F_B * FS + i];
    v.ib = sm[F_INVB * FS + i];
    v.lr = sm[F_LNRHO * FS + i];
    v.lb = sm[F_LNB * FS + i];
    v.phi = sm[F_PHI * FS + i];
    v.h = sm[F_H * FS + i];
    v.A0 = sm[(F_JA0 + 3 * R + 0) * FS + i];
    v.A1 = sm[(F_JA0 + 3 * R + 1) * FS + i];
    v.A2 = sm[(F_JA0 + 3 * R + 2) * FS + i];
    return v;
}

// The values of two nodes in the two halves of packed operands.
__device__ __forceinline__ NodeVals<p2> pack_vals(const NodeVals<float>& a, const NodeVals<float>& b) {
    NodeVals<p2> v;
    v.rho = p2(a.rho, b.rho);
    v.u1 = p2(a.u1, b.u1);
    v.u2 = p2(a.u2, b.u2);
    v.u3 = p2(a.u3, b.u3);
    v.b = p2(a.b, b.b);
    v.ib = p2(a.ib, b.ib);
    v.lr = p2(a.lr, b.lr);
    v.lb = p2(a.lb, b.lb);
    v.phi = p2(a.phi, b.phi);
    v.h = p2(a.h, b.h);
    v.A0 = p2(a.A0, b.A0);
    v.A1 = p2(a.A1, b.A1);
    v.A2 = p2(a.A2, b.A2);
    return v;
}

// Whether the FP32 kernel evaluates its offsets two at a time in packed FP32
// registers.  Chosen per order from the order sweep on GB300 (ms at about
// 6.4e7 nodes, unpacked -> packed): N = 4 3.44 -> 2.92, N = 5 3.64 -> 3.54,
// N = 6 4.32 -> 4.23, N = 8 5.00 -> 4.47 (with two line sets per warp at N = 4,
// 5, 8 for the registers); N = 7 3.210 -> 3.188 with the pre-scaled node
// values (the channel: 0.2183 -> 0.2167 ms; with two line sets per warp it
// was slower, 3.281); N = 3 1.908 -> 1.817, and 1.727 with two line sets.
template <typename C, int N>
struct PackPairs {
    static constexpr bool value =
        std::is_same<C, float>::value && N >= 3;
};

// The FP32 fused Runge-Kutta stage evaluates the surface term inside this
// kernel: every element takes each of its face nodes from its own side (the
// interface flux of surface_flux.cuh), reading the neighbour's trace while it
// loads its own element, so the planes are read once per stage instead of
// once more per direction by the face-centric surface kernel (whose xi and
// eta passes touch every DRAM line).  Each interface is evaluated twice, once
// per side; FP32 has the issue slots for that.  Float-float keeps the
// separate surface kernel and the face accumulator.
template <typename C>
struct FusedSurface {
    static constexpr bool value = std::is_same<C, float>::value;
};

// Face slots of a CTA: slot = el PER_EL + (2 dir + side) NF + i1 + NQ i2, with
// side 0 the face at index 0 along direction dir, side 1 the face at index
// N, and (i1, i2) the node's other two indices in (a, b, c) order.  The face
// buffer holds FIELDS values per slot (neighbour q, its metric row of the
// face direction, phi, rho_ref, p_ref), replaced by the slot's surface
// contribution (5 values) in the face phase.
template <int N>
struct FaceSlots {
    static constexpr int NQ = N + 1;
    static constexpr int NF = NQ * NQ;
    static constexpr int PER_EL = 6 * NF;
    static constexpr int COUNT = PER_EL * Shape<N>::EPB;
    static constexpr int FIELDS = 11;
    static __host__ __device__ __forceinline__ int slot(int el, int dir, int side, int i1, int i2) {
        return el * PER_EL + (2 * dir + side) * NF + i1 + NQ * i2;
    }
    static __host__ __device__ __forceinline__ void decode(int s, int& el, int& dir, int& side, int& i1, int& i2) {
        el = s / PER_EL;
        const int r = s - el * PER_EL;
        const int f = r / NF;
        const int w = r - f * NF;
        dir = f >> 1;
        side = f & 1;
        i1 = w % NQ;
        i2 = w / NQ;
    }
    // (a, b, c) of the node at index A along dir with other indices (i1, i2)
    static __host__ __device__ __forceinline__ void node(int dir, int A, int i1, int i2, int& na, int& nb, int& nc) {
        na = dir == 0 ? A : i1;
        nb = dir == 1 ? A : (dir == 0 ? i1 : i2);
        nc = dir == 2 ? A : i2;
    }
};

// The element across face (dir, side) of element e, or -1 at a slip wall
// (64-bit divisions: evaluated once per element and face, into the CTA's
// neighbour table).
template <typename T>
__host__ __device__ __forceinline__ long long neighbour_element(const VolumeArgs<T>& a, long long e, int dir, int side) {
    const long long Kd = dir == 0 ? a.Kx : dir == 1 ? a.Ky : a.Kz;
    const long long stride = dir == 0 ? 1 : dir == 1 ? a.Kx : a.Kx * a.Ky;
    const long long r = (e / stride) % Kd;  // element index along dir
    if (side) return r + 1 < Kd ? e + stride : (a.bc[dir] ? -1 : e - (Kd - 1) * stride);
    return r > 0 ? e - stride : (a.bc[dir] ? -1 : e + (Kd - 1) * stride);
}

// Global index of the node across face (dir, side) from node (i1, i2) of
// local element el, with the neighbour table nbr[6 el + 2 dir + side]; false
// at a slip wall.
template <int N>
__host__ __device__ __forceinline__ bool face_neighbour(const long long* nbr, int el, int dir, int side, int i1,
                                                        int i2, long long& g) {
    constexpr int NQ = N + 1;
    const long long en = nbr[6 * el + 2 * dir + side];
    if (en < 0) return false;
    int na, nb, nc;
    FaceSlots<N>::node(dir, side ? 0 : N, i1, i2, na, nb, nc);
    g = en * (long long)(NQ * NQ * NQ) + na + NQ * (nb + NQ * nc);
    return true;
}

// Dynamic shared memory of the volume kernel in bytes: the fields, and for
// the FP32 fused stage the face buffer and the neighbour table behind them.
// Kernel modes: 0 writes the volume term to out; 1 is the fused Runge-Kutta
// stage (FP32 and float-float); 2 writes volume + surface to out, the faces
// evaluated in the kernel (FP32).  Modes 1 and 2 in FP32 carry the face
// machinery (FaceMode).
template <typename C, int MODE>
struct FaceMode {
    static constexpr bool value = MODE != 0 && FusedSurface<C>::value;
};

template <typename C, int N, int MODE>
constexpr size_t volume_smem_fields() {
    return sizeof(C) * (size_t)F_COUNT * Slots<N>::SIZE +
           (FaceMode<C, MODE>::value ? sizeof(C) * (size_t)FaceSlots<N>::FIELDS * FaceSlots<N>::COUNT : 0);
}
template <typename C, int N, int MODE>
constexpr size_t volume_smem_nbr_offset() {
    return (volume_smem_fields<C, N, MODE>() + 7) & ~(size_t)7;
}
template <typename C, int N, int MODE>
constexpr size_t volume_smem_bytes() {
    return FaceMode<C, MODE>::value
               ? volume_smem_nbr_offset<C, N, MODE>() + 6 * sizeof(long long) * Shape<N>::EPB
               : volume_smem_fields<C, N, MODE>();
}

// The scalars of one pair (i, m) of a line from which both nodes' shares
// are formed (see pair_flux): cq = Q_{pp'} with p, p' the positions of i and m
// on the line, c_g2 = 1/(gamma - 1).
//   fr      2Q F_rho (mass flux times 2Q_{pp'})
//   fE      2Q F_E
//   Pi, Pm  the momentum flux's scalar factor of A at node i and at node m:
//           Q (p_hat + gravity scaled at b_i) and Q (-p_hat + gravity scaled
//           at b_m), G(m,i) = -G(i,m) b_i/b_m (Sec. 4.1)
//   s       the mean velocity {{u}}, A = Ja_i + Ja_m (twice the averaged metric)
// Node i's share of the momentum is fr s + A Pi, node m's -fr s + A Pm; the
// mass and energy shares are +-fr and +-fE.
//
// Scaling of the per-node values (chosen so that no factor of 2 is applied
// per pair): u holds u/2, so s = u_i + u_m is the mean velocity; b holds
// b2 = 2b = rho/p (1/b and ln b2 as stored); phi holds phi/8; the metric
// terms are unscaled, so A = Ja_i + Ja_m is twice the averaged metric and
// Un = s.A twice the contravariant velocity U.
template <typename T>
struct PairTerms {
    T fr, fE, Pi, Pm, s1, s2, s3, A0, A1, A2;
};

__device__ __forceinline__ bool any_of(bool c) { return c; }
__device__ __forceinline__ bool any_of(m2 c) { return c.x || c.y; }

// Horner evaluation of the degree-4 polynomial of table W (0: kLogMeanRatio,
// 1: kInvLogMeanRatio) at u.
template <int W, typename T>
__device__ __forceinline__ T poly4(T u) {
    constexpr float c0 = W ? kInvLogMeanRatio[0] : kLogMeanRatio[0];
    constexpr float c1 = W ? kInvLogMeanRatio[1] : kLogMeanRatio[1];
    constexpr float c2 = W ? kInvLogMeanRatio[2] : kLogMeanRatio[2];
    constexpr float c3 = W ? kInvLogMeanRatio[3] : kLogMeanRatio[3];
    constexpr float c4 = W ? kInvLogMeanRatio[4] : kLogMeanRatio[4];
    return fma(fma(fma(fma(T(c4), u, T(c3)), u, T(c2)), u, T(c1)), u, T(c0));
}

// NARROW (FP32 only): every node value of the CTA's elements lies within a
// factor kNarrowRatio of every other (checked in the load phase), so the
// logarithmic means come from polynomials, without logarithms or branches.
template <typename T, bool NARROW = false>
__device__ __forceinline__ PairTerms<T> pair_terms(const NodeVals<T>& I, const NodeVals<T>& M, T cq, T c_g2) {
    PairTerms<T> o;
    o.A0 = I.A0 + M.A0;
    o.A1 = I.A1 + M.A1;
    o.A2 = I.A2 + M.A2;
    o.s1 = I.u1 + M.u1;
    o.s2 = I.u2 + M.u2;
    o.s3 = I.u3 + M.u3;
    const T Un = fma(o.s3, o.A2, fma(o.s2, o.A1, o.s1 * o.A0));

    // crl = Q {{rho}}_log, inv_bsum = 1/(b2+ + b2-) = 1/(4{{b}}) and
    // inv_bln = 1/(2{{b}}_log); cqr = Q (rho+ + rho-) serves the pressure
    // mean and the close density branch
    const T rsum = I.rho + M.rho;
    const T bsum = I.b + M.b;
    const T cqr = cq * rsum;
    T crl, inv_bsum, inv_bln;
    constexpr bool FP32 = std::is_same<T, float>::value || std::is_same<T, p2>::value;
    static_assert(FP32 || !NARROW, "the polynomial log means are FP32 only");
    if constexpr (FP32) {
        // With f = (a+ - a-)/(a+ + a-) and u = f^2,
        //   {{rho}}_log = rsum f/(2 atanh f),  1/{{b2}}_log = (2 atanh(f)/f)/bsum,
        // each ratio a degree-4 polynomial in u (relative error below 3e-8
        // for u <= kLogMeanPolyU = 0.16, values within a factor 2.33).  No
        // logarithms: the whole pair costs two reciprocals.
        const T drho = M.rho - I.rho;
        const T fr_ = drho * Num<T>::rcp(rsum);
        const T ur = fr_ * fr_;
        crl = cqr * poly4<0>(ur);
        inv_bsum = Num<T>::rcp(bsum);
        const T db = M.b - I.b;
        const T fb = db * inv_bsum;
        const T ub = fb * fb;
        inv_bln = inv_bsum * poly4<1>(ub);
        if constexpr (!NARROW) {
            // A CTA with a wider spread: pairs beyond the polynomials' range
            // take the logarithm of the ratio x = a_m/a_i of their two values
            // (1/rho_i is the same for every offset of the line, so it is
            // hoisted; 1/b2_i = (1/b_i)/2 is a node value), selected per lane:
            //   {{rho}}_log = drho log2(e)/lg2(x_rho),  1/{{b2}}_log = ln2 lg2(x_b)/db.
            // There |lg2 x| > 1.2, so the absolute error of the hardware
            // lg2 (2^-22) stays near FP32 rounding in relative terms.
            // A warp vote skips them where no lane of the warp needs them
            // (lines along which the values vary little).
            const auto far_r = Num<T>::above(ur, kLogMeanPolyU);
            const auto far_b = Num<T>::above(ub, kLogMeanPolyU);
            if (__any_sync(__activemask(), any_of(far_r) || any_of(far_b))) {
                const T lr = Num<T>::lg2(M.rho * Num<T>::rcp(I.rho));
                crl = sel(far_r, (cq * drho) * (T(kLog2E) * Num<T>::rcp(lr)), crl);
                const T lb = Num<T>::lg2(M.b * (T(0.5) * I.ib));
                inv_bln = sel(far_b, (T(kLn2F) * lb) * Num<T>::rcp(db), inv_bln);
            }
        }
    } else {
        // Log means from the per-node logarithms: far, (a+ - a-)/(ln a+ - ln a-);
        // close (|d| < 0.02, d = ln a+ - ln a-), with x = d/2,
        //     {{a}}_log = {{a}} tanh(x)/x,  1/{{a}}_log = (x/tanh(x))/{{a}},
        // as series in v = d^2 -- no reciprocal for rho, and d's absolute
        // error only enters multiplied by d.  A warp vote skips the branch no
        // lane of the warp needs; a mixed warp evaluates both and selects.
        // Each lane computes the same formula either way.
        const T dlr = M.lr - I.lr;
        const T dlb = M.lb - I.lb;
        const auto cr = Num<T>::close(dlr);
        const auto cb = Num<T>::close(dlb);
        const unsigned mask = __activemask();
        // tanh(x)/x / 2 = 1/2 - v/24 + v^2/240 - 17 v^3/40320
        auto series_r = [&](T v) {
            return fma(v, fma(v, fma(v, T(-17.0 / 40320.0), T(1.0 / 240.0)), T(-1.0 / 24.0)), T(0.5));
        };
        // 2 x/tanh(x) = 2 + v/6 - v^2/360 + v^3/15120
        auto series_b = [&](T v) {
            return fma(v, fma(v, fma(v, T(1.0 / 15120.0), T(-1.0 / 360.0)), T(1.0 / 6.0)), T(2.0));
        };
        if (!__any_sync(mask, cr)) {
            crl = (cq * (M.rho - I.rho)) * Num<T>::rcp_pair(dlr);
        } else if (__all_sync(mask, cr)) {
            crl = cqr * series_r(dlr * dlr);
        } else {
            crl = sel(cr, cqr * series_r(dlr * dlr), (cq * (M.rho - I.rho)) * Num<T>::rcp_pair(dlr));
        }

        // 1/(b2+ + b2-) and, far, 1/(2{{b}}_log) = dlb/db2 from one reciprocal
        if (!__any_sync(mask, cb)) {
            const T db = M.b - I.b;
            const T rb = Num<T>::rcp_pair(db * bsum);
            inv_bsum = db * rb;
            inv_bln = dlb * (bsum * rb);
        } else if (__all_sync(mask, cb)) {
            inv_bsum = Num<T>::rcp_pair(bsum);
            inv_bln = inv_bsum * series_b(dlb * dlb);
        } else {
            const T db = M.b - I.b;
            const T rb = Num<T>::rcp_pair(sel(cb, bsum, db * bsum));
            inv_bsum = sel(cb, rb, db * rb);
            inv_bln = sel(cb, inv_bsum * series_b(dlb * dlb), dlb * (bsum * rb));
        }
    }

    // flux scalars, already multiplied by 2Q_{pp'} (momentum parts by Q, as
    // they multiply A = 2 x averaged metric)
    o.fr = crl * Un;                                    // 2Q F_rho
    const T gq = crl * (bsum * (M.phi - I.phi));        // Q rho_ln {{b}} [[phi]] / 2: gravity
    const T phq = cqr * inv_bsum;                       // Q p_hat, p_hat = {{rho}}/(2{{b}})
    // 1/(2 (gamma-1) {{b}}_log) - {{|u|^2}}/2 + {{phi}} + |{{u}}|^2
    const T hs = I.h + M.h;
    const T Kf = fma(c_g2, inv_bln, fma(o.s3, o.s3, fma(o.s2, o.s2, fma(o.s1, o.s1, hs))));
    o.fE = fma(o.fr, Kf, phq * Un);                     // 2Q F_E
    o.Pi = fma(gq, I.ib, phq);   // own: pressure mean + gravity scaled at b_i
    o.Pm = fma(gq, M.ib, -phq);  // partner: -pressure mean + gravity scaled at b_m
    return o;
}

// One pair (i, m) of a line, evaluated once for both nodes: adds node i's
// share 2Q_{pp'} (F + G(i,m)) to o0..o4 and returns node m's share
// 2Q_{p'p} (F + G(m,i)) = -2Q_{pp'} (F + G(m,i)) in t0..t4; t0 and t4 are
// returned with the opposite sign (the receiver subtracts them), which saves
// two negations per pair.  Both shares still need the 1/w scaling of their
// own node.
template <typename T, bool NARROW = false>
__device__ __forceinline__ void pair_flux(const NodeVals<T>& I, const NodeVals<T>& M, T cq, T c_g2, T& o0, T& o1,
                                          T& o2, T& o3, T& o4, T& t0, T& t1, T& t2, T& t3, T& t4) {
    const PairTerms<T> p = pair_terms<T, NARROW>(I, M, cq, c_g2);
    o0 += p.fr;
    o1 = fma(p.A0, p.Pi, fma(p.fr, p.s1, o1));
    o2 = fma(p.A1, p.Pi, fma(p.fr, p.s2, o2));
    o3 = fma(p.A2, p.Pi, fma(p.fr, p.s3, o3));
    o4 += p.fE;
    t0 = p.fr;  // subtracted by the receiver
    t1 = fma(p.A0, p.Pm, -(p.fr * p.s1));
    t2 = fma(p.A1, p.Pm, -(p.fr * p.s2));
    t3 = fma(p.A2, p.Pm, -(p.fr * p.s3));
    t4 = p.fE;  // subtracted by the receiver
}

// Whether the partner lane forms its momentum share itself from the pair's
// scalars (fr, fE, Pm, s, A moved by shuffles: 2 FMAs per component at the
// receiver) instead of receiving the finished share (a multiply and an FMA at
// the sender, an add at the receiver): three FP64 operations fewer per pair
// for four more shuffles.  For native FP64, bound by its FP64 pipe with issue
// slots to spare; the issue-bound FP32 and float-float kernels keep the
// finished shares.
template <typename C>
struct ReceiverForms {
    static constexpr bool value = std::is_same<C, double>::value;
};

// The face contributions of node (na, nb, nc) of local element el from the
// face phase, added to sv in the fixed order xi, eta, zeta.
template <typename T, int N>
__device__ __forceinline__ void face_sum(const T* __restrict__ fb, int el, int na, int nb, int nc, T (&sv)[5],
                                         unsigned* status) {
    using FSL = FaceSlots<N>;
    auto add_slot = [&](int sl) {
        sl = checked(sl, FSL::COUNT, status);
#pragma unroll
        for (int v = 0; v < 5; ++v) sv[v] += fb[v * FSL::COUNT + sl];
    };
    if (na == 0) add_slot(FSL::slot(el, 0, 0, nb, nc));
    else if (na == N) add_slot(FSL::slot(el, 0, 1, nb, nc));
    if (nb == 0) add_slot(FSL::slot(el, 1, 0, na, nc));
    else if (nb == N) add_slot(FSL::slot(el, 1, 1, na, nc));
    if (nc == 0) add_slot(FSL::slot(el, 2, 0, na, nb));
    else if (nc == N) add_slot(FSL::slot(el, 2, 1, na, nb));
}

// The final write of one node's volume term t0..t4.  MODE 0: to out.  MODE
// 2 (FP32): volume + the node's face contributions to out.  MODE 1: a fused
// Runge-Kutta stage, plus the surface term at face nodes, as a stage update
// of dq and q (the node's own element only, so updating q in place is safe
// where the surface term comes precomputed).
template <typename T, int N, int MODE>
__device__ __forceinline__ void store_node(const VolumeArgs<T>& a, long long g, int na, int nb, int nc, int el,
                                           const T* __restrict__ fb, T t0, T t1, T t2, T t3, T t4) {
    const long long n = a.n;
    constexpr bool FUSED = FaceMode<T, MODE>::value;
    if constexpr (MODE != 1) {
        T* __restrict__ o = a.out;
        if constexpr (FUSED) {
            T sv[5] = {T(0), T(0), T(0), T(0), T(0)};
            face_sum<T, N>(fb, el, na, nb, nc, sv, a.status);
            t0 += sv[0];
            t1 += sv[1];
            t2 += sv[2];
            t3 += sv[3];
            t4 += sv[4];
        }
        o[0 * n + g] = t0;
        o[1 * n + g] = t1;
        o[2 * n + g] = t2;
        o[3 * n + g] = t3;
        o[4 * n + g] = t4;
        return;
    }
    // every load first, through restrict-qualified pointers: loads interleaved
    // with stores through possibly aliasing pointers would each wait for DRAM
    // in turn (measured 1.0 ms against 0.22 ms for the plain FP32 kernel)
    const T* __restrict__ qp = a.rk_q;
    T* __restrict__ qo = FUSED ? a.rk_qout : a.rk_q;
    T* __restrict__ dqp = a.rk_dq;
    T* __restrict__ Sp = a.rk_S;
    const bool face = na == 0 || na == N || nb == 0 || nb == N || nc == 0 || nc == N;
    const bool use_dq = a.rk_A != T(0);
    T qv[5], dqv[5], sv[5];
#pragma unroll
    for (int v = 0; v < 5; ++v) {
        qv[v] = qp[v * n + g];
        dqv[v] = use_dq ? dqp[v * n + g] : T(0);
        sv[v] = (!FUSED && face) ? Sp[v * n + g] : T(0);
    }
    if constexpr (FUSED) face_sum<T, N>(fb, el, na, nb, nc, sv, a.status);
    const T Jg = a.rk_J[g];
    const T sc = -a.rk_dt * Num<T>::rcp(Jg);
    const T tot[5] = {t0, t1, t2, t3, t4};
    T dL[5];
#pragma unroll
    for (int v = 0; v < 5; ++v) dL[v] = (tot[v] + sv[v]) * sc;
    if (a.rk_f != T(0)) {
        const T fdt = a.rk_f * a.rk_dt;
        dL[1] = fma(fdt, qv[2], dL[1]);
        dL[2] = fma(-fdt, qv[1], dL[2]);
    }
#pragma unroll
    for (int v = 0; v < 5; ++v) {
        const T d = use_dq ? fma(a.rk_A, dqv[v], dL[v]) : dL[v];
        dqp[v * n + g] = d;
        qo[v * n + g] = fma(a.rk_B, d, qv[v]);
        if (!FUSED && face) Sp[v * n + g] = T(0);
    }
}

// (p + d) mod Nq for line positions p and offsets -Nq < d < Nq: a mask when
// Nq is a power of two (N = 1, 3, 7), a compare and correction otherwise.
template <int NQ>
__host__ __device__ __forceinline__ int wrap_pos(int p, int d) {
    if constexpr ((NQ & (NQ - 1)) == 0) {
        return (p + d) & (NQ - 1);
    } else {
        int q = p + d;
        if (q >= NQ) q -= NQ;
        if (q < 0) q += NQ;
        return q;
    }
}

// The line a lane works on in a direction phase: the lanes of a warp hold
// 32/Nq whole lines (slot), lane position p on the line; virtual warp vwarp
// takes lines vwarp LPW .. vwarp LPW + LPW - 1 of the CTA (element el = L/NL
// and line L - el NL within it).  Lanes past the last line, or on an element
// beyond e_count, return false and compute on line 0 (their results are
// discarded).
template <int N>
__host__ __device__ __forceinline__ bool lane_line(int vwarp, int lane, int e_count, int& slot, int& p, int& L) {
    using S = Shape<N>;
    slot = lane / S::NQ;
    p = lane - slot * S::NQ;
    L = vwarp * S::LPW + slot;
    const bool valid = (slot < S::LPW) && (L < S::LINES) && (L / S::NL < e_count);
    if (!valid) L = 0;
    return valid;
}

// One direction phase.  R = 0 (xi), 1 (eta), 2 (zeta).  FINAL = 0: add the
// scaled sum to the shared accumulators; 1, 2, 3: add the shared
// accumulators and store the node's result with store_node in MODE FINAL - 1
// (to out; as a fused Runge-Kutta stage update; with the faces, to out).  Offsets
// d = 1..NEAR; the antipodal offset Nq/2 of even Nq is left to
// antipodal_phase.
template <typename T, typename C, int N, int FINAL, bool NARROW = false>
__device__ __forceinline__ void direction_lines(const VolumeArgs<T>& a, C* __restrict__ sm, int e_count,
                                                long long node0, const C (&cq)[Shape<N>::H], C iw, C c_g,
                                                int vwarp, int R) {
    using S = Shape<N>;
    using SL = Slots<N>;
    constexpr int NQ = S::NQ;
    constexpr int FS = SL::SIZE;
    constexpr int NEAR = (S::EVEN && SplitAntipodal<C>::value) ? S::H - 1 : S::H;

    const int lane = threadIdx.x & 31;
    int slot, p, L;
    const bool valid = lane_line<N>(vwarp, lane, e_count, slot, p, L);
    const int el = L / S::NL;
    const int ell = L - el * S::NL;
    int ia, ib, ic;
    line_node<N>(R, ell, p, ia, ib, ic);
    const int i = checked(SL::at(el, ia, ib, ic), FS, a.status);
    const NodeVals<C> I = load_node<N>(sm, i, R);

    C acc0 = C(0.0), acc1 = C(0.0), acc2 = C(0.0), acc3 = C(0.0), acc4 = C(0.0);

    auto offset = [&](int d, C cqd) {
        const int pm = wrap_pos<NQ>(p, d);
        int ma = ia, mb = ib, mc = ic;
        if (R == 0) ma = pm;
        else if (R == 1) mb = pm;
        else mc = pm;
        const NodeVals<C> M = load_node<N>(sm, checked(SL::at(el, ma, mb, mc), FS, a.status), R);
        // the partner share goes to the lane at position p + d; this lane
        // receives from the lane at p - d
        const int src = wrap_pos<NQ>(p, -d) + slot * NQ;
        if constexpr (ReceiverForms<C>::value) {
            const PairTerms<C> pt = pair_terms<C>(I, M, cqd, c_g);
            acc0 += pt.fr;
            acc1 = fma(pt.A0, pt.Pi, fma(pt.fr, pt.s1, acc1));
            acc2 = fma(pt.A1, pt.Pi, fma(pt.fr, pt.s2, acc2));
            acc3 = fma(pt.A2, pt.Pi, fma(pt.fr, pt.s3, acc3));
            acc4 += pt.fE;
            if (S::EVEN && d == S::H) return;  // in-phase antipodal offset: own share only
            // this lane is node m of the pair evaluated by the lane at p - d:
            // -fr, -fE, and -fr s + A Pm for the momentum
            const C rfr = shfl(pt.fr, src), rfE = shfl(pt.fE, src), rPm = shfl(pt.Pm, src);
            const C rs1 = shfl(pt.s1, src), rs2 = shfl(pt.s2, src), rs3 = shfl(pt.s3, src);
            const C rA0 = shfl(pt.A0, src), rA1 = shfl(pt.A1, src), rA2 = shfl(pt.A2, src);
            acc0 -= rfr;
            acc1 = fma(-rfr, rs1, fma(rA0, rPm, acc1));
            acc2 = fma(-rfr, rs2, fma(rA1, rPm, acc2));
            acc3 = fma(-rfr, rs3, fma(rA2, rPm, acc3));
            acc4 -= rfE;
        } else {
            C t0, t1, t2, t3, t4;
            pair_flux<C, NARROW>(I, M, cqd, c_g, acc0, acc1, acc2, acc3, acc4, t0, t1, t2, t3, t4);
            // In-phase antipodal offset (when not split off): both nodes evaluate
            // the pair and keep their own share -- Fig. 1(b)'s two weight-1/2
            // evaluations summed per node.
            if (S::EVEN && d == S::H) return;
            acc0 -= shfl(t0, src);
            acc1 += shfl(t1, src);
            acc2 += shfl(t2, src);
            acc3 += shfl(t3, src);
            acc4 -= shfl(t4, src);
        }
    };
    if constexpr (IsFF<C>::value) {
        // one copy of the (long) float-float pair evaluation: no unrolling,
        // the offset's 2Q/8 read from the operator table each time
#pragma unroll 1
        for (int d = 1; d <= NEAR; ++d) offset(d, Conv<T, C>::in(T(0.5) * a.ops.Q2[p * NQ + wrap_pos<NQ>(p, d)]));
    } else if constexpr (PackPairs<C, N>::value) {
        // offsets d and d + 1 in the two halves of packed FP32 operands: one
        // issue slot for two evaluations' arithmetic
        const NodeVals<p2> I2 = pack_vals(I, I);
        const p2 cg2(c_g, c_g);
        p2 o0(0.0), o1(0.0), o2(0.0), o3(0.0), o4(0.0);
#pragma unroll
        for (int d = 1; d + 1 <= NEAR; d += 2) {
            const int pm = wrap_pos<NQ>(p, d);
            const int pn = wrap_pos<NQ>(p, d + 1);
            int ma = ia, mb = ib, mc = ic, na = ia, nb = ib, nc = ic;
            if (R == 0) { ma = pm; na = pn; }
            else if (R == 1) { mb = pm; nb = pn; }
            else { mc = pm; nc = pn; }
            const NodeVals<p2> M = pack_vals(load_node<N>(sm, checked(SL::at(el, ma, mb, mc), FS, a.status), R),
                                             load_node<N>(sm, checked(SL::at(el, na, nb, nc), FS, a.status), R));
            p2 t0, t1, t2, t3, t4;
            pair_flux<p2, NARROW>(I2, M, p2(cq[d - 1], cq[d]), cg2, o0, o1, o2, o3, o4, t0, t1, t2, t3, t4);
            // partner shares: half x to the lane at p + d, half y to p + d + 1
            // (none for the in-phase antipodal offset of even Nq); when both
            // halves are received they are added to the packed accumulators
            // (one packed add per component instead of two)
            const int src = wrap_pos<NQ>(p, -d) + slot * NQ;
            if (!(S::EVEN && d + 1 == S::H)) {
                const int src2 = wrap_pos<NQ>(p, -d - 1) + slot * NQ;
                o0 = o0 - p2(shfl(t0.v.x, src), shfl(t0.v.y, src2));
                o1 += p2(shfl(t1.v.x, src), shfl(t1.v.y, src2));
                o2 += p2(shfl(t2.v.x, src), shfl(t2.v.y, src2));
                o3 += p2(shfl(t3.v.x, src), shfl(t3.v.y, src2));
                o4 = o4 - p2(shfl(t4.v.x, src), shfl(t4.v.y, src2));
            } else {
                acc0 -= shfl(t0.v.x, src);
                acc1 += shfl(t1.v.x, src);
                acc2 += shfl(t2.v.x, src);
                acc3 += shfl(t3.v.x, src);
                acc4 -= shfl(t4.v.x, src);
            }
        }
        if constexpr (NEAR % 2 == 1) offset(NEAR, cq[NEAR - 1]);
        acc0 += o0.v.x + o0.v.y;
        acc1 += o1.v.x + o1.v.y;
        acc2 += o2.v.x + o2.v.y;
        acc3 += o3.v.x + o3.v.y;
        acc4 += o4.v.x + o4.v.y;
    } else {
#pragma unroll
        for (int d = 1; d <= NEAR; ++d) offset(d, cq[d - 1]);
    }

    C* s_acc = sm + F_ACC0 * FS;
    if constexpr (FINAL == 0) {
        if (valid) {
            s_acc[0 * FS + i] = fma(acc0, iw, s_acc[0 * FS + i]);
            s_acc[1 * FS + i] = fma(acc1, iw, s_acc[1 * FS + i]);
            s_acc[2 * FS + i] = fma(acc2, iw, s_acc[2 * FS + i]);
            s_acc[3 * FS + i] = fma(acc3, iw, s_acc[3 * FS + i]);
            s_acc[4 * FS + i] = fma(acc4, iw, s_acc[4 * FS + i]);
        }
    } else if (valid) {
        // xi phase: lines of a warp are consecutive (b, c) rows, so the block-
        // linear node L*Nq + p is contiguous across lanes: coalesced stores
        static_assert(Layout<N>::ORD0 == 0, "xi lines must be dealt b-fastest");
        const long long g = checked(node0 + (long long)L * NQ + p, a.n, a.status);
        store_node<T, N, FINAL - 1>(a, g, ia, ib, ic, el, reinterpret_cast<const T*>(sm + F_COUNT * FS),
                                     Conv<T, C>::out(fma(acc0, iw, s_acc[0 * FS + i])),
                         Conv<T, C>::out(fma(acc1, iw, s_acc[1 * FS + i])),
                         Conv<T, C>::out(fma(acc2, iw, s_acc[2 * FS + i])),
                         Conv<T, C>::out(fma(acc3, iw, s_acc[3 * FS + i])),
                         Conv<T, C>::out(fma(acc4, iw, s_acc[4 * FS + i])));
    }
}

// Threads per CTA and line sets per warp.  A warp walks REPS sets of lines in
// each direction phase.  Two sets halve the CTA, so that two CTAs can share an
// SM and one CTA's load phase overlaps the other's pair arithmetic.  Chosen
// per precision and order from the order sweep (about 6.4e7 nodes per order)
// on GB300:
//  * float-float: always 2 (256-thread CTAs at N = 7);
//  * FP64: 2 only at N = 7 (111.2 -> 109.4 ms); at N = 2, 4, 5, 6, 8 the
//    halved CTA was 2-7 % slower;
//  * FP32: 2 at N = 3, 4, 5, 6 and 8, where the packed pair evaluation
//    (PackPairs) needs more than the 64 registers a 512-thread CTA pair
//    leaves (N = 6: 4.34 -> 3.98 ms on the order sweep, N = 3: 1.82 ->
//    1.73); at N = 8 one element's 81 lines would otherwise also need an
//    864-thread CTA.  At N = 7, two sets in 256-thread CTAs, four per SM at
//    64 registers: 0.1935 -> 0.1806 ms on the channel, 2.757 -> 2.565 ms on
//    the order sweep, against one set in two 512-thread CTAs per SM.  The
//    kernels that carry the face machinery (FACES: the FP32 fused stage and
//    volume + faces) keep one set in 512-thread CTAs: their face buffer
//    leaves room for three CTAs per SM only, and the face phase's 384 slots
//    per element would take two rounds of 256 threads (volume + faces
//    0.261 -> 0.279 ms with the smaller CTA).
//  * FP64 rechecked with the current kernel: two sets at N = 4, 5, 6 gave
//    61.8 -> 62.7, 75.5 -> 75.4 and 91.7 -> 94.4 ms, so only N = 7 uses them;
//    but two CTAs of one set per SM (MIN_BLOCKS = 2: 72, 64 and 72 registers
//    with 24-128 byte spills) are faster there: 61.8 -> 60.0, 75.5 -> 74.0,
//    91.7 -> 90.2 ms.  Four CTAs per SM at N = 2, 3 (56 and 64 registers)
//    were no faster (34.8 -> 35.3, 44.3 -> 44.3 ms).
template <int N, typename C, bool FACES = false>
struct Launch {
    using S = Shape<N>;
    static constexpr int VWARPS = (S::LINES + S::LPW - 1) / S::LPW;  // warps' worth of lines
    static constexpr bool FP64 = sizeof(C) == 8;
    static constexpr int REPS =
        IsFF<C>::value ? 2 : FP64 ? (N == 7 ? 2 : 1) : ((N >= 3 && !(N == 7 && FACES)) ? 2 : 1);
    static constexpr int WARPS = (VWARPS + REPS - 1) / REPS;
    static constexpr int THREADS = WARPS * 32;
    static constexpr size_t SMEM = sizeof(C) * (size_t)F_COUNT * Slots<N>::SIZE;
    static constexpr bool TWO_FIT = 2 * SMEM <= 227 * 1024;
    // FP32 at N = 2..7: register bounds that keep more CTAs per SM than the
    // unbounded allocation (N = 2: 5 CTAs of 288 threads at 40 registers;
    // N = 3: 8 of 128 at 64; N = 4: 5 of 224 at 56; N = 6: 4 of 224 at 72;
    // N = 5, 7: 4 of 256 at 64), without spills in the plain kernel.  Order
    // sweep (ms, about 6.4e7 nodes): N = 2 1.902 -> 1.877, N = 3 1.522 ->
    // 1.509, N = 4 2.846 -> 2.631 (4 CTAs) -> 2.571 (5), N = 5 3.163 -> 3.026,
    // N = 6 3.694 -> 3.315; five CTAs at N = 5 and 6 were slower (3.11,
    // 3.43).  The kernels with face work (whose face buffer takes more shared
    // memory) keep the general rule below.
    static constexpr int MIN_BLOCKS =
        (sizeof(C) == 4 && !FACES && (N == 2 || N == 4)) ? 5
        : (sizeof(C) == 4 && !FACES && N == 3) ? 8
        : (sizeof(C) == 4 && !FACES && (N == 5 || N == 6 || N == 7)) ? 4
        : ((sizeof(C) == 4 && THREADS <= 512) || IsFF<C>::value || (FP64 && (REPS == 2 || (N >= 4 && N <= 6)))) &&
                  TWO_FIT
            ? 2
            : 1;
};

template <typename T, typename C, int N, int R, int FINAL, bool NARROW, int MODE>
__device__ __forceinline__ void direction_phase(const VolumeArgs<T>& a, C* __restrict__ sm, int e_count,
                                                long long node0, const C (&cq)[Shape<N>::H], C iw, C c_g) {
    using LA = Launch<N, C, FaceMode<C, MODE>::value>;
    const int warp = threadIdx.x >> 5;
    // FP32 at N = 3, 7, 8: the line sets unrolled (order sweep 1.511 ->
    // 1.477, 2.565 -> 2.506 and 3.993 -> 3.948 ms; at N = 4, 5, 6 the
    // unrolled code was 1-2 % slower)
    if constexpr (std::is_same<C, float>::value && (N == 3 || N == 7 || N == 8)) {
#pragma unroll
        for (int rep = 0; rep < LA::REPS; ++rep)
            direction_lines<T, C, N, FINAL, NARROW>(a, sm, e_count, node0, cq, iw, c_g, warp + rep * LA::WARPS, R);
    } else {
#pragma unroll 1
        for (int rep = 0; rep < LA::REPS; ++rep)
            direction_lines<T, C, N, FINAL, NARROW>(a, sm, e_count, node0, cq, iw, c_g, warp + rep * LA::WARPS, R);
    }
}

// Pair k of the antipodal pass: element el, line ell, lower position p
// (the pair is (p, p + Nq/2)); consecutive k walk a line.
template <int N>
__host__ __device__ __forceinline__ void antipodal_pair(int k, int& el, int& p, int& ell) {
    constexpr int H = Shape<N>::H;
    constexpr int PER_EL = Shape<N>::NL * H;
    el = k / PER_EL;
    const int kk = k - el * PER_EL;
    p = kk % H;
    ell = kk / H;
}

// Antipodal pairs (p, p + Nq/2) of every line of direction R, for even Nq.
// Each node belongs to exactly one such pair per direction, so the pairs are
// disjoint: one thread evaluates a pair once and adds both shares to the
// shared accumulators without races (Fig. 1(b)'s two weight-1/2 evaluations
// become one).  There are Nq^3/2 pairs per element; the surplus threads are
// whole warps, which issue nothing.
template <typename T, typename C, int N>
__device__ __forceinline__ void antipodal_phase(const VolumeArgs<T>& a, C* __restrict__ sm, int e_count, C c_g, int R) {
    using S = Shape<N>;
    using SL = Slots<N>;
    constexpr int NQ = S::NQ;
    constexpr int H = S::H;
    constexpr int FS = SL::SIZE;
    constexpr int PER_EL = S::NL * H;
    C* s_acc = sm + F_ACC0 * FS;
    for (int k = threadIdx.x; k < S::EPB * PER_EL; k += Launch<N, C>::THREADS) {
        int el, p, ell;
        antipodal_pair<N>(k, el, p, ell);
        if (el >= e_count) break;
        int ia, ib, ic, ja, jb, jc;
        line_node<N>(R, ell, p, ia, ib, ic);
        line_node<N>(R, ell, p + H, ja, jb, jc);
        const int i = checked(SL::at(el, ia, ib, ic), FS, a.status);
        const int j = checked(SL::at(el, ja, jb, jc), FS, a.status);
        const NodeVals<C> I = load_node<N>(sm, i, R);
        const NodeVals<C> M = load_node<N>(sm, j, R);
        const C cq = Conv<T, C>::in(T(0.5) * a.ops.Q2[p * NQ + p + H]);
        const PairTerms<C> pt = pair_terms<C>(I, M, cq, c_g);
        // both shares straight from the pair's scalars: fr s_k is common to
        // node i (+fr s + A Pi) and node j (-fr s + A Pm)
        const C x1 = pt.fr * pt.s1, x2 = pt.fr * pt.s2, x3 = pt.fr * pt.s3;
        const C iwi = Conv<T, C>::in(a.ops.invw[p]), iwj = Conv<T, C>::in(a.ops.invw[p + H]);
        s_acc[0 * FS + i] = fma(pt.fr, iwi, s_acc[0 * FS + i]);
        s_acc[1 * FS + i] = fma(fma(pt.A0, pt.Pi, x1), iwi, s_acc[1 * FS + i]);
        s_acc[2 * FS + i] = fma(fma(pt.A1, pt.Pi, x2), iwi, s_acc[2 * FS + i]);
        s_acc[3 * FS + i] = fma(fma(pt.A2, pt.Pi, x3), iwi, s_acc[3 * FS + i]);
        s_acc[4 * FS + i] = fma(pt.fE, iwi, s_acc[4 * FS + i]);
        s_acc[0 * FS + j] = fma(-pt.fr, iwj, s_acc[0 * FS + j]);
        s_acc[1 * FS + j] = fma(fma(pt.A0, pt.Pm, -x1), iwj, s_acc[1 * FS + j]);
        s_acc[2 * FS + j] = fma(fma(pt.A1, pt.Pm, -x2), iwj, s_acc[2 * FS + j]);
        s_acc[3 * FS + j] = fma(fma(pt.A2, pt.Pm, -x3), iwj, s_acc[3 * FS + j]);
        s_acc[4 * FS + j] = fma(-pt.fE, iwj, s_acc[4 * FS + j]);
    }
}

// Face phase of the FP32 fused stage: one thread per face slot evaluates the
// interface flux of its face node from the element's own side (the node
// owning the outward normal), with the neighbour's trace loaded into the face
// buffer during the load phase, or a mirror ghost at a slip wall, and leaves
// 1/w_0 times the contribution in the slot (read back by the node's final
// store).  The own state comes from the shared-memory fields (pre-scaled by
// powers of two, so it is the node state exactly).
template <typename T, typename C, int N>
__device__ __forceinline__ void face_phase(const VolumeArgs<T>& a, C* __restrict__ sm, const long long* nbr,
                                           int e_count) {
    using SL = Slots<N>;
    using FSL = FaceSlots<N>;
    constexpr int FS = SL::SIZE;
    constexpr int CNT = FSL::COUNT;
    C* fb = sm + F_COUNT * FS;
    Consts<C> k;
    k.gm1 = a.sk.gm1;
    k.igm1 = a.sk.igm1;
    k.c_g = a.sk.c_g;
    k.gamma = a.sk.gamma;
    k.c_ac = a.sk.c_ac;
    k.c_en = a.sk.c_en;
    const bool perturbed = a.rho_ref != nullptr;
    for (int s = threadIdx.x; s < e_count * FSL::PER_EL; s += Launch<N, C, true>::THREADS) {
        int el, dir, side, i1, i2, na, nb, nc;
        FSL::decode(s, el, dir, side, i1, i2);
        FSL::node(dir, side ? N : 0, i1, i2, na, nb, nc);
        const int sl = checked(SL::at(el, na, nb, nc), FS, a.status);
        FaceNode<C> I;
        I.rho = sm[F_RHO * FS + sl];
        I.u1 = C(2) * sm[F_U1 * FS + sl];
        I.u2 = C(2) * sm[F_U2 * FS + sl];
        I.u3 = C(2) * sm[F_U3 * FS + sl];
        I.uu = fma(I.u3, I.u3, fma(I.u2, I.u2, I.u1 * I.u1));
        I.b = C(0.5) * sm[F_B * FS + sl];
        I.ib = sm[F_INVB * FS + sl];
        I.phi = C(8) * sm[F_PHI * FS + sl];
        I.p = C(0);  // p and E are not used by the interface flux
        I.E = C(0);
        const C j0 = sm[(F_JA0 + 3 * dir + 0) * FS + sl];
        const C j1 = sm[(F_JA0 + 3 * dir + 1) * FS + sl];
        const C j2 = sm[(F_JA0 + 3 * dir + 2) * FS + sl];
        const C sg = side ? C(1) : C(-1);  // outward
        long long g;
        C fi[5], fo[5];
        if (face_neighbour<N>(nbr, el, dir, side, i1, i2, g)) {
            const FaceNode<C> J = node_state<C>(fb[0 * CNT + s], fb[1 * CNT + s], fb[2 * CNT + s], fb[3 * CNT + s],
                                                fb[4 * CNT + s], fb[8 * CNT + s], k.gm1, perturbed,
                                                fb[9 * CNT + s], fb[10 * CNT + s]);
            const C n0 = sg * C(0.5) * (j0 + fb[5 * CNT + s]);
            const C n1 = sg * C(0.5) * (j1 + fb[6 * CNT + s]);
            const C n2 = sg * C(0.5) * (j2 + fb[7 * CNT + s]);
            interface_flux(I, J, n0, n1, n2, k, a.dissipation != 0, fi, fo);
        } else {
            // slip wall: mirror ghost (rho, m - 2 (m.n^) n^, E), same phi
            const C n0 = sg * j0, n1 = sg * j1, n2 = sg * j2;
            const C inn = Num<C>::rcp(sqrt_(fma(n2, n2, fma(n1, n1, n0 * n0))));
            const C h0 = n0 * inn, h1 = n1 * inn, h2 = n2 * inn;
            const C un2 = C(2.0) * fma(I.u3, h2, fma(I.u2, h1, I.u1 * h0));
            FaceNode<C> G = I;
            G.u1 = fma(-un2, h0, I.u1);
            G.u2 = fma(-un2, h1, I.u2);
            G.u3 = fma(-un2, h2, I.u3);
            interface_flux(I, G, n0, n1, n2, k, a.dissipation != 0, fi, fo);
        }
#pragma unroll
        for (int v = 0; v < 5; ++v) fb[v * CNT + s] = a.inv_w0 * fi[v];
    }
}

// The direction phases of a CTA whose values spread wider than kNarrowRatio
// (FP32), kept out of line so that the kernel's own code and registers are
// those of the polynomial path.  Measured on GB300 at N = 7 (4.2e6 nodes):
// with both forms inline the polynomial CTAs ran 11 % slower than a kernel
// holding the polynomial form alone, and the whole launch was no faster than
// per-pair selects between series and per-node logarithms; out of line (with
// the warp vote around the ratio logarithms) they run as fast as in that
// kernel, and the launch is 9 % faster.
template <typename T, typename C, int N, int MODE>
__device__ __noinline__ void wide_phases(const VolumeArgs<T>& a, C* __restrict__ sm, int e_count, long long node0) {
    using S = Shape<N>;
    constexpr int NQ = S::NQ;
    using CV = Conv<T, C>;
    static_assert(!SplitAntipodal<C>::value, "no antipodal pass");
    const int lane = threadIdx.x & 31;
    const int p = lane - (lane / NQ) * NQ;
    C cq[S::H];
#pragma unroll
    for (int d = 1; d <= S::H; ++d) cq[d - 1] = CV::in(T(0.5) * a.ops.Q2[p * NQ + wrap_pos<NQ>(p, d)]);
    const C iw = CV::in(a.ops.invw[p]);
    const C c_g = CV::in(T(2) * a.c_g);
    direction_phase<T, C, N, 1, 0, false, MODE>(a, sm, e_count, node0, cq, iw, c_g);
    __syncthreads();
    direction_phase<T, C, N, 2, 0, false, MODE>(a, sm, e_count, node0, cq, iw, c_g);
    __syncthreads();
    direction_phase<T, C, N, 0, MODE + 1, false, MODE>(a, sm, e_count, node0, cq, iw, c_g);
}

// MODE (store_node): 0 volume to out, 1 fused Runge-Kutta stage, 2 (FP32)
// volume + faces to out; separate instantiations, so that the plain kernel's
// code and registers are those of a store to out.
template <typename T, int N, typename C, int MODE>
__global__ void __launch_bounds__(Launch<N, C, FaceMode<C, MODE>::value>::THREADS,
                                  Launch<N, C, FaceMode<C, MODE>::value>::MIN_BLOCKS)
volume_kernel(const __grid_constant__ VolumeArgs<T> a) {
    using S = Shape<N>;
    using SL = Slots<N>;
    constexpr int NQ = S::NQ;
    constexpr int NP3 = S::NP3;
    constexpr int FS = SL::SIZE;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    C* sm = reinterpret_cast<C*>(smem_raw);
    using CV = Conv<T, C>;
    using LK = Launch<N, C, FaceMode<C, MODE>::value>;
    poison_shared(smem_raw, volume_smem_bytes<C, N, MODE>());  // debug builds only

    const long long e0 = a.e_begin + (long long)blockIdx.x * S::EPB;
    const long long rem = a.e_end - e0;
    const int e_count = rem < S::EPB ? (int)rem : S::EPB;
    const long long node0 = e0 * NP3;

    // FP32 fused stage: the element across each face of the CTA's elements
    // (-1 at a slip wall), one entry per thread
    long long* nbr = nullptr;
    if constexpr (FaceMode<C, MODE>::value) {
        nbr = reinterpret_cast<long long*>(smem_raw + volume_smem_nbr_offset<C, N, MODE>());
        static_assert(6 * S::EPB <= LK::THREADS, "one neighbour entry per thread");
        const int t = threadIdx.x;
        if (t < 6 * e_count) nbr[t] = neighbour_element(a, e0 + t / 6, (t % 6) >> 1, t & 1);
        __syncthreads();
    }

    // ---- load phase: one node per thread, coalesced plane reads -> derived values.
    // The per-node arithmetic runs in P: the I/O type for FP64 and FP32, and
    // float-float for FP64_FF, where the doubles are split on the integer
    // pipe and the divisions and logarithms stay off the FP64 pipe.
    using P = typename std::conditional<IsFF<C>::value, ff, T>::type;
    using PV = Conv<T, P>;
    bool bad = false;
    // NarrowCheck: bit patterns of the smallest and largest density and b2
    // of this thread's nodes (for positive floats the unsigned order of the
    // bits is the order of the values)
    unsigned r_lo = 0xffffffffu, r_hi = 0u, b_lo = 0xffffffffu, b_hi = 0u;
    // FP32 fused stage: the neighbour trace of this thread's first face slot
    // is requested before the element's own planes, so that the latencies of
    // the two sets of loads overlap; it is written to the face buffer after
    // the node loop
    constexpr bool FUSED = FaceMode<C, MODE>::value;
    constexpr int TR = 11;  // trace values: q (5), metric row (3), phi, rho_ref, p_ref
    C trace[FUSED ? TR : 1];
    bool trace_ok = false;
    if constexpr (FUSED) {
        using FSL = FaceSlots<N>;
        const int s = threadIdx.x;
        if (s < e_count * FSL::PER_EL) {
            int el, dir, side, i1, i2;
            FSL::decode(s, el, dir, side, i1, i2);
            long long g;
            if (face_neighbour<N>(nbr, el, dir, side, i1, i2, g)) {
                g = checked(g, a.n, a.status);
                trace_ok = true;
                const long long n = a.n;
#pragma unroll
                for (int v = 0; v < 5; ++v) trace[v] = __ldg(a.q + v * n + g);
#pragma unroll
                for (int c = 0; c < 3; ++c) trace[5 + c] = __ldg(a.Ja + (3 * dir + c) * n + g);
                trace[8] = __ldg(a.phi + g);
                trace[9] = a.rho_ref ? __ldg(a.rho_ref + g) : C(0);
                trace[10] = a.rho_ref ? __ldg(a.p_ref + g) : C(0);
            }
        }
    }
    for (int t = threadIdx.x; t < S::NODES; t += LK::THREADS) {
        const int el = t / NP3;
        const int nd = FaceFirst<C>::value ? face_first_node<N>(t - el * NP3) : t - el * NP3;
        const int na = nd % NQ, nb = (nd / NQ) % NQ, nc = nd / (NQ * NQ);
        const int sl = checked(SL::at(el, na, nb, nc), FS, a.status);
        T rho_t = T(1), m1_t = T(0), m2_t = T(0), m3_t = T(0), E_t = T(1), phi_t = T(0);
        T ja_t[9];
#pragma unroll
        for (int k = 0; k < 9; ++k) ja_t[k] = T(0);
        const bool real = t < e_count * NP3;
        const bool perturbed = a.rho_ref != nullptr;
        T rr_t = T(0), pr_t = T(0);
        if (real) {
            const long long g = checked(FaceFirst<C>::value ? node0 + (long long)el * NP3 + nd : node0 + t, a.n,
                                        a.status);
            const long long n = a.n;
            rho_t = __ldg(a.q + g);
            m1_t = __ldg(a.q + n + g);
            m2_t = __ldg(a.q + 2 * n + g);
            m3_t = __ldg(a.q + 3 * n + g);
            E_t = __ldg(a.q + 4 * n + g);
            phi_t = __ldg(a.phi + g);
#pragma unroll
            for (int k = 0; k < 9; ++k) ja_t[k] = __ldg(a.Ja + k * n + g);
            if (perturbed) {
                rr_t = __ldg(a.rho_ref + g);
                pr_t = __ldg(a.p_ref + g);
            }
        }
        const P m1 = PV::in(m1_t), m2 = PV::in(m2_t), m3 = PV::in(m3_t);
        const P E = PV::in(E_t), phi = PV::in(phi_t);
        // perturbation variables: q holds q - (rho_ref, 0, 0, 0, E_ref) with
        // E_ref = p_ref/(gamma-1) + rho_ref phi, so rho = rho_ref + rho' and
        // p = p_ref + (gamma-1)(E' - rho|u|^2/2 - rho' phi) without the
        // cancellation of E against rho phi and p_ref/(gamma-1)
        const P rho_p = PV::in(rho_t);
        const P rho = perturbed ? PV::in(rr_t) + rho_p : rho_p;
        P ja[9];
#pragma unroll
        for (int k = 0; k < 9; ++k) ja[k] = PV::in(ja_t[k]);
        const P gm1 = PV::in(a.gm1);
        const P irho = Num<P>::rcp(rho);
        const P ih = P(0.5) * irho;
        // v = u/2 (the scaling pair_terms expects) and vv = |u|^2/4
        const P v1 = m1 * ih, v2 = m2 * ih, v3 = m3 * ih;
        const P vv = fma(v3, v3, fma(v2, v2, v1 * v1));
        P pr = perturbed ? fma(gm1, E - fma(P(2.0) * rho, vv, rho_p * phi), PV::in(pr_t))
                         : gm1 * (E - rho * fma(P(2.0), vv, phi));
        if (!real) pr = P(0.5) * gm1;  // padding node: finite values, never stored
        bad |= !positive(rho) || !positive(pr);
        // stored with the scalings pair_terms expects: u/2, b2 = 2b = rho/p,
        // ln b2, phi/8 (1/b and h = phi/2 - |u|^2/4 unscaled)
        const P b2 = rho * Num<P>::rcp(pr);
        const P ib = P(4.0) * pr * ih;
        const P h = P(0.5) * phi - vv;
        sm[F_RHO * FS + sl] = rho;
        sm[F_U1 * FS + sl] = v1;
        sm[F_U2 * FS + sl] = v2;
        sm[F_U3 * FS + sl] = v3;
        sm[F_B * FS + sl] = b2;
        sm[F_INVB * FS + sl] = ib;
        if constexpr (NarrowCheck<C>::value) {
            // no per-node logarithms: the range of the CTA's values instead
            if (real) {
                r_lo = min(r_lo, __float_as_uint(rho));
                r_hi = max(r_hi, __float_as_uint(rho));
                b_lo = min(b_lo, __float_as_uint(b2));
                b_hi = max(b_hi, __float_as_uint(b2));
            }
        } else {
            sm[F_LNRHO * FS + sl] = Num<P>::log_(rho);
            sm[F_LNB * FS + sl] = Num<P>::log_(b2);
        }
        sm[F_PHI * FS + sl] = P(0.125) * phi;
        sm[F_H * FS + sl] = h;
#pragma unroll
        for (int k = 0; k < 9; ++k) sm[(F_JA0 + k) * FS + sl] = ja[k];

        // diagonal pairs of the 2D form: sum_r 2 D_{a_r a_r} Ja^r(i) . f(q_i), nonzero
        // only where a_r is 0 or N; f is the physical flux of Eq. 1
        P f0 = P(0.0), f1 = P(0.0), f2 = P(0.0), f3 = P(0.0), f4 = P(0.0);
        bool with_diag = a.form == 0;
        if constexpr (FaceFirst<C>::value)  // whole warps of interior nodes skip it
            with_diag = with_diag && __any_sync(__activemask(), na == 0 || na == N || nb == 0 || nb == N ||
                                                                    nc == 0 || nc == N);
        if (with_diag) {
            // 2 D_ii of the node's position along each direction (0 inside)
            const P dA = PV::in(a.ops.diag[na]);
            const P dB = PV::in(a.ops.diag[nb]);
            const P dC = PV::in(a.ops.diag[nc]);
            const P V0 = fma(dC, ja[6], fma(dB, ja[3], dA * ja[0]));
            const P V1 = fma(dC, ja[7], fma(dB, ja[4], dA * ja[1]));
            const P V2 = fma(dC, ja[8], fma(dB, ja[5], dA * ja[2]));
            // rho U = m.V; 2 rho U multiplies v = u/2
            const P rU = fma(m3, V2, fma(m2, V1, m1 * V0));
            const P rU2 = P(2.0) * rU;
            f0 = rU;
            f1 = fma(rU2, v1, pr * V0);
            f2 = fma(rU2, v2, pr * V1);
            f3 = fma(rU2, v3, pr * V2);
            // (E + p) U = rho U (gamma/(gamma-1) p/rho + |u|^2/2 + phi)
            f4 = rU * fma(PV::in(a.c_h), ib, fma(P(2.0), vv, phi));
        }
        sm[(F_ACC0 + 0) * FS + sl] = f0;
        sm[(F_ACC0 + 1) * FS + sl] = f1;
        sm[(F_ACC0 + 2) * FS + sl] = f2;
        sm[(F_ACC0 + 3) * FS + sl] = f3;
        sm[(F_ACC0 + 4) * FS + sl] = f4;
    }
    if constexpr (FaceMode<C, MODE>::value) {
        // neighbour traces of this CTA's face slots (walls: none): the
        // prefetched first slot, then any further slots of this thread
        using FSL = FaceSlots<N>;
        constexpr int CNT = FSL::COUNT;
        C* fb = sm + F_COUNT * FS;
        const long long n = a.n;
        if (trace_ok) {
#pragma unroll
            for (int v = 0; v < TR; ++v) fb[v * CNT + threadIdx.x] = trace[v];
        }
        for (int s = threadIdx.x + LK::THREADS; s < e_count * FSL::PER_EL; s += LK::THREADS) {
            int el, dir, side, i1, i2;
            FSL::decode(s, el, dir, side, i1, i2);
            long long g;
            if (!face_neighbour<N>(nbr, el, dir, side, i1, i2, g)) continue;
            g = checked(g, a.n, a.status);
#pragma unroll
            for (int v = 0; v < 5; ++v) fb[v * CNT + s] = __ldg(a.q + v * n + g);
#pragma unroll
            for (int c = 0; c < 3; ++c) fb[(5 + c) * CNT + s] = __ldg(a.Ja + (3 * dir + c) * n + g);
            fb[8 * CNT + s] = __ldg(a.phi + g);
            if (a.rho_ref) {
                fb[9 * CNT + s] = __ldg(a.rho_ref + g);
                fb[10 * CNT + s] = __ldg(a.p_ref + g);
            }
        }
    }
    if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) atomicOr(a.status, 1u);
    constexpr int WARPS = LK::THREADS / 32;
    static_assert(WARPS <= 32, "one range entry per lane");
    __shared__ unsigned s_range[NarrowCheck<C>::value ? 4 : 1][32];
    if constexpr (NarrowCheck<C>::value) {
        r_lo = __reduce_min_sync(0xffffffffu, r_lo);
        r_hi = __reduce_max_sync(0xffffffffu, r_hi);
        b_lo = __reduce_min_sync(0xffffffffu, b_lo);
        b_hi = __reduce_max_sync(0xffffffffu, b_hi);
        if ((threadIdx.x & 31) == 0) {
            const int w = threadIdx.x >> 5;
            s_range[0][w] = r_lo;
            s_range[1][w] = r_hi;
            s_range[2][w] = b_lo;
            s_range[3][w] = b_hi;
        }
    }

    // lane constants: Q_{p,p+d} for every offset, 1/w_p and 1/(gamma - 1)
    const int lane = threadIdx.x & 31;
    const int p = lane - (lane / NQ) * NQ;
    C cq[S::H];
#pragma unroll
    for (int d = 1; d <= S::H; ++d) cq[d - 1] = CV::in(T(0.5) * a.ops.Q2[p * NQ + wrap_pos<NQ>(p, d)]);
    const C iw = CV::in(a.ops.invw[p]);
    const C c_g = CV::in(T(2) * a.c_g);  // 1/(gamma - 1)
    __syncthreads();

    // NarrowCheck: every warp reduces the CTA's ranges from the warps'
    // entries, so all take the same decision.  A non-positive, infinite or
    // NaN value (bits at or above those of +inf) makes the CTA wide.
    bool narrow = false;
    if constexpr (NarrowCheck<C>::value) {
        const bool have = lane < WARPS;
        const unsigned rl = __reduce_min_sync(0xffffffffu, have ? s_range[0][lane] : 0xffffffffu);
        const unsigned rh = __reduce_max_sync(0xffffffffu, have ? s_range[1][lane] : 0u);
        const unsigned bl = __reduce_min_sync(0xffffffffu, have ? s_range[2][lane] : 0xffffffffu);
        const unsigned bh = __reduce_max_sync(0xffffffffu, have ? s_range[3][lane] : 0u);
        narrow = rh < 0x7f800000u && bh < 0x7f800000u &&
                 __uint_as_float(rh) <= kNarrowRatio * __uint_as_float(rl) &&
                 __uint_as_float(bh) <= kNarrowRatio * __uint_as_float(bl);
    }

    if constexpr (IsFF<C>::value) {
        // Float-float: one pair evaluation is ~850 instructions, so the
        // phases run as loops over a runtime direction (not unrolled) to keep
        // a single copy of each loop body in the instruction cache; a last
        // pass stores the sums.
        using LA = Launch<N, C>;
        const int warp = threadIdx.x >> 5;
#pragma unroll 1
        for (int k = 0; k < 3; ++k) {
            const int R = (k == 0) ? 1 : (k == 1) ? 2 : 0;
#pragma unroll 1
            for (int rep = 0; rep < LA::REPS; ++rep)
                direction_lines<T, C, N, 0>(a, sm, e_count, node0, cq, iw, c_g, warp + rep * LA::WARPS, R);
            __syncthreads();
        }
        if constexpr (S::EVEN && SplitAntipodal<C>::value) {
#pragma unroll 1
            for (int k = 0; k < 3; ++k) {
                antipodal_phase<T, C, N>(a, sm, e_count, c_g, (k == 0) ? 1 : (k == 1) ? 2 : 0);
                __syncthreads();
            }
        }
        const C* s_acc = sm + F_ACC0 * FS;
        for (int t = threadIdx.x; t < e_count * NP3; t += LA::THREADS) {
            const int el = t / NP3;
            const int nd = t - el * NP3;
            const int na = nd % NQ, nb = (nd / NQ) % NQ, nc = nd / (NQ * NQ);
            const int sl = checked(SL::at(el, na, nb, nc), FS, a.status);
            const long long g = checked(node0 + t, a.n, a.status);
            store_node<T, N, MODE>(a, g, na, nb, nc, el, nullptr, CV::out(s_acc[0 * FS + sl]),
                                 CV::out(s_acc[1 * FS + sl]),
                             CV::out(s_acc[2 * FS + sl]), CV::out(s_acc[3 * FS + sl]), CV::out(s_acc[4 * FS + sl]));
        }
    } else {
        if constexpr (FaceMode<C, MODE>::value) face_phase<T, C, N>(a, sm, nbr, e_count);
        auto phases = [&](auto narrow_tag) {
            constexpr bool NW = decltype(narrow_tag)::value;
            direction_phase<T, C, N, 1, 0, NW, MODE>(a, sm, e_count, node0, cq, iw, c_g);
            __syncthreads();
            direction_phase<T, C, N, 2, 0, NW, MODE>(a, sm, e_count, node0, cq, iw, c_g);
            __syncthreads();
            if constexpr (S::EVEN && SplitAntipodal<C>::value) {
                antipodal_phase<T, C, N>(a, sm, e_count, c_g, 1);
                __syncthreads();
                antipodal_phase<T, C, N>(a, sm, e_count, c_g, 2);
                __syncthreads();
                antipodal_phase<T, C, N>(a, sm, e_count, c_g, 0);
                __syncthreads();
            }
            direction_phase<T, C, N, 0, MODE + 1, NW, MODE>(a, sm, e_count, node0, cq, iw, c_g);
        };
        // a CTA-uniform branch: the polynomial form inline, the wide one out
        // of line
        if constexpr (NarrowCheck<C>::value) {
            if (narrow) phases(std::true_type{});
            else wide_phases<T, C, N, MODE>(a, sm, e_count, node0);
        } else {
            phases(std::false_type{});
        }
    }
}

template <typename T, int N, typename C, int MODE>
cudaError_t launch_volume_mode(const VolumeArgs<T>& a, cudaStream_t s) {
    using S = Shape<N>;
    const long long K = a.e_end - a.e_begin;
    if (K <= 0) return cudaSuccess;
    const size_t smem = volume_smem_bytes<C, N, MODE>();
    // The dynamic shared-memory limit is an attribute of the function on the
    // current device (and is lost when that device's context is reset), so it
    // is set on every launch: a host-side call, no stream work, and no shared
    // host state between threads or devices.
    cudaError_t err = cudaFuncSetAttribute(volume_kernel<T, N, C, MODE>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    const long long blocks = (K + S::EPB - 1) / S::EPB;
    volume_kernel<T, N, C, MODE><<<(unsigned)blocks, Launch<N, C, FaceMode<C, MODE>::value>::THREADS, smem, s>>>(a);
    return cudaGetLastError();
}

// The fused Runge-Kutta mode is built for FP32 and float-float only (native
// FP64 keeps the separate stage kernel); volume + faces to out for FP32 only.
template <typename T, int N, typename C = T>
cudaError_t launch_volume(const VolumeArgs<T>& a, cudaStream_t s) {
    if (a.rk_q != nullptr) {
        if constexpr (std::is_same<C, double>::value) return cudaErrorNotSupported;
        else return launch_volume_mode<T, N, C, 1>(a, s);
    }
    if (a.with_faces) {
        if constexpr (FusedSurface<C>::value) return launch_volume_mode<T, N, C, 2>(a, s);
        else return cudaErrorNotSupported;
    }
    return launch_volume_mode<T, N, C, 0>(a, s);
}

}  // namespace esdg
