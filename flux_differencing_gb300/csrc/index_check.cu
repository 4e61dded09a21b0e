// Host check of the kernels' index arithmetic: the same __host__ __device__
// functions the volume and surface kernels use to place nodes in shared
// memory, deal lines to lanes, order the load phase, pair antipodal nodes,
// number face slots, find neighbour elements and enumerate surface slots,
// walked exhaustively on the CPU for one order and one mesh.  Every index
// must stay in range, every map that should be a bijection must be one, and
// every node the kernels must visit must be visited exactly once.
#include <cstdio>
#include <string>
#include <vector>

#include "esdg_bench.h"
#include "surface_index.cuh"
#include "volume_kernel.cuh"

namespace {

using esdg::FaceSlots;
using esdg::Shape;
using esdg::Slots;

struct Fail {
    std::string msg;
    bool set(const char* what, long long a = 0, long long b = 0, long long c = 0) {
        if (msg.empty()) {
            char buf[256];
            std::snprintf(buf, sizeof buf, "%s (%lld, %lld, %lld)", what, a, b, c);
            msg = buf;
        }
        return false;
    }
};

// Lines dealt to the lanes of the direction phases: every line of every
// element of a CTA holding e_count elements visited exactly once, at every
// position, over the virtual warps warp + rep WARPS (for each CTA shape:
// FACES, the FP32 kernels with the face machinery).
template <int N, typename C, bool FACES>
bool check_lanes(Fail& f) {
    using S = Shape<N>;
    using LA = esdg::Launch<N, C, FACES>;
    if (LA::WARPS * LA::REPS * S::LPW < S::LINES) return f.set("too few lane lines", LA::WARPS, LA::REPS);
    for (int e_count = 1; e_count <= S::EPB; ++e_count) {
        std::vector<int> seen(S::LINES * S::NQ, 0);
        for (int rep = 0; rep < LA::REPS; ++rep)
            for (int warp = 0; warp < LA::WARPS; ++warp)
                for (int lane = 0; lane < 32; ++lane) {
                    int slot, p, L;
                    const bool valid = esdg::lane_line<N>(warp + rep * LA::WARPS, lane, e_count, slot, p, L);
                    if (L < 0 || L >= S::LINES || p < 0 || p >= S::NQ) return f.set("lane line out of range", L, p);
                    if (valid) ++seen[L * S::NQ + p];
                }
        for (int L = 0; L < S::LINES; ++L)
            for (int p = 0; p < S::NQ; ++p)
                if (seen[L * S::NQ + p] != (L / S::NL < e_count ? 1 : 0))
                    return f.set("lane lines not covered once", e_count, L, p);
    }
    return true;
}

template <int N>
bool check_element(Fail& f) {
    using S = Shape<N>;
    using SL = Slots<N>;
    using FSL = FaceSlots<N>;
    constexpr int NQ = S::NQ;
    constexpr int NP3 = S::NP3;
    // shared-memory slots: injective into one field of SIZE values
    std::vector<int> used(SL::SIZE, 0);
    for (int el = 0; el < S::EPB; ++el)
        for (int c = 0; c < NQ; ++c)
            for (int b = 0; b < NQ; ++b)
                for (int a = 0; a < NQ; ++a) {
                    const int i = SL::at(el, a, b, c);
                    if (i < 0 || i >= SL::SIZE) return f.set("shared-memory slot out of range", el, a + NQ * (b + NQ * c), i);
                    if (used[i]++) return f.set("two nodes share a shared-memory slot", el, a + NQ * (b + NQ * c), i);
                }
    // lines of each direction: (line, position) -> node is a bijection, the
    // position is the node's index along the direction
    for (int R = 0; R < 3; ++R) {
        std::vector<int> seen(NP3, 0);
        for (int ell = 0; ell < S::NL; ++ell)
            for (int p = 0; p < NQ; ++p) {
                int a, b, c;
                esdg::line_node<N>(R, ell, p, a, b, c);
                if (a < 0 || a > N || b < 0 || b > N || c < 0 || c > N) return f.set("line node out of range", R, ell, p);
                if ((R == 0 ? a : R == 1 ? b : c) != p) return f.set("line position mismatch", R, ell, p);
                ++seen[a + NQ * (b + NQ * c)];
            }
        for (int k = 0; k < NP3; ++k)
            if (seen[k] != 1) return f.set("lines do not cover the element once", R, k, seen[k]);
    }
    // the xi lines of a warp are consecutive rows (the coalesced store)
    for (int ell = 0; ell + 1 < S::NL; ++ell) {
        int a0, b0, c0, a1, b1, c1;
        esdg::line_node<N>(0, ell, 0, a0, b0, c0);
        esdg::line_node<N>(0, ell + 1, 0, a1, b1, c1);
        if (b1 + NQ * c1 != b0 + NQ * c0 + 1) return f.set("xi lines not in row order", ell);
    }
    if (!check_lanes<N, double, false>(f) || !check_lanes<N, float, false>(f) || !check_lanes<N, float, true>(f) ||
        !check_lanes<N, esdg::ff, false>(f))
        return false;
    // load order of the FP64 kernel: a permutation, face nodes first
    {
        std::vector<int> seen(NP3, 0);
        const int nface = NP3 - (N - 1) * (N - 1) * (N - 1);
        for (int k = 0; k < NP3; ++k) {
            const int nd = esdg::face_first_node<N>(k);
            if (nd < 0 || nd >= NP3) return f.set("face-first node out of range", k, nd);
            ++seen[nd];
            const int a = nd % NQ, b = (nd / NQ) % NQ, c = nd / (NQ * NQ);
            const bool face = a == 0 || a == N || b == 0 || b == N || c == 0 || c == N;
            if (face != (k < nface)) return f.set("face-first order: face nodes not first", k, nd);
        }
        for (int k = 0; k < NP3; ++k)
            if (seen[k] != 1) return f.set("face-first order is not a permutation", k, seen[k]);
    }
    // antipodal pass (even Nq): every node in exactly one pair per direction
    if constexpr (S::EVEN) {
        constexpr int H = S::H;
        for (int R = 0; R < 3; ++R) {
            std::vector<int> seen(S::EPB * NP3, 0);
            for (int k = 0; k < S::EPB * S::NL * H; ++k) {
                int el, p, ell;
                esdg::antipodal_pair<N>(k, el, p, ell);
                if (el < 0 || el >= S::EPB || p < 0 || p >= H || ell < 0 || ell >= S::NL)
                    return f.set("antipodal pair out of range", k, el, p);
                int a, b, c;
                esdg::line_node<N>(R, ell, p, a, b, c);
                ++seen[el * NP3 + a + NQ * (b + NQ * c)];
                esdg::line_node<N>(R, ell, p + H, a, b, c);
                ++seen[el * NP3 + a + NQ * (b + NQ * c)];
            }
            for (int k = 0; k < S::EPB * NP3; ++k)
                if (seen[k] != 1) return f.set("antipodal pairs do not cover each node once", R, k, seen[k]);
        }
    }
    // face slots of the fused FP32 kernel: decode inverts slot, every slot
    // names a node on its face, and every face node finds its slots
    for (int s = 0; s < FSL::COUNT; ++s) {
        int el, dir, side, i1, i2;
        FSL::decode(s, el, dir, side, i1, i2);
        if (el < 0 || el >= S::EPB || dir < 0 || dir > 2 || i1 < 0 || i1 > N || i2 < 0 || i2 > N)
            return f.set("face slot decodes out of range", s);
        if (FSL::slot(el, dir, side, i1, i2) != s) return f.set("face slot round trip", s);
        int a, b, c;
        FSL::node(dir, side ? N : 0, i1, i2, a, b, c);
        if (a < 0 || a > N || b < 0 || b > N || c < 0 || c > N) return f.set("face slot node out of range", s);
    }
    for (int c = 0; c < NQ; ++c)
        for (int b = 0; b < NQ; ++b)
            for (int a = 0; a < NQ; ++a) {
                const int idx[3][3] = {{a, b, c}, {b, a, c}, {c, a, b}};  // (A, i1, i2) per direction
                for (int d = 0; d < 3; ++d) {
                    const int A = idx[d][0];
                    if (A != 0 && A != N) continue;
                    const int s = FSL::slot(S::EPB - 1, d, A == N ? 1 : 0, idx[d][1], idx[d][2]);
                    if (s < 0 || s >= FSL::COUNT) return f.set("store-side face slot out of range", d, s);
                    int na, nb, nc;
                    FSL::node(d, A, idx[d][1], idx[d][2], na, nb, nc);
                    if (na != a || nb != b || nc != c) return f.set("store-side face slot names another node", d, s);
                }
            }
    return true;
}

// Neighbour elements and face traces of the fused FP32 kernel, and the slots
// of the face-centric surface kernel, on one Kx x Ky x Kz brick.
template <int N>
bool check_mesh(long Kx, long Ky, long Kz, const int* bc, Fail& f) {
    constexpr int NQ = N + 1;
    constexpr long long NP3 = (long long)NQ * NQ * NQ;
    const long long K = (long long)Kx * Ky * Kz;
    const long long n = K * NP3;
    const long long Kd[3] = {Kx, Ky, Kz};
    esdg::VolumeArgs<float> va{};
    va.Kx = Kx;
    va.Ky = Ky;
    va.Kz = Kz;
    for (int d = 0; d < 3; ++d) va.bc[d] = bc[d];
    for (long long e = 0; e < K; ++e) {
        const long long r[3] = {e % Kx, (e / Kx) % Ky, e / (Kx * Ky)};
        for (int dir = 0; dir < 3; ++dir)
            for (int side = 0; side < 2; ++side) {
                const long long en = esdg::neighbour_element(va, e, dir, side);
                const bool boundary = side ? r[dir] == Kd[dir] - 1 : r[dir] == 0;
                if (en < 0) {
                    if (!(bc[dir] && boundary)) return f.set("wall where there is none", e, dir, side);
                    continue;
                }
                if (bc[dir] && boundary) return f.set("neighbour across a wall", e, dir, side);
                if (en >= K) return f.set("neighbour element out of range", e, dir, en);
                if (esdg::neighbour_element(va, en, dir, 1 - side) != e)
                    return f.set("neighbour of the neighbour is not the element", e, dir, side);
                // the node across each face node: on the neighbour's opposite face
                long long nbr[6];
                for (int t = 0; t < 6; ++t) nbr[t] = esdg::neighbour_element(va, e, t >> 1, t & 1);
                for (int i2 = 0; i2 < NQ; ++i2)
                    for (int i1 = 0; i1 < NQ; ++i1) {
                        long long g;
                        if (!esdg::face_neighbour<N>(nbr, 0, dir, side, i1, i2, g))
                            return f.set("face neighbour missing", e, dir, side);
                        if (g < 0 || g >= n) return f.set("face neighbour node out of range", e, dir, g);
                        const long long node = g - en * NP3;
                        const int a = (int)(node % NQ), b = (int)((node / NQ) % NQ), c = (int)(node / (NQ * NQ));
                        const int along = dir == 0 ? a : dir == 1 ? b : c;
                        const int o1 = dir == 0 ? b : a, o2 = dir == 2 ? b : c;
                        if (node < 0 || node >= NP3 || along != (side ? 0 : N) || o1 != i1 || o2 != i2)
                            return f.set("face neighbour is not the node across", e, dir, node);
                    }
            }
    }
    // face-centric surface kernel: each face node of direction DIR written by
    // exactly one slot (as the slot's own node or as the far node), all
    // indices in range
    for (int DIR = 0; DIR < 3; ++DIR) {
        const long long stride = DIR == 0 ? 1 : DIR == 1 ? Kx : (long long)Kx * Ky;
        std::vector<unsigned char> written(n, 0);
        for (long long t = 0;; ++t) {
            long long e, er;
            int fn;
            bool plus;
            if (!esdg::surface_slot<N>(DIR, t, Kx, Ky, Kz, bc[DIR] != 0, e, fn, plus, er)) break;
            if (e < 0 || e >= K || fn < 0 || fn >= NQ * NQ || er < 0 || er >= Kd[DIR])
                return f.set("surface slot out of range", DIR, t, e);
            if (!plus && er != 0) return f.set("minus-face slot not on the first layer", DIR, t, e);
            const int s1 = fn % NQ, s2 = fn / NQ;
            auto fnode = [&](int A) {
                return DIR == 0 ? esdg::face_node<N, 0>(A, s1, s2)
                                : DIR == 1 ? esdg::face_node<N, 1>(A, s1, s2) : esdg::face_node<N, 2>(A, s1, s2);
            };
            const long long gi = e * NP3 + fnode(plus ? N : 0);
            if (gi < 0 || gi >= n) return f.set("surface node out of range", DIR, t, gi);
            ++written[gi];
            const bool interior = plus && (er + 1 < Kd[DIR] || bc[DIR] == 0);
            if (interior) {
                const long long ej = (er + 1 < Kd[DIR]) ? e + stride : e - (Kd[DIR] - 1) * stride;
                if (ej < 0 || ej >= K) return f.set("surface far element out of range", DIR, t, ej);
                const long long gj = ej * NP3 + fnode(0);
                if (gj < 0 || gj >= n) return f.set("surface far node out of range", DIR, t, gj);
                ++written[gj];
            }
        }
        for (long long g = 0; g < n; ++g) {
            const long long node = g % NP3;
            const int a = (int)(node % NQ), b = (int)((node / NQ) % NQ), c = (int)(node / (NQ * NQ));
            const int along = DIR == 0 ? a : DIR == 1 ? b : c;
            const int want = (along == 0 || along == N) ? 1 : 0;
            if (written[g] != want) return f.set("surface face node not written exactly once", DIR, g, written[g]);
        }
    }
    return true;
}

template <int N>
bool check(long Kx, long Ky, long Kz, const int* bc, Fail& f) {
    return check_element<N>(f) && check_mesh<N>(Kx, Ky, Kz, bc, f);
}

}  // namespace

extern "C" int esdg_selftest_index_maps(int N, long Kx, long Ky, long Kz, const int* bc, char* msg, int msglen) {
    if (N < 1 || N > 8 || Kx < 1 || Ky < 1 || Kz < 1 || !bc) return 1;
    if ((long double)Kx * Ky * Kz * (N + 1) * (N + 1) * (N + 1) > 5e7L) return 1;  // host walk: keep it small
    Fail f;
    bool ok = false;
    switch (N) {
        case 1: ok = check<1>(Kx, Ky, Kz, bc, f); break;
        case 2: ok = check<2>(Kx, Ky, Kz, bc, f); break;
        case 3: ok = check<3>(Kx, Ky, Kz, bc, f); break;
        case 4: ok = check<4>(Kx, Ky, Kz, bc, f); break;
        case 5: ok = check<5>(Kx, Ky, Kz, bc, f); break;
        case 6: ok = check<6>(Kx, Ky, Kz, bc, f); break;
        case 7: ok = check<7>(Kx, Ky, Kz, bc, f); break;
        case 8: ok = check<8>(Kx, Ky, Kz, bc, f); break;
    }
    if (!ok && msg && msglen > 0) std::snprintf(msg, (size_t)msglen, "%s", f.msg.c_str());
    return ok ? 0 : 2;
}
