// Index maps of the face-centric surface kernel (surface_kernel.cu), callable
// from host code too so that the index arithmetic can be checked on the CPU.
#pragma once

#include <cuda_runtime.h>

namespace esdg {

// Node index of face node (s1, s2) on the face a_DIR = A of a (N+1)^3 element.
template <int N, int DIR>
__host__ __device__ __forceinline__ int face_node(int A, int s1, int s2) {
    constexpr int NQ = N + 1;
    if constexpr (DIR == 0) return A + NQ * (s1 + NQ * s2);
    else if constexpr (DIR == 1) return s1 + NQ * (A + NQ * s2);
    else return s1 + NQ * (s2 + NQ * A);
}

// Thread t of the direction-DIR launch: slots [0, K (N+1)^2) are the +xi_DIR
// faces of every element (an interface with the next element along DIR,
// wrapped when periodic, or a wall); the slots after them are the -xi_DIR
// faces of the elements with index 0 along DIR when DIR has walls.  Gives
// the element e, its index er along DIR, the face node f and the side;
// false past the last slot.
template <int N>
__host__ __device__ __forceinline__ bool surface_slot(int DIR, long long t, long long Kx, long long Ky,
                                                      long long Kz, bool wall_dir, long long& e, int& f,
                                                      bool& plus_face, long long& er) {
    constexpr int NF = (N + 1) * (N + 1);
    const long long K = Kx * Ky * Kz;
    const long long Kd = DIR == 0 ? Kx : DIR == 1 ? Ky : Kz;
    const long long n_plus = K * NF;
    const long long n_minus = wall_dir ? (K / Kd) * NF : 0;
    if (t < 0 || t >= n_plus + n_minus) return false;
    if (t < n_plus) {
        e = t / NF;
        f = (int)(t - e * NF);
        plus_face = true;
    } else {
        const long long u = t - n_plus;
        const long long k = u / NF;
        f = (int)(u - k * NF);
        // element with index 0 along DIR, k enumerating the other two indices
        if (DIR == 0) e = k * Kx;
        else if (DIR == 1) e = (k % Kx) + (k / Kx) * Kx * Ky;
        else e = k;
        plus_face = false;
    }
    er = (DIR == 0) ? e % Kx : (DIR == 1) ? (e / Kx) % Ky : e / (Kx * Ky);
    return true;
}

}  // namespace esdg
