// Two FP32 values carried as one operand of Blackwell's packed FP32
// instructions (add, multiply and fused multiply-add on float2).  One packed
// instruction does two lanes' worth of FP32 arithmetic in one issue slot; it
// occupies the FMA pipe for two cycles, so it pays where a kernel is bound by
// instruction issue rather than by the FMA pipe -- the FP32 volume kernel,
// which evaluates two line pairs of a thread at once with it.
#pragma once

#include <cuda_runtime.h>

namespace esdg {

struct p2 {
    float2 v;
    p2() = default;
    __device__ __forceinline__ p2(float a, float b) { v = make_float2(a, b); }
    // both halves equal to a compile-time constant
    __device__ __forceinline__ explicit p2(double c) { v = make_float2((float)c, (float)c); }
};

// a pair of predicates, one per half
struct m2 {
    bool x, y;
};

__device__ __forceinline__ p2 pk(float2 f) {
    p2 r;
    r.v = f;
    return r;
}
__device__ __forceinline__ p2 operator+(p2 a, p2 b) { return pk(__fadd2_rn(a.v, b.v)); }
__device__ __forceinline__ p2 operator*(p2 a, p2 b) { return pk(__fmul2_rn(a.v, b.v)); }
__device__ __forceinline__ p2 fma(p2 a, p2 b, p2 c) { return pk(__ffma2_rn(a.v, b.v, c.v)); }
__device__ __forceinline__ p2 operator-(p2 a) { return pk(__fmul2_rn(a.v, make_float2(-1.0f, -1.0f))); }
__device__ __forceinline__ p2 operator-(p2 a, p2 b) { return pk(__ffma2_rn(b.v, make_float2(-1.0f, -1.0f), a.v)); }
__device__ __forceinline__ p2& operator+=(p2& a, p2 b) { return a = a + b; }
__device__ __forceinline__ p2 sel(m2 c, p2 a, p2 b) { return p2(c.x ? a.v.x : b.v.x, c.y ? a.v.y : b.v.y); }

}  // namespace esdg
