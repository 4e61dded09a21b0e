// Float-float arithmetic: a value is the unevaluated sum hi + lo of two FP32
// numbers with |lo| <= ulp(hi)/2, which carries about 48 significant bits.
// The building blocks are the error-free transformations of Dekker (1971) and
// Knuth: two_sum gives a + b = s + e exactly, fast_two_sum does the same when
// |a| >= |b|, and a fused multiply-add gives the exact rounding error of a
// product.  Relative error of one operation is a small multiple of 2^-48
// (the addition is the "sloppy" variant, whose error is bounded relative to
// the operands rather than to the result -- the same kind of bound as a
// difference of rounded FP64 inputs).
//
// Why: GB300 executes FP32 at 64 times its FP64 rate, so FP64-accurate
// arithmetic built from FP32 operations on the FP32 pipes can beat native
// FP64.  The volume kernel uses this type for its pair arithmetic in the
// ESDG_FP64_FF precision (FP64 inputs and outputs).
//
// The algorithms are written for a component type F (float here).  Carrying
// two float-float values per thread in Blackwell's packed FP32 registers
// (add/mul/fma on float2) was measured slower for the volume kernel: the
// packed instructions hold the FMA pipe twice as long, so they only save
// issue slots, and the doubled register footprint spills.
//
// Range: the FP32 exponent range, about 1e-38 .. 3e38; magnitudes below
// about 1e-30 lose relative precision in lo.  Values are assumed finite.
#pragma once

#include <cuda_runtime.h>

namespace esdg {

// the float and double overloads stay visible next to the ones below
using ::fma;
using ::fabs;

__device__ __forceinline__ float sel(bool c, float a, float b) { return c ? a : b; }
__device__ __forceinline__ double sel(bool c, double a, double b) { return c ? a : b; }

// hardware reciprocal estimate
__device__ __forceinline__ float rcp_estimate(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// ---------------------------------------------------------------------------
// float-float over component type F
template <typename F>
struct ffv {
    F hi, lo;
    ffv() = default;
    __host__ __device__ constexpr ffv(F h, F l) : hi(h), lo(l) {}
    // exact split of a compile-time or host constant
    __host__ __device__ constexpr explicit ffv(double d)
        : hi(static_cast<float>(d)), lo(static_cast<float>(d - static_cast<double>(static_cast<float>(d)))) {}
};
using ff = ffv<float>;

__device__ __forceinline__ float ffma_(float a, float b, float c) { return __fmaf_rn(a, b, c); }

template <typename F>
__device__ __forceinline__ void ff_two_sum(F a, F b, F& s, F& e) {
    s = a + b;
    const F bb = s - a;
    e = (a - (s - bb)) + (b - bb);
}

template <typename F>
__device__ __forceinline__ ffv<F> ff_fast(F s, F e) {  // renormalise, |s| >= |e|
    const F h = s + e;
    return ffv<F>(h, e - (h - s));
}

template <typename F>
__device__ __forceinline__ ffv<F> operator+(ffv<F> x, ffv<F> y) {
    F s, e;
    ff_two_sum(x.hi, y.hi, s, e);
    e = e + (x.lo + y.lo);
    return ff_fast(s, e);
}

template <typename F>
__device__ __forceinline__ ffv<F> operator-(ffv<F> x) { return ffv<F>(-x.hi, -x.lo); }
template <typename F>
__device__ __forceinline__ ffv<F> operator-(ffv<F> x, ffv<F> y) { return x + (-y); }

template <typename F>
__device__ __forceinline__ ffv<F> operator*(ffv<F> x, ffv<F> y) {
    const F p = x.hi * y.hi;
    F e = ffma_(x.hi, y.hi, -p);
    e = ffma_(x.hi, y.lo, e);
    e = ffma_(x.lo, y.hi, e);
    return ff_fast(p, e);
}

template <typename F>
__device__ __forceinline__ ffv<F>& operator+=(ffv<F>& x, ffv<F> y) { return x = x + y; }
template <typename F>
__device__ __forceinline__ ffv<F>& operator-=(ffv<F>& x, ffv<F> y) { return x = x - y; }

// x*y + z with the product's rounding error kept and one renormalisation
template <typename F>
__device__ __forceinline__ ffv<F> fma(ffv<F> x, ffv<F> y, ffv<F> z) {
    const F p = x.hi * y.hi;
    F e = ffma_(x.hi, y.hi, -p);
    e = ffma_(x.hi, y.lo, e);
    e = ffma_(x.lo, y.hi, e);
    F s, t;
    ff_two_sum(p, z.hi, s, t);
    t = t + (e + z.lo);
    return ff_fast(s, t);
}

// 1/x: FP32 estimate r of x.hi, then one Newton-Raphson step in float-float,
// r' = r + r (1 - x r); the estimate's error (about 2^-23) squares.
template <typename F>
__device__ __forceinline__ ffv<F> ff_rcp(ffv<F> x) {
    const F r = rcp_estimate(x.hi);
    const F z = F(0.0f);
    const ffv<F> e = ffv<F>(F(1.0f), z) - x * ffv<F>(r, z);
    return ffv<F>(r, z) + ffv<F>(r, z) * e;
}

__device__ __forceinline__ ff sel(bool c, ff a, ff b) { return c ? a : b; }
__device__ __forceinline__ ff fabs(ff x) { return x.hi < 0.0f ? -x : x; }

// sqrt(x) for x > 0: FP32 square root y of x.hi, then one correction
// y + (x - y^2)/(2y) with the residual x - y^2 formed exactly (FMA product
// error); relative error about 2^-47 (Karp and Markstein's method).
__device__ __forceinline__ ff ff_sqrt(ff x) {
    const float y = sqrtf(x.hi);
    const float p = y * y;
    const float pe = __fmaf_rn(y, y, -p);
    const float r = ((x.hi - p) - pe) + x.lo;
    const float c = r * (0.5f * rcp_estimate(y));
    const float h = y + c;
    return ff(h, c - (h - y));
}

// ---------------------------------------------------------------------------
// conversions from and to FP64 with the conversion instructions (FP64 pipe)
__device__ __forceinline__ ff ff_from_double(double d) {
    const float h = __double2float_rn(d);
    return ff(h, __double2float_rn(d - static_cast<double>(h)));
}
__device__ __forceinline__ double ff_to_double(ff x) {
    return static_cast<double>(x.hi) + static_cast<double>(x.lo);
}

// The same conversions on the integer pipe, which keeps them off GB300's
// narrow FP64 pipe.  Split: hi is d with its significand cut to 24 bits
// (exact as a float), lo the remaining 29 bits scaled by 2^(E-1075), i.e.
// hi + lo = d up to the rounding of those 29 bits to a float (< 2^-48 |d|).
// Zeros are exact; magnitudes outside 2^-74 .. 2^128 take the conversion
// instructions instead.
__device__ __forceinline__ ff ff_split(double d) {
    const unsigned hw = static_cast<unsigned>(__double2hiint(d));
    const unsigned lw = static_cast<unsigned>(__double2loint(d));
    const unsigned sign = hw & 0x80000000u;
    const int ef = static_cast<int>((hw >> 20) & 0x7FFu) - 896;  // float biased exponent
    if (ef >= 53 && ef <= 254) {
        const float hi = __uint_as_float(sign | (static_cast<unsigned>(ef) << 23) | ((hw & 0xFFFFFu) << 3) |
                                         (lw >> 29));
        const float lo = __uint2float_rn(lw & 0x1FFFFFFFu) * __uint_as_float(sign | (static_cast<unsigned>(ef - 52) << 23));
        return ff(hi, lo);
    }
    if (((hw & 0x7FFFFFFFu) | lw) == 0u) return ff(__uint_as_float(sign), 0.0f);
    return ff_from_double(d);
}

// A normal float widened to double by moving its bits (exact); zeros and
// subnormals go through the conversion instruction.
__device__ __forceinline__ double ff_widen(float f) {
    const unsigned b = __float_as_uint(f);
    const unsigned e = (b >> 23) & 0xFFu;
    if (e == 0u || e == 0xFFu) return static_cast<double>(f);
    return __hiloint2double(static_cast<int>((b & 0x80000000u) | ((e + 896u) << 20) | ((b & 0x7FFFFFu) >> 3)),
                            static_cast<int>(b << 29));
}
__device__ __forceinline__ double ff_join(ff x) { return ff_widen(x.hi) + ff_widen(x.lo); }

// Natural logarithm of a positive float-float x, with no FP64 instruction.
// Argument reduction by the binary exponent of x.hi: x = 2^e m with m in
// [sqrt(1/2), sqrt(2)), then ln m = 2 atanh(s) = 2 s (1 + s^2/3 + s^4/5 + ...)
// with s = (m - 1)/(m + 1), |s| <= 0.1716 (the series of Abramowitz & Stegun
// 4.1.27).  Terms up to s^8/9 are summed in float-float, the rest (each below
// 2^-26 relative) in FP32; ln 2 enters as a three-part constant so that e ln 2
// is exact to float-float precision.  Absolute error about 2^-48 |ln x|;
// x.hi must be a positive normal float.
__device__ __forceinline__ ff ff_log(ff x) {
    const unsigned hb = __float_as_uint(x.hi);
    int e = static_cast<int>((hb >> 23) & 0xFFu) - 127;
    unsigned mb = (hb & 0x007FFFFFu) | 0x3F800000u;  // m in [1, 2)
    if (mb > 0x3FB504F3u) {                           // m > sqrt(2): use m/2, e + 1
        mb -= 0x00800000u;
        e += 1;
    }
    const float scale = __uint_as_float(static_cast<unsigned>(127 - e) << 23);  // 2^-e, exact
    const ff m(__uint_as_float(mb), x.lo * scale);
    const ff num = m + ff(-1.0f, 0.0f);
    const ff den = m + ff(1.0f, 0.0f);
    const ff s = num * ff_rcp(den);
    const ff z = s * s;
    // tail 1/11 + z/13 + z^2/15 + z^3/17 + z^4/19 in FP32
    const float zf = z.hi;
    float tail = __fmaf_rn(zf, 1.0f / 19.0f, 1.0f / 17.0f);
    tail = __fmaf_rn(zf, tail, 1.0f / 15.0f);
    tail = __fmaf_rn(zf, tail, 1.0f / 13.0f);
    tail = __fmaf_rn(zf, tail, 1.0f / 11.0f);
    ff P = fma(z, ff(tail, 0.0f), ff(1.0 / 9.0));
    P = fma(z, P, ff(1.0 / 7.0));
    P = fma(z, P, ff(1.0 / 5.0));
    P = fma(z, P, ff(1.0 / 3.0));
    P = fma(z, P, ff(1.0f, 0.0f));
    const ff lnm = (s + s) * P;
    // e ln 2 with ln 2 = L1 + L2 + L3: L1 has 16 significant bits, so e L1 is exact
    const float ef = static_cast<float>(e);
    constexpr float L1 = 0.693145751953125f;      // 0x3F317200, 45426 * 2^-16
    constexpr float L2 = 1.428606765330187e-06f;  // ln 2 - L1 rounded to float
    constexpr float L3 = 5.497923148104107e-14f;  // ln 2 - L1 - L2 rounded to float
    const ff eln2 = ff(ef * L1, 0.0f) + (ff(ef, 0.0f) * ff(L2, L3));
    return eln2 + lnm;
}

__device__ __forceinline__ ff shfl_ff(ff v, int src) {
    return ff(__shfl_sync(0xffffffffu, v.hi, src), __shfl_sync(0xffffffffu, v.lo, src));
}

}  // namespace esdg
