// Numeric building blocks shared by the volume, surface and time-stepping
// kernels: reciprocal, closeness tests and logarithm per arithmetic type
// (FP64, FP32, float-float), the non-physical-state test, warp shuffles and
// the conversion between a kernel's I/O type and its arithmetic type.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "floatfloat.cuh"
#include "log_fp64.cuh"

// Debug builds (compiled with -DESDG_DEBUG_CHECKS=1 into a library of their
// own, libesdg_debug.so) range-check every computed shared-memory, face-slot
// and global index of the volume and surface kernels and poison shared memory
// before the kernels fill it; release builds compile both to nothing.
#ifndef ESDG_DEBUG_CHECKS
#define ESDG_DEBUG_CHECKS 0
#endif

namespace esdg {

constexpr unsigned kStatusIndex = 4u;  // ESDG_STATUS_INDEX of esdg.h

// Debug builds: an index outside [0, hi) sets ESDG_STATUS_INDEX in the status
// word and is replaced by 0, so that the access stays in bounds and the kernel
// runs to its end (nothing traps).  Release builds return i unchanged.
template <typename I>
__device__ __forceinline__ I checked(I i, long long hi, unsigned* status) {
#if ESDG_DEBUG_CHECKS
    if (i < 0 || static_cast<long long>(i) >= hi) {
        atomicOr(status, kStatusIndex);
        return I(0);
    }
#endif
    (void)hi;
    (void)status;
    return i;
}

// Debug builds: fill `bytes` of shared memory with all-ones words, a NaN in
// FP32 and in FP64, so that a read of a slot no phase has written shows up as
// NaN in the output.  Called by every thread of the CTA; ends with a barrier.
__device__ __forceinline__ void poison_shared(void* p, size_t bytes) {
#if ESDG_DEBUG_CHECKS
    unsigned* w = static_cast<unsigned*>(p);
    for (size_t k = threadIdx.x; k < bytes / 4; k += blockDim.x) w[k] = 0xffffffffu;
    __syncthreads();
#endif
    (void)p;
    (void)bytes;
}

template <typename T>
struct Num;
template <>
struct Num<double> {
    // 1/x: hardware estimate (rcp.approx.ftz.f64) and one Newton-Raphson step
    // of third order, r' = r (1 + e + e^2) with e = 1 - x r, which cubes the
    // estimate's relative error.  Zeros and infinities never reach a result
    // that is used (the selects pick the other branch).
    static __device__ __forceinline__ double rcp(double x) {
        double r;
        asm("rcp.approx.ftz.f64 %0, %1;" : "=d"(r) : "d"(x));
        const double e = fma(-x, r, 1.0);
        return fma(r, fma(e, e, e), r);
    }
    // 1/x for the pair evaluations of the volume kernel: an estimate from the
    // FP32 reciprocal of x's mantissa, refined by one Newton-Raphson step of
    // second order, r' = r (1 + e), which squares the estimate's relative error.
    // The FP64 estimate above reads only the high word of x and is good to
    // about 2^-20 (measured), so one second-order step would leave 2^-40;
    // the mantissa's top 23 bits through the FP32 reciprocal give about 2^-22,
    // and the step then about 2^-44 -- one FP64 operation fewer than rcp(),
    // the estimate built on the integer and FP32 pipes.  The pair reciprocals
    // scale the pressure mean and the logarithmic means, so their relative
    // error passes into the flux terms unamplified.  For normal |x| in
    // [2^-1020, 2^1020] (the pair quantities are differences and sums of
    // per-node logarithms and of rho/p); the bound is measured on the GPU by
    // the test suite.
    static __device__ __forceinline__ double rcp_estimate(double x) {
        const int hi = __double2hiint(x);
        const unsigned lo = static_cast<unsigned>(__double2loint(x));
        // x = +-M 2^(E - 1023), M in [1, 2): M's top 23 bits as a float
        const float m = __int_as_float(0x3f800000 | ((hi & 0x000fffff) << 3) | static_cast<int>(lo >> 29));
        float rm;
        asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(rm) : "f"(m));  // in (0.5, 1]
        // 1/x = +-rm 2^(1023 - E): rm's exponent field (126 or 127) rebiased
        // for a double, its 23 mantissa bits moved to the top of a double's
        const int rb = __float_as_int(rm);
        const int E = (hi >> 20) & 0x7ff;
        const int ohi = (hi & static_cast<int>(0x80000000u)) | ((rb >> 3) + ((1919 - E) << 20));
        return __hiloint2double(ohi, rb << 29);
    }
    static __device__ __forceinline__ double rcp_pair(double x) {
        const double r = rcp_estimate(x);
        return fma(r, fma(-x, r, 1.0), r);
    }
    // 1/sqrt(x) for positive normal x in [2^-1020, 2^1020] the same way: the
    // FP32 reciprocal square root of the mantissa (times 2 when the binary
    // exponent is odd, so that the exponent halves exactly), then one
    // second-order Newton step y' = y + y (1 - x y^2)/2 (relative error about
    // 3/2 of the estimate's squared: near 2^-43, measured by the test suite).
    static __device__ __forceinline__ double rsqrt_estimate(double x) {
        const int hi = __double2hiint(x);
        const unsigned lo = static_cast<unsigned>(__double2loint(x));
        const int e = ((hi >> 20) & 0x7ff) - 1023;
        const int odd = e & 1;
        // M' = M or 2 M in [1, 4), top 23 mantissa bits, as a float
        const float m = __int_as_float(((127 + odd) << 23) | ((hi & 0x000fffff) << 3) | static_cast<int>(lo >> 29));
        float rm;
        asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(rm) : "f"(m));  // in (0.5, 1]
        // 1/sqrt(x) = rm 2^(-(e - odd)/2)
        const int rb = __float_as_int(rm);
        const int ohi = (rb >> 3) + ((896 - ((e - odd) >> 1)) << 20);
        return __hiloint2double(ohi, rb << 29);
    }
    static __device__ __forceinline__ double rsqrt_pair(double x) {
        const double y = rsqrt_estimate(x);
        return fma(0.5 * y, fma(-x * y, y, 1.0), y);
    }
    // |d| < 0.02 (high word of 0.02 = 0x3F947AE1), tested on the integer pipe
    static __device__ __forceinline__ bool close(double d) {
        return (static_cast<unsigned>(__double2hiint(d)) & 0x7fffffffu) < 0x3F947AE1u;
    }
    // table-driven, 14 FP64 operations (log_fp64.cuh); within 2 ulp
    static __device__ __forceinline__ double log_(double x) { return log_fp64(x); }
    // |f| < 0.01 (high word of 0.01 = 0x3F847AE1): for f = (a+ - a-)/(a+ + a-)
    // this is |ln a+ - ln a-| < 2 atanh(0.01), the same closeness as close()
    static __device__ __forceinline__ bool close_ratio(double f) {
        return (static_cast<unsigned>(__double2hiint(f)) & 0x7fffffffu) < 0x3F847AE1u;
    }
};
template <>
struct Num<float> {
    static __device__ __forceinline__ float rcp(float x) {
        float r;
        asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
        return r;
    }
    static __device__ __forceinline__ float rcp_pair(float x) { return rcp(x); }
    static __device__ __forceinline__ float log_(float x) { return logf(x); }
    // the hardware base-2 logarithm (absolute error about 2^-22)
    static __device__ __forceinline__ float lg2(float x) {
        float r;
        asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
        return r;
    }
    static __device__ __forceinline__ bool above(float u, float lim) { return u > lim; }
    // |f| < 0.1 (0x3DCCCCCD), i.e. |ln a+ - ln a-| < 2 atanh(0.1) ~ 0.2
    static __device__ __forceinline__ bool close_ratio(float f) {
        return (__float_as_uint(f) & 0x7fffffffu) < 0x3DCCCCCDu;
    }
};
// float-float pair arithmetic (ESDG_FP64_FF): thresholds as in FP64, tested on hi
template <>
struct Num<ff> {
    static __device__ __forceinline__ ff rcp(ff x) { return ff_rcp(x); }
    static __device__ __forceinline__ ff rcp_pair(ff x) { return ff_rcp(x); }
    static __device__ __forceinline__ bool close(ff d) {
        return (__float_as_uint(d.hi) & 0x7fffffffu) < 0x3CA3D70Au;  // |d| < 0.02
    }
    static __device__ __forceinline__ ff log_(ff x) { return ff_log(x); }
    static __device__ __forceinline__ bool close_ratio(ff f) {
        return (__float_as_uint(f.hi) & 0x7fffffffu) < 0x3C23D70Au;  // |f| < 0.01
    }
};
// x > 0 (false for NaN), for the non-physical-state check.  FP64: a test of
// the high word on the integer pipe (1 <= hi <= 0x7fefffff), which also takes
// +infinity and the positive numbers below 2^-1042 (high word zero) as not
// positive -- neither is a physical density or pressure.
__device__ __forceinline__ bool positive(double x) {
    return static_cast<unsigned>(__double2hiint(x) - 1) < 0x7fefffffu;
}
__device__ __forceinline__ bool positive(float x) { return x > 0.0f; }
__device__ __forceinline__ bool positive(ff x) { return x.hi > 0.0f; }

template <typename C>
struct IsFF {
    static constexpr bool value = false;
};
template <>
struct IsFF<ff> {
    static constexpr bool value = true;
};

template <typename T>
__device__ __forceinline__ T shfl(T v, int src) {
    return __shfl_sync(0xffffffffu, v, src);
}
template <>
__device__ __forceinline__ ff shfl<ff>(ff v, int src) {
    return shfl_ff(v, src);
}

// Conversion between the I/O type T of the kernel's arguments and the type C
// its pair arithmetic runs in (the same type, or float-float for FP64 I/O).
template <typename T, typename C>
struct Conv {
    static __device__ __forceinline__ C in(T x) { return x; }
    static __device__ __forceinline__ T out(C x) { return x; }
};
template <>
struct Conv<double, ff> {
    static __device__ __forceinline__ ff in(double x) { return ff_split(x); }
    static __device__ __forceinline__ double out(ff x) { return ff_join(x); }
};

}  // namespace esdg
