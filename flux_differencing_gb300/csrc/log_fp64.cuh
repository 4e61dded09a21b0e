// Natural logarithm of a positive normal double in 10 FP64-pipe operations
// (CUDA's log() takes 28 on sm_103a, counted with ncu), for the volume
// kernel's two per-node logarithms, whose only use is in differences
// ln a+ - ln a- of two nodes (the logarithmic means and their closeness test).
//
// Method: table-driven argument reduction, P. T. P. Tang, "Table-driven
// implementation of the logarithm function in IEEE floating-point
// arithmetic", ACM Trans. Math. Softw. 16(4), 1990.  Write x = 2^k m with
// m in [0.75, 1.5) and let F be the nearest point of a grid of spacing 1/512
// on [1, 1.5] (1/1024 on [0.75, 1]).  Then
//     ln x = k ln 2 + ln F + ln(1 + r),   r = (m - F)/F,   |r| <= 2^-10,
// where m - F is exact (Sterbenz's lemma: m and F are within a factor two),
// 1/F and ln F come from a 514-entry table (log_table.inc, 8 KB, written by
// gen_log_table.py from 50-digit arithmetic), and ln(1 + r) is its Taylor
// series to r^5 (the first dropped term, r^6/6, is below 2^-52 |r|).  The
// result is formed as k ln2 + (ln F + ln(1 + r)) with ln 2 and ln F each
// rounded once.
//
// Accuracy for the use made of it: the rounding of ln 2 (below 2^-55) is
// multiplied by k, the same k for both nodes of nearly every pair, so it
// cancels in the difference of two logarithms unless the two values straddle
// a power of two (then it contributes |k+ - k-| 2^-55); the rounding of ln F
// (below 2^-55) and of the inner sum (half an ulp of a number below 0.41)
// are far below the final rounding, half an ulp of the result.  So a
// difference of two of these logarithms is within one ulp of the larger
// result (plus |k+ - k-| 2^-55) of the exact ln(a+/a-), as for correctly
// rounded logarithms; the absolute value carries up to |k| 2^-55 more.
//
// The reduction to [0.75, 1.5) rather than [1, 2) keeps every x near 1 on
// the k = 0 branch, with F = 1 and r = x - 1 exactly when |x - 1| < 2^-11:
// the result keeps its relative accuracy near 1.  Exponent and mantissa are
// taken apart on the integer pipe.  Inputs that are not positive normal
// numbers give a meaningless value without faulting (the table index is
// always in range); the kernel flags such non-physical states separately.
#pragma once

#include <cuda_runtime.h>

namespace esdg {

#include "log_table.inc"

__device__ __forceinline__ double log_fp64(double x) {
    const int hi = __double2hiint(x);
    const int lo = __double2loint(x);
    const int mant = hi & 0x000fffff;                 // top 20 mantissa bits
    const int half = mant >= 0x80000 ? 1 : 0;         // m >= 1.5: reduce m/2, k + 1
    const int j = (mant + 0x400) >> 11;               // nearest of 0..512 (units of 1/512)
    const int ebits = 0x3ff00000 - (half << 20);      // exponent field of m or m/2
    const double m = __hiloint2double(ebits | mant, lo);
    const double F = __hiloint2double(ebits + (j << 11), 0);  // j = 512, halved: exactly 1
    const double2 t = __ldg(&kLogTable[j + half]);    // (1/F, ln F rounded)
    const int k = ((hi >> 20) & 0x7ff) - 1023 + half;
    // (double)k without a conversion instruction: 2^52 + (k + 1024) has k + 1024
    // in its low mantissa word
    const double kd = __hiloint2double(0x43300000, k + 1024) - 4503599627371520.0;
    const double r = (m - F) * t.x;
    const double r2 = r * r;
    // ln(1 + r) = r + r^2 (-1/2 + r/3 - r^2/4 + r^3/5)
    double q = fma(r, 1.0 / 5.0, -0.25);
    q = fma(q, r, 1.0 / 3.0);
    q = fma(q, r, -0.5);
    const double p = fma(r2, q, r);
    return fma(kd, kLn2, t.y + p);
}

}  // namespace esdg
