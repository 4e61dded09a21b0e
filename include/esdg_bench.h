/*
 * esdg_bench.h -- measurement kernels shipped with the volume-term library.
 *
 * Not part of the volume term.  They give the denominators of the volume
 * kernel's roofline on the machine at hand: the FP64 and FP32 vector FMA
 * throughput.  The ESDG GPU paper ("GPU Performance of an Entropy-Stable
 * Discontinuous Galerkin Euler Solver with Non-Conservative Terms", Sec. 4.2,
 * Fig. 3) reports the volume kernel against the FP64 peak of its GPU; this
 * kernel measures that peak instead of quoting a data sheet.
 */
#ifndef ESDG_BENCH_H
#define ESDG_BENCH_H

#ifdef __cplusplus
extern "C" {
#endif

/* Launch `blocks` CTAs of `threads` threads; every thread runs `iters`
 * iterations of 8 independent fused multiply-adds (FP64 when fp64 != 0, FP32
 * otherwise).  The launch performs 16 * iters * blocks * threads floating-
 * point operations.  sink: device buffer of at least `blocks` elements of the
 * chosen type (written only to keep the work observable).  Asynchronous on
 * `stream`.  Returns 0, 1 (bad argument) or 4 (CUDA launch error). */
int esdg_bench_fma(int fp64, long blocks, int threads, int iters, void* sink, void* stream);

/* Self-test of the volume kernel's reciprocal: y[k] = 1/x[k] computed exactly
 * as the kernel computes it, so the test suite can measure its error against
 * correctly rounded division.  fp64 = 1: the FP64 per-node reciprocal
 * (hardware estimate plus one third-order Newton-Raphson step); 2: the FP64
 * pair reciprocal (an estimate from the FP32 reciprocal of the mantissa plus
 * one second-order step); 3: that estimate alone; 4: the FP64 reciprocal
 * square root of the surface flux (y[k] = 1/sqrt(x[k]), x > 0, built the same
 * way); 5: its estimate alone; 0: FP32 (the hardware estimate alone).
 * x, y: device arrays of n doubles (fp64 != 0) or floats.  Asynchronous on
 * `stream`.  Returns 0, 1 (bad argument) or 4 (CUDA launch error). */
int esdg_selftest_rcp(int fp64, long n, const void* x, void* y, void* stream);

/* Self-test of the float-float arithmetic of ESDG_FP64_FF: x[k] and y[k]
 * (doubles) are split into float-float, combined by operation `op`
 * (0: x + y, 1: x - y, 2: x * y, 3: x * y + x, 4: 1 / x, 5: log x for x > 0) in
 * float-float, and
 * the result is written back as a double to out[k], so the test suite can
 * compare it with FP64.  x, y, out: device arrays of n doubles (y unused for
 * ops 4 and 5).  Asynchronous on `stream`.  Returns 0, 1 (bad argument) or 4 (CUDA
 * launch error). */
int esdg_selftest_ff(int op, long n, const double* x, const double* y, double* out, void* stream);

/* Self-test of the FP64 volume kernel's per-node logarithm (the table-driven
 * reduction of Tang, ACM TOMS 16(4), 1990, used for ln rho and ln 2b):
 * y[k] = ln x[k] computed exactly as the kernel computes it, so the test
 * suite can measure its error in ulps against the host's log.  Meaningful
 * for positive normal x; other x give an unspecified value without a fault.
 * x, y: device arrays of n doubles.  Asynchronous on `stream`.  Returns 0,
 * 1 (bad argument) or 4 (CUDA launch error). */
int esdg_selftest_log(long n, const double* x, double* y, void* stream);

/* Host-only check of the kernels' index arithmetic for order N on a
 * Kx x Ky x Kz brick with per-direction boundary kinds bc[3] (0 periodic,
 * 1 slip wall): walks the same index functions the kernels use -- shared-
 * memory slots, the lines dealt to lanes (for every CTA fill and every
 * precision's launch shape), the FP64 load order, the antipodal pairs, the
 * fused kernel's face slots and neighbour traces, the face-centric surface
 * kernel's slots -- and checks that every index is in range, that the maps
 * meant to be bijections are, and that every node is visited exactly as
 * often as the kernels require.  No GPU needed.  msg (may be NULL) receives
 * the first failure.  Returns 0 (all hold), 1 (bad argument; at most 5e7
 * nodes) or 2 (a check failed). */
int esdg_selftest_index_maps(int N, long Kx, long Ky, long Kz, const int* bc, char* msg, int msglen);

#ifdef __cplusplus
}
#endif

#endif /* ESDG_BENCH_H */
