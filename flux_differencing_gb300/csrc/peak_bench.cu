// FMA-throughput kernels for the roofline denominators (see esdg_bench.h).
#include <cuda_runtime.h>

#include "esdg_bench.h"
#include "volume_kernel.cuh"

namespace {

template <typename T>
__global__ void fma_throughput(T* sink, int iters, T a, T b) {
    constexpr int CH = 8;
    T x[CH];
#pragma unroll
    for (int c = 0; c < CH; ++c) x[c] = T(threadIdx.x) * T(1e-3) + T(c);
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int c = 0; c < CH; ++c) x[c] = fma(x[c], a, b);
    }
    T s = T(0);
#pragma unroll
    for (int c = 0; c < CH; ++c) s += x[c];
    // practically never true; keeps the chains observable
    if (s == T(-1.25)) sink[blockIdx.x] = s;
}

}  // namespace

extern "C" int esdg_bench_fma(int fp64, long blocks, int threads, int iters, void* sink, void* stream) {
    if (blocks < 1 || threads < 32 || threads > 1024 || iters < 1 || !sink) return 1;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (fp64)
        fma_throughput<double><<<(unsigned)blocks, threads, 0, s>>>(static_cast<double*>(sink), iters, 0.9999999,
                                                                      1e-7);
    else
        fma_throughput<float><<<(unsigned)blocks, threads, 0, s>>>(static_cast<float*>(sink), iters, 0.9999f,
                                                                     1e-4f);
    return cudaGetLastError() == cudaSuccess ? 0 : 4;
}

namespace {
template <typename T>
__global__ void rcp_selftest(const T* __restrict__ x, T* __restrict__ y, long n) {
    const long k = (long)blockIdx.x * blockDim.x + threadIdx.x;
    if (k < n) y[k] = esdg::Num<T>::rcp(x[k]);
}
// mode 2: the pair reciprocal; 3: its estimate; 4: the reciprocal square
// root of the surface flux; 5: its estimate
__global__ void rcp_selftest_fp64_variant(int mode, const double* __restrict__ x, double* __restrict__ y, long n) {
    const long k = (long)blockIdx.x * blockDim.x + threadIdx.x;
    if (k >= n) return;
    using D = esdg::Num<double>;
    y[k] = mode == 2 ? D::rcp_pair(x[k]) : mode == 3 ? D::rcp_estimate(x[k])
         : mode == 4 ? D::rsqrt_pair(x[k]) : D::rsqrt_estimate(x[k]);
}
}  // namespace

extern "C" int esdg_selftest_rcp(int fp64, long n, const void* x, void* y, void* stream) {
    if (n < 1 || !x || !y || fp64 < 0 || fp64 > 5) return 1;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const unsigned blocks = (unsigned)((n + 255) / 256);
    if (fp64 >= 2)
        rcp_selftest_fp64_variant<<<blocks, 256, 0, s>>>(fp64, static_cast<const double*>(x), static_cast<double*>(y),
                                                          n);
    else if (fp64)
        rcp_selftest<double><<<blocks, 256, 0, s>>>(static_cast<const double*>(x), static_cast<double*>(y), n);
    else
        rcp_selftest<float><<<blocks, 256, 0, s>>>(static_cast<const float*>(x), static_cast<float*>(y), n);
    return cudaGetLastError() == cudaSuccess ? 0 : 4;
}

namespace {
__global__ void ff_selftest(int op, const double* __restrict__ x, const double* __restrict__ y,
                            double* __restrict__ out, long n) {
    const long k = (long)blockIdx.x * blockDim.x + threadIdx.x;
    if (k >= n) return;
    const esdg::ff a = esdg::ff_split(x[k]);
    const esdg::ff b = esdg::ff_split(y[k]);
    esdg::ff r;
    switch (op) {
        case 0: r = a + b; break;
        case 1: r = a - b; break;
        case 2: r = a * b; break;
        case 3: r = esdg::fma(a, b, a); break;
        case 4: r = esdg::ff_rcp(a); break;
        default: r = esdg::ff_log(a); break;
    }
    out[k] = esdg::ff_join(r);
}
}  // namespace

extern "C" int esdg_selftest_ff(int op, long n, const double* x, const double* y, double* out, void* stream) {
    if (n < 1 || op < 0 || op > 5 || !x || !y || !out) return 1;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    ff_selftest<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(op, x, y, out, n);
    return cudaGetLastError() == cudaSuccess ? 0 : 4;
}

namespace {
__global__ void log_selftest(const double* __restrict__ x, double* __restrict__ y, long n) {
    const long k = (long)blockIdx.x * blockDim.x + threadIdx.x;
    if (k < n) y[k] = esdg::Num<double>::log_(x[k]);
}
}  // namespace

extern "C" int esdg_selftest_log(long n, const double* x, double* y, void* stream) {
    if (n < 1 || !x || !y) return 1;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    log_selftest<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(x, y, n);
    return cudaGetLastError() == cudaSuccess ? 0 : 4;
}
