// FMA-throughput kernels for the roofline denominators (see esdg_bench.h).
#include <cuda_runtime.h>

#include "esdg_bench.h"

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
