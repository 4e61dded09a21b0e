// One instantiation of the volume kernel.  The build compiles this file once
// per (order, precision) with -DESDG_INST_N=<1..8> and -DESDG_INST_PREC=<0|1|2>
// (0: FP64, 1: FP32, 2: FP64 I/O with float-float pair arithmetic), so the
// instantiations compile in parallel.
#include "volume_kernel.cuh"

#ifndef ESDG_INST_N
#error "ESDG_INST_N must be defined"
#endif
#ifndef ESDG_INST_PREC
#error "ESDG_INST_PREC must be defined"
#endif

#define ESDG_CAT_(a, b) a##b
#define ESDG_CAT(a, b) ESDG_CAT_(a, b)

namespace esdg {

#if ESDG_INST_PREC == 0
cudaError_t ESDG_CAT(launch_volume_fp64_n, ESDG_INST_N)(const VolumeArgs<double>& a, cudaStream_t s) {
    return launch_volume<double, ESDG_INST_N>(a, s);
}
#elif ESDG_INST_PREC == 1
cudaError_t ESDG_CAT(launch_volume_fp32_n, ESDG_INST_N)(const VolumeArgs<float>& a, cudaStream_t s) {
    return launch_volume<float, ESDG_INST_N>(a, s);
}
#else
cudaError_t ESDG_CAT(launch_volume_fp64ff_n, ESDG_INST_N)(const VolumeArgs<double>& a, cudaStream_t s) {
    return launch_volume<double, ESDG_INST_N, ff>(a, s);
}
#endif

}  // namespace esdg
