// esdg_volume_rhs_noalloc: the volume term for callers that cannot allocate
// device memory.
//
// The handle-based path (esdg_create) allocates one device word per handle
// with cudaMalloc for the kernel's status flags.  Some callers cannot do
// that: applications that hand every byte of device memory to their own pool
// and forbid other allocations, or code that must not call cudaMalloc on a
// busy device because it can synchronise with work on other streams.  This
// entry point needs no handle and allocates nothing: the kernel's status word
// lives in the file-scope array below, which the CUDA runtime places in
// device memory when the library is loaded on a device and keeps there until
// the process exits.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>
#include <string>

#include "esdg.h"
#include "esdg_internal.h"

namespace {

// 64 words (256 bytes): word 0 is the status word of the volume kernel; the
// rest is reserved.  Shared by every call on a device.
constexpr int kScratchWords = 64;
static __device__ __align__(256) unsigned g_noalloc_scratch[kScratchWords];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
// Device address of g_noalloc_scratch per device, with the identifier of the
// context it was looked up in.  A context that is destroyed and created
// again (cudaDeviceReset, or a driver-API caller replacing its context)
// reloads the module, and the array can then sit at another address: the
// identifier shows that, and the address is looked up again.
struct ScratchAddr {
    unsigned long long ctx_id;
    unsigned* addr;
};
ScratchAddr g_scratch[kMaxDevices] = {};

int noalloc_fail(int code, const std::string& msg) {
    esdg::set_unhandled_error(msg);  // reported by esdg_last_error(NULL)
    return code;
}

// The current context's process-unique identifier, through the driver's
// cuCtxGetCurrent and cuCtxGetId (resolved once through the runtime, so the
// library does not link the driver library itself).  False when either is
// unavailable or no context is current yet.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
CtxGetCurrentFn g_ctx_current = nullptr;
CtxGetIdFn g_ctx_id = nullptr;
std::once_flag g_resolve_once;

bool current_context_id(unsigned long long* id) {
    std::call_once(g_resolve_once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult r;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &r) == cudaSuccess &&
            r == cudaDriverEntryPointSuccess)
            g_ctx_current = reinterpret_cast<CtxGetCurrentFn>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &r) == cudaSuccess &&
            r == cudaDriverEntryPointSuccess)
            g_ctx_id = reinterpret_cast<CtxGetIdFn>(f);
    });
    if (!g_ctx_current || !g_ctx_id) return false;
    CUcontext ctx = nullptr;
    if (g_ctx_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
    return g_ctx_id(ctx, id) == CUDA_SUCCESS;
}

// Host code must not pass &g_noalloc_scratch to a kernel: on the host that
// name is only a stand-in.  The real device address is looked up with the
// device current: on the first call on a device (which also loads the module
// there, so that first call should come before any stream capture), and again
// whenever the device's context has changed since.
cudaError_t scratch_address(int dev, unsigned** out) {
    std::lock_guard<std::mutex> lock(g_mutex);
    unsigned long long id = 0;
    const bool have_id = current_context_id(&id);
    if (have_id && g_scratch[dev].addr && g_scratch[dev].ctx_id == id) {
        *out = g_scratch[dev].addr;
        return cudaSuccess;
    }
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    // the lookup above makes the primary context current if none was: take
    // its identifier now; without one the address is looked up every call
    unsigned long long id_after = 0;
    if (current_context_id(&id_after)) {
        g_scratch[dev].ctx_id = id_after;
        g_scratch[dev].addr = static_cast<unsigned*>(p);
    } else {
        g_scratch[dev].addr = nullptr;
    }
    *out = static_cast<unsigned*>(p);
    return cudaSuccess;
}

template <typename T>
cudaError_t launch_noalloc(long K, int N, int form, double gamma, const void* q, const void* Ja, const void* phi,
                           void* out, unsigned* status, cudaStream_t s) {
    esdg::VolumeArgs<T> a{};  // value-initialised: the fused-stage fields stay null
    a.q = static_cast<const T*>(q);
    a.Ja = static_cast<const T*>(Ja);
    a.phi = static_cast<const T*>(phi);
    a.out = static_cast<T*>(out);
    a.n = (long long)K * (N + 1) * (N + 1) * (N + 1);
    a.e_begin = 0;
    a.e_end = K;
    a.gm1 = (T)(gamma - 1.0);
    a.c_g = (T)(1.0 / (2.0 * (gamma - 1.0)));
    a.c_h = (T)(gamma / (2.0 * (gamma - 1.0)));
    a.form = form;
    a.status = status;
    a.rho_ref = nullptr;  // full-state variables
    a.p_ref = nullptr;
    a.rk_q = nullptr;  // writes out
    a.rk_dq = nullptr;
    a.rk_S = nullptr;
    a.rk_J = nullptr;
    a.rk_A = a.rk_B = a.rk_dt = a.rk_f = T(0);
    esdg::fill_op_tables(a.ops, N);
    if constexpr (sizeof(T) == sizeof(double)) {
        switch (N) {
            case 1: return esdg::launch_volume_fp64_n1(a, s);
            case 2: return esdg::launch_volume_fp64_n2(a, s);
            case 3: return esdg::launch_volume_fp64_n3(a, s);
            case 4: return esdg::launch_volume_fp64_n4(a, s);
            case 5: return esdg::launch_volume_fp64_n5(a, s);
            case 6: return esdg::launch_volume_fp64_n6(a, s);
            case 7: return esdg::launch_volume_fp64_n7(a, s);
            case 8: return esdg::launch_volume_fp64_n8(a, s);
        }
    } else {
        switch (N) {
            case 1: return esdg::launch_volume_fp32_n1(a, s);
            case 2: return esdg::launch_volume_fp32_n2(a, s);
            case 3: return esdg::launch_volume_fp32_n3(a, s);
            case 4: return esdg::launch_volume_fp32_n4(a, s);
            case 5: return esdg::launch_volume_fp32_n5(a, s);
            case 6: return esdg::launch_volume_fp32_n6(a, s);
            case 7: return esdg::launch_volume_fp32_n7(a, s);
            case 8: return esdg::launch_volume_fp32_n8(a, s);
        }
    }
    return cudaErrorInvalidValue;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void* a, size_t an, const void* b, size_t bn) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + bn && b0 < a0 + an;
}

}  // namespace

extern "C" int esdg_volume_rhs_noalloc(long K, int N, int precision, int form, double gamma, const void* q,
                                       const void* metrics, const void* phi, void* out, unsigned* status_out,
                                       void* stream) {
    if (N < 1 || N > esdg::kMaxN) return noalloc_fail(ESDG_ERR_UNSUPPORTED, "N must be in 1..8");
    if (precision != ESDG_FP64 && precision != ESDG_FP32)
        return noalloc_fail(ESDG_ERR_UNSUPPORTED, "precision must be ESDG_FP64 or ESDG_FP32");
    if (form != ESDG_FORM_2D && form != ESDG_FORM_SKEW)
        return noalloc_fail(ESDG_ERR_UNSUPPORTED, "form must be ESDG_FORM_2D or ESDG_FORM_SKEW");
    if (!(gamma > 1.0 && gamma < 10.0)) return noalloc_fail(ESDG_ERR_ARG, "gamma must be in (1, 10)");
    if (K < 1) return noalloc_fail(ESDG_ERR_ARG, "K must be >= 1");
    // Largest mesh one call accepts: 2^31 - 1 elements (one grid launch) and
    // 2^40 nodes.  The scratch itself does not grow with the mesh.
    const long double nodes = (long double)K * (N + 1) * (N + 1) * (N + 1);
    if (K > 2147483647L || nodes > (long double)(1LL << 40))
        return noalloc_fail(ESDG_ERR_ARG, "mesh too large for one call: at most 2^31-1 elements and 2^40 nodes");
    if (!q || !metrics || !phi || !out) return noalloc_fail(ESDG_ERR_ARG, "null device pointer");
    if (!aligned16(q) || !aligned16(metrics) || !aligned16(phi) || !aligned16(out))
        return noalloc_fail(ESDG_ERR_ALIGN, "device pointers must be 16-byte aligned");
    const size_t nb = (precision == ESDG_FP64 ? sizeof(double) : sizeof(float)) * (size_t)nodes;
    if (overlaps(out, 5 * nb, q, 5 * nb) || overlaps(out, 5 * nb, metrics, 9 * nb) || overlaps(out, 5 * nb, phi, nb))
        return noalloc_fail(ESDG_ERR_ARG, "out overlaps an input");

    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return noalloc_fail(ESDG_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return noalloc_fail(ESDG_ERR_UNSUPPORTED, "device index out of range");
    unsigned* status = nullptr;
    e = scratch_address(dev, &status);
    if (e != cudaSuccess)
        return noalloc_fail(ESDG_ERR_CUDA, std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(e));

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the status word keeps the previous call's bits: clear it first
    e = cudaMemsetAsync(status, 0, sizeof(unsigned), s);
    if (e == cudaSuccess)
        e = precision == ESDG_FP64 ? launch_noalloc<double>(K, N, form, gamma, q, metrics, phi, out, status, s)
                                   : launch_noalloc<float>(K, N, form, gamma, q, metrics, phi, out, status, s);
    if (e != cudaSuccess) return noalloc_fail(ESDG_ERR_CUDA, std::string("volume kernel launch: ") + cudaGetErrorString(e));
    if (status_out) {
        e = cudaMemcpyAsync(status_out, status, sizeof(unsigned), cudaMemcpyDeviceToHost, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
        if (e != cudaSuccess) return noalloc_fail(ESDG_ERR_CUDA, std::string("reading the status word: ") + cudaGetErrorString(e));
    }
    return ESDG_OK;
}
