// Pipelined host-buffer executor for the volume term (include/esdg.h,
// esdg_pipeline_*).
//
// A caller that holds its state in host memory pays, per evaluation, the
// host-to-device copy of q, the metric terms and phi, the kernel, and the copy
// of the result back.  Done one after another these serialise; here each
// submission goes to the next of `depth` slots, each slot owning device
// buffers and a stream, so the copies of one submission run on the copy
// engines while another submission's kernel runs.  Every submission still
// moves all of its bytes; only the waiting is removed.
//
// Ordering: submissions on one slot are ordered by the slot's stream; a
// submission's output is in the host buffer once esdg_pipeline_wait returns
// (or the slot comes round again and its event has completed).  The handle is
// shared by all slots (its kernels are enqueued on the slot streams).
#include <cuda_runtime.h>

#include <cstring>
#include <string>

#include "esdg.h"
#include "esdg_internal.h"

struct esdg_pipeline_s {
    esdg_handle h = nullptr;
    int depth = 0;
    int next = 0;
    size_t es = 0;
    long long n = 0;
    struct Slot {
        void* q = nullptr;
        void* Ja = nullptr;
        void* phi = nullptr;
        void* out = nullptr;
        cudaStream_t stream = nullptr;
        cudaEvent_t done = nullptr;
        bool used = false;
    } slot[ESDG_PIPELINE_MAX_DEPTH];
    std::string err;
};

namespace {

void release(esdg_pipeline_s* p) {
    for (int k = 0; k < ESDG_PIPELINE_MAX_DEPTH; ++k) {
        auto& s = p->slot[k];
        if (s.stream) cudaStreamSynchronize(s.stream);
        if (s.q) cudaFree(s.q);
        if (s.Ja) cudaFree(s.Ja);
        if (s.phi) cudaFree(s.phi);
        if (s.out) cudaFree(s.out);
        if (s.done) cudaEventDestroy(s.done);
        if (s.stream) cudaStreamDestroy(s.stream);
        s = esdg_pipeline_s::Slot();
    }
}

int pfail(esdg_pipeline_s* p, int code, const std::string& msg) {
    if (p) p->err = msg;
    else esdg::set_unhandled_error(msg);
    return code;
}

}  // namespace

extern "C" {

int esdg_pipeline_create(esdg_handle h, int depth, esdg_pipeline* out) {
    if (!out) return pfail(nullptr, ESDG_ERR_ARG, "out is NULL");
    *out = nullptr;
    if (!h) return pfail(nullptr, ESDG_ERR_ARG, "null handle");
    if (depth < 1 || depth > ESDG_PIPELINE_MAX_DEPTH)
        return pfail(nullptr, ESDG_ERR_ARG, "depth must be in 1..ESDG_PIPELINE_MAX_DEPTH");
    int prec = 0, N = 0;
    long long n = 0;
    esdg_describe(h, &prec, &N, &n);
    auto* p = new esdg_pipeline_s();
    p->h = h;
    p->depth = depth;
    p->es = prec == ESDG_FP32 ? sizeof(float) : sizeof(double);
    p->n = n;
    const size_t nb = p->es * (size_t)n;
    cudaError_t e = cudaSuccess;
    for (int k = 0; k < depth && e == cudaSuccess; ++k) {
        auto& s = p->slot[k];
        e = cudaMalloc(&s.q, 5 * nb);
        if (e == cudaSuccess) e = cudaMalloc(&s.Ja, 9 * nb);
        if (e == cudaSuccess) e = cudaMalloc(&s.phi, nb);
        if (e == cudaSuccess) e = cudaMalloc(&s.out, 5 * nb);
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&s.stream, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s.done, cudaEventDisableTiming);
    }
    if (e != cudaSuccess) {
        const std::string msg = std::string("pipeline buffers: ") + cudaGetErrorString(e);
        release(p);
        delete p;
        return pfail(nullptr, ESDG_ERR_CUDA, msg);
    }
    *out = p;
    return ESDG_OK;
}

int esdg_pipeline_submit(esdg_pipeline p, const void* q_host, const void* metrics_host, const void* phi_host,
                         void* out_host) {
    if (!p) return pfail(nullptr, ESDG_ERR_ARG, "null pipeline");
    if (!q_host || !metrics_host || !phi_host || !out_host) return pfail(p, ESDG_ERR_ARG, "null host pointer");
    auto& s = p->slot[p->next];
    const size_t nb = p->es * (size_t)p->n;
    cudaError_t e = cudaMemcpyAsync(s.q, q_host, 5 * nb, cudaMemcpyHostToDevice, s.stream);
    if (e == cudaSuccess) e = cudaMemcpyAsync(s.Ja, metrics_host, 9 * nb, cudaMemcpyHostToDevice, s.stream);
    if (e == cudaSuccess) e = cudaMemcpyAsync(s.phi, phi_host, nb, cudaMemcpyHostToDevice, s.stream);
    if (e != cudaSuccess) return pfail(p, ESDG_ERR_CUDA, std::string("host-to-device copy: ") + cudaGetErrorString(e));
    if (int rc = esdg_volume_rhs(p->h, s.q, s.Ja, s.phi, s.out, s.stream))
        return pfail(p, rc, std::string("volume term: ") + esdg_last_error(p->h));
    e = cudaMemcpyAsync(out_host, s.out, 5 * nb, cudaMemcpyDeviceToHost, s.stream);
    if (e == cudaSuccess) e = cudaEventRecord(s.done, s.stream);
    if (e != cudaSuccess) return pfail(p, ESDG_ERR_CUDA, std::string("device-to-host copy: ") + cudaGetErrorString(e));
    s.used = true;
    p->next = (p->next + 1) % p->depth;
    return ESDG_OK;
}

int esdg_pipeline_wait(esdg_pipeline p) {
    if (!p) return pfail(nullptr, ESDG_ERR_ARG, "null pipeline");
    for (int k = 0; k < p->depth; ++k) {
        if (!p->slot[k].used) continue;
        const cudaError_t e = cudaEventSynchronize(p->slot[k].done);
        if (e != cudaSuccess) return pfail(p, ESDG_ERR_CUDA, std::string("pipeline wait: ") + cudaGetErrorString(e));
    }
    return ESDG_OK;
}

const char* esdg_pipeline_last_error(esdg_pipeline p) { return p ? p->err.c_str() : ""; }

int esdg_pipeline_destroy(esdg_pipeline p) {
    if (!p) return ESDG_OK;
    release(p);
    delete p;
    return ESDG_OK;
}

}  // extern "C"
