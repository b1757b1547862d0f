// gdn_api.cu -- the exported C ABI: argument checks, the device status word,
// and dispatch to the kernels. Every check runs before any device work is
// queued; a failed check returns its gdn_status and touches nothing.
#include <stdint.h>

#include <cstdlib>
#include <cstring>
#include <mutex>

#include <cuda_runtime.h>

#include "gdn.h"
#include "gdn_internal.h"

namespace {

// Device-side consistency flag, one per device (a __device__ variable has one
// instance per device context). Kernels set it with atomicExch; the host reads
// and clears it in gdn_get_device_status.
__device__ int g_device_status = 0;
__device__ int g_status_taken = 0;  // where the read-and-clear kernel leaves the old value

// Read and clear the status word in one atomic step, so a flag raised by a kernel on another
// stream between a read and a separate clear cannot be lost.
__global__ void take_status_kernel(int *status, int *taken) { *taken = atomicExch(status, 0); }

constexpr int kMaxDevices = 64;
int *g_status_ptr[kMaxDevices] = {nullptr};
int *g_taken_ptr[kMaxDevices] = {nullptr};

std::mutex g_status_mu;  // first use on a device may come from several host threads

int *status_ptr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_status_mu);
    if (!g_status_ptr[dev]) {
        void *p = nullptr, *t = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
        if (cudaGetSymbolAddress(&t, g_status_taken) != cudaSuccess) return nullptr;
        g_taken_ptr[dev] = static_cast<int *>(t);
        g_status_ptr[dev] = static_cast<int *>(p);
    }
    return g_status_ptr[dev];
}

int *taken_ptr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    if (!status_ptr()) return nullptr;
    std::lock_guard<std::mutex> lock(g_status_mu);
    return g_taken_ptr[dev];
}

// gdn_prefill's own workspace for the kernels that need one: one per device, allocated on the
// first call that needs it (and grown when a call needs more). Calls on different streams are
// ordered on the GPU through an event, so they never use it at the same time; inside a stream
// capture the workspace must already be large enough (no allocation, no cross-stream wait).
struct DeviceWorkspace {
    std::mutex mu;
    void *ptr = nullptr;
    size_t bytes = 0;
    cudaEvent_t last = nullptr;   // recorded after the last call that used the workspace
    cudaStream_t last_stream = nullptr;
    bool used = false;
};
DeviceWorkspace g_ws[kMaxDevices];

bool stream_capturing(cudaStream_t s) {
    cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &st) != cudaSuccess) return true;
    return st != cudaStreamCaptureStatusNone;
}

bool force_cluster_kernel() {
    const char *env = getenv("GDN_PREFILL_KERNEL");
    return env && strcmp(env, "cluster") == 0;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool dim_ok(int d) { return d == 32 || d == 64 || d == 128; }
bool chunk_ok(int c) { return c == 16 || c == 32 || c == 64; }

int common_checks(int Hk, int Hv, int dk, int dv, int dtype) {
    if (Hk <= 0 || Hv <= 0 || Hv % Hk != 0 || Hv > 65535) return GDN_ERR_INVALID_ARG;
    if (dtype != GDN_BF16 && dtype != GDN_F32) return GDN_ERR_UNSUPPORTED;
    if (!dim_ok(dk) || !dim_ok(dv)) return GDN_ERR_UNSUPPORTED;
    return GDN_OK;
}

int prefill_checks(const void *q, const void *k, const void *v, const void *g, const void *b,
                   const float *state_in, const float *state_out, const void *out,
                   const int32_t *cu, int B, int T, int Hk, int Hv, int dk, int dv, int chunk,
                   int dtype) {
    if (B < 0 || T < 0 || B > 65535) return GDN_ERR_INVALID_ARG;
    int rc = common_checks(Hk, Hv, dk, dv, dtype);
    if (rc != GDN_OK) return rc;
    if (!chunk_ok(chunk)) return GDN_ERR_UNSUPPORTED;
    if (B == 0) return GDN_OK;
    const long long Ttot = cu ? (long long)T : (long long)B * T;
    if (Ttot > 0x7fffffffLL) return GDN_ERR_INVALID_ARG;
    if (!state_out) return GDN_ERR_INVALID_ARG;
    if (Ttot > 0 && (!q || !k || !v || !g || !b || !out)) return GDN_ERR_INVALID_ARG;
    const void *ptrs[] = {q, k, v, g, b, state_in, state_out, out, cu};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return GDN_ERR_INVALID_ARG;
    return GDN_OK;
}

}  // namespace

extern "C" {

const char *gdn_status_string(int status) {
    switch (status) {
        case GDN_OK: return "GDN_OK";
        case GDN_ERR_INVALID_ARG: return "GDN_ERR_INVALID_ARG";
        case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED";
        case GDN_ERR_CUDA: return "GDN_ERR_CUDA";
        case GDN_ERR_DEVICE_CHECK: return "GDN_ERR_DEVICE_CHECK";
    }
    return "GDN_UNKNOWN_STATUS";
}

int gdn_prefill_path(int B, int T, int Hk, int Hv, int dk, int dv, int chunk, int dtype) {
    // a dummy aligned address stands in for every pointer: only sizes are checked
    static __align__(16) char dummy[16];
    const void *p = dummy;
    int rc = prefill_checks(p, p, p, p, p, nullptr, (const float *)p, p, nullptr, B, T, Hk, Hv, dk,
                            dv, chunk, dtype);
    if (rc != GDN_OK) return rc;
    gdn::PrefillArgs a{};
    a.B = B; a.T = T; a.Hk = Hk; a.Hv = Hv; a.dk = dk; a.dv = dv; a.chunk = chunk; a.dtype = dtype;
    if (gdn::prefill_scan_supported(a)) return 2;
    return gdn::prefill_tc_supported(a) || gdn::prefill_ring_supported(a) ? 1 : 0;
}

// Workspace the tensor-core kernel needs for these sizes, whether or not cu_seqlens is given
// (with cu_seqlens NULL and T <= 8 the token scan runs instead and uses none of it).
size_t gdn_prefill_workspace_size(int B, int T, int Hk, int Hv, int dk, int dv, int chunk, int dtype) {
    static __align__(16) char dummy[16];
    const void *p = dummy;
    if (prefill_checks(p, p, p, p, p, nullptr, (const float *)p, p, nullptr, B, T, Hk, Hv, dk, dv, chunk,
                       dtype) != GDN_OK || B == 0)
        return 0;
    gdn::PrefillArgs a{};
    a.B = B; a.T = T; a.Hk = Hk; a.Hv = Hv; a.dk = dk; a.dv = dv; a.chunk = chunk; a.dtype = dtype;
    if (!gdn::prefill_ring_supported(a)) return 0;
    return gdn::prefill_ring_workspace(a);
}

int gdn_prefill_ws(const void *q, const void *k, const void *v, const void *g, const void *b,
                   const float *state_in, float *state_out, void *out, const int32_t *cu_seqlens,
                   int B, int T, int Hk, int Hv, int dk, int dv, int chunk, int dtype, void *workspace,
                   size_t workspace_bytes, void *stream) {
    int rc = prefill_checks(q, k, v, g, b, state_in, state_out, out, cu_seqlens, B, T, Hk, Hv, dk,
                            dv, chunk, dtype);
    if (rc != GDN_OK) return rc;
    if (B == 0) return GDN_OK;
    int *status = status_ptr();
    if (!status) return GDN_ERR_CUDA;
    gdn::PrefillArgs a{q, k, v, g, b, state_in, state_out, out, cu_seqlens,
                       B, T, Hk, Hv, dk, dv, chunk, dtype, status};
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (gdn::prefill_scan_supported(a)) {
        e = gdn::launch_prefill_scan(a, s);
    } else if (gdn::prefill_ring_supported(a) && !force_cluster_kernel()) {
        const size_t need = gdn::prefill_ring_workspace(a);
        if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
            return GDN_ERR_INVALID_ARG;
        e = gdn::launch_prefill_ring(a, workspace, workspace_bytes, s);
    } else {
        e = gdn::prefill_tc_supported(a) ? gdn::launch_prefill_tc(a, s) : gdn::launch_prefill_simt(a, s);
    }
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

int gdn_prefill_static(const void *q, const void *k, const void *v, const void *g, const void *b,
                       const float *state_in, float *state_out, void *out, const int32_t *cu_seqlens,
                       int B, int T, int Hk, int Hv, int dk, int dv, int chunk, int dtype, void *stream) {
    int rc = prefill_checks(q, k, v, g, b, state_in, state_out, out, cu_seqlens, B, T, Hk, Hv, dk,
                            dv, chunk, dtype);
    if (rc != GDN_OK) return rc;
    if (B == 0) return GDN_OK;
    gdn::PrefillArgs a{q, k, v, g, b, state_in, state_out, out, cu_seqlens, B, T, Hk, Hv, dk, dv, chunk, dtype,
                       nullptr};
    // sizes whose kernels take no scratch: the same kernels as gdn_prefill, nothing allocated
    if (gdn::prefill_scan_supported(a) || !gdn::prefill_ring_supported(a))
        return gdn_prefill_ws(q, k, v, g, b, state_in, state_out, out, cu_seqlens, B, T, Hk, Hv, dk, dv, chunk,
                              dtype, nullptr, 0, stream);
    const size_t need = gdn::prefill_ring_workspace(a, gdn::kStaticChainCtas);
    if (need == 0 || need > gdn::kStaticScratchBytes) return GDN_ERR_UNSUPPORTED;
    void *scratch = gdn::static_scratch();
    a.status = status_ptr();
    if (!scratch || !a.status) return GDN_ERR_CUDA;
    const cudaError_t e = gdn::launch_prefill_ring(a, scratch, gdn::kStaticScratchBytes,
                                                   static_cast<cudaStream_t>(stream), gdn::kStaticChainCtas);
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

int gdn_prefill(const void *q, const void *k, const void *v, const void *g, const void *b,
                const float *state_in, float *state_out, void *out, const int32_t *cu_seqlens,
                int B, int T, int Hk, int Hv, int dk, int dv, int chunk, int dtype, void *stream) {
    int rc = prefill_checks(q, k, v, g, b, state_in, state_out, out, cu_seqlens, B, T, Hk, Hv, dk,
                            dv, chunk, dtype);
    if (rc != GDN_OK) return rc;
    if (B == 0) return GDN_OK;
    gdn::PrefillArgs probe{q, k, v, g, b, state_in, state_out, out, cu_seqlens, B, T, Hk, Hv, dk, dv, chunk, dtype,
                           nullptr};
    const bool ring = !force_cluster_kernel() && !gdn::prefill_scan_supported(probe) && gdn::prefill_ring_supported(probe);
    const size_t need = ring ? gdn::prefill_ring_workspace(probe) : 0;
    if (need == 0)
        return gdn_prefill_ws(q, k, v, g, b, state_in, state_out, out, cu_seqlens, B, T, Hk, Hv, dk, dv, chunk,
                              dtype, nullptr, 0, stream);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDN_ERR_CUDA;
    DeviceWorkspace &w = g_ws[dev];
    std::lock_guard<std::mutex> lock(w.mu);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool capturing = stream_capturing(s);
    if (w.bytes < need) {
        if (capturing) return GDN_ERR_CUDA;  // first use (or growth) must happen outside a capture
        if (w.ptr) {  // the old buffer may still be in use by queued work
            if (w.used && cudaEventSynchronize(w.last) != cudaSuccess) return GDN_ERR_CUDA;
            cudaFree(w.ptr);
            w.ptr = nullptr;
            w.bytes = 0;
        }
        const size_t bytes = (need + (1u << 20) - 1) & ~(size_t)((1u << 20) - 1);
        if (cudaMalloc(&w.ptr, bytes) != cudaSuccess) return GDN_ERR_CUDA;
        w.bytes = bytes;
        if (!w.last && cudaEventCreateWithFlags(&w.last, cudaEventDisableTiming) != cudaSuccess) return GDN_ERR_CUDA;
    }
    if (w.used && !capturing && w.last_stream != s && cudaStreamWaitEvent(s, w.last, 0) != cudaSuccess)
        return GDN_ERR_CUDA;
    rc = gdn_prefill_ws(q, k, v, g, b, state_in, state_out, out, cu_seqlens, B, T, Hk, Hv, dk, dv, chunk, dtype,
                        w.ptr, w.bytes, stream);
    if (rc == GDN_OK && !capturing) {
        if (cudaEventRecord(w.last, s) != cudaSuccess) return GDN_ERR_CUDA;
        w.last_stream = s;
        w.used = true;
    }
    return rc;
}

int gdn_decode_step(const void *q, const void *k, const void *v, const void *g, const void *b,
                    float *state, void *out, int N, int Hk, int Hv, int dk, int dv, int dtype,
                    void *stream) {
    if (N < 0) return GDN_ERR_INVALID_ARG;
    int rc = common_checks(Hk, Hv, dk, dv, dtype);
    if (rc != GDN_OK) return rc;
    if (N == 0) return GDN_OK;
    if ((long long)N * Hv * dv * dk > (1LL << 40)) return GDN_ERR_INVALID_ARG;
    const void *ptrs[] = {q, k, v, g, b, state, out};
    for (const void *p : ptrs)
        if (!p || !aligned16(p)) return GDN_ERR_INVALID_ARG;
    gdn::DecodeArgs a{q, k, v, g, b, state, out, N, Hk, Hv, dk, dv, dtype};
    return gdn::launch_decode(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? GDN_OK
                                                                                   : GDN_ERR_CUDA;
}

int gdn_decode_step_slots(const void *q, const void *k, const void *v, const void *g, const void *b,
                          float *state_pool, const int32_t *slots, void *out, int N, int num_slots,
                          int Hk, int Hv, int dk, int dv, int dtype, void *stream) {
    if (N < 0 || num_slots < 0) return GDN_ERR_INVALID_ARG;
    int rc = common_checks(Hk, Hv, dk, dv, dtype);
    if (rc != GDN_OK) return rc;
    if (N == 0) return GDN_OK;
    if ((long long)num_slots * Hv * dv * dk > (1LL << 40)) return GDN_ERR_INVALID_ARG;
    if (num_slots > 0 && (!state_pool || !aligned16(state_pool))) return GDN_ERR_INVALID_ARG;
    const void *ptrs[] = {q, k, v, g, b, slots, out};
    for (const void *p : ptrs)
        if (!p || !aligned16(p)) return GDN_ERR_INVALID_ARG;
    int *status = status_ptr();
    if (!status) return GDN_ERR_CUDA;
    gdn::DecodeArgs a{q, k, v, g, b, state_pool, out, N, Hk, Hv, dk, dv, dtype};
    a.slots = slots;
    a.num_slots = num_slots;
    a.status = status;
    return gdn::launch_decode(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? GDN_OK
                                                                                   : GDN_ERR_CUDA;
}

int gdn_prepass(const void *q, const void *k, const void *g, const void *b,
                const int32_t *cu_seqlens, int B, int T, int Hk, int Hv, int dk, int chunk,
                int dtype, float *rq, float *rk, float *beta, float *gcum, void *stream) {
    if (B < 0 || T < 0 || B > 65535) return GDN_ERR_INVALID_ARG;
    int rc = common_checks(Hk, Hv, dk, 32, dtype);
    if (rc != GDN_OK) return rc;
    if (!chunk_ok(chunk)) return GDN_ERR_UNSUPPORTED;
    const long long Ttot = cu_seqlens ? (long long)T : (long long)B * T;
    if (Ttot > 0x7fffffffLL) return GDN_ERR_INVALID_ARG;
    if (B == 0 || Ttot == 0) return GDN_OK;
    const void *ptrs[] = {q, k, g, b, rq, rk, beta, gcum};
    for (const void *p : ptrs)
        if (!p || !aligned16(p)) return GDN_ERR_INVALID_ARG;
    if (cu_seqlens && !aligned16(cu_seqlens)) return GDN_ERR_INVALID_ARG;
    int *status = status_ptr();
    if (!status) return GDN_ERR_CUDA;
    gdn::PrepassArgs a{q, k, g, b, cu_seqlens, B, T, Hk, Hv, dk, chunk, dtype, rq, rk, beta, gcum,
                       status};
    return gdn::launch_prepass(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? GDN_OK
                                                                                     : GDN_ERR_CUDA;
}

int gdn_get_device_status(void *stream) {
    int *status = status_ptr();
    int *taken = taken_ptr();
    if (!status || !taken) return GDN_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return GDN_ERR_CUDA;
    take_status_kernel<<<1, 1, 0, s>>>(status, taken);
    if (cudaGetLastError() != cudaSuccess) return GDN_ERR_CUDA;
    int host = 0;
    if (cudaMemcpyAsync(&host, taken, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return GDN_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return GDN_ERR_CUDA;
    return host == 0 ? GDN_OK : GDN_ERR_DEVICE_CHECK;
}

}  // extern "C"
