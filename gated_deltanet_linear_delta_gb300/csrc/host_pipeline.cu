// host_pipeline.cu -- prefill of one sequence whose inputs and outputs live in host memory,
// with the host<->device copies overlapped with the computation.
//
// The recurrent state is carried from one prompt fragment to the next with an unchanged
// result ("Optimiser l'inference sur appareil pour Apple Silicon", section "Limiter la
// memoire temporaire grace au decoupage des prompts"), so a prompt can be processed
// fragment by fragment: while fragment f is computed on the caller's stream, the inputs of
// fragment f+1 are copied in on one library stream and the outputs of fragment f-1 are
// copied out on another. Fragments are whole multiples of the block length, so every block
// is the one a single call would form and the result is bit-identical to one gdn_prefill
// over the whole prompt.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "gdn.h"
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxFragments = 256;

struct DevicePipe {
    std::mutex mu;  // one call enqueues at a time: the events below are shared by calls
    bool ready = false;
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t start = nullptr, done_in[kMaxFragments] = {}, done_k[kMaxFragments] = {}, done_out = nullptr;
    cudaEvent_t join_in = nullptr, join_out = nullptr;  // error path: the caller's stream waits for both
};
DevicePipe g_pipe[kMaxDevices];
std::mutex g_init_mu;

// streams and events of the current device, created on first use (no device memory)
DevicePipe *pipe_for_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    DevicePipe &d = g_pipe[dev];
    std::lock_guard<std::mutex> lock(g_init_mu);
    if (d.ready) return &d;
    if (cudaStreamCreateWithFlags(&d.in, cudaStreamNonBlocking) != cudaSuccess) return nullptr;
    if (cudaStreamCreateWithFlags(&d.out, cudaStreamNonBlocking) != cudaSuccess) return nullptr;
    const unsigned fl = cudaEventDisableTiming;
    if (cudaEventCreateWithFlags(&d.start, fl) != cudaSuccess) return nullptr;
    if (cudaEventCreateWithFlags(&d.done_out, fl) != cudaSuccess) return nullptr;
    if (cudaEventCreateWithFlags(&d.join_in, fl) != cudaSuccess) return nullptr;
    if (cudaEventCreateWithFlags(&d.join_out, fl) != cudaSuccess) return nullptr;
    for (int f = 0; f < kMaxFragments; ++f)
        if (cudaEventCreateWithFlags(&d.done_in[f], fl) != cudaSuccess ||
            cudaEventCreateWithFlags(&d.done_k[f], fl) != cudaSuccess)
            return nullptr;
    d.ready = true;
    return &d;
}

}  // namespace
}  // namespace gdn

extern "C" int gdn_prefill_from_host(const void *q_h, const void *k_h, const void *v_h, const void *g_h,
                                     const void *b_h, const float *state_in_h, float *state_out_h, void *out_h,
                                     void *q_d, void *k_d, void *v_d, void *g_d, void *b_d, float *state_d,
                                     void *out_d, int T, int Hk, int Hv, int dk, int dv, int chunk, int dtype,
                                     int fragment, void *stream) {
    if (T < 0 || fragment <= 0 || chunk <= 0 || fragment % chunk != 0) return GDN_ERR_INVALID_ARG;
    if (!state_out_h || !state_d) return GDN_ERR_INVALID_ARG;
    if (T > 0 && (!q_h || !k_h || !v_h || !g_h || !b_h || !out_h || !q_d || !k_d || !v_d || !g_d || !b_d ||
                  !out_d))
        return GDN_ERR_INVALID_ARG;
    const int nfrag = T == 0 ? 0 : (T + fragment - 1) / fragment;
    if (nfrag > gdn::kMaxFragments) return GDN_ERR_INVALID_ARG;
    // every size check of the device call, before any work is queued
    int rc = gdn_prefill_path(1, T, Hk, Hv, dk, dv, chunk, dtype);
    if (rc < 0) return rc;
    const size_t es = dtype == GDN_BF16 ? 2 : 4;
    const size_t qk_tok = (size_t)Hk * dk * es, v_tok = (size_t)Hv * dv * es, g_tok = (size_t)Hv * es;
    const size_t st_bytes = (size_t)Hv * dv * dk * sizeof(float);

    gdn::DevicePipe *d = gdn::pipe_for_device();
    if (!d) return GDN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(d->mu);
    cudaStream_t sk = static_cast<cudaStream_t>(stream);
    auto ok = [](cudaError_t e) { return e == cudaSuccess; };
    auto c8 = [](const void *p, size_t off) { return static_cast<const char *>(p) + off; };
    auto m8 = [](void *p, size_t off) { return static_cast<char *>(p) + off; };

    // the copies start after the work already queued on the caller's stream
    if (!ok(cudaEventRecord(d->start, sk)) || !ok(cudaStreamWaitEvent(d->in, d->start, 0)) ||
        !ok(cudaStreamWaitEvent(d->out, d->start, 0)))
        return GDN_ERR_CUDA;
    // After the first copy is queued, a failing step still joins both library streams into the
    // caller's stream before returning, so that work the caller queues next (or a synchronisation
    // of its stream) also waits for the copies already in flight into or out of its buffers.
    auto fail = [&](int code) {
        cudaEventRecord(d->join_in, d->in);
        cudaEventRecord(d->join_out, d->out);
        cudaStreamWaitEvent(sk, d->join_in, 0);
        cudaStreamWaitEvent(sk, d->join_out, 0);
        return code;
    };
    if (state_in_h) {
        if (!ok(cudaMemcpyAsync(state_d, state_in_h, st_bytes, cudaMemcpyHostToDevice, d->in))) return fail(GDN_ERR_CUDA);
    } else if (nfrag == 0) {  // an empty prompt passes a zero state through
        if (!ok(cudaMemsetAsync(state_d, 0, st_bytes, d->in))) return fail(GDN_ERR_CUDA);
    }
    for (int f = 0; f < nfrag; ++f) {
        const size_t t0 = (size_t)f * fragment;
        const size_t n = (size_t)(T - (int)t0 < fragment ? T - (int)t0 : fragment);
        const struct { const void *h; void *dv; size_t tok; } in[5] = {
            {q_h, q_d, qk_tok}, {k_h, k_d, qk_tok}, {v_h, v_d, v_tok}, {g_h, g_d, g_tok}, {b_h, b_d, g_tok}};
        for (const auto &x : in)
            if (!ok(cudaMemcpyAsync(m8(x.dv, t0 * x.tok), c8(x.h, t0 * x.tok), n * x.tok, cudaMemcpyHostToDevice,
                                    d->in)))
                return fail(GDN_ERR_CUDA);
        if (!ok(cudaEventRecord(d->done_in[f], d->in)) || !ok(cudaStreamWaitEvent(sk, d->done_in[f], 0)))
            return fail(GDN_ERR_CUDA);
        const bool first = f == 0;
        rc = gdn_prefill(m8(q_d, t0 * qk_tok), m8(k_d, t0 * qk_tok), m8(v_d, t0 * v_tok), m8(g_d, t0 * g_tok),
                         m8(b_d, t0 * g_tok), first && !state_in_h ? nullptr : state_d, state_d,
                         m8(out_d, t0 * v_tok), nullptr, 1, (int)n, Hk, Hv, dk, dv, chunk, dtype, sk);
        if (rc != GDN_OK) return fail(rc);
        if (!ok(cudaEventRecord(d->done_k[f], sk)) || !ok(cudaStreamWaitEvent(d->out, d->done_k[f], 0)) ||
            !ok(cudaMemcpyAsync(m8(out_h, t0 * v_tok), c8(out_d, t0 * v_tok), n * v_tok, cudaMemcpyDeviceToHost,
                                d->out)))
            return fail(GDN_ERR_CUDA);
    }
    if (nfrag == 0 && (!ok(cudaEventRecord(d->done_in[0], d->in)) || !ok(cudaStreamWaitEvent(d->out, d->done_in[0], 0))))
        return fail(GDN_ERR_CUDA);
    if (!ok(cudaMemcpyAsync(state_out_h, state_d, st_bytes, cudaMemcpyDeviceToHost, d->out)) ||
        !ok(cudaEventRecord(d->done_out, d->out)) || !ok(cudaStreamWaitEvent(sk, d->done_out, 0)))
        return fail(GDN_ERR_CUDA);
    return GDN_OK;
}
