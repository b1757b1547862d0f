// gdn_internal.h -- launchers behind the C ABI (host side, not exported).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace gdn {

// gdn_prefill runs sequences of at most this many tokens (no cu_seqlens) as a token scan
constexpr int kPrefillScanMaxT = 8;

struct PrefillArgs {
    const void *q, *k, *v, *g, *b;
    const float *state_in;
    float *state_out;
    void *out;
    const int32_t *cu_seqlens;
    int B, T, Hk, Hv, dk, dv, chunk, dtype;
    int *status;  // device status word
};

struct DecodeArgs {
    const void *q, *k, *v, *g, *b;
    float *state;
    void *out;
    int N, Hk, Hv, dk, dv, dtype;
    const int32_t *slots = nullptr;  // pool entry of each sequence, or null: entry n
    long num_slots = 0;              // pool entries (with slots)
    int *status = nullptr;           // device status word (with slots)
};

struct PrepassArgs {
    const void *q, *k, *g, *b;
    const int32_t *cu_seqlens;
    int B, T, Hk, Hv, dk, chunk, dtype;
    float *rq, *rk, *beta, *gcum;
    int *status;
};

cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t s);
cudaError_t launch_prepass(const PrepassArgs &a, cudaStream_t s);
cudaError_t launch_prefill_simt(const PrefillArgs &a, cudaStream_t s);
cudaError_t launch_prefill_tc(const PrefillArgs &a, cudaStream_t s);
bool prefill_tc_supported(const PrefillArgs &a);
// tensor-core kernel with the one-product state chain and block preparation spread over the GPU;
// needs a device workspace of prefill_ring_workspace(a) bytes (256-byte aligned)
bool prefill_ring_supported(const PrefillArgs &a);
// max_chain_ctas > 0 caps the CTAs that carry states (fewer ring slots, a smaller workspace)
size_t prefill_ring_workspace(const PrefillArgs &a, int max_chain_ctas = 0);
cudaError_t launch_prefill_ring(const PrefillArgs &a, void *ws, size_t ws_bytes, cudaStream_t s,
                                int max_chain_ctas = 0);
// Fixed device scratch of the allocation-free prefill: room for the ring of kStaticChainCtas
// state-carrying CTAs (16 slots of 96 KiB each) plus 1 MiB of per-call tables. static_scratch()
// returns its address on the current device (looked up on the first call per device), or null.
constexpr int kStaticChainCtas = 8;
constexpr size_t kStaticScratchBytes = (size_t)13 << 20;
void *static_scratch();
bool prefill_scan_supported(const PrefillArgs &a);
cudaError_t launch_prefill_scan(const PrefillArgs &a, cudaStream_t s);

}  // namespace gdn
