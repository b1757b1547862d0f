// prefill_static.cu -- fixed device scratch for the allocation-free prefill entry point.
//
// The tensor-core prefill keeps its ring of prepared blocks and its per-call tables in a device
// workspace. gdn_prefill_static takes that workspace from this file-scope array instead, so the
// call never allocates: the array is part of this module's device image and exists once the
// module is loaded on a device. It is sized for the ring of a fixed number of state-carrying CTAs
// plus a table allowance; callers whose sizes need more get an error before anything is queued.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kMaxDevices = 64;

__device__ __align__(256) uint8_t g_prefill_scratch[kStaticScratchBytes];

void *g_scratch_ptr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;  // the first call on a device may come from several host threads

}  // namespace

void *static_scratch() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_prefill_scratch) != cudaSuccess) return nullptr;
        g_scratch_ptr[dev] = p;
    }
    return g_scratch_ptr[dev];
}

}  // namespace gdn
