// gdn_common.cuh -- small device helpers shared by the gated delta rule kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn.h"

namespace gdn {

constexpr float kNormEps = 1e-6f;  // x / sqrt(|x|^2 + eps)

// ---- element I/O -----------------------------------------------------------
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// four consecutive elements starting at p (p 8-byte aligned for bf16, 16 for f32)
__device__ __forceinline__ float4 load4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ float4 load4(const __nv_bfloat16 *p) {
    const uint2 raw = *reinterpret_cast<const uint2 *>(p);
    const __nv_bfloat162 lo = *reinterpret_cast<const __nv_bfloat162 *>(&raw.x);
    const __nv_bfloat162 hi = *reinterpret_cast<const __nv_bfloat162 *>(&raw.y);
    const float2 a = __bfloat1622float2(lo), b = __bfloat1622float2(hi);
    return make_float4(a.x, a.y, b.x, b.y);
}

__device__ __forceinline__ float dot4(float4 a, float4 b) {
    return a.x * b.x + a.y * b.y + a.z * b.z + a.w * b.w;
}

// sum over aligned groups of `width` lanes (width a power of two <= 32)
template <int width>
__device__ __forceinline__ float group_sum(float x) {
#pragma unroll
    for (int o = width / 2; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

__device__ __forceinline__ float warp_sum(float x) { return group_sum<32>(x); }

__device__ __forceinline__ float sigmoidf_(float x) { return 1.0f / (1.0f + expf(-x)); }

// Record a device-side consistency failure (never traps).
__device__ __forceinline__ void flag_error(int *status) {
    if (status) atomicExch(status, (int)GDN_ERR_DEVICE_CHECK);
}

// Bounds of sequence n. Returns false (and flags) when cu_seqlens is inconsistent.
__device__ __forceinline__ bool seq_bounds(const int32_t *cu, int n, int B, long T, long *bos,
                                           long *eos, int *status) {
    if (cu == nullptr) {
        *bos = (long)n * T;
        *eos = *bos + T;
        return true;
    }
    const long a = cu[n], e = cu[n + 1];
    bool ok = (a >= 0) && (e >= a) && (e <= T);
    if (n == 0 && a != 0) ok = false;
    if (n == B - 1 && e != T) ok = false;
    if (!ok) {
        flag_error(status);
        return false;
    }
    *bos = a;
    *eos = e;
    return true;
}

// Packed sequences are taken longest first: CTA row y works on the sequence of rank y, where
// sequence m's rank counts the sequences longer than it (ties: lower index first). With
// sequences of mixed lengths this starts the longest chains of blocks first, so that they do
// not finish alone at the end of the launch. Rank is a permutation even when cu_seqlens is
// inconsistent (such sequences are still reported by seq_bounds). Every thread of the CTA calls
// this (it synchronises the CTA); above kRankMaxSeqs sequences row y keeps sequence y.
constexpr int kRankMaxSeqs = 128;
__device__ __forceinline__ int longest_first(const int32_t *cu, int B, int y) {
    if (cu == nullptr || B > kRankMaxSeqs) return y;
    __shared__ int s_len[kRankMaxSeqs];
    __shared__ int s_pick;
    for (int m = threadIdx.x; m < B; m += blockDim.x) s_len[m] = cu[m + 1] - cu[m];
    __syncthreads();
    for (int m = threadIdx.x; m < B; m += blockDim.x) {
        const int lm = s_len[m];
        int rank = 0;
        for (int o = 0; o < B; ++o) rank += (s_len[o] > lm) || (s_len[o] == lm && o < m);
        if (rank == y) s_pick = m;
    }
    __syncthreads();
    return s_pick;
}

}  // namespace gdn
