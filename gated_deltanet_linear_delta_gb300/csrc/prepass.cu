// prepass.cu -- the per-token quantities of the block (chunk) form, written out.
//
// The block form of the gated delta rule ("Optimiser l'inference sur appareil
// pour Apple Silicon", section "Qwen cree trois formes de charges de
// travail": the updates may be regrouped into blocks) needs, per token, the
// inverse L2 norms of q and k, beta = sigmoid(b) and the cumulative log-gate
// G_t inside the token's block. The prefill kernels compute these on chip and
// never store them; this kernel materialises them so they can be checked on
// their own.
//
// One warp per token. Blocks start at every sequence start and every `chunk`
// tokens after it, so G_t = sum of g over [block start, t].
#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kPrepassThreads = 256;

template <typename TIn>
__global__ void __launch_bounds__(kPrepassThreads)
prepass_kernel(const TIn *__restrict__ q, const TIn *__restrict__ k, const TIn *__restrict__ g,
               const TIn *__restrict__ b, const int32_t *__restrict__ cu, int B, long T, long Ttot,
               int Hk, int Hv, int dk, int chunk, float *__restrict__ rq, float *__restrict__ rk,
               float *__restrict__ beta, float *__restrict__ gcum, int *status) {
    const int lane = threadIdx.x & 31;
    const long t = (long)blockIdx.x * (kPrepassThreads / 32) + (threadIdx.x >> 5);
    if (t >= Ttot) return;

    // the sequence that owns token t: the last n with cu[n] <= t
    long bos;
    if (cu == nullptr) {
        bos = (t / T) * T;
    } else {
        int lo = 0, hi = B - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if ((long)cu[mid] <= t) lo = mid; else hi = mid - 1;
        }
        long e;
        if (!seq_bounds(cu, lo, B, Ttot, &bos, &e, status) || t < bos || t >= e) {
            flag_error(status);
            return;
        }
    }
    const long start = bos + ((t - bos) / chunk) * chunk;

    for (int hk = 0; hk < Hk; ++hk) {
        float sq = 0.f, sk = 0.f;
        const TIn *qr = q + (t * Hk + hk) * (long)dk;
        const TIn *kr = k + (t * Hk + hk) * (long)dk;
        for (int j = lane; j < dk; j += 32) {
            const float a = to_f32(qr[j]), c = to_f32(kr[j]);
            sq += a * a;
            sk += c * c;
        }
        sq = warp_sum(sq);
        sk = warp_sum(sk);
        if (lane == 0) {
            rq[t * Hk + hk] = rsqrtf(sq + kNormEps);
            rk[t * Hk + hk] = rsqrtf(sk + kNormEps);
        }
    }
    for (int h = lane; h < Hv; h += 32) {
        beta[t * Hv + h] = sigmoidf_(to_f32(b[t * Hv + h]));
        float acc = 0.f;
        for (long s = start; s <= t; ++s) acc += to_f32(g[s * Hv + h]);
        gcum[t * Hv + h] = acc;
    }
}

template <typename TIn>
cudaError_t launch_t(const PrepassArgs &a, cudaStream_t s) {
    const long Ttot = a.cu_seqlens ? (long)a.T : (long)a.B * a.T;
    if (Ttot == 0) return cudaSuccess;
    const long blocks = (Ttot + kPrepassThreads / 32 - 1) / (kPrepassThreads / 32);
    prepass_kernel<TIn><<<(unsigned)blocks, kPrepassThreads, 0, s>>>(
        (const TIn *)a.q, (const TIn *)a.k, (const TIn *)a.g, (const TIn *)a.b, a.cu_seqlens, a.B,
        (long)a.T, Ttot, a.Hk, a.Hv, a.dk, a.chunk, a.rq, a.rk, a.beta, a.gcum, a.status);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prepass(const PrepassArgs &a, cudaStream_t s) {
    return a.dtype == GDN_BF16 ? launch_t<__nv_bfloat16>(a, s) : launch_t<float>(a, s);
}

}  // namespace gdn
