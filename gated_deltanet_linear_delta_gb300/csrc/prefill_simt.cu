// prefill_simt.cu -- block (chunk) form of the gated delta rule on CUDA cores.
//
// The updates of a run of C tokens are regrouped into one block ("Optimiser
// l'inference sur appareil pour Apple Silicon", section "Qwen cree trois
// formes de charges de travail"). With Kh, Qh the L2-normalised keys/queries
// of the block, G_t the in-block cumulative log-gate and S0 the entering state:
//     A_ts = beta_t e^{G_t-G_s} kh_t.kh_s  (s<t)      T = (I + A)^-1
//     Z    = diag(beta) (V - diag(e^G) Kh S0^T)        U = T Z
//     P_ts = e^{G_t-G_s} qh_t.kh_s  (s<=t)
//     O    = diag(e^G) Qh S0^T + P U
//     S    = e^{G_L} S0 + U^T diag(e^{G_L-G_t}) Kh
// (U = T diag(beta) V - T diag(beta e^G) Kh S0^T is the usual WY/UT form with
// the S0-dependent product taken before the triangular factor.)
//
// This kernel keeps the whole block in shared memory in fp32 and uses plain
// FMAs. It serves shapes the tensor-core kernel does not take (fp32 I/O,
// dk or dv below 128, blocks of 16 or 32 tokens). One CTA per (value-column
// slab, value head, sequence); the state slab stays in shared memory across
// all blocks of the sequence and is written back once at the end (section
// "Maintenir l'etat recurrent sur la puce").
#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kSimtThreads = 256;

template <int DK, int DVS, int C>
struct SimtSmem {
    static constexpr int KS = DK + 1;  // padded row stride of S, Kh, Qh
    static constexpr int floats = DVS * KS + 2 * C * KS + 3 * C * DVS + 3 * C * C + 4 * C;
    static constexpr size_t bytes = sizeof(float) * floats;
};

template <int DK, int DVS, int C, typename TIn>
__global__ void __launch_bounds__(kSimtThreads)
prefill_simt_kernel(const TIn *__restrict__ q, const TIn *__restrict__ k, const TIn *__restrict__ v,
                    const TIn *__restrict__ g, const TIn *__restrict__ b,
                    const float *state_in, float *state_out,  // may alias (in-place update)
                    TIn *__restrict__ out, const int32_t *__restrict__ cu, int B, long T, long Ttot,
                    int Hk, int Hv, int DV, int *status) {
    using L = SimtSmem<DK, DVS, C>;
    constexpr int KS = L::KS;
    extern __shared__ float smem[];
    float *S = smem;              // [DVS][KS]
    float *Kh = S + DVS * KS;     // [C][KS]
    float *Qh = Kh + C * KS;      // [C][KS]
    float *V = Qh + C * KS;       // [C][DVS]
    float *Z = V + C * DVS;       // [C][DVS]
    float *U = Z + C * DVS;       // [C][DVS]
    float *A = U + C * DVS;       // [C][C]
    float *Tm = A + C * C;        // [C][C]
    float *P = Tm + C * C;        // [C][C]
    float *beta_s = P + C * C;    // [C]
    float *G = beta_s + C;        // [C]
    float *eG = G + C;            // [C] e^{G_t}
    float *dG = eG + C;           // [C] e^{G_L - G_t}

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n = blockIdx.z, h = blockIdx.y, i_base = blockIdx.x * DVS;
    const int hk = h / (Hv / Hk);
    long bos, eos;
    if (!seq_bounds(cu, n, B, cu ? Ttot : T, &bos, &eos, status)) return;

    const long st_off = ((long)n * Hv + h) * DV * (long)DK;
    for (int idx = tid; idx < DVS * DK; idx += kSimtThreads) {
        const int i = idx / DK, j = idx % DK;
        S[i * KS + j] = state_in ? state_in[st_off + (long)(i_base + i) * DK + j] : 0.f;
    }

    for (long c0 = bos; c0 < eos; c0 += C) {
        const int Lc = (int)min((long)C, eos - c0);
        __syncthreads();  // previous block's readers of Kh/V/S are done
        // normalised keys and queries, one warp per row
        for (int t = warp; t < C; t += kSimtThreads / 32) {
            float kr[(DK + 31) / 32], qr[(DK + 31) / 32];
            float sk = 0.f, sq = 0.f;
#pragma unroll
            for (int u = 0; u < (DK + 31) / 32; ++u) {
                const int j = lane + 32 * u;
                kr[u] = qr[u] = 0.f;
                if (t < Lc && j < DK) {
                    const long off = ((c0 + t) * Hk + hk) * (long)DK + j;
                    kr[u] = to_f32(k[off]);
                    qr[u] = to_f32(q[off]);
                }
                sk += kr[u] * kr[u];
                sq += qr[u] * qr[u];
            }
            sk = warp_sum(sk);
            sq = warp_sum(sq);
            const float rk = rsqrtf(sk + kNormEps), rq = rsqrtf(sq + kNormEps);
#pragma unroll
            for (int u = 0; u < (DK + 31) / 32; ++u) {
                const int j = lane + 32 * u;
                if (j < DK) {
                    Kh[t * KS + j] = kr[u] * rk;
                    Qh[t * KS + j] = qr[u] * rq;
                }
            }
        }
        for (int idx = tid; idx < C * DVS; idx += kSimtThreads) {
            const int t = idx / DVS, i = idx % DVS;
            V[idx] = t < Lc ? to_f32(v[((c0 + t) * Hv + h) * (long)DV + i_base + i]) : 0.f;
        }
        if (tid < C) {
            const bool ok = tid < Lc;
            G[tid] = ok ? to_f32(g[(c0 + tid) * Hv + h]) : 0.f;
            beta_s[tid] = ok ? sigmoidf_(to_f32(b[(c0 + tid) * Hv + h])) : 0.f;
        }
        __syncthreads();
        // in-block inclusive cumulative sum of the log-gates (one warp, C <= 64)
        if (warp == 0) {
            float x0 = lane < C ? G[lane] : 0.f;
            float x1 = lane + 32 < C ? G[lane + 32] : 0.f;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y0 = __shfl_up_sync(0xffffffffu, x0, o);
                const float y1 = __shfl_up_sync(0xffffffffu, x1, o);
                if (lane >= o) { x0 += y0; x1 += y1; }
            }
            x1 += __shfl_sync(0xffffffffu, x0, 31);
            __syncwarp();
            if (lane < C) G[lane] = x0;
            if (lane + 32 < C) G[lane + 32] = x1;
        }
        __syncthreads();
        const float GL = G[Lc - 1];
        if (tid < C) {
            eG[tid] = expf(G[tid]);
            dG[tid] = tid < Lc ? expf(GL - G[tid]) : 0.f;
        }
        // A (strictly lower) and P (lower with diagonal)
        for (int idx = tid; idx < C * C; idx += kSimtThreads) {
            const int t = idx / C, s = idx % C;
            float kk = 0.f, qk = 0.f;
            if (s <= t) {
#pragma unroll 8
                for (int j = 0; j < DK; ++j) {
                    const float ks = Kh[s * KS + j];
                    kk += Kh[t * KS + j] * ks;
                    qk += Qh[t * KS + j] * ks;
                }
            }
            const float dec = s <= t ? expf(G[t] - G[s]) : 0.f;
            A[idx] = s < t ? beta_s[t] * dec * kk : 0.f;
            P[idx] = dec * qk;
        }
        __syncthreads();
        // T = (I + A)^-1, forward substitution, one column per thread
        if (tid < C) {
            const int j = tid;
            for (int r = 0; r < j; ++r) Tm[r * C + j] = 0.f;
            Tm[j * C + j] = 1.f;
            for (int r = j + 1; r < C; ++r) {
                float acc = 0.f;
                for (int s = j; s < r; ++s) acc += A[r * C + s] * Tm[s * C + j];
                Tm[r * C + j] = -acc;
            }
        }
        // Z = diag(beta) (V - diag(e^G) Kh S0^T)
        for (int idx = tid; idx < C * DVS; idx += kSimtThreads) {
            const int t = idx / DVS, i = idx % DVS;
            float y = 0.f;
#pragma unroll 8
            for (int j = 0; j < DK; ++j) y += Kh[t * KS + j] * S[i * KS + j];
            Z[idx] = beta_s[t] * (V[idx] - eG[t] * y);
        }
        __syncthreads();
        // U = T Z
        for (int idx = tid; idx < C * DVS; idx += kSimtThreads) {
            const int t = idx / DVS, i = idx % DVS;
            float acc = 0.f;
            for (int s = 0; s <= t; ++s) acc += Tm[t * C + s] * Z[s * DVS + i];
            U[idx] = acc;
        }
        __syncthreads();
        // O = diag(e^G) Qh S0^T + P U
        for (int idx = tid; idx < C * DVS; idx += kSimtThreads) {
            const int t = idx / DVS, i = idx % DVS;
            if (t >= Lc) continue;
            float qs = 0.f;
#pragma unroll 8
            for (int j = 0; j < DK; ++j) qs += Qh[t * KS + j] * S[i * KS + j];
            float pu = 0.f;
            for (int s = 0; s <= t; ++s) pu += P[t * C + s] * U[s * DVS + i];
            out[((c0 + t) * Hv + h) * (long)DV + i_base + i] = from_f32<TIn>(eG[t] * qs + pu);
        }
        __syncthreads();
        // S = e^{G_L} S0 + U^T diag(e^{G_L - G_t}) Kh
        const float gL = expf(GL);
        for (int idx = tid; idx < DVS * DK; idx += kSimtThreads) {
            const int i = idx / DK, j = idx % DK;
            float acc = 0.f;
            for (int t = 0; t < Lc; ++t) acc += U[t * DVS + i] * dG[t] * Kh[t * KS + j];
            S[i * KS + j] = gL * S[i * KS + j] + acc;
        }
    }
    __syncthreads();
    for (int idx = tid; idx < DVS * DK; idx += kSimtThreads) {
        const int i = idx / DK, j = idx % DK;
        state_out[st_off + (long)(i_base + i) * DK + j] = S[i * KS + j];
    }
}

template <int DK, int DVS, int C, typename TIn>
cudaError_t launch_t(const PrefillArgs &a, cudaStream_t s) {
    constexpr size_t bytes = SimtSmem<DK, DVS, C>::bytes;
    auto kern = prefill_simt_kernel<DK, DVS, C, TIn>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    const long Ttot = a.cu_seqlens ? (long)a.T : (long)a.B * a.T;
    dim3 grid(a.dv / DVS, a.Hv, a.B);
    kern<<<grid, kSimtThreads, bytes, s>>>((const TIn *)a.q, (const TIn *)a.k, (const TIn *)a.v,
                                           (const TIn *)a.g, (const TIn *)a.b, a.state_in, a.state_out,
                                           (TIn *)a.out, a.cu_seqlens, a.B, (long)a.T, Ttot, a.Hk,
                                           a.Hv, a.dv, a.status);
    return cudaGetLastError();
}

template <int DK, int DVS, typename TIn>
cudaError_t by_chunk(const PrefillArgs &a, cudaStream_t s) {
    switch (a.chunk) {
        case 16: return launch_t<DK, DVS, 16, TIn>(a, s);
        case 32: return launch_t<DK, DVS, 32, TIn>(a, s);
        case 64: return launch_t<DK, DVS, 64, TIn>(a, s);
    }
    return cudaErrorInvalidValue;
}

template <typename TIn>
cudaError_t by_dims(const PrefillArgs &a, cudaStream_t s) {
    const int dvs = a.dv < 64 ? a.dv : 64;
    if (dvs == 32) {
        if (a.dk == 32) return by_chunk<32, 32, TIn>(a, s);
        if (a.dk == 64) return by_chunk<64, 32, TIn>(a, s);
        if (a.dk == 128) return by_chunk<128, 32, TIn>(a, s);
    } else {
        if (a.dk == 32) return by_chunk<32, 64, TIn>(a, s);
        if (a.dk == 64) return by_chunk<64, 64, TIn>(a, s);
        if (a.dk == 128) return by_chunk<128, 64, TIn>(a, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_prefill_simt(const PrefillArgs &a, cudaStream_t s) {
    if (a.B == 0) return cudaSuccess;
    return a.dtype == GDN_BF16 ? by_dims<__nv_bfloat16>(a, s) : by_dims<float>(a, s);
}

}  // namespace gdn
