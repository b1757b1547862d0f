// decode_step.cu -- one recurrent step of the gated delta rule for N sequences.
//
// Decoding is bound by the bytes moved per token ("Optimiser l'inference sur
// appareil pour Apple Silicon", section "Decodage : minimiser les octets
// deplaces par token"): per (sequence, value head) the fp32 state S
// (dv x dk) is read once and written once, in place. Everything else -- the
// L2 normalisation of q and k, alpha = exp(g), beta = sigmoid(b), the delta
// update and the read-out -- is fused into the same pass (section "Reduire le
// trafic intermediaire et d'etat": the recurrent update is fused with its
// normalisation). Adjacent lanes read adjacent 16-byte pieces of a state row
// (section "Fusionner les lectures du cache d'attention": neighbouring threads
// should ask for neighbouring bytes).
//
// Per row i of S, with kh, qh the normalised key/query of the shared key head:
//     e_i = alpha (S kh)_i,   u_i = beta (v_i - e_i)
//     S_i <- alpha S_i + u_i kh^T
//     o_i = (S_new qh)_i = alpha (S qh)_i + u_i (kh . qh)
// so both dot products S_i.kh and S_i.qh come from the single read of S_i and
// are reduced together across the lanes that hold the row.
//
// Work mapping: a row of dk fp32 is held by LPR = dk/4 lanes, one float4 each;
// a warp covers RPW = 32/LPR rows per pass and R passes, all R loads issued
// before any arithmetic so that 16*R bytes per thread are in flight. All rows
// of one warp belong to one (sequence, head), so the norms are computed once
// per warp.
//
// Slot-indexed variant (kSlots): the states live in a pool of `num_slots`
// [Hv][dv][dk] entries and sequence n updates pool entry slots[n], so a server
// can keep many sessions resident and step any subset of them in one launch.
// A negative slot marks a padding row (state untouched, output zero); a slot
// >= num_slots is a caller error, flagged on the device status word and
// skipped the same way.
#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr int kDecodeThreads = 256;
constexpr int kDecodeRows = 4;  // passes (rows per lane group) per warp
constexpr int kScanMaxT = kPrefillScanMaxT;  // tokens per sequence of the token-scan kernel

template <int DK, int DV, typename TIn, bool kSlots>
__global__ void __launch_bounds__(kDecodeThreads)
decode_step_kernel(const TIn *__restrict__ q, const TIn *__restrict__ k, const TIn *__restrict__ v,
                   const TIn *__restrict__ g, const TIn *__restrict__ b, float *__restrict__ state,
                   TIn *__restrict__ out, int N, int Hk, int Hv, const int32_t *__restrict__ slots,
                   long num_slots, int *status) {
    constexpr int LPR = DK / 4;    // lanes per row
    constexpr int RPW = 32 / LPR;  // rows per warp pass
    constexpr int R = kDecodeRows;
    constexpr int ROWS_PER_WARP = RPW * R;
    static_assert(DV % ROWS_PER_WARP == 0, "a warp must stay within one head");

    const int lane = threadIdx.x & 31;
    const long warp = (long)blockIdx.x * (kDecodeThreads / 32) + (threadIdx.x >> 5);
    const long row0 = warp * ROWS_PER_WARP;
    const long total_rows = (long)N * Hv * DV;
    if (row0 >= total_rows) return;

    const long nh = row0 / DV;  // (sequence, value head) index = n*Hv + h
    const int i0 = (int)(row0 % DV);
    const int h = (int)(nh % Hv);
    const long n = nh / Hv;
    const int hk = h / (Hv / Hk);
    const int grp = lane / LPR;  // row within a pass
    const int c = lane % LPR;    // float4 column

    long sh = nh;  // (pool entry, value head) index of this warp's state
    if (kSlots) {
        const long sl = slots[n];
        if (sl < 0 || sl >= num_slots) {
            if (sl >= num_slots && i0 == 0 && lane == 0) flag_error(status);
#pragma unroll
            for (int r = 0; r < R; ++r)
                if (c == 0) out[nh * DV + i0 + r * RPW + grp] = from_f32<TIn>(0.f);
            return;
        }
        sh = sl * Hv + h;
    }

    // issue the state loads first: they are the bytes that matter
    float *srow[R];
    float4 s[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int i = i0 + r * RPW + grp;
        srow[r] = state + (sh * DV + i) * (long)DK + 4 * c;
        s[r] = __ldcs(reinterpret_cast<const float4 *>(srow[r]));
    }
    const long kq_off = (n * Hk + hk) * (long)DK + 4 * c;
    const float4 k4 = load4(k + kq_off);
    const float4 q4 = load4(q + kq_off);
    float vi[R];
#pragma unroll
    for (int r = 0; r < R; ++r) vi[r] = to_f32(v[nh * DV + i0 + r * RPW + grp]);
    const float alpha = expf(to_f32(g[nh]));
    const float beta = sigmoidf_(to_f32(b[nh]));

    // L2 norms of the shared key head (every lane group holds a full copy)
    const float ssk = group_sum<LPR>(dot4(k4, k4));
    const float ssq = group_sum<LPR>(dot4(q4, q4));
    const float skq = group_sum<LPR>(dot4(k4, q4));
    const float rk = rsqrtf(ssk + kNormEps), rq = rsqrtf(ssq + kNormEps);
    const float4 kh = make_float4(k4.x * rk, k4.y * rk, k4.z * rk, k4.w * rk);
    const float4 qh = make_float4(q4.x * rq, q4.y * rq, q4.z * rq, q4.w * rq);
    const float kq = skq * rk * rq;

#pragma unroll
    for (int r = 0; r < R; ++r) {
        const float sk = group_sum<LPR>(dot4(s[r], kh));
        const float sq = group_sum<LPR>(dot4(s[r], qh));
        const float u = beta * (vi[r] - alpha * sk);
        float4 o4;
        o4.x = alpha * s[r].x + u * kh.x;
        o4.y = alpha * s[r].y + u * kh.y;
        o4.z = alpha * s[r].z + u * kh.z;
        o4.w = alpha * s[r].w + u * kh.w;
        __stcs(reinterpret_cast<float4 *>(srow[r]), o4);
        if (c == 0) out[nh * DV + i0 + r * RPW + grp] = from_f32<TIn>(alpha * sq + u * kq);
    }
}

// A few tokens per sequence (1 <= T <= kScanMaxT), the shape of checking a short run of
// speculated tokens: each state row is read once from state_in (or zero), all T tokens
// are applied in order while it sits in registers, and it is written once to state_out
// (which may be state_in: each lane reads its pieces of a row before it writes them). The
// T steps cost one pass over the state instead of T.
//
// The key and query norms of a token are the same for every row of a head, so each CTA
// computes them once (one warp per token) into shared memory before the scan.
//
// Since every token adds two dot products per row, the row is spread over only
// kScanLanes = 8 lanes (DK/32 float4 pieces each, interleaved so that the 8 lanes read
// 128 contiguous bytes at a time): a 3-step shuffle reduction then serves the 4 rows of a
// warp pass at once, where 32 lanes per row would take 5 steps for one row.
constexpr int kScanLanes = 8;
constexpr int kScanPasses = 2;

template <int DK, int DV, typename TIn>
__global__ void __launch_bounds__(kDecodeThreads, 3)
scan_tokens_kernel(const TIn *__restrict__ q, const TIn *__restrict__ k, const TIn *__restrict__ v,
                   const TIn *__restrict__ g, const TIn *__restrict__ b, const float *state_in,
                   float *state_out, TIn *__restrict__ out, int B, int T, int Hk, int Hv) {
    constexpr int LPR = kScanLanes;
    constexpr int CPL = DK / (4 * LPR);  // float4 pieces per lane
    constexpr int RPW = 32 / LPR;        // rows per warp pass
    constexpr int R = kScanPasses;
    constexpr int ROWS_PER_WARP = RPW * R;
    static_assert(CPL >= 1 && DV % ROWS_PER_WARP == 0, "a warp must stay within one head");

    // warps of this CTA that share a head (a CTA holds one head, or two when DV = 32)
    constexpr int GW = DV / ROWS_PER_WARP < kDecodeThreads / 32 ? DV / ROWS_PER_WARP : kDecodeThreads / 32;
    __shared__ float s_nrm[kDecodeThreads / 32 / GW][kScanMaxT][3];  // per head and token: rk, rq, k.q

    const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
    const long warp = (long)blockIdx.x * (kDecodeThreads / 32) + wib;
    const long row0 = warp * ROWS_PER_WARP;
    const bool valid = row0 < (long)B * Hv * DV;
    const long nh = row0 / DV;
    const int i0 = (int)(row0 % DV);
    const int h = (int)(nh % Hv);
    const long n = nh / Hv;
    const int hk = h / (Hv / Hk);
    const int grp = lane / LPR;  // row within a pass
    const int c = lane % LPR;    // piece j of this lane covers columns 4 (c + LPR j) .. +3

    float4 s[R][CPL];
    if (valid) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const long off = (nh * DV + i0 + r * RPW + grp) * (long)DK;
#pragma unroll
            for (int j = 0; j < CPL; ++j)
                s[r][j] = state_in ? __ldcs(reinterpret_cast<const float4 *>(state_in + off + 4 * (c + LPR * j)))
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        // the norms of this head's tokens, once per CTA: warp w of the head takes tokens w, w + GW, ...
        for (int t = wib % GW; t < T; t += GW) {
            const long kq_off = ((n * T + t) * Hk + hk) * (long)DK;
            float pkk = 0.f, pqq = 0.f, pkq = 0.f;
#pragma unroll
            for (int j = 0; j < DK / 32; ++j) {
                const float kx = to_f32(k[kq_off + lane + 32 * j]), qx = to_f32(q[kq_off + lane + 32 * j]);
                pkk += kx * kx;
                pqq += qx * qx;
                pkq += kx * qx;
            }
            pkk = warp_sum(pkk);
            pqq = warp_sum(pqq);
            pkq = warp_sum(pkq);
            if (lane == 0) {
                s_nrm[wib / GW][t][0] = rsqrtf(pkk + kNormEps);
                s_nrm[wib / GW][t][1] = rsqrtf(pqq + kNormEps);
                s_nrm[wib / GW][t][2] = pkq;
            }
        }
    }
    __syncthreads();
    if (!valid) return;
#pragma unroll 1
    for (int t = 0; t < T; ++t) {
        const long tok = n * T + t;
        const long kq_off = (tok * Hk + hk) * (long)DK;
        float4 kh[CPL], qh[CPL];
#pragma unroll
        for (int j = 0; j < CPL; ++j) {
            kh[j] = load4(k + kq_off + 4 * (c + LPR * j));
            qh[j] = load4(q + kq_off + 4 * (c + LPR * j));
        }
        float vi[R];
#pragma unroll
        for (int r = 0; r < R; ++r) vi[r] = to_f32(v[(tok * Hv + h) * DV + i0 + r * RPW + grp]);
        const float alpha = expf(to_f32(g[tok * Hv + h]));
        const float beta = sigmoidf_(to_f32(b[tok * Hv + h]));
        const float rk = s_nrm[wib / GW][t][0], rq = s_nrm[wib / GW][t][1];
        const float kq = s_nrm[wib / GW][t][2] * rk * rq;
#pragma unroll
        for (int j = 0; j < CPL; ++j) {
            kh[j] = make_float4(kh[j].x * rk, kh[j].y * rk, kh[j].z * rk, kh[j].w * rk);
            qh[j] = make_float4(qh[j].x * rq, qh[j].y * rq, qh[j].z * rq, qh[j].w * rq);
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float psk = 0.f, psq = 0.f;
#pragma unroll
            for (int j = 0; j < CPL; ++j) {
                psk += dot4(s[r][j], kh[j]);
                psq += dot4(s[r][j], qh[j]);
            }
            const float sk = group_sum<LPR>(psk), sq = group_sum<LPR>(psq);
            const float u = beta * (vi[r] - alpha * sk);
#pragma unroll
            for (int j = 0; j < CPL; ++j) {
                s[r][j].x = alpha * s[r][j].x + u * kh[j].x;
                s[r][j].y = alpha * s[r][j].y + u * kh[j].y;
                s[r][j].z = alpha * s[r][j].z + u * kh[j].z;
                s[r][j].w = alpha * s[r][j].w + u * kh[j].w;
            }
            if (c == 0) out[(tok * Hv + h) * DV + i0 + r * RPW + grp] = from_f32<TIn>(alpha * sq + u * kq);
        }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const long off = (nh * DV + i0 + r * RPW + grp) * (long)DK;
#pragma unroll
        for (int j = 0; j < CPL; ++j) __stcs(reinterpret_cast<float4 *>(state_out + off + 4 * (c + LPR * j)), s[r][j]);
    }
}

template <int DK, int DV, typename TIn>
cudaError_t launch_t(const DecodeArgs &a, cudaStream_t s) {
    const auto kern = a.slots ? decode_step_kernel<DK, DV, TIn, true> : decode_step_kernel<DK, DV, TIn, false>;
    constexpr int ROWS_PER_WARP = (32 / (DK / 4)) * kDecodeRows;
    const long rows = (long)a.N * a.Hv * DV;
    const long warps = (rows + ROWS_PER_WARP - 1) / ROWS_PER_WARP;
    const long blocks = (warps + kDecodeThreads / 32 - 1) / (kDecodeThreads / 32);
    if (blocks > 0x7fffffffL) return cudaErrorInvalidConfiguration;
    kern<<<(unsigned)blocks, kDecodeThreads, 0, s>>>(
        (const TIn *)a.q, (const TIn *)a.k, (const TIn *)a.v, (const TIn *)a.g, (const TIn *)a.b,
        a.state, (TIn *)a.out, a.N, a.Hk, a.Hv, a.slots, a.num_slots, a.status);
    return cudaGetLastError();
}

template <typename TIn>
cudaError_t dispatch_dims(const DecodeArgs &a, cudaStream_t s) {
#define GDN_DECODE_CASE(DKV, DVV) \
    if (a.dk == DKV && a.dv == DVV) return launch_t<DKV, DVV, TIn>(a, s);
    GDN_DECODE_CASE(32, 32) GDN_DECODE_CASE(32, 64) GDN_DECODE_CASE(32, 128)
    GDN_DECODE_CASE(64, 32) GDN_DECODE_CASE(64, 64) GDN_DECODE_CASE(64, 128)
    GDN_DECODE_CASE(128, 32) GDN_DECODE_CASE(128, 64) GDN_DECODE_CASE(128, 128)
#undef GDN_DECODE_CASE
    return cudaErrorInvalidValue;
}

template <int DK, int DV, typename TIn>
cudaError_t launch_scan_t(const PrefillArgs &a, cudaStream_t s) {
    constexpr int ROWS_PER_WARP = (32 / kScanLanes) * kScanPasses;
    const long rows = (long)a.B * a.Hv * DV;
    const long warps = (rows + ROWS_PER_WARP - 1) / ROWS_PER_WARP;
    const long blocks = (warps + kDecodeThreads / 32 - 1) / (kDecodeThreads / 32);
    if (blocks > 0x7fffffffL) return cudaErrorInvalidConfiguration;
    scan_tokens_kernel<DK, DV, TIn><<<(unsigned)blocks, kDecodeThreads, 0, s>>>(
        (const TIn *)a.q, (const TIn *)a.k, (const TIn *)a.v, (const TIn *)a.g, (const TIn *)a.b,
        a.state_in, a.state_out, (TIn *)a.out, a.B, a.T, a.Hk, a.Hv);
    return cudaGetLastError();
}

template <typename TIn>
cudaError_t dispatch_scan(const PrefillArgs &a, cudaStream_t s) {
#define GDN_SCAN_CASE(DKV, DVV) \
    if (a.dk == DKV && a.dv == DVV) return launch_scan_t<DKV, DVV, TIn>(a, s);
    GDN_SCAN_CASE(32, 32) GDN_SCAN_CASE(32, 64) GDN_SCAN_CASE(32, 128)
    GDN_SCAN_CASE(64, 32) GDN_SCAN_CASE(64, 64) GDN_SCAN_CASE(64, 128)
    GDN_SCAN_CASE(128, 32) GDN_SCAN_CASE(128, 64) GDN_SCAN_CASE(128, 128)
#undef GDN_SCAN_CASE
    return cudaErrorInvalidValue;
}

}  // namespace

bool prefill_scan_supported(const PrefillArgs &a) {
    return a.cu_seqlens == nullptr && a.T >= 1 && a.T <= kScanMaxT;
}

cudaError_t launch_prefill_scan(const PrefillArgs &a, cudaStream_t s) {
    if (a.B == 0) return cudaSuccess;
    return a.dtype == GDN_BF16 ? dispatch_scan<__nv_bfloat16>(a, s) : dispatch_scan<float>(a, s);
}

cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t s) {
    if (a.N == 0) return cudaSuccess;
    return a.dtype == GDN_BF16 ? dispatch_dims<__nv_bfloat16>(a, s) : dispatch_dims<float>(a, s);
}

}  // namespace gdn
