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
#include <algorithm>
#include <atomic>

#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "tc_ops.cuh"

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
// (which may be state_in). The T steps cost one pass over the state instead of T.
//
// The CTAs are persistent and take one (sequence, value head) state at a time: its rows are
// spread over the CTA's 8 warps (8 lanes per row), and while they are updated in registers
// the next head's state is already on its way into shared memory (one bulk copy), so the
// HBM reads of one head overlap the arithmetic of the previous one.
//
// Everything a token contributes that is the same for every row of a head -- the normalised
// key and query (fp32), v, alpha, beta and kh . qh -- is computed once per head into shared
// memory (one warp per token), so the per-row work of a token is two dot products, one
// paired reduction and the update. Each lane holds DK/32 float4 pieces of its row,
// interleaved so that the 8 lanes of a row read 128 contiguous bytes at a time. The two
// reductions of a row share one 3-step shuffle tree: at the first step each lane keeps one
// of the two sums and sends the other, so every step moves one value.
constexpr int kScanLanes = 8;
constexpr int kScanWarps = kDecodeThreads / 32;
constexpr long long kScanWait = 4000000000LL;  // SM cycles before a wait for a state copy gives up

template <int DK, int DV>
struct ScanSmem {
    float4 state[DV * DK / 4];          // the next head's state (bulk copy)
    float4 kq[kScanMaxT][2][DK / 4];    // per token: kh, qh (normalised)
    float v[kScanMaxT][DV];             // per token: v
    float sc[kScanMaxT][4];             // per token: alpha, beta, kh . qh
    uint64_t bar;
};

template <int DK, int DV, typename TIn>
__global__ void __launch_bounds__(kDecodeThreads, 2)
scan_tokens_kernel(const TIn *__restrict__ q, const TIn *__restrict__ k, const TIn *__restrict__ v,
                   const TIn *__restrict__ g, const TIn *__restrict__ b, const float *state_in,
                   float *state_out, TIn *__restrict__ out, int B, int T, int Hk, int Hv, int *status) {
    constexpr int LPR = kScanLanes;
    constexpr int CPL = DK / (4 * LPR);  // float4 pieces per lane
    constexpr int RPW = 32 / LPR;        // rows per warp pass
    constexpr int R = DV / (RPW * kScanWarps);  // passes: the CTA's warps cover the DV rows of a head
    static_assert(CPL >= 1 && R >= 1 && R * RPW * kScanWarps == DV, "the CTA must cover one head");
    static_assert(LPR == 8, "the paired reduction below is a 3-step tree");
    constexpr uint32_t kStateBytes = DV * DK * 4;

    extern __shared__ __align__(128) uint8_t scan_smem_raw[];
    ScanSmem<DK, DV> &sm = *reinterpret_cast<ScanSmem<DK, DV> *>(scan_smem_raw);
    const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
    const int grp = lane / LPR;  // row within a pass
    const int c = lane % LPR;    // piece j of this lane covers columns 4 (c + LPR j) .. +3
    const long heads = (long)B * Hv;
    const bool low = (c & 4) == 0;  // after the first reduction step: low lanes hold S.kh, high lanes S.qh

    if (threadIdx.x == 0) {
        tc::mbar_init(&sm.bar, 1);
        tc::fence_mbar_init();
    }
    __syncthreads();
    long nh = blockIdx.x;
    if (threadIdx.x == 0 && state_in && nh < heads) {
        tc::mbar_expect_tx(&sm.bar, kStateBytes);
        tc::bulk_load(sm.state, state_in + nh * (long)(DV * DK), kStateBytes, &sm.bar);
    }
    for (uint32_t it = 0; nh < heads; ++it, nh += gridDim.x) {
        const int h = (int)(nh % Hv);
        const long n = nh / Hv;
        const int hk = h / (Hv / Hk);
        // this head's tokens: warp w takes tokens w, w + 8, ...
        for (int t = wib; t < T; t += kScanWarps) {
            const long tok = n * T + t;
            const long kq_off = (tok * Hk + hk) * (long)DK;
            float kx[DK / 32], qx[DK / 32];
            float pkk = 0.f, pqq = 0.f, pkq = 0.f;
#pragma unroll
            for (int j = 0; j < DK / 32; ++j) {
                kx[j] = to_f32(k[kq_off + lane + 32 * j]);
                qx[j] = to_f32(q[kq_off + lane + 32 * j]);
                pkk += kx[j] * kx[j];
                pqq += qx[j] * qx[j];
                pkq += kx[j] * qx[j];
            }
            pkk = warp_sum(pkk);
            pqq = warp_sum(pqq);
            pkq = warp_sum(pkq);
            const float rk = rsqrtf(pkk + kNormEps), rq = rsqrtf(pqq + kNormEps);
            float *kh = reinterpret_cast<float *>(sm.kq[t][0]), *qh = reinterpret_cast<float *>(sm.kq[t][1]);
#pragma unroll
            for (int j = 0; j < DK / 32; ++j) {
                kh[lane + 32 * j] = kx[j] * rk;
                qh[lane + 32 * j] = qx[j] * rq;
            }
#pragma unroll
            for (int j = 0; j < (DV + 31) / 32; ++j)
                if (lane + 32 * j < DV) sm.v[t][lane + 32 * j] = to_f32(v[(tok * Hv + h) * DV + lane + 32 * j]);
            if (lane == 0) {
                sm.sc[t][0] = expf(to_f32(g[tok * Hv + h]));
                sm.sc[t][1] = sigmoidf_(to_f32(b[tok * Hv + h]));
                sm.sc[t][2] = pkq * rk * rq;
            }
        }
        // the state of this head: from the bulk copy (or zero)
        bool failed = false;
        if (state_in) failed = !tc::mbar_wait(&sm.bar, it & 1, kScanWait);
        float4 s[R][CPL];
        const int rbase = wib * (R * RPW) + grp;  // row of pass r: rbase + r * RPW
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int j = 0; j < CPL; ++j)
                s[r][j] = state_in ? sm.state[(rbase + r * RPW) * (DK / 4) + c + LPR * j] : make_float4(0.f, 0.f, 0.f, 0.f);
        // every thread has read the buffer (and the token values are visible): the next head's copy may start
        if (__syncthreads_or(failed)) {
            if (threadIdx.x == 0) {
                flag_error(status);
                tc::mbar_wait(&sm.bar, it & 1, kScanWait);  // the copy must land before the CTA leaves
            }
            return;
        }
        if (threadIdx.x == 0 && state_in && nh + gridDim.x < heads) {
            tc::fence_async_smem();
            tc::mbar_expect_tx(&sm.bar, kStateBytes);
            tc::bulk_load(sm.state, state_in + (nh + gridDim.x) * (long)(DV * DK), kStateBytes, &sm.bar);
        }
#pragma unroll 1
        for (int t = 0; t < T; ++t) {
            const float alpha = sm.sc[t][0], beta = sm.sc[t][1], kq = sm.sc[t][2];
            float4 kh[CPL], qh[CPL];
#pragma unroll
            for (int j = 0; j < CPL; ++j) {
                kh[j] = sm.kq[t][0][c + LPR * j];
                qh[j] = sm.kq[t][1][c + LPR * j];
            }
            const long orow = ((n * T + t) * Hv + h) * DV;
            // the R rows are independent: each stage below runs over all of them, so their
            // dependent chains (dots, shuffle steps, update) interleave
            float x[R], send[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                float pk2[2] = {0.f, 0.f}, pq2[2] = {0.f, 0.f};  // two chains each: shorter dependences
#pragma unroll
                for (int j = 0; j < CPL; ++j) {
                    pk2[j & 1] += dot4(s[r][j], kh[j]);
                    pq2[j & 1] += dot4(s[r][j], qh[j]);
                }
                const float psk = pk2[0] + pk2[1], psq = pq2[0] + pq2[1];
                x[r] = low ? psk : psq;  // paired reduction over the row's 8 lanes: keep one sum, send the other
                send[r] = low ? psq : psk;
            }
#pragma unroll
            for (int r = 0; r < R; ++r) x[r] += __shfl_xor_sync(0xffffffffu, send[r], 4);
#pragma unroll
            for (int r = 0; r < R; ++r) x[r] += __shfl_xor_sync(0xffffffffu, x[r], 2);
#pragma unroll
            for (int r = 0; r < R; ++r) x[r] += __shfl_xor_sync(0xffffffffu, x[r], 1);
#pragma unroll
            for (int r = 0; r < R; ++r) send[r] = __shfl_xor_sync(0xffffffffu, x[r], 4);
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const float sk = low ? x[r] : send[r], sq = low ? send[r] : x[r];
                const int row = rbase + r * RPW;
                const float u = beta * (sm.v[t][row] - alpha * sk);
#pragma unroll
                for (int j = 0; j < CPL; ++j) {
                    s[r][j].x = fmaf(alpha, s[r][j].x, u * kh[j].x);
                    s[r][j].y = fmaf(alpha, s[r][j].y, u * kh[j].y);
                    s[r][j].z = fmaf(alpha, s[r][j].z, u * kh[j].z);
                    s[r][j].w = fmaf(alpha, s[r][j].w, u * kh[j].w);
                }
                if (c == 0) out[orow + row] = from_f32<TIn>(fmaf(alpha, sq, u * kq));
            }
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const long off = (nh * DV + rbase + r * RPW) * (long)DK;
#pragma unroll
            for (int j = 0; j < CPL; ++j) __stcs(reinterpret_cast<float4 *>(state_out + off + 4 * (c + LPR * j)), s[r][j]);
        }
        __syncthreads();  // the token values of this head are read before the next head's overwrite them
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
    const long heads = (long)a.B * a.Hv;
    constexpr int kBytes = (int)sizeof(ScanSmem<DK, DV>);
    const auto kern = scan_tokens_kernel<DK, DV, TIn>;
    // resident CTAs per device for this instantiation, found once per device (0: not yet)
    static std::atomic<int> resident[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    int ctas = resident[dev].load(std::memory_order_relaxed);
    if (ctas == 0) {
        int sms = 0, per_sm = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kBytes);
        if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kDecodeThreads, kBytes);
        if (e != cudaSuccess) return e;
        ctas = sms * std::max(per_sm, 1);
        resident[dev].store(ctas, std::memory_order_relaxed);
    }
    const long blocks = std::min<long>(heads, (long)ctas);
    kern<<<(unsigned)blocks, kDecodeThreads, kBytes, s>>>(
        (const TIn *)a.q, (const TIn *)a.k, (const TIn *)a.v, (const TIn *)a.g, (const TIn *)a.b,
        a.state_in, a.state_out, (TIn *)a.out, a.B, a.T, a.Hk, a.Hv, a.status);
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
