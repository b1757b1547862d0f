// prefill_tc.cu -- block (chunk) form of the gated delta rule on the sm_103a
// tensor cores: TMA tile loads, tcgen05.mma into tensor memory (TMEM), fp32
// state carried on chip across all blocks of a sequence.
//
// The pages describe two evaluation orders of the recurrence: a direct token
// scan, or regrouping the updates into blocks that expose matrix products
// ("Optimiser l'inference sur appareil pour Apple Silicon", section "Qwen cree
// trois formes de charges de travail"), and they keep the recurrent state on
// chip for the whole scan, written back once (section "Maintenir l'etat
// recurrent sur la puce"). This kernel is the block order for dk = dv = 128,
// blocks of C = 64 tokens, bf16 I/O.
//
// Notation for one block of L <= 64 tokens of value head h, entering state S
// (dv x dk, fp32), raw bf16 tiles K, Q (C x dk) and V (C x dv), per-token
// rk, rq (inverse L2 norms), beta = sigmoid(b), G = in-block cumulative g,
// e_t = exp(G_t), d_t = exp(G_{L-1} - G_t), gamma = exp(G_{L-1}):
//   Gram:  [K; Q] K^T                      -> A_ts = beta_t rk_t rk_s e^{G_t-G_s} (K K^T)_ts, s < t
//                                             P_ts = rq_t rk_s e^{G_t-G_s} (Q K^T)_ts,         s <= t
//   solve: T = (I + A)^-1                  (blocked forward substitution, fp32, CUDA cores)
//          PT = P T                        (tensor cores)
//   chain: [Y; Y_q] = [K; Q] S^T           Z = diag(beta) (V - diag(e rk) Y)
//          [U; O_p] = [T; PT] Z            (so U = T diag(beta) V - T diag(beta e rk) K S^T,
//                                           O_p = P U)
//          O   = diag(e rq) Y_q + O_p      -> out (bf16)
//          S^T <- gamma S^T + K^T diag(d rk) U
// The raw K, Q, V tiles enter the MMAs exactly (bf16); every computed operand
// (S, T, PT, P, Z, U) is split into bf16 hi + lo parts and multiplied as
// hi*hi + hi*lo + lo*hi (or raw*hi + raw*lo), so each product keeps about
// 16 significant bits while the accumulation is fp32 in TMEM. The state itself
// stays in fp32 registers (thread j holds column j of S) and is never rounded.
//
// Rows t >= L of a partial block have beta = 0, rk = rq = 0 and d = 0, so they
// contribute nothing; their outputs are not stored.
#include <cuda.h>

#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "tc_ops.cuh"

namespace gdn {
namespace {

using namespace tc;

constexpr int C = 64;       // block length
constexpr int DK = 128;     // key dim
constexpr int DV = 128;     // value dim
constexpr int kThreads = 128;
constexpr long long kWaitBudget = 4000000000LL;  // SM cycles (about 2 s) before a wait gives up

// shared memory map, byte offsets from a 1 KiB aligned base
constexpr uint32_t OFF_KQ = 0;        // 32 KiB [kb 0..1][rows: K 0..63 | Q 64..127][128 B], TMA
constexpr uint32_t OFF_V = 32768;     // 16 KiB [kb 0..1][t 0..63][128 B], TMA
constexpr uint32_t OFF_SHI = 49152;   // 32 KiB S hi, MN-major [i-block 0..1][j 0..127][128 B]
constexpr uint32_t OFF_SLO = 81920;   // 32 KiB S lo
constexpr uint32_t OFF_PHI = 114688;  // 16 KiB P hi, K-major [t 0..127][128 B] (rows 64.. zero)
constexpr uint32_t OFF_PLO = 131072;  // 16 KiB P lo
constexpr uint32_t OFF_THI = 147456;  // 16 KiB [T; PT] hi, K-major [t 0..127][128 B]
constexpr uint32_t OFF_TLO = 163840;  // 16 KiB [T; PT] lo
constexpr uint32_t OFF_Z = 180224;    // 36 KiB: Z / U~ hi (16 KiB) + lo (16 KiB), MN-major
                                      //         [i-block 0..1][t 0..63][128 B];
                                      //         during the solve: A, T fp32 [64][64] + scratch
constexpr uint32_t OFF_SC = 217088;   // per-token scalars, 6 x 64 fp32
constexpr uint32_t OFF_BAR = OFF_SC + 6 * 64 * 4;
constexpr uint32_t SMEM_USED = OFF_BAR + 64;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;  // alignment slack
static_assert(SMEM_BYTES <= 232448, "over the 227 KiB opt-in limit");

// TMEM columns (512 allocated): Gram / PT, [Y; Y_q], [U; O_p], K^T U~
constexpr uint32_t TM_G = 0, TM_Y = 64, TM_U = 192, TM_S = 320;

constexpr uint32_t ID_N64 = idesc_bf16(128, 64, 0, 0);        // Gram
constexpr uint32_t ID_N64_BMN = idesc_bf16(128, 64, 0, 1);    // PT
constexpr uint32_t ID_N128_BMN = idesc_bf16(128, 128, 0, 1);  // Y, U
constexpr uint32_t ID_N128_AMN_BMN = idesc_bf16(128, 128, 1, 1);  // K^T U~

struct TcParams {
    const __nv_bfloat16 *g, *b;
    const float *state_in;
    float *state_out;
    __nv_bfloat16 *out;
    const int32_t *cu;
    int B, Hk, Hv;
    long T, Ttot;
    int *status;
};

// T = (I + A)^-1 for a unit lower-triangular 64 x 64 matrix, A strictly lower, row-major fp32.
// Diagonal 16 x 16 blocks by forward substitution (one column per thread), then the
// off-diagonal blocks by block diagonals: T_ij = -T_ii sum_{k=j}^{i-1} A_ik T_kj.
__device__ void solve_unit_lower(const float *sA, float *sT, float *sX, int tid) {
    if (tid < 64) {
        const int b = tid >> 4, c = tid & 15;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            float acc = (r == c) ? 1.f : 0.f;
#pragma unroll
            for (int s = 0; s < r; ++s) acc -= sA[(16 * b + r) * 64 + 16 * b + s] * x[s];
            x[r] = acc;
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) sT[(16 * b + r) * 64 + 16 * b + c] = x[r];
        for (int i = 0; i < b; ++i)
#pragma unroll
            for (int r = 0; r < 16; ++r) sT[(16 * i + r) * 64 + 16 * b + c] = 0.f;
    }
    __syncthreads();
    for (int d = 1; d < 4; ++d) {
        const int nb = 4 - d;
        for (int e = tid; e < nb * 256; e += kThreads) {
            const int blk = e >> 8, r = (e >> 4) & 15, c = e & 15;
            const int i = d + blk, j = blk;
            float acc = 0.f;
            for (int k = j; k < i; ++k)
#pragma unroll
                for (int m = 0; m < 16; ++m) acc += sA[(16 * i + r) * 64 + 16 * k + m] * sT[(16 * k + m) * 64 + 16 * j + c];
            sX[e] = acc;
        }
        __syncthreads();
        for (int e = tid; e < nb * 256; e += kThreads) {
            const int blk = e >> 8, r = (e >> 4) & 15, c = e & 15;
            const int i = d + blk, j = blk;
            float acc = 0.f;
#pragma unroll
            for (int m = 0; m < 16; ++m) acc += sT[(16 * i + r) * 64 + 16 * i + m] * sX[(blk << 8) + (m << 4) + c];
            sT[(16 * i + r) * 64 + 16 * j + c] = -acc;
        }
        __syncthreads();
    }
}

// S (thread j holds S[:, j]) -> hi/lo bf16, MN-major B operand rows j
__device__ __forceinline__ void store_state_hilo(uint8_t *sm, int j, const float (&S)[DV]) {
#pragma unroll
    for (int mb = 0; mb < 2; ++mb)
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            uint4 hi, lo;
            pack8_hilo(&S[mb * 64 + 8 * c], hi, lo);
            *reinterpret_cast<uint4 *>(sm + OFF_SHI + mb * 16384 + swz(j, c)) = hi;
            *reinterpret_cast<uint4 *>(sm + OFF_SLO + mb * 16384 + swz(j, c)) = lo;
        }
}

__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *sm = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const uint32_t sb = smem_u32(sm);
    float *rk_s = reinterpret_cast<float *>(sm + OFF_SC);
    float *rq_s = rk_s + 64, *beta_s = rq_s + 64, *G_s = beta_s + 64, *eG_s = G_s + 64, *dG_s = eG_s + 64;
    uint64_t *bar_tma = reinterpret_cast<uint64_t *>(sm + OFF_BAR);
    uint64_t *bar_mma = bar_tma + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar_mma + 1);
    int *abort_s = reinterpret_cast<int *>(tmem_slot + 1);
    float *sA = reinterpret_cast<float *>(sm + OFF_Z);
    float *sT = sA + 64 * 64;
    float *sX = sT + 64 * 64;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.x, n = blockIdx.y;
    const int hk = h / (p.Hv / p.Hk);
    long bos, eos;
    if (!seq_bounds(p.cu, n, p.B, p.cu ? p.Ttot : p.T, &bos, &eos, p.status)) return;

    if (tid == 0) {
        mbar_init(bar_tma, 1);
        mbar_init(bar_mma, 1);
        fence_mbar_init();
        *abort_s = 0;
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
    }
    if (warp == 0) tmem_alloc(tmem_slot, 512);
    {  // rows 64..127 of the P operand stay zero
        const uint4 z = make_uint4(0, 0, 0, 0);
        for (int i = tid; i < 512; i += kThreads) {
            reinterpret_cast<uint4 *>(sm + OFF_PHI + 8192)[i] = z;
            reinterpret_cast<uint4 *>(sm + OFF_PLO + 8192)[i] = z;
        }
    }
    float S[DV];  // column tid of the state
    const long st_off = ((long)n * p.Hv + h) * (long)DV * DK;
#pragma unroll
    for (int i = 0; i < DV; ++i) S[i] = p.state_in ? p.state_in[st_off + (long)i * DK + tid] : 0.f;
    store_state_hilo(sm, tid, S);
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    uint32_t ph_tma = 0, ph_mma = 0;
    bool aborted = false;

    auto wait_mma = [&]() {
        if (!mbar_wait(bar_mma, ph_mma, kWaitBudget)) *abort_s = 1;
        ph_mma ^= 1;
        tc_fence_after();
    };
    auto sync_for_mma = [&]() {  // make generic smem writes and TMEM reads visible before an MMA
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
    };

    for (long c0 = bos; c0 < eos; c0 += C) {
        const int L = (int)min((long)C, eos - c0);
        if (tid == 0) {
            mbar_expect_tx(bar_tma, 6 * 8192);
#pragma unroll
            for (int kb = 0; kb < 2; ++kb) {
                tma_load_3d(sm + OFF_KQ + kb * 16384, &tm_k, kb * 64, hk, (int)c0, bar_tma);
                tma_load_3d(sm + OFF_KQ + kb * 16384 + 8192, &tm_q, kb * 64, hk, (int)c0, bar_tma);
                tma_load_3d(sm + OFF_V + kb * 8192, &tm_v, kb * 64, h, (int)c0, bar_tma);
            }
        }
        if (tid < C) {
            const bool ok = tid < L;
            G_s[tid] = ok ? to_f32(p.g[(c0 + tid) * p.Hv + h]) : 0.f;
            beta_s[tid] = ok ? sigmoidf_(to_f32(p.b[(c0 + tid) * p.Hv + h])) : 0.f;
        }
        if (!mbar_wait(bar_tma, ph_tma, kWaitBudget)) *abort_s = 1;
        ph_tma ^= 1;
        __syncthreads();
        if (*abort_s) { aborted = true; break; }

        // inverse norms: warps 0-1 the K rows, warps 2-3 the Q rows
        {
            const int t = tid & 63;
            const uint32_t base = OFF_KQ + (tid >= 64 ? 8192u : 0u);
            float ss = 0.f;
#pragma unroll
            for (int kb = 0; kb < 2; ++kb)
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    float x[8];
                    unpack8(*reinterpret_cast<const uint4 *>(sm + base + kb * 16384 + swz(t, c)), x);
#pragma unroll
                    for (int e = 0; e < 8; ++e) ss += x[e] * x[e];
                }
            (tid >= 64 ? rq_s : rk_s)[t] = t < L ? rsqrtf(ss + kNormEps) : 0.f;
        }
        if (warp == 0) {  // in-block inclusive cumulative log-gate
            float x0 = G_s[lane], x1 = G_s[lane + 32];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y0 = __shfl_up_sync(0xffffffffu, x0, o);
                const float y1 = __shfl_up_sync(0xffffffffu, x1, o);
                if (lane >= o) { x0 += y0; x1 += y1; }
            }
            x1 += __shfl_sync(0xffffffffu, x0, 31);
            G_s[lane] = x0;
            G_s[lane + 32] = x1;
        }
        __syncthreads();
        const float GL = G_s[L - 1];
        if (tid < C) {
            eG_s[tid] = expf(G_s[tid]);
            dG_s[tid] = tid < L ? expf(GL - G_s[tid]) : 0.f;
        }

        // ---- Gram: [K; Q] K^T ----
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const uint32_t off = OFF_KQ + (s >> 2) * 16384 + (s & 3) * 32;
                mma_bf16(tmem + TM_G, desc_sw128(sb + off, 16, 1024), desc_sw128(sb + off, 16, 1024), ID_N64, s > 0);
            }
            mma_commit(bar_mma);
        }
        wait_mma();
        __syncthreads();
        if (*abort_s) { aborted = true; break; }

        // ---- A (fp32, for the solve) and P (hi/lo operand) ----
        {
            const int t = tid & 63;
            float row[64];
            {
                float v0[32], v1[32];
                tmem_ld32(tmem + TM_G + lane_off, v0);
                tmem_ld32(tmem + TM_G + lane_off + 32, v1);
#pragma unroll
                for (int s = 0; s < 32; ++s) { row[s] = v0[s]; row[32 + s] = v1[s]; }
            }
            const float Gt = G_s[t];
            if (tid < 64) {
                const float bt = beta_s[t] * rk_s[t];
#pragma unroll
                for (int s = 0; s < 64; ++s) {
                    const float a = bt * rk_s[s] * expf(Gt - G_s[s]) * row[s];
                    sA[t * 64 + s] = s < t ? a : 0.f;
                }
            } else {
                const float qt = rq_s[t];
#pragma unroll
                for (int s = 0; s < 64; ++s) {
                    const float pv = qt * rk_s[s] * expf(Gt - G_s[s]) * row[s];
                    row[s] = s <= t ? pv : 0.f;
                }
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint4 hi, lo;
                    pack8_hilo(&row[8 * c], hi, lo);
                    *reinterpret_cast<uint4 *>(sm + OFF_PHI + swz(t, c)) = hi;
                    *reinterpret_cast<uint4 *>(sm + OFF_PLO + swz(t, c)) = lo;
                }
            }
        }
        __syncthreads();

        // ---- T = (I + A)^-1, rows 0..63 of the [T; PT] operand ----
        solve_unit_lower(sA, sT, sX, tid);
        if (tid < 64) {
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                uint4 hi, lo;
                pack8_hilo(&sT[tid * 64 + 8 * c], hi, lo);
                *reinterpret_cast<uint4 *>(sm + OFF_THI + swz(tid, c)) = hi;
                *reinterpret_cast<uint4 *>(sm + OFF_TLO + swz(tid, c)) = lo;
            }
        }
        sync_for_mma();

        // ---- PT = P T (B = T rows as an MN-major operand) ----
        if (tid == 0) {
            tc_fence_after();
            const uint32_t a_op[3] = {OFF_PHI, OFF_PHI, OFF_PLO}, b_op[3] = {OFF_THI, OFF_TLO, OFF_THI};
            int first = 1;
#pragma unroll
            for (int m = 0; m < 3; ++m)
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    mma_bf16(tmem + TM_G, desc_sw128(sb + a_op[m] + s * 32, 16, 1024),
                             desc_sw128(sb + b_op[m] + s * 2048, 8192, 1024), ID_N64_BMN, !first);
                    first = 0;
                }
            mma_commit(bar_mma);
        }
        wait_mma();
        if (tid < 64) {  // rows 64..127 of [T; PT]
            float v0[32], v1[32];
            tmem_ld32(tmem + TM_G + lane_off, v0);
            tmem_ld32(tmem + TM_G + lane_off + 32, v1);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                uint4 hi, lo;
                pack8_hilo(c < 4 ? &v0[8 * c] : &v1[8 * (c - 4)], hi, lo);
                *reinterpret_cast<uint4 *>(sm + OFF_THI + swz(64 + tid, c)) = hi;
                *reinterpret_cast<uint4 *>(sm + OFF_TLO + swz(64 + tid, c)) = lo;
            }
        }
        sync_for_mma();
        if (*abort_s) { aborted = true; break; }

        // ---- [Y; Y_q] = [K; Q] S^T ----
        if (tid == 0) {
            tc_fence_after();
            int first = 1;
#pragma unroll
            for (int m = 0; m < 2; ++m)
#pragma unroll
                for (int s = 0; s < 8; ++s) {
                    const uint32_t a_off = OFF_KQ + (s >> 2) * 16384 + (s & 3) * 32;
                    const uint32_t b_off = (m == 0 ? OFF_SHI : OFF_SLO) + s * 2048;
                    mma_bf16(tmem + TM_Y, desc_sw128(sb + a_off, 16, 1024), desc_sw128(sb + b_off, 16384, 1024),
                             ID_N128_BMN, !first);
                    first = 0;
                }
            mma_commit(bar_mma);
        }
        wait_mma();
        // ---- Z = diag(beta) (V - diag(e rk) Y), rows t (warps 0-1) ----
        if (tid < 64) {
            const int t = tid;
            const float bt = beta_s[t], et = eG_s[t] * rk_s[t];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                float y[32];
                tmem_ld32(tmem + TM_Y + lane_off + 32 * q4, y);
                const int kb = q4 >> 1;
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    const int c = (q4 & 1) * 4 + cc;
                    float v8[8], z[8];
                    unpack8(*reinterpret_cast<const uint4 *>(sm + OFF_V + kb * 8192 + swz(t, c)), v8);
#pragma unroll
                    for (int e = 0; e < 8; ++e) z[e] = bt * (v8[e] - et * y[cc * 8 + e]);
                    uint4 hi, lo;
                    pack8_hilo(z, hi, lo);
                    *reinterpret_cast<uint4 *>(sm + OFF_Z + kb * 8192 + swz(t, c)) = hi;
                    *reinterpret_cast<uint4 *>(sm + OFF_Z + 16384 + kb * 8192 + swz(t, c)) = lo;
                }
            }
        }
        sync_for_mma();

        // ---- [U; O_p] = [T; PT] Z ----
        if (tid == 0) {
            tc_fence_after();
            const uint32_t a_op[3] = {OFF_THI, OFF_THI, OFF_TLO}, b_op[3] = {OFF_Z, OFF_Z + 16384, OFF_Z};
            int first = 1;
#pragma unroll
            for (int m = 0; m < 3; ++m)
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    mma_bf16(tmem + TM_U, desc_sw128(sb + a_op[m] + s * 32, 16, 1024),
                             desc_sw128(sb + b_op[m] + s * 2048, 8192, 1024), ID_N128_BMN, !first);
                    first = 0;
                }
            mma_commit(bar_mma);
        }
        wait_mma();
        if (tid < 64) {
            // U~ = diag(d rk) U, hi/lo, over the consumed Z operand
            const int t = tid;
            const float sc = dG_s[t] * rk_s[t];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                float u[32];
                tmem_ld32(tmem + TM_U + lane_off + 32 * q4, u);
                const int kb = q4 >> 1;
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    const int c = (q4 & 1) * 4 + cc;
                    float z[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) z[e] = sc * u[cc * 8 + e];
                    uint4 hi, lo;
                    pack8_hilo(z, hi, lo);
                    *reinterpret_cast<uint4 *>(sm + OFF_Z + kb * 8192 + swz(t, c)) = hi;
                    *reinterpret_cast<uint4 *>(sm + OFF_Z + 16384 + kb * 8192 + swz(t, c)) = lo;
                }
            }
        } else {
            // O = diag(e rq) Y_q + O_p, rows t = tid - 64
            const int t = tid - 64;
            const float sc = eG_s[t] * rq_s[t];
            __nv_bfloat16 *orow = p.out + ((c0 + t) * p.Hv + h) * (long)DV;
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                float yq[32], op[32];
                tmem_ld32(tmem + TM_Y + lane_off + 32 * q4, yq);
                tmem_ld32(tmem + TM_U + lane_off + 32 * q4, op);
                if (t < L) {
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        float o[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) o[e] = sc * yq[cc * 8 + e] + op[cc * 8 + e];
                        *reinterpret_cast<uint4 *>(orow + 32 * q4 + 8 * cc) = pack8(o);
                    }
                }
            }
        }
        sync_for_mma();

        // ---- S^T update: K^T U~ ----
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int m = 0; m < 2; ++m)
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    mma_bf16(tmem + TM_S, desc_sw128(sb + OFF_KQ + s * 2048, 16384, 1024),
                             desc_sw128(sb + OFF_Z + m * 16384 + s * 2048, 8192, 1024), ID_N128_AMN_BMN,
                             (m | s) != 0);
                }
            mma_commit(bar_mma);
        }
        wait_mma();
        {
            const float gam = expf(GL);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                float d[32];
                tmem_ld32(tmem + TM_S + lane_off + 32 * q4, d);
#pragma unroll
                for (int e = 0; e < 32; ++e) S[32 * q4 + e] = gam * S[32 * q4 + e] + d[e];
            }
        }
        store_state_hilo(sm, tid, S);
        sync_for_mma();
        if (*abort_s) { aborted = true; break; }
    }

    if (aborted) {
        if (tid == 0) flag_error(p.status);
    } else {
#pragma unroll
        for (int i = 0; i < DV; ++i) p.state_out[st_off + (long)i * DK + tid] = S[i];
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

// ---- host side ------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encoder() {
    static EncodeTiledFn fn = []() -> EncodeTiledFn {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<EncodeTiledFn>(f);
    }();
    return fn;
}

// [tokens][heads][dim] bf16 -> 3-D map, box (64 elements, 1 head, 64 tokens), 128B swizzle
bool make_map(CUtensorMap *m, const void *base, int dim, int heads, long tokens) {
    EncodeTiledFn enc = encoder();
    if (!enc) return false;
    const cuuint64_t gdim[3] = {(cuuint64_t)dim, (cuuint64_t)heads, (cuuint64_t)tokens};
    const cuuint64_t gstride[2] = {(cuuint64_t)dim * 2, (cuuint64_t)heads * dim * 2};
    const cuuint32_t box[3] = {64, 1, 64};
    const cuuint32_t estride[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), gdim, gstride, box, estride,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool prefill_tc_supported(const PrefillArgs &a) {
    const long Ttot = a.cu_seqlens ? (long)a.T : (long)a.B * a.T;
    return a.dtype == GDN_BF16 && a.dk == DK && a.dv == DV && a.chunk == C && Ttot > 0;
}

cudaError_t launch_prefill_tc(const PrefillArgs &a, cudaStream_t s) {
    const long Ttot = a.cu_seqlens ? (long)a.T : (long)a.B * a.T;
    CUtensorMap mq, mk, mv;
    if (!make_map(&mq, a.q, DK, a.Hk, Ttot) || !make_map(&mk, a.k, DK, a.Hk, Ttot) ||
        !make_map(&mv, a.v, DV, a.Hv, Ttot))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    TcParams p{(const __nv_bfloat16 *)a.g, (const __nv_bfloat16 *)a.b, a.state_in, a.state_out,
               (__nv_bfloat16 *)a.out, a.cu_seqlens, a.B, a.Hk, a.Hv, (long)a.T, Ttot, a.status};
    prefill_tc_kernel<<<dim3(a.Hv, a.B), kThreads, SMEM_BYTES, s>>>(mq, mk, mv, p);
    return cudaGetLastError();
}

}  // namespace gdn
