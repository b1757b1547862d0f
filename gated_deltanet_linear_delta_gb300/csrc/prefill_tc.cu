// prefill_tc.cu -- block (chunk) form of the gated delta rule on the sm_103a
// tensor cores: TMA tile loads, tcgen05.mma into tensor memory (TMEM), the fp32
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
// Per block of L <= 64 tokens of value head h, entering state S (dv x dk, fp32),
// with Kh, Qh the L2-normalised key/query rows, G the in-block cumulative log-gate,
// e_t = exp(G_t), d_t = exp(G_{L-1} - G_t), gamma = exp(G_{L-1}):
//   A_ts = beta_t e^{G_t-G_s} kh_t.kh_s (s < t),  P_ts = e^{G_t-G_s} qh_t.kh_s (s <= t)
//   T  = (I + A)^-1,  Tb = T diag(beta),  Tw = T diag(beta e)
//   W  = Tw Kh                           (C x dk)
//   U^T = V^T Tb^T - S W^T               (dv x C)      <- first state-dependent product
//   S  <- gamma S + U^T Kt,  Kt = diag(d) Kh           <- second state-dependent product
//   O^T = S Qt^T + U^T P^T,  Qt = diag(e) Qh           (dv x C)
// The state product is transposed so that the 128 state rows sit on the 128 TMEM
// lanes: one thread owns one row of S in fp32 registers for the whole sequence,
// and an fp16 copy of S is the A operand of the MMAs straight from TMEM.
//
// Work split: one thread-block cluster of P CTAs per value head (P = 4 when every head's
// cluster fits on the GPU at once, else 2, else 1; 512 threads each). Rank 0 carries the state.
//   * F = 0: every CTA prepares blocks (TMA of the raw K, Q, V tiles, norms and gates, fp16
//     conversion, the Gram MMA, A and P, the blocked triangular solve on CUDA cores, W by MMA);
//     helper ranks send their blocks' operands into the state CTA's shared memory by
//     distributed-shared-memory bulk copies, and rank 0's own threads 0..255 prepare the rest.
//     Threads 256..511 of rank 0 own the state (two threads per row) and issue its MMAs: per
//     block two dependent MMA round trips (U^T, then the state update) plus the output products.
//   * F = 1 (P >= 3): rank 0 prepares no blocks. Its K, Q, V tiles come by TMA and the helpers
//     send only Tb (as bf16 hi + lo), P, W and the block scalars; one thread issues every MMA,
//     256 threads hold the state, 128 write the outputs and 96 convert the Q rows.
// Stages and sent slots are handed over with mbarriers (full / empty, local or cluster scope);
// MMA completion is tracked with tcgen05.commit. The ring kernel (prefill_ring.cu) is the
// default for these sizes; this one runs when GDN_PREFILL_KERNEL=cluster.
//
// Numerics: MMAs multiply fp16 operands into fp32 accumulators, except where raw bf16 tiles
// (K, V) meet an operand that fp16 cannot carry exactly enough: there that operand (Tb, and U
// diag(d rk) in the state update) is split into bf16 hi + lo (about 16 significant bits) and
// both halves are multiplied. fp16 operands are scaled by an exact power of two before rounding
// (per block for V, Tb, Tw, W and P from their maxima; per row of S and U in the chain), which
// keeps every value in fp16's normal range and each product to about 2^-11 relative. Raw q/k
// are normalised before rounding.
//
// Rows t >= L of a partial block get zero kh, qh, beta, d, so they contribute
// nothing; their outputs are not stored.
#include <cuda.h>
#include <cstdio>
#include <cstdlib>
#include <cuda_fp16.h>

#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "tc_ops.cuh"

namespace gdn {
namespace {

using namespace tc;

constexpr int C = 64;     // block length
constexpr int DK = 128;   // key dim
constexpr int DV = 128;   // value dim
constexpr int kThreads = 512;
constexpr int kWG = 256;  // threads per warpgroup pair ("prep" 0..255, "chain" 256..511)
constexpr long long kWaitBudget = 4000000000LL;  // SM cycles (about 2 s) before a wait gives up

// ---- shared memory map (byte offsets from a 1 KiB aligned base) ----
// operand stage s (two of them), handed from prep to chain
constexpr uint32_t ST_KQ = 0;       // 32 KiB [kb 0..1][rows: Kh 0..63 | Qh 64..127][128 B] fp16
constexpr uint32_t ST_V = 32768;    // 16 KiB [i-block 0..1][t 0..63][128 B] fp16, scaled V
constexpr uint32_t ST_TB = 49152;   //  8 KiB [t][s] fp16, scaled Tb           } fp32 T during the solve
constexpr uint32_t ST_P = 57344;    //  8 KiB [t][s] fp16, scaled P            }
constexpr uint32_t ST_W = 65536;    // 16 KiB MN-major [j 0..127][64 t] fp16, scaled -W; fp32 A during the solve
constexpr uint32_t ST_SC = 81920;   //  1 KiB block scalars (below)
constexpr uint32_t STAGE = 82944;
// stage scalars (float index)
// SC_RK[t] = d_t rk_t and SC_RQ[t] = e_t rq_t turn raw K, Q rows into Kt, Qt; SC_SV = sig_v (V's scale)
constexpr int SC_RK = 0, SC_RQ = 64, SC_GAMMA = 128, SC_X1 = 129, SC_X2 = 130, SC_PO = 131, SC_L = 132, SC_SV = 133;
// What a helper sends when the state CTA converts the raw K, Q, V tiles itself: Tb, P, W and the scalars
constexpr uint32_t ST_SENT = ST_TB, SENT_BYTES = STAGE - ST_TB;
// A helper of a chain-only state CTA sends Tb as two bf16 tiles, Tb = hi + lo (hi = bf16(Tb),
// lo = bf16(Tb - hi), about 16 significant bits), which multiply the raw bf16 V tile directly;
// hi sits in the V region, which such a helper does not use, so the part sent is contiguous:
// [Tb hi | Tb lo | P | W | scalars].
constexpr uint32_t ST_TBH = ST_V + 8192;
constexpr uint32_t ST_RSENT = ST_TBH, RSENT_BYTES = STAGE - ST_TBH;
// shared memory of a chain-only state CTA (1 KiB aligned base as above)
constexpr uint32_t CO_RAW = 0;                          // [2] raw K|Q (32 KiB) and V (16 KiB); Q rows to fp16
constexpr uint32_t CO_RAW_BYTES = 49152;
constexpr uint32_t CO_SENT = 2 * CO_RAW_BYTES;          // [3] what the helpers send
constexpr uint32_t SN_TBH = ST_TBH - ST_RSENT, SN_TBL = ST_TB - ST_RSENT, SN_P = ST_P - ST_RSENT,
                   SN_W = ST_W - ST_RSENT, SN_SC = ST_SC - ST_RSENT;
constexpr uint32_t CO_SCL = CO_SENT + 3 * RSENT_BYTES;  // for O: row scales [2][128] x 2, P scale [2], L [2]
// prep-private
constexpr uint32_t RAW = 2 * STAGE;   // 48 KiB raw bf16 tiles: [kb][K rows 0..63 | Q rows 64..127] (32K), V (32K, 40K)
constexpr uint32_t TW = RAW + 49152;  //  8 KiB [t][s] fp16, scaled Tw; solve scratch X before
constexpr uint32_t PSC = TW + 8192;   // prep scalars (float index below)
constexpr int PS_G = 0, PS_BETA = 64, PS_AA = 128, PS_BB = 192, PS_EE = 256, PS_BE = 320, PS_DD = 384,
              PS_SS = 448 /* [2][128] */, PS_FACT = 704, PS_GMIN = 705, PS_GMAX = 706, PS_RK = 712, PS_RQ = 776,
              PS_RKB = 840, PS_RED = 904 /* [sites][8 warps][4] */;
constexpr int RED_V = 0, RED_TP = 1, RED_W = 2;  // reduction sites
constexpr uint32_t CSC = PSC + 4 * (PS_RED + 3 * 32);  // chain scratch: [2 sites][2 halves][128] floats
constexpr uint32_t BAR = CSC + 4 * 512;
constexpr uint32_t SMEM_USED = BAR + 256;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;  // alignment slack
static_assert(SMEM_BYTES <= 232448, "over the 227 KiB opt-in limit");
static_assert(CO_SCL + 4 * 528 <= CSC, "chain-only map overlaps the chain scratch");
static_assert(RSENT_BYTES % 1024 == 0, "sent slots keep the 1 KiB swizzle alignment");

// ---- TMEM columns (512 allocated) ----
constexpr uint32_t TM_GW = 0;     // prep: Gram, then W^T          (64)
constexpr uint32_t TM_X1 = 64;    // chain: V^T Tb^T               (64)
constexpr uint32_t TM_X2 = 128;   // chain: S (-W)^T, then U^T P^T (64)
constexpr uint32_t TM_Q = 192;    // chain: S Qh^T                 (64)
constexpr uint32_t TM_S = 256;    // chain: U~^T Kh                (128)
constexpr uint32_t TM_AS = 384;   // chain: fp16 S, A operand      (64 = 128 fp16)
constexpr uint32_t TM_AU = 448;   // chain: fp16 U^T               (32)
// a state CTA that prepares no blocks (its cluster's other CTAs do) keeps Q and O apart
// (X2 and O share columns: O(k) is issued after C has read X2(k), X2(k+1) after O has read O(k));
// AUH/AUL: bf16 hi/lo of U diag(d rk) for the state update, AUF: fp16 U for the outputs
constexpr uint32_t CT_X1 = 0, CT_X2O = 64, CT_Q = 128, CT_S = 192, CT_AS = 320, CT_AUH = 384, CT_AUL = 416,
                   CT_AUF = 448;

constexpr uint32_t ID_GRAM_BF16 = idesc_bf16(128, 64, 0, 0);
constexpr uint32_t ID_W = idesc_f16(128, 64, 1, 0);
constexpr uint32_t ID_X1 = idesc_f16(128, 64, 1, 0);
constexpr uint32_t ID_X2 = idesc_f16(128, 64, 0, 1);
constexpr uint32_t ID_Q = idesc_f16(128, 64, 0, 0);
constexpr uint32_t ID_S = idesc_f16(128, 128, 0, 1);
constexpr uint32_t ID_O = idesc_f16(128, 64, 0, 0);
constexpr uint32_t ID_X1_BF16 = idesc_bf16(128, 64, 1, 0);   // raw V^T x Tb hi/lo
constexpr uint32_t ID_S_BF16 = idesc_bf16(128, 128, 0, 1);   // U diag(d rk) hi/lo x raw K

struct TcParams {
    const __nv_bfloat16 *g, *b;
    const float *state_in;
    float *state_out;
    __nv_bfloat16 *out;
    const int32_t *cu;
    int B, Hk, Hv;
    long T, Ttot;
    int *status;
    int P;  // CTAs per value head (a thread-block cluster); rank 0 carries the state
    int F;  // first rank that prepares blocks: block k is prepared by rank F + k % (P - F)
};

// fp32 64 x 64 row-major with the column index XOR-swizzled by the row (keeps float4 groups)
__device__ __forceinline__ int sw(int t, int s) { return t * 64 + (s ^ ((t & 7) << 2)); }

// T = (I + A)^-1, A strictly lower 64 x 64 (swizzled fp32); 256 threads of one warpgroup pair.
// Diagonal 16 x 16 blocks by forward substitution (one column per thread), then the block
// diagonals T_ij = -T_ii sum_{k=j}^{i-1} A_ik T_kj, each thread owning 4 adjacent outputs.
__device__ void solve_unit_lower(const float *sA, float *sT, float *sX, int p, int bar_id) {
    if (p < 64) {
        const int b = p >> 4, c = p & 15;
        float x[16];  // column c of the block inverse, right-looking: independent updates per step
#pragma unroll
        for (int r = 0; r < 16; ++r) x[r] = (r == c) ? 1.f : 0.f;
#pragma unroll
        for (int s = 0; s < 15; ++s)
#pragma unroll
            for (int r = s + 1; r < 16; ++r) x[r] -= sA[sw(16 * b + r, 16 * b + s)] * x[s];
#pragma unroll
        for (int r = 0; r < 16; ++r) sT[sw(16 * b + r, 16 * b + c)] = x[r];
        for (int i = 0; i < b; ++i)
#pragma unroll
            for (int r = 0; r < 16; ++r) sT[sw(16 * i + r, 16 * b + c)] = 0.f;
    }
    bar_sync(bar_id, kWG);
    // Level d (blocks i = j + d): X_ij = sum_{k=j}^{i-1} A_ik T_kj, T_ij = -T_ii X_ij.
    // The X phase gives each (block, term k) its own 64 threads (4 adjacent outputs each), so
    // 192..256 threads work in every phase; the T phase adds the d partial products.
    // One copy of the level code (instruction fetch is a shared, contended resource when every
    // SM runs this), with the (block, term) split done without a division.
#pragma unroll 1
    for (int d = 1; d < 4; ++d) {
        const int nb = 4 - d;                   // blocks in this level
        const int slot = p >> 6;                // (block, term) pair handled by this thread
        const bool act = slot < nb * d;
        const int blk = d == 1 ? slot : (d == 2 ? slot >> 1 : 0), kk = slot - blk * d;
        const int r = (p >> 2) & 15, c0 = (p & 3) * 4;
        if (act) {
            const int i = d + blk, j = blk, k = j + kk;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f), acc2 = acc;
#pragma unroll
            for (int m = 0; m < 16; m += 2) {
                const float a = sA[sw(16 * i + r, 16 * k + m)], a2 = sA[sw(16 * i + r, 16 * k + m + 1)];
                const float4 t4 = *reinterpret_cast<const float4 *>(sT + sw(16 * k + m, 16 * j + c0));
                const float4 u4 = *reinterpret_cast<const float4 *>(sT + sw(16 * k + m + 1, 16 * j + c0));
                acc.x += a * t4.x; acc.y += a * t4.y; acc.z += a * t4.z; acc.w += a * t4.w;
                acc2.x += a2 * u4.x; acc2.y += a2 * u4.y; acc2.z += a2 * u4.z; acc2.w += a2 * u4.w;
            }
            *reinterpret_cast<float4 *>(sX + slot * 256 + r * 16 + c0) =
                make_float4(acc.x + acc2.x, acc.y + acc2.y, acc.z + acc2.z, acc.w + acc2.w);
        }
        bar_sync(bar_id, kWG);
        if (p < nb * 64) {
            const int tb = p >> 6, i = d + tb, j = tb;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int m = 0; m < 16; ++m) {
                const float a = sT[sw(16 * i + r, 16 * i + m)];
                float4 x4 = *reinterpret_cast<const float4 *>(sX + (tb * d) * 256 + m * 16 + c0);
#pragma unroll
                for (int q = 1; q < 3; ++q) {
                    if (q < d) {
                        const float4 y4 = *reinterpret_cast<const float4 *>(sX + (tb * d + q) * 256 + m * 16 + c0);
                        x4.x += y4.x; x4.y += y4.y; x4.z += y4.z; x4.w += y4.w;
                    }
                }
                acc.x += a * x4.x; acc.y += a * x4.y; acc.z += a * x4.z; acc.w += a * x4.w;
            }
            *reinterpret_cast<float4 *>(sT + sw(16 * i + r, 16 * j + c0)) = make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
        }
        bar_sync(bar_id, kWG);
    }
}

template <bool kChainOnly>  // rank 0 carries the state and prepares no blocks (F = 1)
__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *sm = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    const uint32_t sb = smem_u32(sm);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + BAR);
    uint64_t *bar_tma = bars + 0, *bar_prep = bars + 1, *bar_full = bars + 2, *bar_empty = bars + 4;
    uint64_t *bar_x = bars + 6, *bar_fin_p = bars + 7, *bar_s = bars + 8, *bar_o = bars + 9;
    uint64_t *bar_fin_c = bars + 11;  // a group's last MMAs, waited for before leaving after a give-up
    // handshakes of the state CTA when it prepares no blocks (kChainOnly)
    uint64_t *bar_as = bars + 12;  // fp16 S for the next block stored (8 warps)
    uint64_t *bar_u = bars + 13;   // [2] fp16 U of block k and the row scales stored (8 warps)
    uint64_t *bar_of = bars + 15;  // [2] output accumulators of block k read (4 warps)
    uint64_t *bar_tl = bars + 17;  // [2] raw K, Q, V tiles of raw slot k&1 loaded (TMA)
    uint64_t *bar_rd = bars + 19;  // [2] block k complete: raw tiles converted, helper's part landed (3 warps)
    uint64_t *bar_sent = bars + 21;  // [3] a helper's part landed in sent slot k%3 (bulk copy)
    uint64_t *bar_uo = bars + 24;    // [2] fp16 U of block k and what O needs of block k stored (8 warps)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 10);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int P = p.P, F = p.F, NP = P - F;
    const int rank = P > 1 ? (int)cluster_ctarank() : 0;
    const int h = blockIdx.x / P, n = longest_first(p.cu, p.B, blockIdx.y);
    const int hk = h / (p.Hv / p.Hk);
    long bos, eos;
    if (!seq_bounds(p.cu, n, p.B, p.cu ? p.Ttot : p.T, &bos, &eos, p.status)) return;
    const int nchunks = (int)((eos - bos + C - 1) / C);

    if (tid == 0) {
        mbar_init(bar_tma, 1);
        mbar_init(bar_prep, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar_full + s, 1);
            mbar_init(bar_empty + s, 1);
        }
        mbar_init(bar_x, 1);
        mbar_init(bar_fin_p, 1);
        mbar_init(bar_s, 1);
        mbar_init(bar_o, 1);
        mbar_init(bar_fin_c, 1);
        mbar_init(bar_as, 8);
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar_u + s, 8);
            mbar_init(bar_of + s, 4);
            mbar_init(bar_tl + s, 1);
            mbar_init(bar_rd + s, 3);
            mbar_init(bar_uo + s, 8);
        }
        for (int j = 0; j < 3; ++j) mbar_init(bar_sent + j, 1);
        if (kChainOnly && rank == 0)
            for (int j = 0; j < 5; ++j) reinterpret_cast<int *>(sm + CO_SCL + 4 * 516)[j] = 0;  // load/release counts
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(tmem_slot, 512);
    tc_fence_before();
    __syncthreads();
    if (P > 1) cluster_sync();  // every CTA's barriers are initialised before any remote arrive
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;  // this warp's TMEM lane quarter
    const int half = (tid >> 7) & 1;                              // which half of a row this thread owns
    const int r = tid & 127;                                      // TMEM lane = row

    if (tid < kWG && rank >= F && !(kChainOnly && rank == 0)) {
        // ======================= prep =======================
        // This CTA prepares blocks first, first + NP, ...; rank 0 writes them straight into its
        // stage k & 1, the other ranks into a local buffer (alternating two) that one bulk copy
        // moves into rank 0's stage once the chain has released it.
        const int pt = tid;
        const int first = rank - F;
        const bool local = rank == 0;
        // helpers of a chain-only state CTA leave Kt, Qt and V to it (it loads the raw tiles itself)
        const bool send_raw = kChainOnly && !local;
        uint32_t nwait[2] = {0u, 0u};  // completed waits on empty[0], empty[1]
        // Every wait gives up after kWaitBudget cycles and sets `ab` in the waiting thread; the group
        // leaves the loop together at the next bar_any. Tiles requested and not yet waited for are
        // waited for (bounded) before the CTA may leave.
        bool ab = false, failed = false;
        int tma_issued = 0, tma_waited = 0;
        float *ps = reinterpret_cast<float *>(sm + PSC);
        float *red = ps + PS_RED;
        uint32_t ph_prep = 0;
        // (a helper of a state-only CTA needs no V: the state CTA multiplies the raw V tile itself)
        auto issue_tma = [&](int c_tok) {
            mbar_expect_tx(bar_tma, (send_raw ? 4 : 6) * 8192);
#pragma unroll
            for (int kb = 0; kb < 2; ++kb) {
                tma_load_3d(sm + RAW + kb * 16384, &tm_k, kb * 64, hk, c_tok, bar_tma);
                tma_load_3d(sm + RAW + kb * 16384 + 8192, &tm_q, kb * 64, hk, c_tok, bar_tma);
                if (!send_raw) tma_load_3d(sm + RAW + 32768 + kb * 8192, &tm_v, kb * 64, h, c_tok, bar_tma);
            }
        };
        if (pt == 0 && first < nchunks) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            issue_tma((int)(bos + (long)first * C));
            tma_issued = 1;
        }
        // gates of the next block, fetched one block ahead and kept in bf16 until used, so that
        // the load's latency overlaps a whole block of work
        __nv_bfloat16 g_nx = __float2bfloat16(0.f), b_nx = __float2bfloat16(0.f);
        if (pt < C && first < nchunks && bos + (long)first * C + pt < eos) {
            g_nx = p.g[(bos + (long)first * C + pt) * p.Hv + h];
            b_nx = p.b[(bos + (long)first * C + pt) * p.Hv + h];
        }
        int jb = 0;  // this CTA's job count
        for (int k = first; k < nchunks; k += NP, ++jb) {
            const long c0 = bos + (long)k * C;
            const int L = (int)min((long)C, eos - c0);
            const int s = k & 1;               // rank 0's stage for block k
            const int sl = local ? s : jb & 1;  // where this CTA builds it
            uint8_t *st = sm + sl * STAGE;
            const uint32_t stb = sb + sl * STAGE;
            float *stsc = reinterpret_cast<float *>(st + ST_SC);
            float *sA = reinterpret_cast<float *>(st + ST_W);
            float *sT = reinterpret_cast<float *>(st + ST_TB);
            float *sX = reinterpret_cast<float *>(sm + TW);
            if (pt < C) {
                ps[PS_G + pt] = pt < L ? __bfloat162float(g_nx) : 0.f;
                ps[PS_BETA + pt] = pt < L ? sigmoidf_(__bfloat162float(b_nx)) : 0.f;
                const long cn = c0 + (long)NP * C + pt;
                if (k + NP < nchunks && cn < eos) {
                    g_nx = p.g[cn * p.Hv + h];
                    b_nx = p.b[cn * p.Hv + h];
                }
            }
            if (!mbar_wait(bar_tma, jb & 1, kWaitBudget)) ab = true;  // every reader of the tiles waits (asleep)
            tma_waited = jb + 1;
            if (pt == 0) {  // Gram [K; Q] K^T on the raw bf16 tiles (exact products), overlapping the norms
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint64_t d = desc_sw128(sb + RAW + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024);
                    mma_bf16(tmem + TM_GW, d, d, ID_GRAM_BF16, ks > 0);
                }
                mma_commit(bar_prep);
            }
            if (bar_any(1, kWG, ab)) { failed = true; break; }
            // ---- row norms (half a row per thread), V maximum; warp 0 also scans the gates ----
            const int row = r & 63;  // K rows for r < 64, Q rows for r >= 64
            const uint32_t raw_row = RAW + half * 16384;  // stacked row r of K-block `half`
            uint4 raw8[8];
            float ssq = 0.f;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                raw8[c] = *reinterpret_cast<const uint4 *>(sm + raw_row + swz(r, c));
                float x[8];
                unpack8(raw8[c], x);
#pragma unroll
                for (int e = 0; e < 8; ++e) ssq += x[e] * x[e];
            }
            ps[PS_SS + half * 128 + r] = ssq;
            const int vt = pt >> 2, vq = (pt & 3) * 4;  // V: row vt, chunks vq..vq+3 of 16
            uint4 rawv[4];
            float vmax = 0.f;
            if (!send_raw) {
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                const int c = vq + cc;
                rawv[cc] = *reinterpret_cast<const uint4 *>(sm + RAW + 32768 + (c >> 3) * 8192 + swz(vt, c & 7));
                float x[8];
                unpack8(rawv[cc], x);
#pragma unroll
                for (int e = 0; e < 8; ++e) vmax = fmaxf(vmax, fabsf(x[e]));
            }
            }
            vmax = warp_max(vt < L ? vmax : 0.f);
            if (lane == 0) red[RED_V * 32 + warp * 4] = vmax;
            if (warp == 0) {
                float x0 = ps[PS_G + lane], x1 = ps[PS_G + lane + 32];
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float y0 = __shfl_up_sync(0xffffffffu, x0, o);
                    const float y1 = __shfl_up_sync(0xffffffffu, x1, o);
                    if (lane >= o) { x0 += y0; x1 += y1; }
                }
                x1 += __shfl_sync(0xffffffffu, x0, 31);
                ps[PS_G + lane] = x0;
                ps[PS_G + lane + 32] = x1;
                float mn = fminf(x0, x1), mx = fmaxf(x0, x1);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                }
                if (lane == 0) {
                    ps[PS_GMIN] = mn;
                    ps[PS_GMAX] = mx;
                }
            }
            bar_sync(1, kWG);
            const float GL = ps[PS_G + L - 1];
            const float rnorm = row < L ? rsqrtf(ps[PS_SS + r] + ps[PS_SS + 128 + r] + kNormEps) : 0.f;
            float vm = 0.f;
#pragma unroll
            for (int w = 0; w < 8; ++w) vm = fmaxf(vm, red[RED_V * 32 + w * 4]);
            const float sig_v = pow2_scale(vm);
            if (half == 0) (r < 64 ? ps + PS_RK : ps + PS_RQ)[row] = rnorm;
            const float qscale = r < 64 ? rnorm : rnorm * expf(ps[PS_G + row]);  // Kh rows; Qt = e rq Q rows
            if (pt < C) {  // per-token exp factors, computed once
                const float gmin = ps[PS_GMIN], gmax = ps[PS_GMAX];
                const float G = ps[PS_G + pt];
                ps[PS_AA + pt] = expf(G - gmin);
                ps[PS_BB + pt] = expf(gmin - G);
                ps[PS_RKB + pt] = expf(gmin - G) * (pt < L ? rsqrtf(ps[PS_SS + pt] + ps[PS_SS + 128 + pt] + kNormEps) : 0.f);
                const float e = expf(G);
                ps[PS_EE + pt] = e;
                ps[PS_BE + pt] = ps[PS_BETA + pt] * e;
                ps[PS_DD + pt] = pt < L ? expf(GL - G) : 0.f;
                if (pt == 0) ps[PS_FACT] = (gmax - gmin) < 80.f ? 1.f : 0.f;  // a_t b_s = e^{G_t-G_s} safely
            }
            // ---- rank 0: wait until the chain released this stage (block k-2), then write fp16 operands ----
            if (local && k >= 2) {
                if (pt == 0 && !mbar_wait(bar_empty + s, nwait[s] & 1, kWaitBudget)) ab = true;
                ++nwait[s];
                if (bar_any(1, kWG, ab)) { failed = true; break; }
            }
            if (!send_raw || r < 64) {  // Kh rows (W needs them here), Qt rows
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    float x[8];
                    unpack8(raw8[c], x);
                    *reinterpret_cast<uint4 *>(st + ST_KQ + half * 16384 + swz(r, c)) = pack8_f16(x, qscale);
                }
            }
            if (!send_raw) {
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    const int c = vq + cc;
                    float x[8];
                    unpack8(rawv[cc], x);
                    *reinterpret_cast<uint4 *>(st + ST_V + (c >> 3) * 8192 + swz(vt, c & 7)) =
                        pack8_f16(x, vt < L ? sig_v : 0.f);
                }
            }
            fence_async_smem();
            tc_fence_before();
            bar_sync(1, kWG);
            if (pt == 0 && !mbar_wait(bar_prep, ph_prep, kWaitBudget)) ab = true;  // Gram done: raw tiles free
            ph_prep ^= 1;
            if (bar_any(1, kWG, ab)) { failed = true; break; }
            tc_fence_after();
            if (pt == 0 && k + NP < nchunks) {  // this CTA's next tiles
                issue_tma((int)(c0 + (long)NP * C));
                tma_issued = jb + 2;
            }
            // ---- A rows (fp32, swizzled, for the solve); P rows stay in registers ----
            const bool factor = ps[PS_FACT] != 0.f;
            float pv[32];
            float mp = 0.f;
            {
                float v0[16], v1[16];
                tmem_ld16(tmem + TM_GW + lane_off + 32 * half, v0);
                tmem_ld16(tmem + TM_GW + lane_off + 32 * half + 16, v1);
                const float at = ps[PS_AA + row], Gt = ps[PS_G + row];
                const float nt = r < 64 ? ps[PS_RK + row] * ps[PS_BETA + row] : ps[PS_RQ + row];
                const float bt = nt * at;
                if (factor) {  // uniform branch: e^{G_t-G_s} = a_t b_s
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        pv[e] = (e < 16 ? v0[e] : v1[e - 16]) * bt * ps[PS_RKB + 32 * half + e];
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        pv[e] = (e < 16 ? v0[e] : v1[e - 16]) * nt * ps[PS_RK + 32 * half + e] *
                                expf(Gt - ps[PS_G + 32 * half + e]);
                }
                if (r < 64) {
#pragma unroll
                    for (int e4 = 0; e4 < 8; ++e4) {
                        const int s2 = 32 * half + 4 * e4;
                        float4 a4;
                        a4.x = s2 + 0 < row ? pv[4 * e4 + 0] : 0.f;
                        a4.y = s2 + 1 < row ? pv[4 * e4 + 1] : 0.f;
                        a4.z = s2 + 2 < row ? pv[4 * e4 + 2] : 0.f;
                        a4.w = s2 + 3 < row ? pv[4 * e4 + 3] : 0.f;
                        *reinterpret_cast<float4 *>(sA + sw(row, s2)) = a4;
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        pv[e] = 32 * half + e <= row ? pv[e] : 0.f;
                        mp = fmaxf(mp, fabsf(pv[e]));
                    }
                }
            }
            tc_fence_before();
            bar_sync(1, kWG);
            // ---- T = (I + A)^-1 ----
            solve_unit_lower(sA, sT, sX, pt, 1);
            // ---- Tb, Tw (thread: row t, 16 columns), P scale; one reduction round ----
            const int tt = pt >> 2, q = pt & 3;
            float tb[16], tw[16];
            float mb = 0.f, mw = 0.f;
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
                const float4 t4 = *reinterpret_cast<const float4 *>(sT + sw(tt, 16 * q + 4 * c4));
                const float tv[4] = {t4.x, t4.y, t4.z, t4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int s2 = 16 * q + 4 * c4 + e;
                    tb[4 * c4 + e] = tv[e] * ps[PS_BETA + s2];
                    tw[4 * c4 + e] = tv[e] * ps[PS_BE + s2];
                    mb = fmaxf(mb, fabsf(tb[4 * c4 + e]));
                    mw = fmaxf(mw, fabsf(tw[4 * c4 + e]));
                }
            }
            mb = warp_max(mb);
            mw = warp_max(mw);
            mp = warp_max(mp);
            if (lane == 0) {
                red[RED_TP * 32 + warp * 4 + 0] = mb;
                red[RED_TP * 32 + warp * 4 + 1] = mw;
                red[RED_TP * 32 + warp * 4 + 2] = mp;
            }
            bar_sync(1, kWG);  // also: every read of T is done before Tb and P overwrite it
            float mbb = 0.f, mww = 0.f, mpp = 0.f;
#pragma unroll
            for (int w = 0; w < 8; ++w) {
                mbb = fmaxf(mbb, red[RED_TP * 32 + w * 4 + 0]);
                mww = fmaxf(mww, red[RED_TP * 32 + w * 4 + 1]);
                mpp = fmaxf(mpp, red[RED_TP * 32 + w * 4 + 2]);
            }
            const float sig_b = pow2_scale(mbb), sig_w = pow2_scale(mww), sig_p = pow2_scale(mpp);
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                if (send_raw) {  // Tb = hi + lo in bf16, unscaled
                    float lo[8];
                    const uint4 hi = pack8(&tb[8 * cc]);
                    float hv[8];
                    unpack8(hi, hv);
#pragma unroll
                    for (int e = 0; e < 8; ++e) lo[e] = tb[8 * cc + e] - hv[e];
                    *reinterpret_cast<uint4 *>(st + ST_TBH + swz(tt, 2 * q + cc)) = hi;
                    *reinterpret_cast<uint4 *>(st + ST_TB + swz(tt, 2 * q + cc)) = pack8(lo);
                } else {
                    *reinterpret_cast<uint4 *>(st + ST_TB + swz(tt, 2 * q + cc)) = pack8_f16(&tb[8 * cc], sig_b);
                }
                *reinterpret_cast<uint4 *>(sm + TW + swz(tt, 2 * q + cc)) = pack8_f16(&tw[8 * cc], sig_w);
            }
            if (r >= 64) {
#pragma unroll
                for (int cc = 0; cc < 4; ++cc)
                    *reinterpret_cast<uint4 *>(st + ST_P + swz(row, 4 * half + cc)) = pack8_f16(&pv[8 * cc], sig_p);
            }
            fence_async_smem();
            bar_sync(1, kWG);
            // ---- W^T = Kh^T Tw^T (scaled by sig_w) ----
            if (pt == 0) {
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_f16_ss(tmem + TM_GW, desc_sw128(stb + ST_KQ + ks * 2048, 16384, 1024),
                               desc_sw128(sb + TW + ks * 32, 16, 1024), ID_W, ks > 0);
                mma_commit(bar_prep);
            }
            if (pt == 0 && !mbar_wait(bar_prep, ph_prep, kWaitBudget)) ab = true;
            ph_prep ^= 1;
            if (bar_any(1, kWG, ab)) { failed = true; break; }
            tc_fence_after();
            {  // thread (j = r, half): W^T row j over t in this half -> MN-major row j of the -W operand
                float w0[16], w1[16];
                tmem_ld16(tmem + TM_GW + lane_off + 32 * half, w0);
                tmem_ld16(tmem + TM_GW + lane_off + 32 * half + 16, w1);
                float m = 0.f;
#pragma unroll
                for (int e = 0; e < 16; ++e) m = fmaxf(m, fmaxf(fabsf(w0[e]), fabsf(w1[e])));
                m = warp_max(m);
                if (lane == 0) red[RED_W * 32 + warp * 4] = m;
                bar_sync(1, kWG);
                float mm = 0.f;
#pragma unroll
                for (int w = 0; w < 8; ++w) mm = fmaxf(mm, red[RED_W * 32 + w * 4]);
                const float inv_w = 1.f / sig_w;
                const float sig_ww = pow2_scale(mm * inv_w);
                const float f = -sig_ww * inv_w;
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    *reinterpret_cast<uint4 *>(st + ST_W + swz(r, 4 * half + cc)) = pack8_f16(&w0[8 * cc], f);
                    *reinterpret_cast<uint4 *>(st + ST_W + swz(r, 4 * half + 2 + cc)) = pack8_f16(&w1[8 * cc], f);
                }
                if (!send_raw) {  // thread (row r < 64 of Kh, K-block half): scale by d_r in place
                    const int kr = r & 63, kh = (r >> 6) + 2 * half;  // 64 rows x 4 chunk groups
                    const float dr = ps[PS_DD + kr];
#pragma unroll
                    for (int c2 = 0; c2 < 2; ++c2) {
                        const int kb = kh >> 1, c = (kh & 1) * 4 + 2 * c2;
#pragma unroll
                        for (int cc = 0; cc < 2; ++cc) {
                            uint4 *pk = reinterpret_cast<uint4 *>(st + ST_KQ + kb * 16384 + swz(kr, c + cc));
                            uint4 v = *pk;
                            __half2 *hv = reinterpret_cast<__half2 *>(&v);
                            const __half2 d2 = __float2half2_rn(dr);
#pragma unroll
                            for (int e = 0; e < 4; ++e) hv[e] = __hmul2(hv[e], d2);
                            *pk = v;
                        }
                    }
                }
                if (pt < C) {
                    stsc[SC_RK + pt] = ps[PS_DD + pt] * ps[PS_RK + pt];
                    stsc[SC_RQ + pt] = ps[PS_EE + pt] * ps[PS_RQ + pt];
                }
                if (pt == 0) {
                    stsc[SC_GAMMA] = expf(GL);
                    stsc[SC_X1] = send_raw ? 1.f : 1.f / (sig_v * sig_b);
                    stsc[SC_X2] = 1.f / sig_ww;
                    stsc[SC_PO] = 1.f / sig_p;
                    stsc[SC_SV] = sig_v;
                    reinterpret_cast<int *>(stsc)[SC_L] = L;
                }
            }
            fence_async_smem();
            tc_fence_before();
            bar_sync(1, kWG);
            if (local) {
                if (pt == 0) mbar_arrive(bar_full + s);
            } else if (pt == 0 && send_raw) {
                // Tb, P, W and the scalars go to rank 0's sent slot k % 3, which is free once block
                // k-3 is consumed; one producer per slot (NP = 3), so the releases come in order.
                // (This buffer was last copied out two jobs ago, block k-6; the previous job's wait,
                // block k-6 consumed, already implied that copy had landed.)
                bool ok = true;
                if (k >= 3) {
                    ok = mbar_wait_cluster(bar_empty, nwait[0] & 1, kWaitBudget);
                    ++nwait[0];
                }
                if (!ok) {
                    ab = true;
                } else {
                    const uint32_t j = (uint32_t)(k % 3);
                    const uint32_t full_r = mapa_shared(smem_u32(bar_sent + j), 0);
                    mbar_arrive_expect_tx_cluster(full_r, RSENT_BYTES);
                    bulk_copy_to_cluster(mapa_shared(sb + CO_SENT + j * RSENT_BYTES, 0), st + ST_RSENT, RSENT_BYTES, full_r);
                }
            } else if (pt == 0) {
                // rank 0's stage s is free once the chain has finished block k-2. (This buffer was last
                // copied out two jobs ago, block k - 2 NP; the previous job's wait, block k - NP - 2
                // finished, already implied that copy had landed: NP >= 2 for every rank > 0.)
                bool ok = true;
                if (k >= 2) {
                    ok = mbar_wait_cluster(bar_empty + s, nwait[s] & 1, kWaitBudget);
                    ++nwait[s];
                }
                if (!ok) {
                    ab = true;
                } else {
                    const uint32_t full_r = mapa_shared(smem_u32(bar_full + s), 0);
                    const uint32_t dst_r = mapa_shared(sb + s * STAGE, 0);
                    mbar_arrive_expect_tx_cluster(full_r, STAGE);
#pragma unroll
                    for (uint32_t off = 0; off < STAGE; off += 16384)
                        bulk_copy_to_cluster(dst_r + off, st + off, min(16384u, STAGE - off), full_r);
                }
            }
            if (!local && bar_any(1, kWG, ab)) { failed = true; break; }
        }
        if (failed && pt == 0) {  // nothing of this group may still be in flight when the CTA leaves
            for (int j = tma_waited; j < tma_issued; ++j) mbar_wait(bar_tma, j & 1, kWaitBudget);
            mma_commit(bar_fin_p);
            mbar_wait(bar_fin_p, 0, kWaitBudget);
            flag_error(p.status);
        }
    } else if (kChainOnly && rank == 0) {
        // ============ state CTA of a cluster whose other CTAs prepare every block ============
        // Issuing tcgen05.mma holds the issuing thread until the tensor pipe has nearly finished
        // the batch, and a cluster-scope arrive waits for the thread's own outstanding global
        // stores; so each job has its own threads:
        //   C (threads 256..511): the state, two threads per row as above, waits on mbarriers only;
        //   I (thread 0): issues every MMA;
        //   O (threads 128..255, one row each): the bf16 outputs; its first thread also starts the
        //     raw tile loads of block k+2 and returns block k's sent slot once block k's MMAs are done;
        //   M (threads 32..127): converts the Q rows of each raw tile to Qt in fp16.
        // Operands between SMs move at about 21 B per cycle, TMA from L2 much faster, so the raw
        // K, Q, V tiles come by TMA and a helper sends only Tb (hi, lo), P, W and the scalars (41 KiB)
        // into one of three sent slots: its copy has two block periods to land. K and V are used raw
        // (bf16): Tb and U diag(d rk) are split into bf16 hi + lo to multiply them.
        // Per block k:  I: X1(k) X2(k) Q(k) -> C: U(k) -> I: S(k), O(k) -> C: state update, fp16 S(k+1)
        //   -> I: X1(k+1) X2(k+1) Q(k+1);  O: outputs of block k, loads block k+2.
        float *sgs = reinterpret_cast<float *>(sm + CO_SCL);  // [2][128] row scale of fp16 S(k)
        float *sgu = sgs + 256;                               // [2][128] row scale of fp16 U(k)
        float *spo = sgu + 256;                               // [2] P scale; [2] L (as int)
        int *req = reinterpret_cast<int *>(spo + 4);          // [2] raw loads requested per raw slot, [3] releases per sent slot
        auto raw_b = [&](int k) { return sb + CO_RAW + (uint32_t)(k & 1) * CO_RAW_BYTES; };
        auto sent_b = [&](int k) { return sb + CO_SENT + (uint32_t)(k % 3) * RSENT_BYTES; };
        auto load_raw = [&](int k) {  // raw bf16 K, Q, V tiles of block k into raw slot k&1
            uint8_t *rs = sm + CO_RAW + (k & 1) * CO_RAW_BYTES;
            const int c_tok = (int)(bos + (long)k * C);
            mbar_expect_tx(bar_tl + (k & 1), 6 * 8192);
#pragma unroll
            for (int kb = 0; kb < 2; ++kb) {
                tma_load_3d(rs + ST_KQ + kb * 16384, &tm_k, kb * 64, hk, c_tok, bar_tl + (k & 1));
                tma_load_3d(rs + ST_KQ + kb * 16384 + 8192, &tm_q, kb * 64, hk, c_tok, bar_tl + (k & 1));
                tma_load_3d(rs + ST_V + kb * 8192, &tm_v, kb * 64, h, c_tok, bar_tl + (k & 1));
            }
            ++req[k & 1];
        };
        if (tid == 0) {
            // ---------------- I ----------------
            bool ab = false;
            auto iwait = [&](uint64_t *bar, uint32_t ph) {
                if (!ab && !mbar_wait_spin(bar, ph, kWaitBudget)) ab = true;
                if (!ab) tc_fence_after();
                return !ab;
            };
            auto issue_x1 = [&](int k) {  // V^T (Tb hi + Tb lo)^T
#pragma unroll 1
                for (int ks = 0; ks < 4; ++ks) {
                    const uint64_t a = desc_sw128(raw_b(k) + ST_V + ks * 2048, 8192, 1024);
                    mma_bf16(tmem + CT_X1, a, desc_sw128(sent_b(k) + SN_TBH + ks * 32, 16, 1024), ID_X1_BF16, ks > 0);
                    mma_bf16(tmem + CT_X1, a, desc_sw128(sent_b(k) + SN_TBL + ks * 32, 16, 1024), ID_X1_BF16, 1);
                }
            };
            auto issue_x2 = [&](int k) {  // S (-W)^T
#pragma unroll 1
                for (int ks = 0; ks < 8; ++ks)
                    mma_f16_ts(tmem + CT_X2O, tmem + CT_AS + 8 * ks,
                               desc_sw128(sent_b(k) + SN_W + ks * 2048, 8192, 1024), ID_X2, ks > 0);
                mma_commit(bar_x);
            };
            auto issue_q = [&](int k) {  // S Qt^T
#pragma unroll 1
                for (int ks = 0; ks < 8; ++ks)
                    mma_f16_ts(tmem + CT_Q, tmem + CT_AS + 8 * ks,
                               desc_sw128(raw_b(k) + ST_KQ + (ks >> 2) * 16384 + 8192 + (ks & 3) * 32, 16, 1024), ID_Q,
                               ks > 0);
            };
            if (nchunks > 0) {
                if (iwait(bar_rd, 0)) issue_x1(0);
                if (iwait(bar_as, 0)) {
                    issue_x2(0);
                    issue_q(0);
                }
            }
            for (int k = 0; k < nchunks && !ab; ++k) {
                if (!iwait(bar_u + (k & 1), (k >> 1) & 1)) break;  // U diag(d rk) hi/lo stored; X1(k), X2(k) read
#pragma unroll 1
                for (int ks = 0; ks < 4; ++ks) {  // (hi + lo)^T K
                    const uint64_t b = desc_sw128(raw_b(k) + ST_KQ + ks * 2048, 16384, 1024);
                    mma_bf16_ts(tmem + CT_S, tmem + CT_AUH + 8 * ks, b, ID_S_BF16, ks > 0);
                    mma_bf16_ts(tmem + CT_S, tmem + CT_AUL + 8 * ks, b, ID_S_BF16, 1);
                }
                mma_commit(bar_s);
                if (!iwait(bar_uo + (k & 1), (k >> 1) & 1)) break;  // fp16 U stored
#pragma unroll 1
                for (int ks = 0; ks < 4; ++ks)  // U^T P^T
                    mma_f16_ts(tmem + CT_X2O, tmem + CT_AUF + 8 * ks, desc_sw128(sent_b(k) + SN_P + ks * 32, 16, 1024),
                               ID_O, ks > 0);
                mma_commit(bar_o);  // every MMA of block k
                if (k + 1 < nchunks) {
                    if (!iwait(bar_rd + ((k + 1) & 1), ((k + 1) >> 1) & 1)) break;
                    issue_x1(k + 1);
                    if (!iwait(bar_as, (k + 1) & 1)) break;             // fp16 S(k+1) stored
                    if (!iwait(bar_of + (k & 1), (k >> 1) & 1)) break;  // O(k) and Q(k) read
                    issue_x2(k + 1);
                    issue_q(k + 1);
                }
            }
            mma_commit(bar_fin_c);  // nothing issued here may still run when the CTA leaves
            mbar_wait(bar_fin_c, 0, kWaitBudget);
            if (ab) flag_error(p.status);
        } else if (tid >= 32 && tid < 128) {
            // ---------------- M ----------------
            bool ab = false, failed = false;
            if (tid == 32) {
                prefetch_tmap(&tm_q);
                prefetch_tmap(&tm_k);
                prefetch_tmap(&tm_v);
                for (int k = 0; k < 2 && k < nchunks; ++k) load_raw(k);
            }
            for (int k = 0; k < nchunks; ++k) {
                if (!ab && !mbar_wait(bar_tl + (k & 1), (k >> 1) & 1, kWaitBudget)) ab = true;
                if (!ab && !mbar_wait(bar_sent + k % 3, (k / 3) & 1, kWaitBudget)) ab = true;
                if (bar_any(4, 96, ab)) {
                    failed = true;
                    break;
                }
                uint8_t *rs = sm + CO_RAW + (k & 1) * CO_RAW_BYTES;
                const float *stsc = reinterpret_cast<const float *>(sm + CO_SENT + (k % 3) * RSENT_BYTES + SN_SC);
                // Q rows 64..127 of the two 64-column halves: 1024 chunks of 16 B, consecutive threads on
                // consecutive chunks (row = chunk / 8; the swizzle only permutes chunks within a row)
#pragma unroll
                for (int i0 = 0; i0 < 11; i0 += 4) {
                    uint4 v[4];
                    float f[4];
                    uint32_t off[4];
#pragma unroll
                    for (int ii = 0; ii < 4; ++ii) {
                        const int m = (tid - 32) + 96 * (i0 + ii);
                        const int row = 64 + ((m >> 3) & 63);
                        off[ii] = (uint32_t)((m >> 9) * 16384 + row * 128 + (m & 7) * 16);
                        f[ii] = stsc[SC_RQ + row - 64];
                        if (m < 1024) v[ii] = *reinterpret_cast<const uint4 *>(rs + off[ii]);
                    }
#pragma unroll
                    for (int ii = 0; ii < 4; ++ii) {
                        const int m = (tid - 32) + 96 * (i0 + ii);
                        if (m < 1024) {
                            float x[8];
                            unpack8(v[ii], x);
                            *reinterpret_cast<uint4 *>(rs + off[ii]) =
                                f[ii] != 0.f ? pack8_f16(x, f[ii]) : make_uint4(0u, 0u, 0u, 0u);
                        }
                    }
                }
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_rd + (k & 1));
            }
            if (failed && tid == 32) flag_error(p.status);
        } else if (tid >= 128 && tid < kWG) {
            // ---------------- O ----------------
            const int i = tid & 127;
            bool ab = false, failed = false;
            for (int k = 0; k < nchunks; ++k) {
                const long c0 = bos + (long)k * C;
                if (!ab && !mbar_wait(bar_o, k & 1, kWaitBudget)) ab = true;
                if (!ab && !mbar_wait(bar_uo + (k & 1), (k >> 1) & 1, kWaitBudget)) ab = true;  // scales from C
                __syncwarp();
                tc_fence_after();
                const float fq = 1.f / sgs[(k & 1) * 128 + i], fo = spo[k & 1] / sgu[(k & 1) * 128 + i];
                const int L = reinterpret_cast<const int *>(spo)[2 + (k & 1)];
                uint32_t opk[32];  // outputs t = 0..63 of row i, bf16 pairs
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint32_t qa[16], oa[16];
                    tmem_ld16_nw(tmem + CT_Q + lane_off + 16 * q, qa);
                    tmem_ld16_nw(tmem + CT_X2O + lane_off + 16 * q, oa);
                    tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const float o0 = __uint_as_float(qa[2 * c]) * fq + __uint_as_float(oa[2 * c]) * fo;
                        const float o1 = __uint_as_float(qa[2 * c + 1]) * fq + __uint_as_float(oa[2 * c + 1]) * fo;
                        opk[8 * q + c] = bf2_bits(__floats2bfloat162_rn(o0, o1));
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_of + (k & 1));
                if (tid == 128 && !ab) {
                    // every MMA of block k is done (bar_o) and C read its scalars before fp16 U (bar_uo);
                    // M read them before block k was ready: raw slot k&1 and sent slot k%3 are free
                    if (k + 2 < nchunks) load_raw(k + 2);
                    if (k + 3 < nchunks) {
                        ++req[2 + k % 3];
                        mbar_arrive_cluster(mapa_shared(smem_u32(bar_empty), (uint32_t)(F + (k + 3) % NP)));
                    }
                }
                if (bar_any(3, 128, ab)) {
                    failed = true;
                    break;
                }
                __nv_bfloat16 *ob = p.out + (c0 * p.Hv + h) * (long)DV + i;
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const int t = 2 * c;
                    if (t < L) ob[(long)t * p.Hv * DV] = __ushort_as_bfloat16((unsigned short)(opk[c] & 0xffffu));
                    if (t + 1 < L) ob[(long)(t + 1) * p.Hv * DV] = __ushort_as_bfloat16((unsigned short)(opk[c] >> 16));
                }
            }
            if (failed && tid == 128) flag_error(p.status);
        } else if (tid >= kWG) {
            // ---------------- C ----------------
            const int i = r;
            float *cx = reinterpret_cast<float *>(sm + CSC);
            float S[64];
            const long st_off = ((long)n * p.Hv + h) * (long)DV * DK + (long)i * DK + 64 * half;
            if (p.state_in) {
#pragma unroll
                for (int j = 0; j < 64; j += 4) {
                    const float4 v = *reinterpret_cast<const float4 *>(p.state_in + st_off + j);
                    S[j] = v.x; S[j + 1] = v.y; S[j + 2] = v.z; S[j + 3] = v.w;
                }
            } else {
#pragma unroll
                for (int j = 0; j < 64; ++j) S[j] = 0.f;
            }
            bool ab = false, failed = false;
            auto cwait = [&](uint64_t *bar, uint32_t ph) {
                if (!ab && !mbar_wait_spin(bar, ph, kWaitBudget)) ab = true;
                __syncwarp();
                tc_fence_after();
            };
            auto warp_arrive = [&](uint64_t *bar) {  // this warp's TMEM stores (and smem writes) are done
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar);
            };
            auto row_scale = [&](float m, int site) {
                cx[site * 256 + half * 128 + i] = m;
                bar_sync(6 + (warp & 3), 64);  // the two halves of a row sit in warps w and w+4
                return pow2_scale(fmaxf(cx[site * 256 + i], cx[site * 256 + 128 + i]));
            };
            auto smax = [&]() {
                float m = 0.f;
#pragma unroll
                for (int j = 0; j < 64; ++j) m = fmaxf(m, fabsf(S[j]));
                return m;
            };
            auto store_state_f16 = [&](float sc) {
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) {
                    uint32_t rr[8];
#pragma unroll
                    for (int c = 0; c < 8; ++c) rr[c] = h2_bits(sc * S[16 * c8 + 2 * c], sc * S[16 * c8 + 2 * c + 1]);
                    tmem_st8(tmem + CT_AS + lane_off + 32 * half + 8 * c8, rr);
                }
            };
            float sig_s = row_scale(smax(), 0);
            if (nchunks > 0) {
                store_state_f16(sig_s);
                warp_arrive(bar_as);
            }
            for (int k = 0; k < nchunks; ++k) {
                const float *stsc = reinterpret_cast<const float *>(sm + CO_SENT + (k % 3) * RSENT_BYTES + SN_SC);
                cwait(bar_rd + (k & 1), (k >> 1) & 1);  // block k's scalars (long since there)
                cwait(bar_x, k & 1);                     // X1(k), X2(k)
                const float f1 = stsc[SC_X1], f2 = stsc[SC_X2] / sig_s, gam = stsc[SC_GAMMA];
                float u[32];  // U^T[i][t], t in [32 half, 32 half + 32)
                float m = 0.f;
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    uint32_t a[16], bx[16];
                    tmem_ld16_nw(tmem + CT_X1 + lane_off + 32 * half + 16 * q, a);
                    tmem_ld16_nw(tmem + CT_X2O + lane_off + 32 * half + 16 * q, bx);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e) u[16 * q + e] = __uint_as_float(a[e]) * f1 + __uint_as_float(bx[e]) * f2;
                }
                // the state update's operand first: U diag(d rk) as bf16 hi + lo (no scaling needed)
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    uint32_t rh[8], rl[8];
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const int e = 16 * q + 2 * c;
                        const float x0 = u[e] * stsc[SC_RK + 32 * half + e], x1 = u[e + 1] * stsc[SC_RK + 32 * half + e + 1];
                        const __nv_bfloat162 hb = __floats2bfloat162_rn(x0, x1);
                        const float2 hf = __bfloat1622float2(hb);
                        rh[c] = bf2_bits(hb);
                        rl[c] = bf2_bits(__floats2bfloat162_rn(x0 - hf.x, x1 - hf.y));
                    }
                    tmem_st8(tmem + CT_AUH + lane_off + 16 * half + 8 * q, rh);
                    tmem_st8(tmem + CT_AUL + lane_off + 16 * half + 8 * q, rl);
                }
                warp_arrive(bar_u + (k & 1));
                // then fp16 U for the outputs (row scale), and what O needs of this block
#pragma unroll
                for (int e = 0; e < 32; ++e) m = fmaxf(m, fabsf(u[e]));
                const float sig_u = row_scale(m, 1);
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    uint32_t ru[8];
#pragma unroll
                    for (int c = 0; c < 8; ++c) ru[c] = h2_bits(sig_u * u[16 * q + 2 * c], sig_u * u[16 * q + 2 * c + 1]);
                    tmem_st8(tmem + CT_AUF + lane_off + 16 * half + 8 * q, ru);
                }
                if (half == 0) {
                    sgs[(k & 1) * 128 + i] = sig_s;
                    sgu[(k & 1) * 128 + i] = sig_u;
                }
                if (tid == kWG) {
                    spo[k & 1] = stsc[SC_PO];
                    reinterpret_cast<int *>(spo)[2 + (k & 1)] = reinterpret_cast<const int *>(stsc)[SC_L];
                }
                warp_arrive(bar_uo + (k & 1));
                cwait(bar_s, k & 1);  // (hi + lo)^T K
#pragma unroll
                for (int q2 = 0; q2 < 2; ++q2) {
                    uint32_t d0[16], d1[16];
                    tmem_ld16_nw(tmem + CT_S + lane_off + 64 * half + 32 * q2, d0);
                    tmem_ld16_nw(tmem + CT_S + lane_off + 64 * half + 32 * q2 + 16, d1);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        S[32 * q2 + e] = gam * S[32 * q2 + e] + __uint_as_float(d0[e]);
                        S[32 * q2 + 16 + e] = gam * S[32 * q2 + 16 + e] + __uint_as_float(d1[e]);
                    }
                }
                sig_s = row_scale(smax(), 0);
                if (k + 1 < nchunks) {
                    store_state_f16(sig_s);
                    warp_arrive(bar_as);
                }
                if (bar_any(2, kWG, ab)) {
                    failed = true;
                    break;
                }
            }
            if (failed) {
                if (tid == kWG) flag_error(p.status);
            } else {
#pragma unroll
                for (int j = 0; j < 64; j += 4)
                    *reinterpret_cast<float4 *>(p.state_out + st_off + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
            }
        }
    } else if (tid >= kWG && rank == 0) {
        // ======================= chain =======================
        const int i = r;             // state row (TMEM lane)
        const bool issuer = (tid == kWG);
        float *cx = reinterpret_cast<float *>(sm + CSC);  // [2 sites][2 halves][128]
        float S[64];                 // S[i][64 half .. 64 half + 63]
        const long st_off = ((long)n * p.Hv + h) * (long)DV * DK + (long)i * DK + 64 * half;
        if (p.state_in) {
#pragma unroll
            for (int j = 0; j < 64; j += 4) {
                const float4 v = *reinterpret_cast<const float4 *>(p.state_in + st_off + j);
                S[j] = v.x; S[j + 1] = v.y; S[j + 2] = v.z; S[j + 3] = v.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 64; ++j) S[j] = 0.f;
        }
        // One thread polls the mbarrier (sleeping), the other 255 wait on the group barrier. A wait
        // that gives up sets `ab` in the issuer, which stops issuing; the group leaves the loop
        // together at its next bar_any.
        bool ab = false, failed = false;
        auto group_wait = [&](uint64_t *bar, uint32_t phase) {
            if (issuer && !ab && !mbar_wait(bar, phase, kWaitBudget)) ab = true;
            bar_sync(2, kWG);
        };
        // per-row power-of-two scale: both halves' maxima through shared memory
        auto row_scale = [&](float m, int site) {
            cx[site * 256 + half * 128 + i] = m;
            bar_sync(2, kWG);
            return pow2_scale(fmaxf(cx[site * 256 + i], cx[site * 256 + 128 + i]));
        };
        auto smax = [&]() {
            float m = 0.f;
#pragma unroll
            for (int j = 0; j < 64; ++j) m = fmaxf(m, fabsf(S[j]));
            return m;
        };
        auto store_state_f16 = [&](float sc) {  // 64 values of row i -> 32 columns of the A operand
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8) {
                uint32_t rr[8];
#pragma unroll
                for (int c = 0; c < 8; ++c) rr[c] = h2_bits(sc * S[16 * c8 + 2 * c], sc * S[16 * c8 + 2 * c + 1]);
                tmem_st8(tmem + TM_AS + lane_off + 32 * half + 8 * c8, rr);
            }
        };
        auto issue_x2 = [&](int k) {  // S(-W)^T for block k: the state's critical product
            const uint32_t stb = sb + (k & 1) * STAGE;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                mma_f16_ts(tmem + TM_X2, tmem + TM_AS + 8 * ks, desc_sw128(stb + ST_W + ks * 2048, 8192, 1024), ID_X2,
                           ks > 0);
            mma_commit(bar_x);
        };
        auto issue_q = [&](int k) {  // S Qt^T for block k (outputs only)
            const uint32_t stb = sb + (k & 1) * STAGE;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                mma_f16_ts(tmem + TM_Q, tmem + TM_AS + 8 * ks,
                           desc_sw128(stb + ST_KQ + (ks >> 2) * 16384 + 8192 + (ks & 3) * 32, 16, 1024), ID_Q, ks > 0);
        };
        auto issue_x1 = [&](int k) {  // V^T Tb^T for block k (state independent)
            const uint32_t stb = sb + (k & 1) * STAGE;
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                mma_f16_ss(tmem + TM_X1, desc_sw128(stb + ST_V + ks * 2048, 8192, 1024),
                           desc_sw128(stb + ST_TB + ks * 32, 16, 1024), ID_X1, ks > 0);
        };

        float sig_s = row_scale(smax(), 0);
        bool x1_next = false;  // issuer only: the next block's V^T Tb^T is already issued
        if (nchunks > 0) {
            group_wait(bar_full + 0, 0);
            store_state_f16(sig_s);
            tmem_wait_st();
            tc_fence_before();
            bar_sync(2, kWG);
            if (issuer && !ab) {
                tc_fence_after();
                issue_x1(0);
                issue_x2(0);
            }
        }
        for (int k = 0; k < nchunks; ++k) {
            const long c0 = bos + (long)k * C;
            const float *stsc = reinterpret_cast<const float *>(sm + (k & 1) * STAGE + ST_SC);
            group_wait(bar_full + (k & 1), (k >> 1) & 1);  // scalars of block k
            // ---- E1: U^T = X1 / (sig_v sig_b) + X2 / (sig_s sig_ww) -> fp16 U~^T, U^T (columns t of this half) ----
            group_wait(bar_x, k & 1);
            tc_fence_after();
            const float f1 = stsc[SC_X1], f2 = stsc[SC_X2] / sig_s;
            float u[32];  // U^T[i][t], t in [32 half, 32 half + 32)
            float m = 0.f;
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                uint32_t a[16], bx[16];
                tmem_ld16_nw(tmem + TM_X1 + lane_off + 32 * half + 16 * q, a);
                tmem_ld16_nw(tmem + TM_X2 + lane_off + 32 * half + 16 * q, bx);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const float uv = __uint_as_float(a[e]) * f1 + __uint_as_float(bx[e]) * f2;
                    u[16 * q + e] = uv;
                    m = fmaxf(m, fabsf(uv));
                }
            }
            const float sig_u = row_scale(m, 1);
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                uint32_t ru[8];
#pragma unroll
                for (int c = 0; c < 8; ++c) ru[c] = h2_bits(sig_u * u[16 * q + 2 * c], sig_u * u[16 * q + 2 * c + 1]);
                tmem_st8(tmem + TM_AU + lane_off + 16 * half + 8 * q, ru);
            }
            tmem_wait_st();
            tc_fence_before();
            if (bar_any(2, kWG, ab)) { failed = true; break; }
            if (issuer) {
                tc_fence_after();
                const uint32_t stb = sb + (k & 1) * STAGE;
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)  // U^T Kt  (B = diag(d) Kh rows, MN-major)
                    mma_f16_ts(tmem + TM_S, tmem + TM_AU + 8 * ks, desc_sw128(stb + ST_KQ + ks * 2048, 16384, 1024),
                               ID_S, ks > 0);
                mma_commit(bar_s);
                issue_q(k);  // outputs: behind the state update in the tensor pipe
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)  // U^T P^T
                    mma_f16_ts(tmem + TM_X2, tmem + TM_AU + 8 * ks, desc_sw128(stb + ST_P + ks * 32, 16, 1024), ID_O,
                               ks > 0);
                mma_commit(bar_o);  // covers Q and O
                // the next block's state-independent V^T Tb^T, now if its operands are already there
                // (TM_X1 was read in E1); otherwise just before the next S(-W)^T
                x1_next = false;
                if (k + 1 < nchunks && mbar_try_wait(bar_full + ((k + 1) & 1), ((k + 1) >> 1) & 1)) {
                    issue_x1(k + 1);
                    x1_next = true;
                }
            }
            // ---- E2: state update (columns j of this half), next A operand, outputs ----
            group_wait(bar_s, k & 1);
            tc_fence_after();
            const float gam = stsc[SC_GAMMA];
            const float inv_u = 1.f / sig_u;
#pragma unroll
            for (int q2 = 0; q2 < 2; ++q2) {
                uint32_t d0[16], d1[16];
                tmem_ld16_nw(tmem + TM_S + lane_off + 64 * half + 32 * q2, d0);
                tmem_ld16_nw(tmem + TM_S + lane_off + 64 * half + 32 * q2 + 16, d1);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    S[32 * q2 + e] = gam * S[32 * q2 + e] + __uint_as_float(d0[e]) * inv_u;
                    S[32 * q2 + 16 + e] = gam * S[32 * q2 + 16 + e] + __uint_as_float(d1[e]) * inv_u;
                }
            }
            const float sig_s_old = sig_s;
            sig_s = row_scale(smax(), 0);
            const bool more = k + 1 < nchunks;
            group_wait(bar_o, k & 1);  // Q and O of block k: A_S is free
            tc_fence_after();
            if (more) store_state_f16(sig_s);
            uint32_t opk[16];  // outputs for t in [32 half, 32 half + 32), bf16 pairs
            {
                const float fq = 1.f / sig_s_old, fo = stsc[SC_PO] * inv_u;
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    uint32_t qa[16], oa[16];
                    tmem_ld16_nw(tmem + TM_Q + lane_off + 32 * half + 16 * q, qa);
                    tmem_ld16_nw(tmem + TM_X2 + lane_off + 32 * half + 16 * q, oa);
                    tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const float o0 = __uint_as_float(qa[2 * c]) * fq + __uint_as_float(oa[2 * c]) * fo;
                        const float o1 = __uint_as_float(qa[2 * c + 1]) * fq + __uint_as_float(oa[2 * c + 1]) * fo;
                        opk[8 * q + c] = bf2_bits(__floats2bfloat162_rn(o0, o1));
                    }
                }
            }
            const int L = reinterpret_cast<const int *>(stsc)[SC_L];
            tmem_wait_st();
            tc_fence_before();
            if (bar_any(2, kWG, ab)) { failed = true; break; }
            if (issuer && k + 2 < nchunks) {  // every MMA of block k has completed, scalars read:
                const int to = F + (k + 2) % NP;  // release stage k & 1 to the producer of block k + 2
                if (to == 0)
                    mbar_arrive(bar_empty + (k & 1));
                else
                    mbar_arrive_cluster(mapa_shared(smem_u32(bar_empty + (k & 1)), (uint32_t)to));
            }
            if (issuer) {
                if (more) {
                    if (!x1_next) {
                        if (!mbar_wait(bar_full + ((k + 1) & 1), ((k + 1) >> 1) & 1, kWaitBudget)) ab = true;
                        tc_fence_after();
                        if (!ab) issue_x1(k + 1);
                    }
                    tc_fence_after();
                    if (!ab) issue_x2(k + 1);
                }
            }
            // outputs of block k (off the state's critical path)
            __nv_bfloat16 *ob = p.out + (c0 * p.Hv + h) * (long)DV + i;
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const int t = 32 * half + 2 * c;
                if (t < L) ob[(long)t * p.Hv * DV] = __ushort_as_bfloat16((unsigned short)(opk[c] & 0xffffu));
                if (t + 1 < L) ob[(long)(t + 1) * p.Hv * DV] = __ushort_as_bfloat16((unsigned short)(opk[c] >> 16));
            }
        }
        if (failed) {
            if (issuer) {  // nothing of this group may still be in flight when the CTA leaves
                mma_commit(bar_fin_c);
                mbar_wait(bar_fin_c, 0, kWaitBudget);
                flag_error(p.status);
            }
        } else {
#pragma unroll
            for (int j = 0; j < 64; j += 4)
                *reinterpret_cast<float4 *>(p.state_out + st_off + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (P > 1) cluster_sync();  // no CTA leaves while another may still touch its shared memory
    if (kChainOnly) {
        // After a give-up, raw loads and helper copies may still be in flight into the state CTA; they
        // land (bounded waits) before any CTA of the cluster leaves. At most one is outstanding per slot.
        if (rank == 0 && tid == 32) {
            const int *req = reinterpret_cast<const int *>(sm + CO_SCL + 4 * 516);
            for (int s = 0; s < 2; ++s)
                if (req[s] > 0) mbar_wait(bar_tl + s, (uint32_t)(req[s] - 1) & 1, kWaitBudget);
            for (int j = 0; j < 3; ++j) {
                const int ncp = (j < nchunks ? 1 : 0) + req[2 + j];
                if (ncp > 0) mbar_wait(bar_sent + j, (uint32_t)(ncp - 1) & 1, kWaitBudget);
            }
        }
        __syncthreads();
        cluster_sync();
    }
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

// CTAs per value head. The block chain of one head is sequential, but preparing a block
// (norms, gates, the triangular solve, W) is not: with few heads the other SMs prepare blocks
// for the state-carrying CTA of their cluster. P = 4 when every head's cluster fits on the
// GPU at once, else 2, else 1; F = 1 (rank 0 only carries the state) needs P >= 3.
// GDN_PREFILL_CLUSTER="P,F" overrides the choice (a tuning knob; invalid values are ignored).
void pick_cluster(long heads, int *P, int *F) {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    *P = 1;
    *F = 0;
    for (int cand : {4, 2}) {
        if (heads * cand > sms) continue;
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = cand;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.gridDim = dim3((unsigned)(heads * cand), 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = SMEM_BYTES;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int nclusters = 0;
        if (cudaOccupancyMaxActiveClusters(&nclusters, prefill_tc_kernel<false>, &cfg) != cudaSuccess) {
            cudaGetLastError();
            continue;
        }
        if (nclusters >= heads) {
            *P = cand;
            break;
        }
    }
    *F = *P >= 3 ? 1 : 0;
    if (const char *env = getenv("GDN_PREFILL_CLUSTER")) {
        int pp = 0, ff = 0;
        if (sscanf(env, "%d,%d", &pp, &ff) == 2 && (pp == 1 || pp == 2 || pp == 4) && (ff == 0 || (ff == 1 && pp >= 3))) {
            *P = pp;
            *F = ff;
        }
    }
}

cudaError_t launch_prefill_tc(const PrefillArgs &a, cudaStream_t s) {
    const long Ttot = a.cu_seqlens ? (long)a.T : (long)a.B * a.T;
    CUtensorMap mq, mk, mv;
    if (!make_map(&mq, a.q, DK, a.Hk, Ttot) || !make_map(&mk, a.k, DK, a.Hk, Ttot) ||
        !make_map(&mv, a.v, DV, a.Hv, Ttot))
        return cudaErrorInvalidValue;
    for (auto fn : {prefill_tc_kernel<false>, prefill_tc_kernel<true>}) {
        const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
        if (e != cudaSuccess) return e;
    }
    int P = 1, F = 0;
    pick_cluster((long)a.B * a.Hv, &P, &F);
    TcParams p{(const __nv_bfloat16 *)a.g, (const __nv_bfloat16 *)a.b, a.state_in, a.state_out,
               (__nv_bfloat16 *)a.out, a.cu_seqlens, a.B, a.Hk, a.Hv, (long)a.T, Ttot, a.status, P, F};
    if (P == 1) {
        prefill_tc_kernel<false><<<dim3(a.Hv, a.B), kThreads, SMEM_BYTES, s>>>(mq, mk, mv, p);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = P;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.gridDim = dim3((unsigned)(a.Hv * P), (unsigned)a.B, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = s;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return F ? cudaLaunchKernelEx(&cfg, prefill_tc_kernel<true>, mq, mk, mv, p)
             : cudaLaunchKernelEx(&cfg, prefill_tc_kernel<false>, mq, mk, mv, p);
}

}  // namespace gdn
