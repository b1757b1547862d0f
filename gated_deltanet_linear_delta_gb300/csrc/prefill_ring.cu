// prefill_ring.cu -- block (chunk) form of the gated delta rule with the state chain cut to
// one dependent tensor-core product per block, fed by block preparation spread over the GPU.
//
// The pages describe two evaluation orders of the recurrence: a direct token scan, or
// regrouping the updates into blocks that expose matrix products and token parallelism
// ("Optimiser l'inference sur appareil pour Apple Silicon", section "Qwen cree trois formes
// de charges de travail"), and they keep the recurrent state on chip for a whole scan,
// written back once (section "Maintenir l'etat recurrent sur la puce"). This kernel is the
// block order for dk = dv = 128, blocks of C = 64 tokens, bf16 I/O, fp32 state.
//
// Per block of L <= 64 tokens of value head h, entering state S (dv x dk, fp32), with Kh, Qh
// the L2-normalised key/query rows, G the in-block cumulative log-gate, e_t = exp(G_t),
// d_t = exp(G_{L-1} - G_t), gamma = exp(G_{L-1}), T = (I + A)^-1 with
// A_ts = beta_t e^{G_t-G_s} kh_t.kh_s (s < t), P_ts = e^{G_t-G_s} qh_t.kh_s (s <= t),
// Tb = T diag(beta), Tw = T diag(beta e), W = Tw Kh, the block's update is affine in S:
//     S   <- gamma S + S N + V^T B,      N = -W^T diag(d) Kh         (dk x dk)
//                                        B = Tb^T diag(d) Kh         (C x dk)
//     O^T  = S Z + V^T E,                Z = Qt^T - W^T P^T, Qt = diag(e) Qh   (dk x C)
//                                        E = Tb^T P^T                (C x C)
// (substituting U^T = V^T Tb^T - S W^T into the usual WY/UT update and read-out). Only S N
// depends on the previous block, so the state's dependent chain is one MMA per block.
//
// One launch holds two kinds of CTA, all resident at once (cooperative launch):
//  * chain CTAs (one per state chain at a time): the fp32 state in registers, per block four
//    tcgen05 MMAs (S N and S Z with an fp16 copy of S in TMEM; V^T B and V^T E on the raw bf16
//    V tile with B, E as bf16 hi + lo pairs, B sent as B^T rows), the state update and the bf16
//    outputs;
//  * prep CTAs: take (block, value head) units from a global counter, compute norms, gates, A,
//    P, the triangular solve and N, Z, B, E, and write them into a per-chain ring of slots in
//    device memory that the chain CTA bulk-copies in. With more chains than chain CTAs a
//    pipeline takes the value heads of one key head in a row and does the key-side work once.
// Ring protocol: slot k of chain CTA i holds its step s = k (mod slots) once
// slot_seq[i][k] == s + 1 (release/acquire at GPU scope); the chain publishes consumed[i] =
// s + 1 when step s's copy has landed, and a prep CTA writes step s only once step s - slots
// is consumed. Units are handed out in step order, so every wait is for a unit handed out
// earlier, and a prep CTA publishes what it has written before it waits for a slot: no cycle.
//
// Numerics (per-operand rounding validated against the fp64 token scan): N, Z, W and P in fp16;
// K in fp16 as sigma K (exact: a power-of-two sigma from the tile's largest magnitude); S in fp16
// with an exact power-of-two scale per row for the MMAs, fp32 everywhere else; B and E (which
// carry v into the state and the outputs) as bf16 hi + lo pairs against the raw bf16 V tile;
// T diag(beta e rk) and diag(d rk) T diag(beta) as fp16 hi + lo (W and B cancel to a small
// fraction of their terms when keys are nearly parallel), with rk divided by a power of two
// kappa >= max rk so that keys of any norm keep them out of fp16's subnormals; every scale is
// taken back in fp32; every accumulator fp32.
//
// Rows t >= L of a partial block get zero kh, qh, beta and d, so they contribute nothing; their
// outputs are not stored. Every wait is bounded; a wait that runs out sets the device status
// word and a launch-wide abort flag, and every role leaves after draining its own asynchronous
// copies and MMAs.
#include <cuda.h>
#include <type_traits>
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
constexpr int kThreads = 384;
constexpr int kSlots = 16;                         // ring slots per chain CTA
constexpr long long kWaitDefault = 4000000000LL;  // SM cycles (about 2 s) before a wait gives up
constexpr long long kDrainBudget = 2000000000LL;  // waits for the CTA's own copies/MMAs when leaving

// ---- ring slot image: one block's operands in the chain CTA's shared-memory layouts ----
constexpr uint32_t RS_N = 0;        // 32 KiB fp16 N, MN-major [j 0..127][n]: n-blocks of 16 KiB
constexpr uint32_t RS_Z = 32768;    // 16 KiB fp16 Z, MN-major [j][t]
constexpr uint32_t RS_BE = 49152;   // 48 KiB: the V-side operands as bf16 hi + lo pairs:
constexpr uint32_t RS_BH = 49152;   //   16 KiB B^T hi, K-major [n 0..127][t 0..63]
constexpr uint32_t RS_BL = 65536;   //   16 KiB B^T lo
constexpr uint32_t RS_EH = 81920;   //    8 KiB E hi, MN-major [t 0..63][s 0..63]
constexpr uint32_t RS_EL = 90112;   //    8 KiB E lo
constexpr uint32_t RS_BYTES = 98304;
constexpr uint32_t RS_HEAD = RS_EH;  // a stage is loaded in two parts: [0, RS_HEAD) and the E images
// Once a step's MMAs are done, its stage's E region (16 KiB) holds that step's bf16 outputs,
// [dv block 0..1][t][128 B] with the 128-byte swizzle, for one tensor store per dv block.
constexpr uint32_t CH_OUT = RS_EH;
static_assert((size_t)kStaticChainCtas * kSlots * RS_BYTES + ((size_t)1 << 20) <= kStaticScratchBytes,
              "the fixed scratch holds the ring of its chain CTAs plus 1 MiB of tables");

// ---- chain CTA shared memory (byte offsets from a 1 KiB aligned base) ----
constexpr uint32_t CH_V = RS_BYTES;                  // raw V tile [i-block 0..1][t][128 B], 16 KiB
constexpr uint32_t CH_STAGE = RS_BYTES + 16384;      // two stages
constexpr uint32_t CH_XCH = 2 * CH_STAGE;            // [2 parities][2 halves][128 rows] int8 row exponents
constexpr uint32_t CH_SC = CH_XCH + 512;             // gamma [2] of the step, [2] of the stage; staged-output info [2][4]
constexpr uint32_t CH_BAR = CH_SC + 64;
constexpr uint32_t CH_END = CH_BAR + 256;
static_assert(CH_STAGE % 1024 == 0 && CH_V % 1024 == 0, "chain stages need 1 KiB alignment");

// ---- prep CTA: two independent pipelines, each in its own shared-memory slice ----
// (image offsets below are byte offsets within a ring slot image; they are staged in dead buffers)
constexpr uint32_t PP_RAW = 0;        // 32 KiB [kb 0..1][K rows 0..63 | Q rows 64..127][128 B] bf16; K rows -> fp16 (scaled)
constexpr uint32_t PP_P = 32768;      //  8 KiB fp16 P [t][s]
constexpr uint32_t PP_AT = 40960;     // 34 KiB: A fp32 [64][68] | T fp32 [64][68]; then Tw' lo; then the staged [B|E] head, N
constexpr uint32_t PP_T = PP_AT + 17408;
constexpr uint32_t PP_TWLO = PP_AT;   //  8 KiB fp16 Tw' lo [t][s], in A's place once the solve is done
constexpr uint32_t PP_TT = 75776;     // 32 KiB: Tw' [t][s] | Tb [m][s] | Tb' hi [s][t] | Tb' lo (fp16); then [B|E] tail, Z
constexpr uint32_t PP_SC = 108544;    //  4 KiB scalars
constexpr uint32_t PP_BAR = 112640;   // mbarriers
constexpr uint32_t PP_BYTES = 113664;  // a multiple of 1 KiB: the swizzled tiles of both slices stay aligned
constexpr uint32_t PR_END = 2 * PP_BYTES;
constexpr uint32_t BE_HEAD = 34816;   // bytes of the [B|E] image staged in AT; the rest goes to TT
constexpr uint32_t Z_STAGE = 14336;   // Z image offset in TT (after the [B|E] tail)
static_assert(2 * 24576 - BE_HEAD <= Z_STAGE && Z_STAGE + 16384 <= 32768, "staging overlaps");
static_assert(32768 <= PP_TT - PP_AT, "N image does not fit in AT");
static_assert(PP_BYTES % 1024 == 0 && PP_TT % 1024 == 0 && PP_P % 1024 == 0 && PP_TWLO % 1024 == 0,
              "128B-swizzled tiles need 1 KiB alignment");
static_assert(PP_TWLO + 8192 <= PP_T, "Tw' lo overlaps T");
static_assert(PP_BAR + 256 <= PP_BYTES, "pipeline slice overflow");
constexpr int LS = 68;                // row stride (floats) of A and T

constexpr uint32_t SMEM_USED = CH_END > PR_END ? CH_END : PR_END;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;  // alignment slack
static_assert(SMEM_BYTES <= 232448, "over the 227 KiB opt-in limit");

// prep scalars (float index into PP_SC)
constexpr int PS_RK = 0, PS_RQ = 64, PS_G = 128, PS_BETA = 192, PS_E = 256, PS_D = 320, PS_AA = 384;
constexpr int PS_BBRK = 448;   // e^{gmin - G_s} rk_s
constexpr int PS_TWF = 512;    // beta_s e_s rk_s / kappa   (Tw' columns)
constexpr int PS_DRK = 576;    // d_s rk_s / kappa          (Tb' rows, W^T d columns)
constexpr int PS_ER = 640;     // e_t rq_t                   (Qt rows)
constexpr int PS_MISC = 704;   // gmin, gmax, factor flag, gamma, 1 / sigma, 1 / sigma_q, kappa
constexpr int PS_RED = 720;    // [4 warps] tile maxima, [4 warps] rk maxima
constexpr int PS_UNIT = 768;   // int[3][16]: unit records, unit h in [h & 1]; [2]: the next group's first
constexpr int PS_MAIL = 752;   // int[4]: to the publisher: [0] ring CTA (-1: stop), [1] step, [2] gamma bits, [3] failed
// unit record (int offsets)
// U_VI: the unit's place among the r value heads of its key head when one pipeline prepares all r
// in a row and shares the key-side work; U_LAST: the group's last unit
constexpr int U_VALID = 0, U_S = 1, U_RI = 2, U_H = 3, U_HK = 4, U_TOK = 5, U_L = 6, U_VI = 7, U_LAST = 8;
// pipeline mbarriers (index into PP_BAR)
constexpr int PB_UREADY = 0, PB_TMA = 1, PB_G = 2, PB_M1REQ = 3, PB_M1 = 4, PB_M2REQ = 5, PB_M2 = 6, PB_RAWFREE = 7,
              PB_BEREADY = 8, PB_BEREAD = 9, PB_NZREADY = 10, PB_STGFREE = 11, PB_FIN = 12, PB_COUNT = 13;

// ---- TMEM columns (512 allocated) ----
constexpr uint32_t CT_D1 = 0, CT_O1 = 128, CT_D2 = 192, CT_O2 = 320, CT_S16 = 384;  // chain (S16: two buffers)
// prep pipeline (256 columns each): Gram, then W^T (fp32) -> WTd' | WT (fp16 A operands) in [0, 64);
// B^T (M = 128) in [64, 128), E (M = 64) in [128, 192); then N in [64, 192) and W^T P^T in [192, 256)
constexpr uint32_t PT_G = 0, PT_WT = 0, PT_B = 64, PT_E = 128, PT_N = 64, PT_WP = 192;

constexpr uint32_t ID_VB = idesc_bf16(128, 128, 1, 0);  // V^T x B (hi or lo; B as B^T rows)
constexpr uint32_t ID_VE = idesc_bf16(128, 64, 1, 1);   // V^T x E (hi or lo)
constexpr uint32_t ID_SN = idesc_f16(128, 128, 0, 1);   // S16 (TMEM) x N
constexpr uint32_t ID_SZ = idesc_f16(128, 64, 0, 1);    // S16 (TMEM) x Z
constexpr uint32_t ID_GRAM = idesc_bf16(128, 64, 0, 0); // [K; Q] K^T on raw tiles
constexpr uint32_t ID_GRAM16 = idesc_f16(128, 64, 0, 0); // [K'; Q'] K'^T on the converted tiles
constexpr uint32_t ID_WT = idesc_f16(128, 64, 1, 0);    // K'^T Tw'^T (K' = sigma K in fp16)
constexpr uint32_t ID_B = idesc_f16(128, 64, 1, 1);     // K'^T Tb' = sigma B^T (Tb' hi or lo, fp16)
constexpr uint32_t ID_E = idesc_f16(64, 64, 1, 0);      // Tb^T P^T
constexpr uint32_t ID_N = idesc_f16(128, 128, 0, 1);    // (W^T diag(d rk)) K', A from TMEM
constexpr uint32_t ID_WP = idesc_f16(128, 64, 0, 0);    // W^T P^T, A from TMEM

struct RingWs {       // device pointers into the workspace
    int *ctl;         // [0] next prep unit, [32] abort, [64] most steps of any group
    int *consumed;    // [NC * 32]: chain CTA i's count at [32 i]
    int *slot_seq;    // [NC * 32]: slot k of chain CTA i at [32 i + k]
    float *slot_sc;   // [NC * kSlots * 4]: gamma of the block in the slot
    int *seq_rank;    // [B] sequence of rank k (longest first when B <= kRankMax)
    int *nblk;        // [B] blocks of each sequence (0: empty or inconsistent)
    int *first_step;  // [G][npos + 1] first step of each list position of a group
    int *total_steps; // [G]
    uint8_t *ring;    // [NC][kSlots][RS_BYTES]
};

struct RingParams {
    const __nv_bfloat16 *g, *b;
    const float *state_in;
    float *state_out;
    __nv_bfloat16 *out;
    const int32_t *cu;
    int B, Hk, Hv, r;  // r = Hv / Hk value heads per key head
    long T, Ttot;
    int NC, G, npos;   // chain CTAs, groups of r chain CTAs, list positions per group
    int *status;
    long long wait_budget;
    RingWs w;
};

constexpr int kRankMax = 1024;  // sequences ranked by length (longest first) up to this count

// ---- small helpers ----

// exponent e with m < 2^e (frexp convention), clamped; -128 for m = 0 or non-finite
__device__ __forceinline__ int row_exp(float m) {
    if (!(m > 0.f) || !isfinite(m)) return -128;
    int e;
    frexpf(m, &e);
    return max(-100, min(100, e));
}

// four consecutive per-row scalars from the 16-byte aligned scalar area (index a multiple of 4)
__device__ __forceinline__ float4 ps4(const float *ps, int i) { return *reinterpret_cast<const float4 *>(ps + i); }

// the power of two 2^e just above m (m < 2^e), clamped; 1 for m <= 0 or non-finite
__device__ __forceinline__ float pow2_above(float m) {
    if (!(m > 0.f) || !isfinite(m)) return 1.f;
    int e;
    frexpf(m, &e);
    return ldexpf(1.f, max(-100, min(100, e)));
}

__device__ __forceinline__ void set_abort(const RingParams &p) {
    atomicExch(p.w.ctl + 32, 1);
    flag_error(p.status);
}
__device__ __forceinline__ bool aborted(const RingParams &p) { return ld_relaxed_gpu(p.w.ctl + 32) != 0; }

// bounded wait on an mbarrier phase; false when the budget runs out
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t par, long long budget) {
    return mbar_wait(bar, par, budget);
}

// T = (I + A)^-1, A strictly lower 64 x 64 fp32 with row stride LS; 128 threads of named barrier
// `bar_id`, in four barrier-separated phases: (1) the four diagonal 16x16 blocks by forward
// substitution (one column per thread, loads issued two steps ahead); (2) inside each 32x32
// diagonal block, T10 = -T11 (A10 T00) (64 threads per block, four per output column: thread q
// holds rows q, q+4, q+8, q+12, and the column of the inner product is exchanged by shuffles in
// the quad); (3) the 32x32 lower-left block, X = A_HL T_LL and then T_HL = -T_HH X, 2 x 4 outputs
// per thread with X passed through the (zero) upper-right block. Block-triangular zeros are
// skipped; every stage issues its shared-memory loads before its FMAs.
__device__ void solve128(const float *sA, float *sT, int p, int bar_id) {
    if (p < 64) {
        const int b = p >> 4, c = p & 15;
        const float *Ab = sA + 16 * b * LS + 16 * b;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) x[r] = (r == c) ? 1.f : 0.f;
        float a[8][16];
#pragma unroll
        for (int s = 0; s < 2; ++s)
#pragma unroll
            for (int r = s + 1; r < 16; ++r) a[s][r] = Ab[r * LS + s];
#pragma unroll
        for (int s = 0; s < 15; ++s) {
            if (s + 2 < 15) {
#pragma unroll
                for (int r = s + 3; r < 16; ++r) a[(s + 2) & 7][r] = Ab[r * LS + s + 2];
            }
#pragma unroll
            for (int r = s + 1; r < 16; ++r) x[r] = fmaf(-a[s & 7][r], x[s], x[r]);
        }
        float *Tb = sT + 16 * b * LS + 16 * b + c;
#pragma unroll
        for (int r = 0; r < 16; ++r) Tb[r * LS] = x[r];
        // zeros above the diagonal blocks (the 32-block zeros are written in step 3's layout too)
#pragma unroll
        for (int i = 0; i < 3; ++i)
            if (i < b)
#pragma unroll
                for (int r = 0; r < 16; ++r) sT[(16 * i + r) * LS + 16 * b + c] = 0.f;
    }
    bar_sync(bar_id, 128);
    {   // step 2: blocks (1,0) and (3,2); thread (col, q) of its 64: rows q, q+4, q+8, q+12 of column col
        const int lane = p & 31, q = p & 3, col = (p >> 2) & 15, j = 2 * (p >> 6), i = j + 1;
        const float *Ar = sA + (16 * i + q) * LS + 16 * j;
        const float *Tc = sT + 16 * j * LS + 16 * j + col;
        float t[16];
        float4 a[4][4];
#pragma unroll
        for (int m = 0; m < 16; ++m) t[m] = Tc[m * LS];
#pragma unroll
        for (int rr = 0; rr < 4; ++rr)
#pragma unroll
            for (int m4 = 0; m4 < 4; ++m4) a[rr][m4] = *reinterpret_cast<const float4 *>(Ar + 4 * rr * LS + 4 * m4);
        float xs[4];
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) {
            float e0 = 0.f, e1 = 0.f;
#pragma unroll
            for (int m4 = 0; m4 < 4; ++m4) {
                float &e = (m4 & 1) ? e1 : e0;
                e = fmaf(a[rr][m4].x, t[4 * m4], e);
                e = fmaf(a[rr][m4].y, t[4 * m4 + 1], e);
                e = fmaf(a[rr][m4].z, t[4 * m4 + 2], e);
                e = fmaf(a[rr][m4].w, t[4 * m4 + 3], e);
            }
            xs[rr] = e0 + e1;
        }
        const float *Tr = sT + (16 * i + q) * LS + 16 * i;
        float4 tt[4][4];
#pragma unroll
        for (int rr = 0; rr < 4; ++rr)
#pragma unroll
            for (int m4 = 0; m4 < 4; ++m4) tt[rr][m4] = *reinterpret_cast<const float4 *>(Tr + 4 * rr * LS + 4 * m4);
        float X[16];
#pragma unroll
        for (int m = 0; m < 16; ++m) X[m] = __shfl_sync(0xffffffffu, xs[m >> 2], (lane & ~3) | (m & 3));
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) {
            float e0 = 0.f, e1 = 0.f;
#pragma unroll
            for (int m4 = 0; m4 < 4; ++m4) {
                float &e = (m4 & 1) ? e1 : e0;
                e = fmaf(tt[rr][m4].x, X[4 * m4], e);
                e = fmaf(tt[rr][m4].y, X[4 * m4 + 1], e);
                e = fmaf(tt[rr][m4].z, X[4 * m4 + 2], e);
                e = fmaf(tt[rr][m4].w, X[4 * m4 + 3], e);
            }
            sT[(16 * i + q + 4 * rr) * LS + 16 * j + col] = -(e0 + e1);
        }
    }
    bar_sync(bar_id, 128);
    // step 3: X = A[32:64, 0:32] T[0:32, 0:32] (T lower: X[:, n] sums k >= 16*(n/16) only), kept in
    // registers as a 2 x 4 tile (rows 2*rg, 2*rg + 1; columns 4*cg .. 4*cg + 3); then
    // T[32+r, n] = -sum_{k <= r} T[32+r, 32+k] X[k, n], the X rows exchanged through shared memory.
    const int cg = p & 7, rg = p >> 3, c0 = 4 * cg, r0 = 2 * rg;
    float acc[2][4];
#pragma unroll
    for (int u = 0; u < 2; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) acc[u][v] = 0.f;
    {
        const int k0 = c0 & 16;  // T[k][c] = 0 for k < 16 when c >= 16
#pragma unroll 4
        for (int k4 = k0; k4 < 32; k4 += 4) {
            const float4 a0 = *reinterpret_cast<const float4 *>(sA + (32 + r0) * LS + k4);
            const float4 a1 = *reinterpret_cast<const float4 *>(sA + (33 + r0) * LS + k4);
            const float av0[4] = {a0.x, a0.y, a0.z, a0.w}, av1[4] = {a1.x, a1.y, a1.z, a1.w};
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const float4 t4 = *reinterpret_cast<const float4 *>(sT + (k4 + kk) * LS + c0);
                acc[0][0] = fmaf(av0[kk], t4.x, acc[0][0]); acc[0][1] = fmaf(av0[kk], t4.y, acc[0][1]);
                acc[0][2] = fmaf(av0[kk], t4.z, acc[0][2]); acc[0][3] = fmaf(av0[kk], t4.w, acc[0][3]);
                acc[1][0] = fmaf(av1[kk], t4.x, acc[1][0]); acc[1][1] = fmaf(av1[kk], t4.y, acc[1][1]);
                acc[1][2] = fmaf(av1[kk], t4.z, acc[1][2]); acc[1][3] = fmaf(av1[kk], t4.w, acc[1][3]);
            }
        }
    }
    // X goes to the (still zero) upper-right block T[0:32, 32:64] as scratch: row r of X at T[r][32..63]
#pragma unroll
    for (int u = 0; u < 2; ++u)
        *reinterpret_cast<float4 *>(sT + (r0 + u) * LS + 32 + c0) = make_float4(acc[u][0], acc[u][1], acc[u][2], acc[u][3]);
    bar_sync(bar_id, 128);
#pragma unroll
    for (int u = 0; u < 2; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) acc[u][v] = 0.f;
    {
        const int kend = r0 + 2;  // T[32+r][32+k] = 0 for k > r
#pragma unroll 2
        for (int k4 = 0; k4 < kend; k4 += 4) {
            const float4 h0 = *reinterpret_cast<const float4 *>(sT + (32 + r0) * LS + 32 + k4);
            const float4 h1 = *reinterpret_cast<const float4 *>(sT + (33 + r0) * LS + 32 + k4);
            const float hv0[4] = {h0.x, h0.y, h0.z, h0.w}, hv1[4] = {h1.x, h1.y, h1.z, h1.w};
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const float4 x4 = *reinterpret_cast<const float4 *>(sT + (k4 + kk) * LS + 32 + c0);
                acc[0][0] = fmaf(hv0[kk], x4.x, acc[0][0]); acc[0][1] = fmaf(hv0[kk], x4.y, acc[0][1]);
                acc[0][2] = fmaf(hv0[kk], x4.z, acc[0][2]); acc[0][3] = fmaf(hv0[kk], x4.w, acc[0][3]);
                acc[1][0] = fmaf(hv1[kk], x4.x, acc[1][0]); acc[1][1] = fmaf(hv1[kk], x4.y, acc[1][1]);
                acc[1][2] = fmaf(hv1[kk], x4.z, acc[1][2]); acc[1][3] = fmaf(hv1[kk], x4.w, acc[1][3]);
            }
        }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u)
        *reinterpret_cast<float4 *>(sT + (32 + r0 + u) * LS + c0) =
            make_float4(-acc[u][0], -acc[u][1], -acc[u][2], -acc[u][3]);
    bar_sync(bar_id, 128);
    // the scratch block back to zero
#pragma unroll
    for (int u = 0; u < 2; ++u)
        *reinterpret_cast<float4 *>(sT + (r0 + u) * LS + 32 + c0) = make_float4(0.f, 0.f, 0.f, 0.f);
    bar_sync(bar_id, 128);
}

// Chain id of list position `pos` of chain CTA (group m, member v). Chains are numbered
// (sequence rank, key head, member) with sequences longest first; position pos hands the G
// groups the next G (sequence, key head) items, left to right at even positions and right to
// left at odd ones, so that a group that took a longer item at one position takes a shorter
// one at the next (serpentine order: the groups' total steps stay close).
__device__ __forceinline__ long chain_id(const RingParams &p, int m, int v, int pos) {
    const int mm = (pos & 1) ? p.G - 1 - m : m;
    return ((long)pos * p.G + mm) * p.r + v;
}

// ---- the plan: sequence order, block counts, step tables; counters zeroed ----
__global__ void __launch_bounds__(1024) ring_plan_kernel(const RingParams p) {
    __shared__ int s_len[kRankMax];
    const int tid = threadIdx.x, nt = blockDim.x;
    for (int x = tid; x < 128; x += nt) p.w.ctl[x] = 0;
    for (int x = tid; x < p.NC * 32; x += nt) {
        p.w.consumed[x] = 0;
        p.w.slot_seq[x] = 0;
    }
    const bool rank = p.B <= kRankMax;
    for (int n = tid; n < p.B; n += nt) {
        long bos, eos;
        const bool ok = seq_bounds(p.cu, n, p.B, p.cu ? p.Ttot : p.T, &bos, &eos, p.status);
        const long len = ok ? eos - bos : 0;
        p.w.nblk[n] = (int)((len + C - 1) / C);
        if (rank) s_len[n] = ok ? (int)min(len, (long)0x7fffffff) : -1;
        if (!rank) p.w.seq_rank[n] = n;
    }
    __syncthreads();
    if (rank) {
        for (int n = tid; n < p.B; n += nt) {
            const int ln = s_len[n];
            int k = 0;
            for (int o = 0; o < p.B; ++o) k += (s_len[o] > ln) || (s_len[o] == ln && o < n);
            p.w.seq_rank[k] = n;
        }
    }
    __syncthreads();
    const long nchains = (long)p.B * p.Hv;
    for (int m = tid; m < p.G; m += nt) {
        int acc = 0;
        int *fs = p.w.first_step + (long)m * (p.npos + 1);
        for (int pos = 0; pos < p.npos; ++pos) {
            fs[pos] = acc;
            const long c = chain_id(p, m, 0, pos);
            if (c < nchains) acc += p.w.nblk[p.w.seq_rank[c / p.Hv]];
        }
        fs[p.npos] = acc;
        p.w.total_steps[m] = acc;
        atomicMax(p.w.ctl + 64, acc);
    }
    // empty sequences pass their state through (sequences with inconsistent bounds are skipped)
    for (int n = 0; n < p.B; ++n) {
        if (p.w.nblk[n] != 0) continue;
        long bos, eos;
        if (!seq_bounds(p.cu, n, p.B, p.cu ? p.Ttot : p.T, &bos, &eos, nullptr)) continue;
        const long base = (long)n * p.Hv * DV * DK;
        if (p.state_in == p.state_out) continue;
        for (long x = tid; x < (long)p.Hv * DV * DK / 4; x += nt) {
            const float4 v = p.state_in ? reinterpret_cast<const float4 *>(p.state_in + base)[x]
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
            reinterpret_cast<float4 *>(p.state_out + base)[x] = v;
        }
    }
}


struct ChainInfo {
    int n, h, nb;
    long bos, len;
};
__device__ __forceinline__ ChainInfo chain_info(const RingParams &p, long c, int nb) {
    ChainInfo ci;
    ci.n = p.w.seq_rank[c / p.Hv];
    ci.h = (int)(c % p.Hv);
    ci.nb = nb;
    if (p.cu) {
        ci.bos = p.cu[ci.n];
        ci.len = (long)p.cu[ci.n + 1] - ci.bos;
    } else {
        ci.bos = (long)ci.n * p.T;
        ci.len = p.T;
    }
    return ci;
}

__device__ __forceinline__ uint8_t *ring_slot(const RingParams &p, int i, int s) {
    return p.w.ring + ((long)i * kSlots + s % kSlots) * RS_BYTES;
}

// ======================= chain CTA =======================
__device__ void chain_cta(const CUtensorMap *tm_v, const CUtensorMap *tm_o, const RingParams &p, uint8_t *sm,
                          uint32_t sb, uint32_t tmem) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int i = blockIdx.x, m = i / p.r, v = i % p.r;
    const int *fs = p.w.first_step + (long)m * (p.npos + 1);
    const int total = p.w.total_steps[m];
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + CH_BAR);
    uint64_t *full = bars + 0, *freeb = bars + 2, *d1 = bars + 4, *o1 = bars + 5, *s16 = bars + 6,
             *d2free = bars + 7, *o12free = bars + 8, *scb = bars + 9, *fin = bars + 11;
    uint64_t *fulle = bars + 12;    // [2] the stage's E images landed
    uint64_t *ostaged = bars + 14;  // [2] the step's outputs staged in the stage's E region (256 arrivals)
    // [2][4] per stage: 1 if the staged outputs are to be stored (a full block), their first token, head
    int *oinfo = reinterpret_cast<int *>(sm + CH_SC + 16);
    float *gam = reinterpret_cast<float *>(sm + CH_SC);  // [2] gamma of step s at [s & 1], for the epilogue
    float *gst = gam + 2;                                 // [2] gamma of the block in stage st
    const long long budget = p.wait_budget;

    if (tid == 0) {
        // ---------------- loader: ring slot (bulk copies) + raw V tile (TMA) per step ----------------
        // A stage is refilled in two parts: everything but the E images as soon as the step two
        // before is done, then -- once the outputs that step staged in the E region have been
        // read out by their tensor store -- the E images, which are needed last.
        prefetch_tmap(tm_v);
        prefetch_tmap(tm_o);
        int s = 0, issued = 0;
        bool ok = true;
        // tensor store of the outputs step j staged (if it was a full block); false when the wait ran out
        auto store_outputs = [&](int j, long long lim) {
            const int sj = j & 1;
            if (!wait_bar(ostaged + sj, (j >> 1) & 1, lim)) return false;
            if (oinfo[4 * sj]) {
                const int tok = oinfo[4 * sj + 1], hh = oinfo[4 * sj + 2];
                tma_store_3d(tm_o, sm + sj * CH_STAGE + CH_OUT, 0, hh, tok);
                tma_store_3d(tm_o, sm + sj * CH_STAGE + CH_OUT + 8192, 64, hh, tok);
                bulk_commit();
                bulk_wait_read_all();
            }
            return true;
        };
        int e_issued = 0;
        for (int pos = 0; pos < p.npos && ok; ++pos) {
            const int nb = fs[pos + 1] - fs[pos];
            if (nb == 0) continue;
            const ChainInfo ci = chain_info(p, chain_id(p, m, v, pos), nb);
            for (int b = 0; b < nb && ok; ++b, ++s) {
                const int st = s & 1;
                if (s >= 2 && !wait_bar(freeb + st, ((s - 2) >> 1) & 1, budget)) { ok = false; break; }
                const int *seq = p.w.slot_seq + 32 * i + s % kSlots;
                const long long t0 = clock64();
                int spins = 0;
                while (ld_acquire_gpu(seq) != s + 1) {
                    if (((++spins) & 63) == 0 && (aborted(p) || clock64() - t0 > budget)) { ok = false; break; }
                    __nanosleep(64);
                }
                if (!ok) break;
                fence_async_global();
                uint8_t *stage = sm + st * CH_STAGE;
                // the block's gamma, read before the slot can be rewritten (that waits for `consumed`)
                gst[st] = p.w.slot_sc[((long)i * kSlots + s % kSlots) * 4];
                mbar_expect_tx(full + st, RS_HEAD + 16384);
                bulk_load(stage, ring_slot(p, i, s), RS_HEAD, full + st);
                const int tok = (int)(ci.bos + (long)b * C);
                tma_load_3d(stage + CH_V, tm_v, 0, ci.h, tok, full + st);
                tma_load_3d(stage + CH_V + 8192, tm_v, 64, ci.h, tok, full + st);
                issued = s + 1;
                if (s >= 2 && !store_outputs(s - 2, budget)) { ok = false; break; }
                mbar_expect_tx(fulle + st, RS_BYTES - RS_HEAD);
                bulk_load(stage + RS_HEAD, ring_slot(p, i, s) + RS_HEAD, RS_BYTES - RS_HEAD, fulle + st);
                e_issued = s + 1;
            }
        }
        // the last two steps' outputs (after a failure: whatever was staged, within a bounded wait)
        for (int j = max(0, issued - 2); j < issued; ++j)
            if (!store_outputs(j, ok ? budget : kDrainBudget / 8)) ok = false;
        bulk_wait_all();
        // copies still landing must land before the CTA leaves (after a failure: the issuer may
        // have stopped waiting for them)
        for (int j = issued - 2; j < issued; ++j)
            if (j >= 0) wait_bar(full + (j & 1), (j >> 1) & 1, kDrainBudget);
        for (int j = e_issued - 2; j < e_issued; ++j)
            if (j >= 0) wait_bar(fulle + (j & 1), (j >> 1) & 1, kDrainBudget);
        if (!ok) set_abort(p);
    } else if (tid == 32) {
        // ---------------- issuer: every MMA ----------------
        // This thread shares its scheduler with two busy epilogue warps, so it issues as few
        // instructions as it can: the loops are unrolled and every shared-memory descriptor is a
        // per-stage base plus a constant (a descriptor's address field counts 16-byte units).
        const uint64_t dN = desc_sw128(sb + RS_N, 16384, 1024), dZ = desc_sw128(sb + RS_Z, 8192, 1024);
        const uint64_t dBH = desc_sw128(sb + RS_BH, 16, 1024), dBL = desc_sw128(sb + RS_BL, 16, 1024);
        const uint64_t dEH = desc_sw128(sb + RS_EH, 8192, 1024), dEL = desc_sw128(sb + RS_EL, 8192, 1024);
        const uint64_t dV = desc_sw128(sb + CH_V, 8192, 1024);
        int s = 0;
        bool ok = true;
        for (int pos = 0; pos < p.npos && ok; ++pos) {
            const int nb = fs[pos + 1] - fs[pos];
            for (int b = 0; b < nb; ++b, ++s) {
                const int st = s & 1;
                const uint64_t so = st ? (uint64_t)(CH_STAGE >> 4) : 0ull;  // stage offset in descriptor units
                if (!wait_bar(full + st, (s >> 1) & 1, budget)) { ok = false; break; }
                if (s > 0 && !wait_bar(d2free, (s - 1) & 1, budget)) { ok = false; break; }
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {  // V^T (B hi + B lo)
                    const uint64_t a = dV + so + ks * (2048 >> 4);
                    mma_bf16(tmem + CT_D2, a, dBH + so + ks * (32 >> 4), ID_VB, ks > 0);
                    mma_bf16(tmem + CT_D2, a, dBL + so + ks * (32 >> 4), ID_VB, 1);
                }
                if (!wait_bar(s16, s & 1, budget)) { ok = false; break; }
                tc_fence_after();
                // gamma of this step for the epilogue; scb(s + 2) cannot complete before the epilogue
                // has waited for scb(s): it follows s16(s + 2), which the epilogue gives in step s + 1
                gam[s & 1] = gst[st];
                mbar_arrive(scb + (s & 1));
                const uint32_t a16 = tmem + CT_S16 + 64 * (s & 1);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)  // S N: the state's dependent product
                    mma_f16_ts(tmem + CT_D1, a16 + 8 * ks, dN + so + ks * (2048 >> 4), ID_SN, ks > 0);
                mma_commit(d1);
                if (s > 0 && !wait_bar(o12free, (s - 1) & 1, budget)) { ok = false; break; }
                if (!wait_bar(fulle + st, (s >> 1) & 1, budget)) { ok = false; break; }
                // Both copies of the slot have landed (their reads are complete once the barrier
                // phases have flipped), so its producer may reuse the slot for step s + kSlots. A
                // relaxed store suffices and keeps this thread going: a release here would also wait
                // for the MMAs still in flight (about 2k cycles per step).
                st_relaxed_gpu(p.w.consumed + 32 * i, s + 1);
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {  // V^T (E hi + E lo)
                    const uint64_t a = dV + so + ks * (2048 >> 4);
                    mma_bf16(tmem + CT_O2, a, dEH + so + ks * (2048 >> 4), ID_VE, ks > 0);
                    mma_bf16(tmem + CT_O2, a, dEL + so + ks * (2048 >> 4), ID_VE, 1);
                }
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)  // S Z
                    mma_f16_ts(tmem + CT_O1, a16 + 8 * ks, dZ + so + ks * (2048 >> 4), ID_SZ, ks > 0);
                mma_commit(o1);
                mma_commit(freeb + st);
            }
        }
        mma_commit(fin);  // nothing issued here may still run when the CTA leaves
        wait_bar(fin, 0, kDrainBudget);
        if (!ok) set_abort(p);
    } else if (warp >= 4) {
        // ---------------- epilogue: the state (two threads per row), outputs ----------------
        const int r = 32 * (warp & 3) + lane, hf = (warp - 4) >> 2;
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const int pair_bar = 1 + (warp & 3);
        int8_t *xch = reinterpret_cast<int8_t *>(sm + CH_XCH);
        float S[64];
        float srow = 1.f;  // 1 / scale of the fp16 copy of S used by the current step
        bool ok = true;
        // the next non-empty list position at or after `pos`, or npos
        auto next_pos = [&](int pos) {
            while (pos < p.npos && fs[pos + 1] == fs[pos]) ++pos;
            return pos;
        };
        auto load_state = [&](const ChainInfo &ci) {
            if (p.state_in) {
                const float4 *src = reinterpret_cast<const float4 *>(
                    p.state_in + (((long)ci.n * p.Hv + ci.h) * DV + r) * DK + 64 * hf);
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                    const float4 x = src[q];
                    S[4 * q] = x.x; S[4 * q + 1] = x.y; S[4 * q + 2] = x.z; S[4 * q + 3] = x.w;
                }
            } else {
#pragma unroll
                for (int e = 0; e < 64; ++e) S[e] = 0.f;
            }
        };
        // fp16 copy of S (row scale shared by the two halves) into TMEM buffer `buf`; false to leave
        auto publish_s16 = [&](int par, int buf, bool good) {
            float m4[4] = {0.f, 0.f, 0.f, 0.f};  // four partial maxima: a short dependent chain
#pragma unroll
            for (int e = 0; e < 64; ++e) m4[e & 3] = fmaxf(m4[e & 3], fabsf(S[e]));
            const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
            xch[(par * 2 + hf) * 128 + r] = good ? (int8_t)max(-127, row_exp(mx)) : (int8_t)127;
            bar_sync(pair_bar, 64);
            const int eo = xch[(par * 2 + (hf ^ 1)) * 128 + r];
            const int em = xch[(par * 2 + hf) * 128 + r];
            // the two warps of a pair see the same rows' flags, so they leave together
            if (__any_sync(0xffffffffu, eo == 127 || em == 127)) return false;
            const int e = max(eo, em);
            const float scale = e == -127 ? 1.f : ldexpf(1.f, 14 - e);
            uint32_t pk[32];
#pragma unroll
            for (int e2 = 0; e2 < 32; ++e2) pk[e2] = h2_bits(S[2 * e2] * scale, S[2 * e2 + 1] * scale);
            tmem_st32(tmem + lane_off + CT_S16 + 64 * buf + 32 * hf, pk);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(s16);
            srow = 1.f / scale;
            return true;
        };
        int pos = next_pos(0);
        int s = 0;
        if (pos < p.npos) {
            const ChainInfo ci = chain_info(p, chain_id(p, m, v, pos), fs[pos + 1] - fs[pos]);
            load_state(ci);
            ok = publish_s16(0, 0, true);
        }
        while (ok && pos < p.npos) {
            const ChainInfo ci = chain_info(p, chain_id(p, m, v, pos), fs[pos + 1] - fs[pos]);
            for (int b = 0; b < ci.nb; ++b, ++s) {
                const int L = (int)min((long)C, ci.len - (long)b * C);
                // every decision is taken by the whole warp (TMEM loads and stores are warp-collective)
                bool good = wait_bar(scb + (s & 1), (s >> 1) & 1, budget);
                const float gamma = good ? gam[s & 1] : 0.f;
                good = __all_sync(0xffffffffu, good && wait_bar(d1, s & 1, budget));
                tc_fence_after();
                if (good) {
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        uint32_t a[32], c2[32];
                        tmem_ld32_nw(tmem + lane_off + CT_D1 + 64 * hf + 32 * q, a);
                        tmem_ld32_nw(tmem + lane_off + CT_D2 + 64 * hf + 32 * q, c2);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            S[32 * q + e] = fmaf(gamma, S[32 * q + e],
                                                 fmaf(srow, __uint_as_float(a[e]), __uint_as_float(c2[e])));
                    }
                }
                tc_fence_before();
                mbar_arrive(d2free);
                const float srow_step = srow;
                const bool last = b == ci.nb - 1;
                int npos_ = pos;
                if (last && good) {
                    float4 *dst = reinterpret_cast<float4 *>(p.state_out + (((long)ci.n * p.Hv + ci.h) * DV + r) * DK +
                                                             64 * hf);
#pragma unroll
                    for (int q = 0; q < 16; ++q)
                        dst[q] = make_float4(S[4 * q], S[4 * q + 1], S[4 * q + 2], S[4 * q + 3]);
                }
                if (last) {
                    npos_ = next_pos(pos + 1);
                    if (npos_ < p.npos)
                        load_state(chain_info(p, chain_id(p, m, v, npos_), fs[npos_ + 1] - fs[npos_]));
                }
                if (s + 1 < total) {
                    if (!publish_s16((s + 1) & 1, (s + 1) & 1, good)) good = false;
                }
                // outputs of this step
                const bool good_o = __all_sync(0xffffffffu, good && wait_bar(o1, s & 1, budget));
                tc_fence_after();
                const int so = s & 1;
                if (good_o) {
                    uint32_t a[32], c2[32];
                    tmem_ld32_nw(tmem + lane_off + CT_O1 + 32 * hf, a);
                    tmem_ld32_nw(tmem + lane_off + CT_O2 + 32 * hf, c2);
                    tmem_wait_ld();
                    tc_fence_before();
                    mbar_arrive(o12free);
                    if (L == C) {  // a full block: into the stage's E region, for one tensor store per dv block
                        uint8_t *ob = sm + so * CH_STAGE + CH_OUT + (r >> 6) * 8192 + ((r & 7) << 1);
                        const int ch = (r & 63) >> 3;
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            const int t = 32 * hf + e;
                            *reinterpret_cast<__nv_bfloat16 *>(ob + t * 128 + ((ch ^ (t & 7)) << 4)) =
                                __float2bfloat16_rn(fmaf(srow_step, __uint_as_float(a[e]), __uint_as_float(c2[e])));
                        }
                        fence_async_smem();
                        if (r == 0 && hf == 0) {
                            oinfo[4 * so] = 1;
                            oinfo[4 * so + 1] = (int)(ci.bos + (long)b * C);
                            oinfo[4 * so + 2] = ci.h;
                        }
                    } else {  // a partial block: only its L rows, straight to global memory
                        __nv_bfloat16 *op = p.out + ((ci.bos + (long)b * C + 32 * hf) * p.Hv + ci.h) * DV + r;
                        const long tstride = (long)p.Hv * DV;
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            if (32 * hf + e < L)
                                op[e * tstride] = __float2bfloat16_rn(
                                    fmaf(srow_step, __uint_as_float(a[e]), __uint_as_float(c2[e])));
                        if (r == 0 && hf == 0) oinfo[4 * so] = 0;
                    }
                } else {
                    tc_fence_before();
                    mbar_arrive(o12free);
                    if (r == 0 && hf == 0) oinfo[4 * so] = 0;
                }
                mbar_arrive(ostaged + so);
                if (!good || !good_o) { ok = false; break; }
                if (last) {  // (the loop's own increment of s is skipped by the break)
                    pos = npos_;
                    ++s;
                    break;
                }
            }
        }
        if (!ok) set_abort(p);
    }
}

// ======================= prep CTA: two pipelines =======================
// Each pipeline owns a 110 KiB slice of shared memory and 256 TMEM columns and prepares one
// (block, value head) unit at a time with three roles: the control thread (units, TMA, every MMA),
// 128 math threads (norms, gates, A and P, the solve, operand tiles, epilogues) and the publisher
// thread (bulk copies of the staged ring image, the slot's flag). Two pipelines per SM overlap
// one another's latencies; within a pipeline the roles hand over through mbarriers, one phase
// per unit each.
struct Pipe {
    uint8_t *sm;   // the pipeline's shared-memory slice
    uint32_t sb;   // its shared address
    uint32_t tm;   // its TMEM base (256 columns)
    float *ps;
    int *pu, *mail;
    uint64_t *bar;
};

__device__ __forceinline__ Pipe make_pipe(uint8_t *sm0, uint32_t sb0, uint32_t tmem, int pipe) {
    Pipe P;
    P.sm = sm0 + pipe * PP_BYTES;
    P.sb = sb0 + pipe * PP_BYTES;
    P.tm = tmem + 256u * pipe;
    P.ps = reinterpret_cast<float *>(P.sm + PP_SC);
    P.pu = reinterpret_cast<int *>(P.ps + PS_UNIT);
    P.mail = reinterpret_cast<int *>(P.ps + PS_MAIL);
    P.bar = reinterpret_cast<uint64_t *>(P.sm + PP_BAR);
    return P;
}

// the unit handed out as number u: (step s, group m, value head v of the group), or none left
__device__ bool unit_of(const RingParams &p, long u, int max_steps, int *rec) {
    const int v = (int)(u % p.r);
    const long mg = u / p.r;
    const int m = (int)(mg % p.G);
    const long s = mg / p.G;
    if (s >= max_steps) return false;
    rec[U_VALID] = 0;
    if (s >= p.w.total_steps[m]) return true;  // this group has no step s: skip it
    const int *fs = p.w.first_step + (long)m * (p.npos + 1);
    int lo = 0, hi = p.npos - 1;  // the last position whose first step is <= s
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (fs[mid] <= s) lo = mid; else hi = mid - 1;
    }
    const ChainInfo ci = chain_info(p, chain_id(p, m, v, lo), fs[lo + 1] - fs[lo]);
    const int b = (int)(s - fs[lo]);
    rec[U_VALID] = 1;
    rec[U_S] = (int)s;
    rec[U_RI] = m * p.r + v;
    rec[U_H] = ci.h;
    rec[U_HK] = ci.h / p.r;
    rec[U_TOK] = (int)(ci.bos + (long)b * C);
    rec[U_L] = (int)min((long)C, ci.len - (long)b * C);
    return true;
}

// ---- control thread: units, tile loads, every MMA ----
template <bool SHARE>
__device__ void prep_control(const CUtensorMap *tm_q, const CUtensorMap *tm_k, const RingParams &p, const Pipe &P) {
    const long long budget = p.wait_budget;
    const int max_steps = p.w.ctl[64];
    uint64_t *B = P.bar;
    bool ok = true;
    int tma_pending = 0;
    prefetch_tmap(tm_q);
    prefetch_tmap(tm_k);
    // The first unit of the next group with work into rec (rec[U_VALID] = 0: none left). With SHARE,
    // units come from the counter r at a time: the r value heads of one key head at one step,
    // prepared in a row with the key-side work done once (fewer instructions per unit, one more unit
    // latency before a step's last value head: taken when there are more chains than state CTAs,
    // i.e. when throughput matters more than latency). Without it a group is one unit.
    auto grab = [&](int *rec) {
        bool any = false;
        while (!any) {
            if (aborted(p)) break;
            const long u = atomicAdd(p.w.ctl + 0, SHARE ? p.r : 1);
            if (!unit_of(p, u, max_steps, rec)) break;
            any = rec[U_VALID] != 0;
        }
        if (!any) rec[U_VALID] = 0;
        if constexpr (SHARE) {
            rec[U_VI] = 0;
            rec[U_LAST] = 0;
        }
    };
    int *const gnext = P.pu + 32;  // the next group's first unit (SHARE)
    grab(P.pu);
    uint32_t g = 0;  // groups started
    for (uint32_t h = 0; ok; ++h) {
        int *rec = P.pu + 16 * (h & 1);
        const bool any = rec[U_VALID] != 0;
        const int vi = SHARE ? rec[U_VI] : 0;
        mbar_arrive(B + PB_UREADY);
        if (!any) break;
        if (vi == 0) {
            // the raw buffer is free once the previous group's last reader (its last Z epilogue) is
            // done, which is after its last second MMA batch: the Gram below overwrites its TMEM operands
            if (g > 0 && !wait_bar(B + PB_RAWFREE, (g - 1) & 1, budget)) { ok = false; break; }
            mbar_expect_tx(B + PB_TMA, 4 * 8192);
#pragma unroll
            for (int kb = 0; kb < 2; ++kb) {
                tma_load_3d(P.sm + PP_RAW + kb * 16384, tm_k, kb * 64, rec[U_HK], rec[U_TOK], B + PB_TMA);
                tma_load_3d(P.sm + PP_RAW + kb * 16384 + 8192, tm_q, kb * 64, rec[U_HK], rec[U_TOK], B + PB_TMA);
            }
            // the next group, found while this one is prepared (without SHARE straight into the other
            // record: the math threads read it at the start of the unit before this one, which ended
            // before RAWFREE above)
            grab(SHARE ? gnext : P.pu + 16 * ((h + 1) & 1));
            tma_pending = 1 + (int)(g & 1);
            if (!wait_bar(B + PB_TMA, g & 1, kDrainBudget)) { ok = false; break; }
            tma_pending = 0;
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {  // Gram [K; Q] K^T on the raw bf16 tiles (exact products)
                const uint64_t d = desc_sw128(P.sb + PP_RAW + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024);
                mma_bf16(P.tm + PT_G, d, d, ID_GRAM, ks > 0);
            }
        } else {
            // the same tiles, now K' and Q' in fp16: the Gram again (times sigma^2 on the K rows,
            // sigma sigma_q on the Q rows), once the previous unit's second batch has left TMEM
            if (!wait_bar(B + PB_M2, (h - 1) & 1, kDrainBudget)) { ok = false; break; }
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint64_t d = desc_sw128(P.sb + PP_RAW + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024);
                mma_f16_ss(P.tm + PT_G, d, d, ID_GRAM16, ks > 0);
            }
        }
        mma_commit(B + PB_G);
        if (!wait_bar(B + PB_M1REQ, h & 1, budget)) { ok = false; break; }
        tc_fence_after();
#pragma unroll 1
        for (int ks = 0; ks < 4; ++ks) {  // (sigma / kappa) W^T = K'^T Tw'^T (Tw' hi + lo)
            const uint64_t ak = desc_sw128(P.sb + PP_RAW + ks * 2048, 16384, 1024);
            mma_f16_ss(P.tm + PT_WT, ak, desc_sw128(P.sb + PP_TT + ks * 32, 16, 1024), ID_WT, ks > 0);
            mma_f16_ss(P.tm + PT_WT, ak, desc_sw128(P.sb + PP_TWLO + ks * 32, 16, 1024), ID_WT, 1);
        }
#pragma unroll 1
        for (int ks = 0; ks < 4; ++ks) {  // (sigma / kappa) B^T = K'^T Tb' (hi + lo)
            const uint64_t ak = desc_sw128(P.sb + PP_RAW + ks * 2048, 16384, 1024);
            mma_f16_ss(P.tm + PT_B, ak, desc_sw128(P.sb + PP_TT + 16384 + ks * 2048, 8192, 1024), ID_B, ks > 0);
            mma_f16_ss(P.tm + PT_B, ak, desc_sw128(P.sb + PP_TT + 24576 + ks * 2048, 8192, 1024), ID_B, 1);
        }
#pragma unroll 1
        for (int ks = 0; ks < 4; ++ks)  // E = Tb^T P^T
            mma_f16_ss(P.tm + PT_E, desc_sw128(P.sb + PP_TT + 8192 + ks * 2048, 8192, 1024),
                       desc_sw128(P.sb + PP_P + ks * 32, 16, 1024), ID_E, ks > 0);
        mma_commit(B + PB_M1);
        if (!wait_bar(B + PB_M2REQ, h & 1, budget)) { ok = false; break; }
        tc_fence_after();
#pragma unroll 1
        for (int ks = 0; ks < 4; ++ks)  // (sigma / kappa) N = -(W^T diag(d rk / kappa)) K', A = WTd' from TMEM
            mma_f16_ts(P.tm + PT_N, P.tm + PT_WT + 8 * ks, desc_sw128(P.sb + PP_RAW + ks * 2048, 16384, 1024), ID_N,
                       ks > 0);
#pragma unroll 1
        for (int ks = 0; ks < 4; ++ks)  // W^T P^T, A = WT from TMEM
            mma_f16_ts(P.tm + PT_WP, P.tm + PT_WT + 32 + 8 * ks, desc_sw128(P.sb + PP_P + ks * 32, 16, 1024), ID_WP,
                       ks > 0);
        mma_commit(B + PB_M2);
        if constexpr (SHARE) {  // the next unit's record: this group's next value head, or the next group's first
            int *nrec = P.pu + 16 * ((h + 1) & 1);
            if (vi + 1 < p.r) {
#pragma unroll
                for (int f = 0; f < 16; ++f) nrec[f] = rec[f];
                nrec[U_RI] = rec[U_RI] + 1;
                nrec[U_H] = rec[U_H] + 1;
                nrec[U_VI] = vi + 1;
                nrec[U_LAST] = vi + 2 == p.r;
            } else {
#pragma unroll
                for (int f = 0; f < 16; ++f) nrec[f] = gnext[f];
                ++g;
            }
        } else {
            ++g;
        }
    }
    if (tma_pending) wait_bar(B + PB_TMA, (uint32_t)(tma_pending - 1), kDrainBudget);  // tiles still landing
    mma_commit(B + PB_FIN);
    wait_bar(B + PB_FIN, 0, kDrainBudget);
    if (!ok) set_abort(p);
}

// ---- publisher thread: staged images -> ring slot, then the slot's flag ----
// It waits for a ring slot only after publishing everything before, so no prep CTA holds a
// written, unpublished block while it waits.
__device__ void prep_publisher(const RingParams &p, const Pipe &P) {
    const long long budget = p.wait_budget;
    uint64_t *B = P.bar;
    bool ok = true;
    for (uint32_t h = 0;; ++h) {
        if (!wait_bar(B + PB_BEREADY, h & 1, budget)) { ok = false; break; }
        const int ri = P.mail[0], us = P.mail[1];
        if (ri < 0) break;
        const int *cons = p.w.consumed + 32 * ri;
        const long long t0 = clock64();
        int spins = 0;
        while (ld_acquire_gpu(cons) < us - kSlots + 1) {
            if (((++spins) & 63) == 0 && (aborted(p) || clock64() - t0 > budget)) { ok = false; break; }
            __nanosleep(64);
        }
        if (!ok) break;
        uint8_t *slot = ring_slot(p, ri, us);
        fence_async_global();
        bulk_store(slot + RS_BE, P.sm + PP_AT, BE_HEAD);
        bulk_store(slot + RS_BE + BE_HEAD, P.sm + PP_TT, 2 * 24576 - BE_HEAD);
        bulk_commit();
        bulk_wait_read_all();
        mbar_arrive(B + PB_BEREAD);
        if (!wait_bar(B + PB_NZREADY, h & 1, budget)) { ok = false; break; }
        if (P.mail[3] != 0) break;  // the math threads gave up inside this unit
        bulk_store(slot + RS_N, P.sm + PP_AT, 32768);
        bulk_store(slot + RS_Z, P.sm + PP_TT + Z_STAGE, 16384);
        bulk_commit();
        bulk_wait_all();
        fence_async_global();
        p.w.slot_sc[((long)ri * kSlots + us % kSlots) * 4] = __int_as_float(P.mail[2]);
        st_release_gpu(p.w.slot_seq + 32 * ri + us % kSlots, us + 1);
        mbar_arrive(B + PB_STGFREE);
    }
    bulk_wait_all();
    if (!ok) set_abort(p);
}

// ---- math threads (128) ----
template <bool SHARE>
__device__ void prep_math(const RingParams &p, const Pipe &P, int mt, int bar_id) {
    const int warp = mt >> 5, lane = mt & 31;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const long long budget = p.wait_budget;
    uint64_t *B = P.bar;
    float *ps = P.ps;
    uint8_t *sm = P.sm;
    float *sA = reinterpret_cast<float *>(sm + PP_AT);
    float *sT = reinterpret_cast<float *>(sm + PP_T);
    bool failed = false;
    for (uint32_t h = 0;; ++h) {
        bool ab = !wait_bar(B + PB_UREADY, h & 1, budget);
        if (bar_any(bar_id, 128, ab)) { failed = true; break; }
        const int *ur = P.pu + 16 * (h & 1);
        if (ur[U_VALID] == 0) break;
        const int us = ur[U_S], ri = ur[U_RI], hv = ur[U_H], tok0 = ur[U_TOK], L = ur[U_L];
        const int vi = SHARE ? ur[U_VI] : 0;  // > 0: the key-side work of this key head is done
        const bool last_of_group = SHARE ? ur[U_LAST] != 0 : true;
        // ---- gates: loads issued now, used once the tiles and the Gram are ready (their latency hides) ----
        // (raw 16-bit values: converting them here would wait for the loads)
        unsigned short g0 = 0, g1 = 0, bl = 0;
        const unsigned short *gr = reinterpret_cast<const unsigned short *>(p.g);
        const unsigned short *br = reinterpret_cast<const unsigned short *>(p.b);
        if (warp == 0) {
            if (lane < L) g0 = gr[(long)(tok0 + lane) * p.Hv + hv];
            if (lane + 32 < L) g1 = gr[(long)(tok0 + lane + 32) * p.Hv + hv];
        } else if (warp == 1 || warp == 2) {
            const int t = mt - 32;
            if (t < L) bl = br[(long)(tok0 + t) * p.Hv + hv];
        }
        ab = !wait_bar(B + PB_G, h & 1, budget);
        if (bar_any(bar_id, 128, ab)) { failed = true; break; }
        tc_fence_after();
        if (warp == 0) {
            float x0 = __uint_as_float((uint32_t)g0 << 16), x1 = __uint_as_float((uint32_t)g1 << 16);
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y0 = __shfl_up_sync(0xffffffffu, x0, o);
                const float y1 = __shfl_up_sync(0xffffffffu, x1, o);
                if (lane >= o) { x0 += y0; x1 += y1; }
            }
            x1 += __shfl_sync(0xffffffffu, x0, 31);
            ps[PS_G + lane] = x0;
            ps[PS_G + lane + 32] = x1;
            float mn = fminf(x0, lane + 32 < L ? x1 : x0), mx = fmaxf(x0, lane + 32 < L ? x1 : x0);
            if (lane >= L) { mn = 3.0e38f; mx = -3.0e38f; }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            }
            if (lane == 0) {
                ps[PS_MISC + 0] = mn;
                ps[PS_MISC + 1] = mx;
            }
        } else if (warp == 1 || warp == 2) {
            const int t = mt - 32;
            ps[PS_BETA + t] = t < L ? sigmoidf_(__uint_as_float((uint32_t)bl << 16)) : 0.f;
        }
        bar_sync(bar_id, 128);
        if (mt < 64) {
            const float gmin = ps[PS_MISC + 0], gmax = ps[PS_MISC + 1];
            const float G = ps[PS_G + mt], GL = ps[PS_G + L - 1];
            ps[PS_E + mt] = expf(G);
            ps[PS_AA + mt] = expf(G - gmin);
            ps[PS_D + mt] = mt < L ? expf(GL - G) : 0.f;
            if (mt == 0) {
                ps[PS_MISC + 2] = (gmax - gmin) < 80.f ? 1.f : 0.f;  // e^{G_t-G_s} = a_t b_s safely
                ps[PS_MISC + 3] = expf(GL);
            }
        }
        if (vi == 0) {  // row norms of [K; Q] (row mt) and the largest magnitude of the K (and Q) tile
            float ssq = 0.f, kmax = 0.f;
#pragma unroll
            for (int kb = 0; kb < 2; ++kb)
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    float x[8];
                    unpack8(*reinterpret_cast<const uint4 *>(sm + PP_RAW + kb * 16384 + swz(mt, c)), x);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        ssq = fmaf(x[e], x[e], ssq);
                        kmax = fmaxf(kmax, fabsf(x[e]));
                    }
                }
            const int row = mt & 63;
            const float rn = row < L ? rsqrtf(ssq + kNormEps) : 0.f;
            (mt < 64 ? ps + PS_RK : ps + PS_RQ)[row] = rn;
            kmax = warp_max((SHARE || mt < 64) && row < L ? kmax : 0.f);
            const float rkmax = warp_max(mt < 64 ? rn : 0.f);
            if (lane == 0) {
                ps[PS_RED + warp] = kmax;
                ps[PS_RED + 4 + warp] = rkmax;
            }
        }
        // iq = 1 / sigma_q when the Z epilogue reads Q'; kappa: a power of two at or above every rk
        float iq = 1.f, sigma = 1.f, sigma_q = 1.f, kappa;
        if (vi == 0) {
            bar_sync(bar_id, 128);
            // K' = sigma K (and, with SHARE, Q' = sigma_q Q) stay below 2^14 in fp16; every product
            // with them is taken back in fp32 in its epilogue (the fp16 operands keep their natural range)
            sigma = pow2_scale(fmaxf(ps[PS_RED + 0], ps[PS_RED + 1]));  // K rows: warps 0, 1
            // rk enters the fp16 operands Tw', Tb' and W^T diag(d rk) as rk / kappa (at most 1): for
            // keys of large norm rk itself would put them among fp16's subnormals
            kappa = pow2_above(fmaxf(ps[PS_RED + 4], ps[PS_RED + 5]));
            if constexpr (SHARE) {
                sigma_q = pow2_scale(fmaxf(ps[PS_RED + 2], ps[PS_RED + 3]));
                iq = 1.f / sigma_q;
            }
        } else {
            iq = ps[PS_MISC + 5];
            kappa = ps[PS_MISC + 6];
        }
        if (mt < 64) {  // the gate-dependent row scalars (rk, rq and the scales are the key head's)
            const float rk = ps[PS_RK + mt], rkk = rk * (1.f / kappa);
            ps[PS_BBRK + mt] = expf(ps[PS_MISC + 0] - ps[PS_G + mt]) * rk;
            ps[PS_TWF + mt] = ps[PS_BETA + mt] * ps[PS_E + mt] * rkk;
            ps[PS_DRK + mt] = ps[PS_D + mt] * rkk;
            ps[PS_ER + mt] = SHARE ? ps[PS_E + mt] * ps[PS_RQ + mt] * iq : ps[PS_E + mt] * ps[PS_RQ + mt];  // Qt rows
            if (mt == 0 && vi == 0) {
                ps[PS_MISC + 4] = 1.f / sigma;
                ps[PS_MISC + 6] = kappa;
                if constexpr (SHARE) ps[PS_MISC + 5] = iq;
            }
        }
        if (vi == 0) {
            // K (and with SHARE Q) rows -> fp16, in place (the Gram that read them is complete); rows
            // beyond L (the next sequence, or past the end) become zero. A group's later units use them.
            const int t = mt & 63, kb = mt >> 6;
            const float sg = t < L ? sigma : 0.f;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                uint4 *pk = reinterpret_cast<uint4 *>(sm + PP_RAW + kb * 16384 + swz(t, c));
                float x[8];
                unpack8(*pk, x);
                *pk = pack8_f16(x, sg);
            }
            if constexpr (SHARE) {
                const float sq = t < L ? sigma_q : 0.f;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint4 *pq = reinterpret_cast<uint4 *>(sm + PP_RAW + kb * 16384 + swz(64 + t, c));
                    float y[8];
                    unpack8(*pq, y);
                    *pq = pack8_f16(y, sq);
                }
            }
        }
        fence_async_smem();
        // the previous unit's staged images must be read out before A, T and the tiles overwrite them
        ab = h > 0 && !wait_bar(B + PB_STGFREE, (h - 1) & 1, budget);
        if (bar_any(bar_id, 128, ab)) { failed = true; break; }
        {  // A rows (fp32) and P rows (fp16) from the Gram: thread mt reads Gram row mt
            const int row = mt & 63;
            const bool isq = mt >= 64;
            float nt = isq ? ps[PS_RQ + row] : ps[PS_RK + row] * ps[PS_BETA + row];
            if (SHARE && vi > 0) {  // a group's later units: the fp16 Gram carries sigma^2 (K rows), sigma sigma_q (Q rows)
                const float isg = ps[PS_MISC + 4];
                nt *= isq ? isg * iq : isg * isg;
            }
            uint32_t gv[2][32];
            tmem_ld32_nw(P.tm + lane_off + PT_G, gv[0]);
            tmem_ld32_nw(P.tm + lane_off + PT_G + 32, gv[1]);
            tmem_wait_ld();
            float x[64];
            if (ps[PS_MISC + 2] != 0.f) {  // e^{G_t-G_s} = a_t b_s (uniform over the CTA)
                const float at = nt * ps[PS_AA + row];
#pragma unroll
                for (int e4 = 0; e4 < 16; ++e4) {
                    const float4 bb = ps4(ps, PS_BBRK + 4 * e4);
                    const float bv[4] = {bb.x, bb.y, bb.z, bb.w};
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int e = 4 * e4 + u;
                        x[e] = __uint_as_float(gv[e >> 5][e & 31]) * at * bv[u];
                    }
                }
            } else {  // a gate range too wide to factor: one exponential per element
                const float Gt = ps[PS_G + row];
#pragma unroll
                for (int e4 = 0; e4 < 16; ++e4) {
                    const float4 r4 = ps4(ps, PS_RK + 4 * e4), g4 = ps4(ps, PS_G + 4 * e4);
                    const float rv[4] = {r4.x, r4.y, r4.z, r4.w}, gg[4] = {g4.x, g4.y, g4.z, g4.w};
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int e = 4 * e4 + u;
                        x[e] = __uint_as_float(gv[e >> 5][e & 31]) * nt * rv[u] * __expf(Gt - gg[u]);
                    }
                }
            }
            if (isq) {
#pragma unroll
                for (int e = 0; e < 64; ++e) x[e] = e <= row ? x[e] : 0.f;
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    *reinterpret_cast<uint4 *>(sm + PP_P + swz(row, c)) = pack8_f16(&x[8 * c], 1.f);
            } else {
#pragma unroll
                for (int e = 0; e < 64; ++e) x[e] = e < row ? x[e] : 0.f;
#pragma unroll
                for (int e4 = 0; e4 < 16; ++e4)
                    *reinterpret_cast<float4 *>(sA + row * LS + 4 * e4) =
                        make_float4(x[4 * e4], x[4 * e4 + 1], x[4 * e4 + 2], x[4 * e4 + 3]);
            }
        }
        tc_fence_before();
        bar_sync(bar_id, 128);
        solve128(sA, sT, mt, bar_id);
        // Tw' [t][s] and Tb' = diag(d rk / kappa) T diag(beta) as fp16 hi + lo, Tb [m][s] fp16. Tw' takes
        // a lo part too: with nearly parallel keys W = Tw Kh cancels to a small fraction of its terms,
        // and a single fp16 Tw' left the state's error at ~1e-3 of its norm.
        {
            const int tt = mt >> 1, hh = mt & 1;
            const float drk = ps[PS_DRK + tt];
            auto split16 = [](const float *x, uint4 &hi, uint4 &lo) {  // x = hi + lo + O(2^-22 |x|)
                hi = pack8_f16(x, 1.f);
                const __half2 *h2 = reinterpret_cast<const __half2 *>(&hi);
                float r[8];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = __half22float2(h2[e]);
                    r[2 * e] = x[2 * e] - f.x;
                    r[2 * e + 1] = x[2 * e + 1] - f.y;
                }
                lo = pack8_f16(r, 1.f);
            };
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8) {
                float tw[8], tb[8], tp[8];
#pragma unroll
                for (int c4 = 0; c4 < 2; ++c4) {
                    const int s0 = 32 * hh + 8 * c8 + 4 * c4;
                    const float4 t4 = *reinterpret_cast<const float4 *>(sT + tt * LS + s0);
                    const float tv[4] = {t4.x, t4.y, t4.z, t4.w};
                    const float4 b4 = ps4(ps, PS_BETA + s0), w4 = ps4(ps, PS_TWF + s0);
                    const float bev[4] = {b4.x, b4.y, b4.z, b4.w}, twv[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        tb[4 * c4 + e] = tv[e] * bev[e];
                        tw[4 * c4 + e] = tv[e] * twv[e];
                        tp[4 * c4 + e] = tb[4 * c4 + e] * drk;
                    }
                }
                const int c = 4 * hh + c8;
                uint4 hi, lo;
                split16(tw, hi, lo);
                *reinterpret_cast<uint4 *>(sm + PP_TT + swz(tt, c)) = hi;
                *reinterpret_cast<uint4 *>(sm + PP_TWLO + swz(tt, c)) = lo;
                *reinterpret_cast<uint4 *>(sm + PP_TT + 8192 + swz(tt, c)) = pack8_f16(tb, 1.f);
                split16(tp, hi, lo);
                *reinterpret_cast<uint4 *>(sm + PP_TT + 16384 + swz(tt, c)) = hi;
                *reinterpret_cast<uint4 *>(sm + PP_TT + 24576 + swz(tt, c)) = lo;
            }
        }
        fence_async_smem();
        tc_fence_before();
        bar_sync(bar_id, 128);
        if (mt == 0) mbar_arrive(B + PB_M1REQ);
        ab = !wait_bar(B + PB_M1, h & 1, budget);
        if (bar_any(bar_id, 128, ab)) { failed = true; break; }
        tc_fence_after();
        {  // W^T row j -> WTd' = W^T diag(d rk / kappa) and WT (fp16) as TMEM A operands, in place
            const int j = mt;
            uint32_t w0[32], w1[32];
            tmem_ld32_nw(P.tm + lane_off + PT_WT, w0);
            tmem_ld32_nw(P.tm + lane_off + PT_WT + 32, w1);
            tmem_wait_ld();
            (void)j;
            uint32_t a[32], b[32];
            const float isg = ps[PS_MISC + 4] * ps[PS_MISC + 6];  // kappa / sigma
#pragma unroll
            for (int e2 = 0; e2 < 8; ++e2) {
                const float4 d0 = ps4(ps, PS_DRK + 4 * e2), d1 = ps4(ps, PS_DRK + 32 + 4 * e2);
                const float dv0[4] = {d0.x, d0.y, d0.z, d0.w}, dv1[4] = {d1.x, d1.y, d1.z, d1.w};
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int e = 2 * e2 + u;
                    const float x0 = __uint_as_float(w0[2 * e]) * isg, x1 = __uint_as_float(w0[2 * e + 1]) * isg;
                    const float y0 = __uint_as_float(w1[2 * e]) * isg, y1 = __uint_as_float(w1[2 * e + 1]) * isg;
                    a[e] = h2_bits(x0 * dv0[2 * u], x1 * dv0[2 * u + 1]);
                    a[16 + e] = h2_bits(y0 * dv1[2 * u], y1 * dv1[2 * u + 1]);
                    b[e] = h2_bits(x0, x1);
                    b[16 + e] = h2_bits(y0, y1);
                }
            }
            tmem_st32(P.tm + lane_off + PT_WT, a);
            tmem_st32(P.tm + lane_off + PT_WT + 32, b);
        }
        // the [B^T | E] image (bf16 hi + lo), staged in AT and then TT: image byte o -> stage address
        auto stage_be = [&](uint32_t o) { return o < BE_HEAD ? sm + PP_AT + o : sm + PP_TT + (o - BE_HEAD); };
        {  // B^T row n (all 128 lanes), taken back by kappa / sigma: K-major [n][t]
            const int n = mt;
            const float isg = ps[PS_MISC + 4] * ps[PS_MISC + 6];  // kappa / sigma
            uint32_t bv[2][32];
            tmem_ld32_nw(P.tm + lane_off + PT_B, bv[0]);
            tmem_ld32_nw(P.tm + lane_off + PT_B + 32, bv[1]);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                float x[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = __uint_as_float(bv[c >> 2][8 * (c & 3) + e]) * isg;
                uint4 hi, lo;
                pack8_hilo(x, hi, lo);
                *reinterpret_cast<uint4 *>(stage_be(swz(n, c))) = hi;
                *reinterpret_cast<uint4 *>(stage_be(16384 + swz(n, c))) = lo;
            }
        }
        {  // E row t (M = 64: warp w holds rows 16 w .. 16 w + 15 in lanes 0..15): MN-major [t][s]
            const int t = 16 * warp + lane;
            uint32_t ev[2][32];
            tmem_ld32_nw(P.tm + lane_off + PT_E, ev[0]);
            tmem_ld32_nw(P.tm + lane_off + PT_E + 32, ev[1]);
            tmem_wait_ld();
            if (lane < 16) {
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    float x[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) x[e] = __uint_as_float(ev[c >> 2][8 * (c & 3) + e]);
                    uint4 hi, lo;
                    pack8_hilo(x, hi, lo);
                    *reinterpret_cast<uint4 *>(stage_be(32768 + swz(t, c))) = hi;
                    *reinterpret_cast<uint4 *>(stage_be(40960 + swz(t, c))) = lo;
                }
            }
        }
        tmem_wait_st();
        fence_async_smem();
        tc_fence_before();
        bar_sync(bar_id, 128);
        if (mt == 0) {
            P.mail[0] = ri;
            P.mail[1] = us;
            mbar_arrive(B + PB_M2REQ);
            mbar_arrive(B + PB_BEREADY);
        }
        ab = !wait_bar(B + PB_M2, h & 1, budget);
        if (bar_any(bar_id, 128, ab)) { failed = true; break; }
        tc_fence_after();
        // Z row j: Z[j][t] = e_t rq_t Q[t][j] - (W^T P^T)[j][t] -> fp16 image (MN-major [j][t]) in TT,
        // Q read raw (bf16) or, with SHARE, as Q' (fp16; ER carries 1 / sigma_q)
        auto z_epilogue = [&](auto q_is_f16) {
            const int j = mt, qb = j >> 6, qc = (j & 63) >> 3, qe = j & 7;
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                uint32_t wv[32];
                tmem_ld32_nw(P.tm + lane_off + PT_WP + 32 * q, wv);
                tmem_wait_ld();
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    float x[8];
                    const float4 r0 = ps4(ps, PS_ER + 32 * q + 8 * cc), r1 = ps4(ps, PS_ER + 32 * q + 8 * cc + 4);
                    const float er[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int t = 32 * q + 8 * cc + e, row = 64 + t;
                        const uint8_t *qa = sm + PP_RAW + qb * 16384 + row * 128 + ((qc ^ (row & 7)) << 4) + 2 * qe;
                        float qf;
                        if constexpr (decltype(q_is_f16)::value)
                            qf = __half2float(*reinterpret_cast<const __half *>(qa));
                        else
                            qf = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(qa));
                        x[e] = er[e] * qf - __uint_as_float(wv[8 * cc + e]);
                    }
                    *reinterpret_cast<uint4 *>(sm + PP_TT + Z_STAGE + swz(j, 4 * q + cc)) = pack8_f16(x, 1.f);
                }
            }
        };
        z_epilogue(std::integral_constant<bool, SHARE>{});
        bar_sync(bar_id, 128);
        if (mt == 0 && last_of_group) mbar_arrive(B + PB_RAWFREE);  // the tiles' last reader is done
        ab = !wait_bar(B + PB_BEREAD, h & 1, budget);  // AT holds the [B|E] head until it is read out
        if (bar_any(bar_id, 128, ab)) { failed = true; break; }
        {  // N row j -> fp16 (-N), MN-major [j][n] image in AT
            const int j = mt;
            const float nsg = -ps[PS_MISC + 4] * ps[PS_MISC + 6];  // -kappa / sigma
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t nv[32];
                tmem_ld32_nw(P.tm + lane_off + PT_N + 32 * q, nv);
                tmem_wait_ld();
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    float x[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) x[e] = __uint_as_float(nv[8 * cc + e]);
                    const int n0 = 32 * q + 8 * cc, blk = n0 >> 6, c = (n0 & 63) >> 3;
                    *reinterpret_cast<uint4 *>(sm + PP_AT + blk * 16384 + swz(j, c)) = pack8_f16(x, nsg);
                }
            }
        }
        fence_async_smem();
        tc_fence_before();
        bar_sync(bar_id, 128);
        if (mt == 0) {
            P.mail[2] = __float_as_int(ps[PS_MISC + 3]);
            mbar_arrive(B + PB_NZREADY);
        }
    }
    if (mt == 0) {  // stop the publisher: at its next unit, or (after a failure) wherever it waits
        P.mail[0] = -1;
        if (failed) P.mail[3] = 1;
        mbar_arrive(B + PB_BEREADY);
        if (failed) mbar_arrive(B + PB_NZREADY);
    }
    if (failed && mt == 0) set_abort(p);
}

template <bool SHARE>
__device__ void prep_cta(const CUtensorMap *tm_q, const CUtensorMap *tm_k, const RingParams &p, uint8_t *sm,
                         uint32_t sb, uint32_t tmem) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (warp < 8) {
        const int pipe = warp >> 2;
        prep_math<SHARE>(p, make_pipe(sm, sb, tmem, pipe), tid & 127, 1 + pipe);
    } else if (lane == 0 && warp < 10) {
        prep_control<SHARE>(tm_q, tm_k, p, make_pipe(sm, sb, tmem, warp - 8));
    } else if (lane == 0) {
        prep_publisher(p, make_pipe(sm, sb, tmem, warp - 10));
    }
}

// SHARE: a preparing pipeline takes the r value heads of a key head at a step in a row (see prep_control)
template <bool SHARE>
__global__ void __launch_bounds__(kThreads, 1)
prefill_ring_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                    const RingParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *sm = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    const uint32_t sb = smem_u32(sm);
    const bool chain = blockIdx.x < (unsigned)p.NC;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + (chain ? CH_BAR : PP_BAR));
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + (chain ? CH_BAR + 240 : PP_BAR + 240));
    const int tid = threadIdx.x, warp = tid >> 5;
    if (tid == 0) {
        if (chain) {
            for (int j = 0; j < 4; ++j) mbar_init(bars + j, 1);       // full[2], free[2]
            mbar_init(bars + 4, 1);                                    // d1
            mbar_init(bars + 5, 1);                                    // o1
            mbar_init(bars + 6, 256);                                  // s16
            mbar_init(bars + 7, 256);                                  // d2free
            mbar_init(bars + 8, 256);                                  // o12free
            mbar_init(bars + 9, 1);                                    // scb[2]
            mbar_init(bars + 10, 1);
            mbar_init(bars + 11, 1);                                   // fin
            mbar_init(bars + 12, 1);                                   // fulle[2]
            mbar_init(bars + 13, 1);
            mbar_init(bars + 14, 256);                                 // ostaged[2]
            mbar_init(bars + 15, 256);
        } else {
            for (int pipe = 0; pipe < 2; ++pipe) {
                uint64_t *pb = reinterpret_cast<uint64_t *>(sm + pipe * PP_BYTES + PP_BAR);
                for (int j = 0; j < PB_COUNT; ++j) mbar_init(pb + j, 1);
                reinterpret_cast<int *>(sm + pipe * PP_BYTES + PP_SC)[PS_MAIL + 3] = 0;
            }
        }
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(tmem_slot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (chain)
        chain_cta(&tm_v, &tm_o, p, sm, sb, tmem);
    else
        prep_cta<SHARE>(&tm_q, &tm_k, p, sm, sb, tmem);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
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

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// how the launch splits into chain CTAs and prep CTAs
struct RingShape {
    int sms, NC, G, npos;
};
bool ring_shape(const PrefillArgs &a, RingShape *sh, int max_chain_ctas) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    if (cudaDeviceGetAttribute(&sh->sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
    const int r = a.Hv / a.Hk;
    const long chains = (long)a.B * a.Hv;
    // 9/38 of the SMs (36 of 152) carry states; the rest prepare blocks (measured on 16 packed
    // sequences with key sharing: 36 state CTAs beat 32, 34, 38, 40 and 44 by 1-7%; 30 and 50 are
    // 10-20% slower; a single sequence needs one CTA per head, which 36 covers for 32 heads). A
    // multiple of r, so that the value heads of one key head sit in consecutive chain CTAs at the
    // same steps.
    long nc = std::min<long>(chains, std::max(1, sh->sms * 9 / 38));
    if (max_chain_ctas > 0) nc = std::min<long>(nc, max_chain_ctas);
    nc = std::max<long>(r, nc / r * r);
    if (nc + 8 > sh->sms) return false;
    sh->NC = (int)nc;
    sh->G = (int)(nc / r);
    sh->npos = (int)((chains + nc - 1) / nc);
    return true;
}

struct WsLayout {
    size_t ctl, consumed, slot_seq, slot_sc, seq_rank, nblk, first_step, total_steps, ring, bytes;
};
WsLayout ws_layout(const PrefillArgs &a, const RingShape &sh) {
    WsLayout L;
    size_t o = 0;
    L.ctl = o; o += 128 * 4;
    L.consumed = o; o += (size_t)sh.NC * 32 * 4;
    L.slot_seq = o; o += (size_t)sh.NC * 32 * 4;
    L.slot_sc = o; o += align_up((size_t)sh.NC * kSlots * 4 * 4, 128);
    L.seq_rank = o; o += align_up((size_t)a.B * 4, 128);
    L.nblk = o; o += align_up((size_t)a.B * 4, 128);
    L.first_step = o; o += align_up((size_t)sh.G * (sh.npos + 1) * 4, 128);
    L.total_steps = o; o += align_up((size_t)sh.G * 4, 128);
    o = align_up(o, 1024);
    L.ring = o; o += (size_t)sh.NC * kSlots * RS_BYTES;
    L.bytes = o;
    return L;
}

}  // namespace

bool prefill_ring_supported(const PrefillArgs &a) {
    const long Ttot = a.cu_seqlens ? (long)a.T : (long)a.B * a.T;
    if (!(a.dtype == GDN_BF16 && a.dk == DK && a.dv == DV && a.chunk == C && Ttot > 0)) return false;
    RingShape sh;
    return ring_shape(a, &sh, 0);
}

size_t prefill_ring_workspace(const PrefillArgs &a, int max_chain_ctas) {
    RingShape sh;
    if (!ring_shape(a, &sh, max_chain_ctas)) return 0;
    return ws_layout(a, sh).bytes;
}

cudaError_t launch_prefill_ring(const PrefillArgs &a, void *ws, size_t ws_bytes, cudaStream_t s,
                                int max_chain_ctas) {
    RingShape sh;
    if (!ring_shape(a, &sh, max_chain_ctas)) return cudaErrorInvalidValue;
    const WsLayout L = ws_layout(a, sh);
    if (!ws || ws_bytes < L.bytes || (reinterpret_cast<uintptr_t>(ws) & 255u)) return cudaErrorInvalidValue;
    const long Ttot = a.cu_seqlens ? (long)a.T : (long)a.B * a.T;
    CUtensorMap mq, mk, mv, mo;
    if (!make_map(&mq, a.q, DK, a.Hk, Ttot) || !make_map(&mk, a.k, DK, a.Hk, Ttot) ||
        !make_map(&mv, a.v, DV, a.Hv, Ttot) || !make_map(&mo, a.out, DV, a.Hv, Ttot))
        return cudaErrorInvalidValue;
    // key-side sharing pays when there are more chains than state CTAs (throughput-bound)
    const bool share = a.Hv > a.Hk && (long)a.B * a.Hv > sh.NC;
    auto kernel = share ? prefill_ring_kernel<true> : prefill_ring_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    uint8_t *w = static_cast<uint8_t *>(ws);
    RingParams p{};
    p.g = (const __nv_bfloat16 *)a.g;
    p.b = (const __nv_bfloat16 *)a.b;
    p.state_in = a.state_in;
    p.state_out = a.state_out;
    p.out = (__nv_bfloat16 *)a.out;
    p.cu = a.cu_seqlens;
    p.B = a.B;
    p.Hk = a.Hk;
    p.Hv = a.Hv;
    p.r = a.Hv / a.Hk;
    p.T = a.T;
    p.Ttot = Ttot;
    p.NC = sh.NC;
    p.G = sh.G;
    p.npos = sh.npos;
    p.status = a.status;
    p.wait_budget = kWaitDefault;
    if (const char *env = getenv("GDN_TEST_WAIT_CYCLES")) {  // test hook: a short limit makes the waits run out
        const long long x = atoll(env);
        if (x > 0) p.wait_budget = x;
    }
    p.w.ctl = reinterpret_cast<int *>(w + L.ctl);
    p.w.consumed = reinterpret_cast<int *>(w + L.consumed);
    p.w.slot_seq = reinterpret_cast<int *>(w + L.slot_seq);
    p.w.slot_sc = reinterpret_cast<float *>(w + L.slot_sc);
    p.w.seq_rank = reinterpret_cast<int *>(w + L.seq_rank);
    p.w.nblk = reinterpret_cast<int *>(w + L.nblk);
    p.w.first_step = reinterpret_cast<int *>(w + L.first_step);
    p.w.total_steps = reinterpret_cast<int *>(w + L.total_steps);
    p.w.ring = w + L.ring;
    ring_plan_kernel<<<1, 1024, 0, s>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeCooperative;
    attr.val.cooperative = 1;
    cfg.gridDim = dim3((unsigned)sh.sms, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = s;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, mq, mk, mv, mo, p);
}

}  // namespace gdn
