/*
 * gdn.h -- C ABI of the GB300 (sm_103a) gated delta rule layer.
 *
 * The layer keeps, per sequence and value head, a fixed-size matrix state
 * S in R^{dv x dk}. A learned gate decides how much of the old state to keep
 * and a delta update writes the current token into it; every token depends on
 * the state left by the previous one ("Optimiser l'inference sur appareil
 * pour Apple Silicon", section "Qwen cree trois formes de charges de
 * travail"). With qh = q/sqrt(|q|^2+1e-6), kh likewise, alpha = exp(g),
 * beta = sigmoid(b), one token does
 *
 *     S <- alpha S (I - beta kh kh^T) + beta v kh^T,      o = S qh
 *
 * (the read-out uses the updated state). State and gate arithmetic is fp32
 * because rounding accumulates over sequential updates, while q/k/v stay in
 * bf16 (same page, section "Maintenir l'etat recurrent sur la puce").
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All array arguments are DEVICE pointers owned by the caller; the library
 *    never frees or keeps them. Every pointer must be 16-byte aligned.
 *  - Packed token layouts, row-major:
 *        q, k   [Ttot][Hk][dk]        v, out [Ttot][Hv][dv]
 *        g, b   [Ttot][Hv]            (g: log-decay; b: beta logit)
 *        state  [B][Hv][dv][dk] fp32  (row i of S is contiguous)
 *  - Value head h reads key head h / (Hv/Hk) (consecutive value heads share
 *    a key head); Hv must be a multiple of Hk.
 *  - `dtype` (gdn_dtype) is the element type of q, k, v, g, b and out; the
 *    state is always fp32.
 *  - q and k are raw: the library L2-normalises them per head.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream). Calls are
 *    asynchronous on it and never synchronise it, except
 *    gdn_get_device_status.
 *  - Argument errors are reported by the return value before any device work
 *    is queued; nothing aborts or exits the process.
 *  - Inconsistent device-side data that the host cannot see (cu_seqlens not
 *    starting at 0, decreasing, or not ending at T) is reported through the
 *    library's device status word; the affected sequences are skipped.
 */
#ifndef GDN_GB300_H
#define GDN_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define GDN_API __attribute__((visibility("default")))
#else
#define GDN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = -1,  /* null pointer, bad size, misaligned pointer */
    GDN_ERR_UNSUPPORTED = -2,  /* valid but unsupported dk/dv/chunk/dtype    */
    GDN_ERR_CUDA = -3,         /* a CUDA runtime/driver call failed          */
    GDN_ERR_DEVICE_CHECK = -4  /* a kernel found inconsistent device data    */
} gdn_status;

typedef enum { GDN_BF16 = 0, GDN_F32 = 1 } gdn_dtype;

/*
 * gdn_prefill -- run the recurrence over whole prompts (chunked prefill).
 *
 * Evaluates the same function as the token scan by regrouping each run of
 * `chunk` tokens into a block whose updates become matrix products ("Qwen cree
 * trois formes de charges de travail": blocks expose matrix operations and
 * token-level parallelism). Within a block of L tokens starting from state
 * S0, with G_t the in-block cumulative log-gate:
 *     A_ts = beta_t e^{G_t-G_s} kh_t.kh_s (s<t),   T = (I + A)^-1,
 *     U    = T diag(beta) V - T diag(beta e^G) Kh S0^T,
 *     O    = diag(e^G) Qh S0^T + P U,   P_ts = e^{G_t-G_s} qh_t.kh_s (s<=t),
 *     S    = e^{G_L} S0 + U^T diag(e^{G_L-G_t}) Kh.
 * The state enters from state_in and leaves in state_out, so a long prompt may
 * be cut into fragments whose state is carried from one call to the next with
 * an unchanged result ("Limiter la memoire temporaire grace au decoupage des
 * prompts").
 *
 *   q, k, v, g, b : packed inputs (layouts above), Ttot tokens.
 *   state_in      : [B][Hv][dv][dk] fp32 initial states, or NULL for zeros.
 *   state_out     : [B][Hv][dv][dk] fp32 final states; may equal state_in
 *                   (in-place update). A zero-length sequence copies its
 *                   initial state through.
 *   out           : [Ttot][Hv][dv] outputs, dtype `dtype`.
 *   cu_seqlens    : device int32 [B+1] sequence offsets (0 = cu[0] <= ... <=
 *                   cu[B] = T), or NULL: B sequences of T tokens each
 *                   (Ttot = B*T).
 *   B, T          : sequence count; tokens per sequence (cu_seqlens NULL) or
 *                   total packed tokens (cu_seqlens given).
 *   Hk, Hv, dk, dv: head counts and head dimensions; dk, dv in {32, 64, 128}.
 *   chunk         : block length, one of 16, 32, 64. The tensor-core kernels take bf16 with
 *                   dk = dv = 128 and chunk 64; every other supported combination (chunk 16
 *                   or 32, fp32, dk or dv of 32 or 64) runs a CUDA-core block kernel that is
 *                   correct but is not a performance path (gdn_prefill_path returns 0 for it).
 * Sequences of at most 8 tokens each (cu_seqlens NULL, T <= 8: a few tokens
 * per sequence, e.g. checking a run of speculated tokens) are evaluated as a
 * token scan instead: every state row is read once, takes the T updates in
 * order in registers, and is written once, so T steps cost one pass over the
 * state. The result is the same function (only the rounding order differs).
 * Accuracy: the tensor-core kernel multiplies fp16 or bf16 operands into fp32 accumulators,
 * with power-of-two scales chosen at run time (so the fp16 operands stay in range whatever the
 * scale of q, k, v and the state) and operands that carry v into the state, or that cancel,
 * split into hi + lo pairs. Against an fp64 token scan the final states stay within 1e-3
 * (relative Frobenius) and the outputs within 2e-2 x RMS (max-abs) plus their one rounding to
 * the output dtype; measured on random inputs, slow and fast gates, q and k scaled by 1e-3 to
 * 300, v and states by 1e-4 to 1e4, and nearly parallel keys with beta near 1.
 * The tensor-core path needs device scratch (see gdn_prefill_workspace_size); gdn_prefill
 * keeps one workspace per device for it, allocated by the first call that needs it and grown
 * (after the work using the old one has finished) when a call needs more. Calls on different
 * streams are ordered on the GPU so that they never use it at once. Inside a stream capture
 * no allocation and no cross-stream ordering can be made: make one call of the same sizes (or
 * larger) outside the capture first, and do not let a captured prefill run at the same time as
 * another prefill of the same device; otherwise use gdn_prefill_ws with a workspace per stream.
 * Returns GDN_OK, GDN_ERR_INVALID_ARG, GDN_ERR_UNSUPPORTED or GDN_ERR_CUDA (also when the
 * workspace cannot be allocated, or would have to be inside a stream capture).
 */
GDN_API int gdn_prefill(const void *q, const void *k, const void *v, const void *g, const void *b,
                const float *state_in, float *state_out, void *out, const int32_t *cu_seqlens,
                int B, int T, int Hk, int Hv, int dk, int dv, int chunk, int dtype, void *stream);

/*
 * gdn_prefill_workspace_size -- bytes of device workspace gdn_prefill_ws needs for these
 * sizes, with or without cu_seqlens (0: the kernel for these sizes needs none, or the sizes are
 * invalid).
 *
 * The tensor-core prefill (dk = dv = 128, chunk 64, bf16) splits the GPU into CTAs that carry
 * the states and CTAs that prepare blocks for them, which hand each block's operands over
 * through a ring of slots in device memory; the workspace holds that ring (a fixed 96 KiB per
 * slot, 16 slots per state-carrying CTA) plus per-call tables that grow with B and Hv. It is
 * scratch: nothing in it outlives a call. Host-only, no device work.
 */
GDN_API size_t gdn_prefill_workspace_size(int B, int T, int Hk, int Hv, int dk, int dv, int chunk,
                                          int dtype);

/*
 * gdn_prefill_ws -- gdn_prefill with a caller-owned workspace.
 *
 * Same arguments and result as gdn_prefill, plus `workspace`: DEVICE memory of at least
 * gdn_prefill_workspace_size(...) bytes, 256-byte aligned (as cudaMalloc returns), which the
 * call uses as scratch until its work on `stream` has finished. Calls whose work may overlap
 * on the GPU must use different workspaces. When the size function returns 0, `workspace`
 * may be NULL. Returns GDN_ERR_INVALID_ARG when the workspace is missing, too small or
 * misaligned; otherwise as gdn_prefill.
 */
GDN_API int gdn_prefill_ws(const void *q, const void *k, const void *v, const void *g, const void *b,
                           const float *state_in, float *state_out, void *out, const int32_t *cu_seqlens,
                           int B, int T, int Hk, int Hv, int dk, int dv, int chunk, int dtype,
                           void *workspace, size_t workspace_bytes, void *stream);

/*
 * gdn_prefill_static -- gdn_prefill that allocates no memory at call time.
 *
 * An addition of this library: the pages that define the operation have no counterpart of it.
 * It is for callers that must not allocate device memory while they run, for instance a
 * serving loop whose memory is fixed when it starts (cudaMalloc and cudaFree can synchronise
 * the device and fail once memory is fragmented or taken) or a host framework that hands its
 * kernels no workspace. Same arguments and result as gdn_prefill. The tensor-core path (dk =
 * dv = 128, chunk 64, bf16, more than 8 tokens per sequence or cu_seqlens given) takes its
 * scratch from one fixed 13 MiB array in the library's device image (one copy per device,
 * present once the library's code is loaded there) and runs with at most 8 state-carrying
 * CTAs, so it is slower than gdn_prefill on large batches; all other sizes run the same
 * scratch-free kernels as gdn_prefill. Nothing is allocated: no cudaMalloc, no cudaFree, no
 * allocating library routine.
 *   Limit: the scratch holds the ring of 8 state-carrying CTAs (12 MiB) and 1 MiB of per-call
 * tables, which take about 4*B*Hk + 8*B bytes plus 5 KiB (B up to about 14,000 at Hk = 16). A
 * call whose sizes need more (that, or Hv/Hk > 8) returns GDN_ERR_UNSUPPORTED before anything
 * is queued.
 *   Set-up: the first call on each device, with that device current, looks up the scratch's
 * device address (cudaGetSymbolAddress, which may load the library's device code on that
 * device) and keeps it; make that first call before any stream capture. Every call clears
 * the scratch's counters itself (in its first kernel), so no call depends on what an earlier
 * one left there.
 *   Races: all calls on one device share the one scratch. Calls whose work may overlap on the
 * GPU (different streams without ordering between them, or several host threads) race on it
 * and give wrong results; calls queued on one stream are ordered and safe.
 * Returns GDN_OK, GDN_ERR_INVALID_ARG, GDN_ERR_UNSUPPORTED or GDN_ERR_CUDA.
 */
GDN_API int gdn_prefill_static(const void *q, const void *k, const void *v, const void *g, const void *b,
                               const float *state_in, float *state_out, void *out, const int32_t *cu_seqlens,
                               int B, int T, int Hk, int Hv, int dk, int dv, int chunk, int dtype, void *stream);

/*
 * gdn_decode_step -- one recurrent step for N independent sequences.
 *
 * Decoding is bound by the bytes moved per token ("Decodage : minimiser les
 * octets deplaces par token"); this step reads each head's fp32 state once
 * and writes it once, in place, fusing normalisation, gates, update and
 * read-out in one launch (same page, section "Reduire le trafic
 * intermediaire et d'etat": the recurrent update is fused with its
 * normalisation so no intermediate goes through memory).
 *
 *   q, k  : [N][Hk][dk];  v : [N][Hv][dv];  g, b : [N][Hv]   (dtype `dtype`)
 *   state : [N][Hv][dv][dk] fp32, updated in place.
 *   out   : [N][Hv][dv] (dtype `dtype`), o = S_new qh.
 *   N     : sequences (N = 0 is a no-op returning GDN_OK).
 * Returns GDN_OK, GDN_ERR_INVALID_ARG, GDN_ERR_UNSUPPORTED or GDN_ERR_CUDA.
 */
GDN_API int gdn_decode_step(const void *q, const void *k, const void *v, const void *g, const void *b,
                    float *state, void *out, int N, int Hk, int Hv, int dk, int dv, int dtype,
                    void *stream);

/*
 * gdn_decode_step_slots -- one decode step for N sequences whose states sit in
 * a pool of resident sessions.
 *
 * The same step as gdn_decode_step (one read and one write of each state, in
 * place), but sequence n updates pool entry slots[n] instead of entry n, so a
 * server can keep many sessions' states in one allocation and step any subset
 * of them, in any order, in one launch. The pages keep each session's state on
 * the device between tokens and move only what a token needs ("Decodage :
 * minimiser les octets deplaces par token"); the indexing adds no state traffic.
 *
 *   q, k, v, g, b, out : as for gdn_decode_step ([N][...]).
 *   state_pool : [num_slots][Hv][dv][dk] fp32, entries slots[n] updated in
 *                place; every other entry is left untouched.
 *   slots      : device int32 [N]. slots[n] < 0 marks a padding row: its state
 *                is not touched and out[n] is written as zeros. Two sequences
 *                must not name the same entry (their updates would race).
 *                slots[n] >= num_slots is treated like padding and sets the
 *                device status word (GDN_ERR_DEVICE_CHECK, see
 *                gdn_get_device_status).
 *   N, num_slots : sequences in this step (0 = no-op) and pool entries.
 * Returns GDN_OK, GDN_ERR_INVALID_ARG, GDN_ERR_UNSUPPORTED or GDN_ERR_CUDA.
 */
GDN_API int gdn_decode_step_slots(const void *q, const void *k, const void *v, const void *g,
                          const void *b, float *state_pool, const int32_t *slots, void *out,
                          int N, int num_slots, int Hk, int Hv, int dk, int dv, int dtype,
                          void *stream);

/*
 * gdn_prefill_from_host -- gdn_prefill of ONE sequence whose inputs and outputs are in
 * host memory, with the copies overlapped with the computation.
 *
 * The state is carried from one prompt fragment to the next with an unchanged result
 * ("Limiter la memoire temporaire grace au decoupage des prompts"), so the prompt is
 * processed in fragments of `fragment` tokens: while fragment f is computed on `stream`,
 * fragment f+1's inputs are copied in and fragment f-1's outputs copied out on two streams
 * the library keeps per device. With every fragment longer than 8 tokens the result is
 * bit-identical to gdn_prefill on the whole prompt (the same blocks, the state carried in
 * fp32 through device memory).
 *
 *   q_h, k_h, v_h, g_h, b_h, out_h : host arrays, layouts as for gdn_prefill with B = 1
 *                   (page-locked memory lets the copies overlap; pageable memory works but
 *                   the copies then do not overlap).
 *   state_in_h    : host [Hv][dv][dk] fp32 initial state, or NULL for zeros.
 *   state_out_h   : host [Hv][dv][dk] fp32 final state (may equal state_in_h).
 *   q_d .. out_d, state_d : caller-owned DEVICE buffers of the full prompt's sizes (and
 *                   one state); the library copies into and computes in them. They must
 *                   not be in use by other work while the call's work is in flight.
 *   T             : tokens of the prompt (0: the state passes through).
 *   fragment      : tokens per fragment, a positive multiple of `chunk`; at most 256
 *                   fragments.
 *   Other arguments as for gdn_prefill.
 * The call is asynchronous on `stream`: its copies start after the work already queued on
 * `stream`, and work queued on `stream` afterwards starts after the last copy (so
 * synchronising `stream` means the host outputs are written). Calls from several host
 * threads on one device are serialised while they queue work.
 * Returns GDN_OK, GDN_ERR_INVALID_ARG, GDN_ERR_UNSUPPORTED or GDN_ERR_CUDA. Argument and
 * size errors are returned before anything is queued. An error from a CUDA call made while
 * queueing may leave the copies and launches queued before it in flight; the call still makes
 * `stream` wait for them before it returns, so the caller's buffers are free once `stream`'s
 * later work runs (or `stream` is synchronised).
 */
GDN_API int gdn_prefill_from_host(const void *q_h, const void *k_h, const void *v_h, const void *g_h,
                          const void *b_h, const float *state_in_h, float *state_out_h, void *out_h,
                          void *q_d, void *k_d, void *v_d, void *g_d, void *b_d, float *state_d,
                          void *out_d, int T, int Hk, int Hv, int dk, int dv, int chunk, int dtype,
                          int fragment, void *stream);

/*
 * gdn_prepass -- the per-token quantities of the block form, materialised.
 *
 * gdn_prefill computes these inside its kernels and never writes them; this
 * entry point exposes the same computation for inspection and testing:
 *   rq, rk : [Ttot][Hk] fp32, 1/sqrt(|q_t|^2 + 1e-6) and likewise for k;
 *   beta   : [Ttot][Hv] fp32, sigmoid(b_t);
 *   gcum   : [Ttot][Hv] fp32, sum of g over t's block up to and including t,
 *            blocks starting at every sequence start and every `chunk` tokens.
 * Other arguments as for gdn_prefill (dk in {32, 64, 128}).
 */
GDN_API int gdn_prepass(const void *q, const void *k, const void *g, const void *b,
                const int32_t *cu_seqlens, int B, int T, int Hk, int Hv, int dk, int chunk,
                int dtype, float *rq, float *rk, float *beta, float *gcum, void *stream);

/*
 * gdn_prefill_path -- which kernel gdn_prefill would launch for these sizes with
 * cu_seqlens NULL: 2 = token scan (T <= 8 tokens per sequence), 1 = tensor-core
 * block kernel (tcgen05/TMEM/TMA), 0 = CUDA-core block kernel (with cu_seqlens
 * given, T is the packed total and a 2 stands for the block kernel 1 or 0 would name),
 * negative = the gdn_status gdn_prefill would return. Host-only, no device work.
 */
GDN_API int gdn_prefill_path(int B, int T, int Hk, int Hv, int dk, int dv, int chunk, int dtype);

/*
 * gdn_get_device_status -- synchronise `stream`, then return and clear the
 * device status word: GDN_OK, or GDN_ERR_DEVICE_CHECK if a kernel found
 * inconsistent device data since the last call; GDN_ERR_CUDA if the
 * synchronisation itself failed.
 * There is one status word per device, shared by every stream and every call
 * on that device: a flag raised by work on another stream is reported to
 * whichever caller reads the word first. The word is read and cleared in one
 * atomic step (a one-thread kernel on `stream`), so no flag is lost between
 * the read and the clear.
 */
GDN_API int gdn_get_device_status(void *stream);

/* gdn_status_string -- static, human-readable name of a gdn_status value. */
GDN_API const char *gdn_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* GDN_GB300_H */
