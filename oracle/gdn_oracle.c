/*
 * gdn_oracle.c -- plain, slow fp64 CPU reference for the gated delta rule.
 *
 * TEST INFRASTRUCTURE. Only the test-suite, the smoke check and the CPU
 * baseline leg of the benchmark may load this code. The CUDA library never
 * links, includes or calls it, and it shares no code with the CUDA library.
 *
 * What it computes (the pages describe the layer in words only; the exact
 * recurrence below is the standard gated delta rule that the description
 * fixes):
 *   - "Optimiser l'inference sur appareil pour Apple Silicon",
 *     section "Qwen cree trois formes de charges de travail": a fixed-size
 *     matrix state; a learned gate decides how much of the old state to keep;
 *     a delta update writes the current token; every token depends on the
 *     state left by the previous one; prefill may either scan the tokens
 *     directly or regroup the updates into blocks that expose matrix products.
 *   - same page, section "Maintenir l'etat recurrent sur la puce": the state
 *     is a matrix carried through the whole scan and written back once; state
 *     and gate are kept in 32-bit floats (here: 64-bit, the oracle is exact
 *     up to rounding order).
 *
 * Per sequence n and value head h (key head hk = h / (Hv/Hk)):
 *     qh = q / sqrt(|q|^2 + 1e-6),   kh = k / sqrt(|k|^2 + 1e-6)
 *     alpha = exp(g),                beta = 1 / (1 + exp(-b))
 *     S <- alpha * S                 (gate: how much old state survives)
 *     e  = S kh                      (what the state currently recalls for kh)
 *     S <- S + beta (v - e) kh^T     (delta write of the current token)
 *     o  = S qh                      (read-out after the update)
 * i.e. S <- alpha S (I - beta kh kh^T) + beta v kh^T, o = S qh.
 *
 * Layouts (row-major, element counts):
 *     q, k        [Ttot][Hk][dk]
 *     v, out      [Ttot][Hv][dv]
 *     g, b        [Ttot][Hv]          (g = log-decay, b = beta logit)
 *     state       [B][Hv][dv][dk]     (S in R^{dv x dk}, so that S kh in R^dv)
 *     cu_seqlens  int32 [B+1] or NULL (NULL: sequence n owns tokens
 *                                      [n*T, (n+1)*T), Ttot = B*T)
 *
 * Three evaluations are provided; they share only the argument plumbing:
 *   oracle_gdn_sequential : the token-by-token scan above (the definition);
 *   oracle_gdn_chunked    : the block (WY / UT) regrouping, chunk size C,
 *                           with the unit-lower-triangular inverse taken by
 *                           forward substitution;
 *   oracle_gdn_prepass    : the per-token quantities the block form needs
 *                           (inverse norms, beta, in-chunk cumulative gate).
 *
 * ORACLE_MUTATION (compile-time, default 0) plants a known mistake so that
 * the test-suite can show its pins catch it. Production of expected values
 * always uses the unmutated build.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef ORACLE_MUTATION
#define ORACLE_MUTATION 0
#endif

#define GDN_NORM_EPS 1e-6

typedef struct {
    const double *q, *k, *v, *g, *b;
    const double *state_in;
    double *state_out, *out;
    const int32_t *cu_seqlens;
    int B, T, Hk, Hv, dk, dv, chunk;
} gdn_problem;

static void seq_bounds(const gdn_problem *p, int n, long *bos, long *eos)
{
    if (p->cu_seqlens) {
        *bos = p->cu_seqlens[n];
        *eos = p->cu_seqlens[n + 1];
    } else {
        *bos = (long)n * p->T;
        *eos = (long)(n + 1) * p->T;
    }
}

/* x / sqrt(sum x^2 + eps) */
static void l2_normalise(const double *x, int d, double *y)
{
    double ss = 0.0;
    for (int j = 0; j < d; ++j) ss += x[j] * x[j];
    double r = 1.0 / sqrt(ss + GDN_NORM_EPS);
#if ORACLE_MUTATION == 5
    r = 1.0; /* planted: normalisation dropped */
#endif
    for (int j = 0; j < d; ++j) y[j] = x[j] * r;
}

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* ------------------------------------------------------------------ */
/* Definition: token-by-token scan for one (sequence, value head).     */
/* ------------------------------------------------------------------ */
static void scan_one(const gdn_problem *p, int n, int h)
{
    const int dk = p->dk, dv = p->dv, Hk = p->Hk, Hv = p->Hv;
#if ORACLE_MUTATION == 4
    const int hk = h % Hk; /* planted: interleaved instead of grouped head sharing */
#else
    const int hk = h / (Hv / Hk);
#endif
    long bos, eos;
    seq_bounds(p, n, &bos, &eos);

    double *S = (double *)calloc((size_t)dv * dk, sizeof(double));
    double *qh = (double *)malloc(sizeof(double) * dk);
    double *kh = (double *)malloc(sizeof(double) * dk);
    double *e = (double *)malloc(sizeof(double) * dv);
    if (p->state_in)
        memcpy(S, p->state_in + ((size_t)n * Hv + h) * dv * dk, sizeof(double) * dv * dk);

    for (long t = bos; t < eos; ++t) {
        l2_normalise(p->q + ((size_t)t * Hk + hk) * dk, dk, qh);
        l2_normalise(p->k + ((size_t)t * Hk + hk) * dk, dk, kh);
        const double alpha = exp(p->g[(size_t)t * Hv + h]);
        const double beta = sigmoid(p->b[(size_t)t * Hv + h]);
        const double *vt = p->v + ((size_t)t * Hv + h) * dv;
        double *ot = p->out + ((size_t)t * Hv + h) * dv;

#if ORACLE_MUTATION == 3
        /* planted: read-out taken before the update */
        for (int i = 0; i < dv; ++i) {
            double acc = 0.0;
            for (int j = 0; j < dk; ++j) acc += S[(size_t)i * dk + j] * qh[j];
            ot[i] = acc;
        }
#endif
        /* gate */
#if ORACLE_MUTATION != 1
        for (size_t ij = 0; ij < (size_t)dv * dk; ++ij) S[ij] *= alpha;
#endif
        /* recall e = S kh */
        for (int i = 0; i < dv; ++i) {
            double acc = 0.0;
            for (int j = 0; j < dk; ++j) acc += S[(size_t)i * dk + j] * kh[j];
            e[i] = acc;
        }
        /* delta write */
        for (int i = 0; i < dv; ++i) {
#if ORACLE_MUTATION == 2
            const double u = beta * (vt[i] + e[i]); /* planted: wrong sign */
#else
            const double u = beta * (vt[i] - e[i]);
#endif
            for (int j = 0; j < dk; ++j) S[(size_t)i * dk + j] += u * kh[j];
        }
#if ORACLE_MUTATION != 3
        /* read-out after the update */
        for (int i = 0; i < dv; ++i) {
            double acc = 0.0;
            for (int j = 0; j < dk; ++j) acc += S[(size_t)i * dk + j] * qh[j];
            ot[i] = acc;
        }
#endif
    }
    memcpy(p->state_out + ((size_t)n * Hv + h) * dv * dk, S, sizeof(double) * dv * dk);
    free(S);
    free(qh);
    free(kh);
    free(e);
}

/* ------------------------------------------------------------------ */
/* Block (chunk) regrouping for one (sequence, value head).            */
/*                                                                     */
/* Within a chunk of L tokens starting from state S0, with             */
/*   G_t = sum_{s<=t} g_s (in-chunk, inclusive), gamma_t = exp(G_t):   */
/*   A_ts = beta_t exp(G_t-G_s) kh_t.kh_s   (s<t), 0 otherwise          */
/*   Tm   = (I + A)^-1                       (unit lower triangular)    */
/*   W    = Tm diag(beta gamma) Kh          [L x dk]                    */
/*   U'   = Tm diag(beta) V                 [L x dv]                    */
/*   U    = U' - W S0^T                     [L x dv]                    */
/*   P_ts = exp(G_t-G_s) qh_t.kh_s           (s<=t), 0 otherwise         */
/*   O    = diag(gamma) Qh S0^T + P U                                   */
/*   S    = gamma_L S0 + U^T diag(exp(G_L - G_t)) Kh                    */
/* ------------------------------------------------------------------ */
static void chunked_one(const gdn_problem *p, int n, int h)
{
    const int dk = p->dk, dv = p->dv, Hk = p->Hk, Hv = p->Hv, C = p->chunk;
    const int hk = h / (Hv / Hk);
    long bos, eos;
    seq_bounds(p, n, &bos, &eos);

    double *S = (double *)calloc((size_t)dv * dk, sizeof(double));
    double *Kh = (double *)malloc(sizeof(double) * C * dk);
    double *Qh = (double *)malloc(sizeof(double) * C * dk);
    double *V = (double *)malloc(sizeof(double) * C * dv);
    double *beta = (double *)malloc(sizeof(double) * C);
    double *G = (double *)malloc(sizeof(double) * C);
    double *A = (double *)calloc((size_t)C * C, sizeof(double));
    double *Tm = (double *)calloc((size_t)C * C, sizeof(double));
    double *P = (double *)calloc((size_t)C * C, sizeof(double));
    double *W = (double *)malloc(sizeof(double) * C * dk);
    double *U = (double *)malloc(sizeof(double) * C * dv);
    double *Snew = (double *)malloc(sizeof(double) * dv * dk);
    if (p->state_in)
        memcpy(S, p->state_in + ((size_t)n * Hv + h) * dv * dk, sizeof(double) * dv * dk);

    for (long c0 = bos; c0 < eos; c0 += C) {
        const int L = (int)((eos - c0) < C ? (eos - c0) : C);
        double run = 0.0;
        for (int t = 0; t < L; ++t) {
            const long tok = c0 + t;
            l2_normalise(p->q + ((size_t)tok * Hk + hk) * dk, dk, Qh + (size_t)t * dk);
            l2_normalise(p->k + ((size_t)tok * Hk + hk) * dk, dk, Kh + (size_t)t * dk);
            memcpy(V + (size_t)t * dv, p->v + ((size_t)tok * Hv + h) * dv, sizeof(double) * dv);
            beta[t] = sigmoid(p->b[(size_t)tok * Hv + h]);
            run += p->g[(size_t)tok * Hv + h];
            G[t] = run;
        }
        /* A (strictly lower) and P (lower incl. diagonal) */
        for (int t = 0; t < L; ++t)
            for (int s = 0; s < L; ++s) {
                double kk = 0.0, qk = 0.0;
                for (int j = 0; j < dk; ++j) {
                    kk += Kh[(size_t)t * dk + j] * Kh[(size_t)s * dk + j];
                    qk += Qh[(size_t)t * dk + j] * Kh[(size_t)s * dk + j];
                }
                const double dec = exp(G[t] - G[s]);
                A[(size_t)t * C + s] = (s < t) ? beta[t] * dec * kk : 0.0;
#if ORACLE_MUTATION == 6
                P[(size_t)t * C + s] = (s < t) ? dec * qk : 0.0; /* planted: diagonal dropped */
#else
                P[(size_t)t * C + s] = (s <= t) ? dec * qk : 0.0;
#endif
            }
        /* Tm = (I + A)^-1 by forward substitution, one column at a time */
        for (int col = 0; col < L; ++col) {
            for (int r = 0; r < L; ++r) Tm[(size_t)r * C + col] = 0.0;
            Tm[(size_t)col * C + col] = 1.0;
            for (int r = col + 1; r < L; ++r) {
                double acc = 0.0;
                for (int s = col; s < r; ++s) acc += A[(size_t)r * C + s] * Tm[(size_t)s * C + col];
                Tm[(size_t)r * C + col] = -acc;
            }
        }
        /* W = Tm diag(beta gamma) Kh ; U = Tm diag(beta) V - W S^T */
        for (int t = 0; t < L; ++t) {
            for (int j = 0; j < dk; ++j) {
                double acc = 0.0;
                for (int s = 0; s <= t; ++s)
                    acc += Tm[(size_t)t * C + s] * beta[s] * exp(G[s]) * Kh[(size_t)s * dk + j];
                W[(size_t)t * dk + j] = acc;
            }
            for (int i = 0; i < dv; ++i) {
                double acc = 0.0;
                for (int s = 0; s <= t; ++s) acc += Tm[(size_t)t * C + s] * beta[s] * V[(size_t)s * dv + i];
                double ws = 0.0;
                for (int j = 0; j < dk; ++j) ws += W[(size_t)t * dk + j] * S[(size_t)i * dk + j];
                U[(size_t)t * dv + i] = acc - ws;
            }
        }
        /* O = diag(gamma) Qh S^T + P U */
        for (int t = 0; t < L; ++t) {
            double *ot = p->out + ((size_t)(c0 + t) * Hv + h) * dv;
            for (int i = 0; i < dv; ++i) {
                double qs = 0.0;
                for (int j = 0; j < dk; ++j) qs += Qh[(size_t)t * dk + j] * S[(size_t)i * dk + j];
                double pu = 0.0;
                for (int s = 0; s <= t; ++s) pu += P[(size_t)t * C + s] * U[(size_t)s * dv + i];
                ot[i] = exp(G[t]) * qs + pu;
            }
        }
        /* S = gamma_L S + U^T diag(exp(G_L - G_t)) Kh */
        const double GL = G[L - 1];
        for (int i = 0; i < dv; ++i)
            for (int j = 0; j < dk; ++j) {
                double acc = 0.0;
                for (int t = 0; t < L; ++t)
#if ORACLE_MUTATION == 7
                    acc += U[(size_t)t * dv + i] * exp(G[t] - GL) * Kh[(size_t)t * dk + j]; /* planted */
#else
                    acc += U[(size_t)t * dv + i] * exp(GL - G[t]) * Kh[(size_t)t * dk + j];
#endif
                Snew[(size_t)i * dk + j] = exp(GL) * S[(size_t)i * dk + j] + acc;
            }
        memcpy(S, Snew, sizeof(double) * dv * dk);
    }
    memcpy(p->state_out + ((size_t)n * Hv + h) * dv * dk, S, sizeof(double) * dv * dk);
    free(S); free(Kh); free(Qh); free(V); free(beta); free(G);
    free(A); free(Tm); free(P); free(W); free(U); free(Snew);
}

/* ------------------------------------------------------------------ */
/* Work distribution over (sequence, value head) pairs.                */
/* ------------------------------------------------------------------ */
typedef void (*unit_fn)(const gdn_problem *, int, int);

typedef struct {
    const gdn_problem *p;
    unit_fn fn;
    int next;
    pthread_mutex_t lock;
} work_queue;

static void *worker(void *arg)
{
    work_queue *wq = (work_queue *)arg;
    const int units = wq->p->B * wq->p->Hv;
    for (;;) {
        pthread_mutex_lock(&wq->lock);
        const int u = wq->next++;
        pthread_mutex_unlock(&wq->lock);
        if (u >= units) break;
        wq->fn(wq->p, u / wq->p->Hv, u % wq->p->Hv);
    }
    return NULL;
}

static int run_all(const gdn_problem *p, unit_fn fn, int threads)
{
    if (p->B < 0 || p->Hk <= 0 || p->Hv <= 0 || p->dk <= 0 || p->dv <= 0) return -1;
    if (p->Hv % p->Hk != 0) return -1;
    work_queue wq;
    wq.p = p;
    wq.fn = fn;
    wq.next = 0;
    pthread_mutex_init(&wq.lock, NULL);
    if (threads < 1) threads = 1;
    if (threads == 1) {
        worker(&wq);
    } else {
        pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * threads);
        for (int i = 0; i < threads; ++i) pthread_create(&tid[i], NULL, worker, &wq);
        for (int i = 0; i < threads; ++i) pthread_join(tid[i], NULL);
        free(tid);
    }
    pthread_mutex_destroy(&wq.lock);
    return 0;
}

int oracle_gdn_sequential(const double *q, const double *k, const double *v, const double *g,
                          const double *b, const double *state_in, double *state_out,
                          double *out, const int32_t *cu_seqlens, int B, int T, int Hk, int Hv,
                          int dk, int dv, int threads)
{
    gdn_problem p = {q, k, v, g, b, state_in, state_out, out, cu_seqlens, B, T, Hk, Hv, dk, dv, 1};
    return run_all(&p, scan_one, threads);
}

int oracle_gdn_chunked(const double *q, const double *k, const double *v, const double *g,
                       const double *b, const double *state_in, double *state_out, double *out,
                       const int32_t *cu_seqlens, int B, int T, int Hk, int Hv, int dk, int dv,
                       int chunk, int threads)
{
    if (chunk <= 0) return -1;
    gdn_problem p = {q, k, v, g, b, state_in, state_out, out, cu_seqlens, B, T, Hk, Hv, dk, dv, chunk};
    return run_all(&p, chunked_one, threads);
}

/*
 * Per-token quantities of the block form, for every packed token t:
 *   rq[t][hk] = 1/sqrt(|q_t|^2 + eps), rk likewise       ([Ttot][Hk])
 *   beta[t][h] = sigmoid(b_t)                            ([Ttot][Hv])
 *   gcum[t][h] = sum of g over the tokens of t's chunk   ([Ttot][Hv])
 *                up to and including t; chunks start at every
 *                sequence start and every `chunk` tokens after it.
 */
int oracle_gdn_prepass(const double *q, const double *k, const double *g, const double *b,
                       const int32_t *cu_seqlens, int B, int T, int Hk, int Hv, int dk,
                       int chunk, double *rq, double *rk, double *beta, double *gcum)
{
    if (chunk <= 0 || Hk <= 0 || Hv <= 0 || Hv % Hk != 0) return -1;
    gdn_problem p;
    memset(&p, 0, sizeof(p));
    p.cu_seqlens = cu_seqlens;
    p.T = T;
    for (int n = 0; n < B; ++n) {
        long bos, eos;
        seq_bounds(&p, n, &bos, &eos);
        for (long t = bos; t < eos; ++t) {
            for (int hk = 0; hk < Hk; ++hk) {
                double sq = 0.0, sk = 0.0;
                for (int j = 0; j < dk; ++j) {
                    const double a = q[((size_t)t * Hk + hk) * dk + j];
                    const double c = k[((size_t)t * Hk + hk) * dk + j];
                    sq += a * a;
                    sk += c * c;
                }
                rq[(size_t)t * Hk + hk] = 1.0 / sqrt(sq + GDN_NORM_EPS);
                rk[(size_t)t * Hk + hk] = 1.0 / sqrt(sk + GDN_NORM_EPS);
            }
            const long pos = t - bos;
            for (int h = 0; h < Hv; ++h) {
                beta[(size_t)t * Hv + h] = sigmoid(b[(size_t)t * Hv + h]);
                const double prev = (pos % chunk == 0) ? 0.0 : gcum[(size_t)(t - 1) * Hv + h];
                gcum[(size_t)t * Hv + h] = prev + g[(size_t)t * Hv + h];
            }
        }
    }
    return 0;
}
