/*
 * linattn_oracle.c -- fp64 CPU oracle for causal linear attention with a
 * fixed dk x dv state per head.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link,
 * load or call this file.  Its only users are the tests under tests/, the
 * smoke() check in __graft_entry__.py and the cpu_baseline leg of bench.py.
 * It shares no code, header, table or constant with the CUDA library.
 *
 * Everything here is the plain token-by-token definition, in double
 * precision, with no chunking, blocking or reordering beyond the sums the
 * definition writes out.  Source of every formula: the web page
 * "From GPT-2 to Kimi K3, explained" (three copies: Chinese translation,
 * Chinese summary, German translation), sections named per function.
 *
 * Conventions (row convention of the page's listings): the state of one
 * (sequence, head) is S in R^{dk x dv}, stored row-major, S[c*dv + j];
 * a read is o = S^T q (the page's "o = q @ S"), a write adds k u^T
 * (the page's "S = S + k.transpose(-1,-2) @ u").
 *
 * Packed layouts (tokens of all sequences back to back, as cu_seqlens says):
 *   q, k         [ntok][H][dk]
 *   v, o         [ntok][H][dv]
 *   beta_logits  [ntok][H]
 *   gate_logits  [ntok][H][dk]      (NULL: no decay, alpha = 1)
 *                [ntok][H]          with ORACLE_SCALAR_GATE (one decay per
 *                                   token and head, all key channels)
 *   S, init/final[N][H][dk][dv]
 *   z            [N][H][dk]          (ELU+1 normaliser)
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Prologue options; values chosen independently of the CUDA library and
 * mapped by the Python wrapper.  */
#define ORACLE_L2NORM_K 1u
#define ORACLE_L2NORM_Q 2u
#define ORACLE_SILU_QK 4u
#define ORACLE_SCALAR_GATE 8u

/* ---------------------------------------------------------------- prologue */

/* phi(x) = elu(x) + 1, the positive feature map applied to q and k
 * separately ("From GPT-2 to Kimi K3, explained", section Linear attention,
 * the forward() that replaces the KV cache: k = F.elu(k)+1, q = F.elu(q)+1). */
static double elu_plus_one(double x) { return x > 0.0 ? x + 1.0 : exp(x); }

/* silu(x) = x * sigmoid(x) (section DeltaNet (Fast Weight Programmers):
 * q, k = F.normalize(F.silu(.))). */
static double sigmoid(double x) {
    if (x >= 0.0) return 1.0 / (1.0 + exp(-x));
    double e = exp(x);
    return e / (1.0 + e);
}

/* softplus(x) = log(1 + e^x), written so that neither branch overflows. */
static double softplus(double x) {
    return (x > 0.0 ? x : 0.0) + log1p(exp(-fabs(x)));
}

/* x / max(||x||_2, 1e-12), the F.normalize default used on the page. */
static void l2_normalize(double *x, int n) {
    double s = 0.0;
    for (int i = 0; i < n; ++i) s += x[i] * x[i];
    double nrm = sqrt(s);
    if (nrm < 1e-12) nrm = 1e-12;
    for (int i = 0; i < n; ++i) x[i] /= nrm;
}

/* Feature preparation for the delta rule: optional silu, then optional L2
 * normalisation (DeltaNet (Fast Weight Programmers): normalize(silu(x))). */
static void prep_qk(const double *src, double *dst, int n, int do_silu, int do_norm) {
    for (int i = 0; i < n; ++i) dst[i] = do_silu ? src[i] * sigmoid(src[i]) : src[i];
    if (do_norm) l2_normalize(dst, n);
}

/* --------------------------------------------------------------- threading */

typedef struct {
    int64_t n_pairs;
    int tid, nthreads;
    void (*fn)(void *ctx, int64_t pair);
    void *ctx;
} worker_arg;

static void *worker_main(void *p) {
    worker_arg *a = (worker_arg *)p;
    for (int64_t i = a->tid; i < a->n_pairs; i += a->nthreads) a->fn(a->ctx, i);
    return NULL;
}

/* Runs fn over the independent (sequence, head) pairs.  Each pair is
 * computed by exactly one thread with the same arithmetic as a serial run,
 * so the thread count changes timing only, never a result. */
static void for_each_pair(int64_t n_pairs, int nthreads, void (*fn)(void *, int64_t), void *ctx) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > n_pairs) nthreads = (int)(n_pairs > 0 ? n_pairs : 1);
    if (nthreads == 1) {
        for (int64_t i = 0; i < n_pairs; ++i) fn(ctx, i);
        return;
    }
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    worker_arg *args = (worker_arg *)malloc(sizeof(worker_arg) * (size_t)nthreads);
    for (int t = 0; t < nthreads; ++t) {
        args[t].n_pairs = n_pairs;
        args[t].tid = t;
        args[t].nthreads = nthreads;
        args[t].fn = fn;
        args[t].ctx = ctx;
        pthread_create(&th[t], NULL, worker_main, &args[t]);
    }
    for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
    free(th);
    free(args);
}

/* ------------------------------------------------- ELU+1 linear attention */

typedef struct {
    const double *q, *k, *v;
    double *o;
    const int64_t *cu;
    int H, dk, dv;
    const double *init_S, *init_z;
    double *final_S, *final_z;
} linear_ctx;

/* Causal ELU+1 linear attention, one (sequence, head), token by token
 * ("From GPT-2 to Kimi K3, explained", section Linear attention):
 *   S_t = S_{t-1} + phi(k_t) v_t^T,   z_t = z_{t-1} + phi(k_t),
 *   o_t = S_t^T phi(q_t) / (z_t^T phi(q_t)).
 * The page keeps the division by the summed q.k scores ("we still divide by
 * the sum"); phi > 0 makes the denominator positive, so no epsilon. */
static void linear_pair(void *vctx, int64_t pair) {
    const linear_ctx *c = (const linear_ctx *)vctx;
    const int H = c->H, dk = c->dk, dv = c->dv;
    const int64_t n = pair / H, h = pair % H;
    double *S = (double *)calloc((size_t)dk * dv, sizeof(double));
    double *z = (double *)calloc((size_t)dk, sizeof(double));
    double *fq = (double *)malloc(sizeof(double) * (size_t)dk);
    double *fk = (double *)malloc(sizeof(double) * (size_t)dk);
    const int64_t sbase = (n * H + h) * (int64_t)dk * dv, zbase = (n * H + h) * (int64_t)dk;
    if (c->init_S) memcpy(S, c->init_S + sbase, sizeof(double) * (size_t)dk * dv);
    if (c->init_z) memcpy(z, c->init_z + zbase, sizeof(double) * (size_t)dk);
    for (int64_t t = c->cu[n]; t < c->cu[n + 1]; ++t) {
        const double *qt = c->q + (t * H + h) * dk, *kt = c->k + (t * H + h) * dk;
        const double *vt = c->v + (t * H + h) * dv;
        double *ot = c->o + (t * H + h) * dv;
        for (int i = 0; i < dk; ++i) { fq[i] = elu_plus_one(qt[i]); fk[i] = elu_plus_one(kt[i]); }
        for (int i = 0; i < dk; ++i) {
            z[i] += fk[i];
            for (int j = 0; j < dv; ++j) S[i * dv + j] += fk[i] * vt[j];
        }
        double den = 0.0;
        for (int i = 0; i < dk; ++i) den += fq[i] * z[i];
        for (int j = 0; j < dv; ++j) {
            double num = 0.0;
            for (int i = 0; i < dk; ++i) num += fq[i] * S[i * dv + j];
            ot[j] = num / den;
        }
    }
    if (c->final_S) memcpy(c->final_S + sbase, S, sizeof(double) * (size_t)dk * dv);
    if (c->final_z) memcpy(c->final_z + zbase, z, sizeof(double) * (size_t)dk);
    free(S); free(z); free(fq); free(fk);
}

int la_oracle_linear(const double *q, const double *k, const double *v, double *o,
                     const int64_t *cu_seqlens, int N, int H, int dk, int dv,
                     const double *init_S, const double *init_z, double *final_S,
                     double *final_z, int nthreads) {
    if (!q || !k || !v || !o || !cu_seqlens || N < 1 || H < 1 || dk < 1 || dv < 1) return 1;
    for (int n = 0; n < N; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n]) return 1;
    linear_ctx c = {q, k, v, o, cu_seqlens, H, dk, dv, init_S, init_z, final_S, final_z};
    for_each_pair((int64_t)N * H, nthreads, linear_pair, &c);
    return 0;
}

/* ------------------------------------------------- (gated) delta rule */

typedef struct {
    const double *q, *k, *v, *beta_logits, *gate_logits;
    double *o;
    const int64_t *cu;
    int H, dk, dv;
    double scale;
    unsigned flags;
    const double *init_S;
    double *final_S;
} delta_ctx;

/* Gated delta rule with one decay per key channel, one (sequence, head),
 * token by token.  With S' = Diag(alpha_t) S_{t-1}:
 *   u_t = beta_t (v_t - S'^T k_t)         the delta: only what is new
 *   S_t = S' + k_t u_t^T                  same outer-product write
 *   o_t = scale * S_t^T q_t               read, no denominator
 * Sources ("From GPT-2 to Kimi K3, explained"):
 *   - the recurrent step and the naive prefill loop: sections
 *     DeltaNet (Fast Weight Programmers) and
 *     DeltaNet (Parallelizing Linear Transformers with Delta Rule);
 *   - the decay of the old state before the write: section Gated DeltaNet
 *     (Mamba-2's cache = alpha * S_old + S_new; alpha = 1 gives the pure
 *     delta rule, alpha = 0 clears the memory);
 *   - one decay per key channel: section KDA / Kimi Linear
 *     (alpha.reshape(nb, C, d)).
 * beta_t = sigmoid(beta_logit) (the page's sigmoid(w_beta x)), one value per
 * token and head; alpha_t = exp(-softplus(gate_logit)) per key channel.
 * With the decay first, the step equals the Householder form of the
 * chunkwise section, S_t = S_{t-1} Diag(alpha)(I - beta k k^T) + beta v k^T
 * in the column convention. */
static void delta_pair(void *vctx, int64_t pair) {
    const delta_ctx *c = (const delta_ctx *)vctx;
    const int H = c->H, dk = c->dk, dv = c->dv;
    const int64_t n = pair / H, h = pair % H;
    double *S = (double *)calloc((size_t)dk * dv, sizeof(double));
    double *qq = (double *)malloc(sizeof(double) * (size_t)dk);
    double *kk = (double *)malloc(sizeof(double) * (size_t)dk);
    double *alpha = (double *)malloc(sizeof(double) * (size_t)dk);
    double *u = (double *)malloc(sizeof(double) * (size_t)dv);
    const int64_t sbase = (n * H + h) * (int64_t)dk * dv;
    const int silu = (c->flags & ORACLE_SILU_QK) != 0;
    if (c->init_S) memcpy(S, c->init_S + sbase, sizeof(double) * (size_t)dk * dv);
    for (int64_t t = c->cu[n]; t < c->cu[n + 1]; ++t) {
        prep_qk(c->q + (t * H + h) * dk, qq, dk, silu, (c->flags & ORACLE_L2NORM_Q) != 0);
        prep_qk(c->k + (t * H + h) * dk, kk, dk, silu, (c->flags & ORACLE_L2NORM_K) != 0);
        const double *vt = c->v + (t * H + h) * dv;
        double *ot = c->o + (t * H + h) * dv;
        const double beta = sigmoid(c->beta_logits[t * H + h]);
        /* one decay per key channel (section KDA / Kimi Linear), or one per
         * token and head for every channel (section Gated DeltaNet) */
        const int scalar_gate = (c->flags & ORACLE_SCALAR_GATE) != 0;
        for (int i = 0; i < dk; ++i)
            alpha[i] = !c->gate_logits ? 1.0
                       : exp(-softplus(scalar_gate ? c->gate_logits[t * H + h]
                                                   : c->gate_logits[(t * H + h) * dk + i]));
        /* S' = Diag(alpha) S */
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j) S[i * dv + j] *= alpha[i];
        /* u = beta (v - S'^T k) */
        for (int j = 0; j < dv; ++j) {
            double old = 0.0;
            for (int i = 0; i < dk; ++i) old += kk[i] * S[i * dv + j];
            u[j] = beta * (vt[j] - old);
        }
        /* S = S' + k u^T */
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j) S[i * dv + j] += kk[i] * u[j];
        /* o = scale S^T q */
        for (int j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int i = 0; i < dk; ++i) acc += qq[i] * S[i * dv + j];
            ot[j] = c->scale * acc;
        }
    }
    if (c->final_S) memcpy(c->final_S + sbase, S, sizeof(double) * (size_t)dk * dv);
    free(S); free(qq); free(kk); free(alpha); free(u);
}

int la_oracle_delta(const double *q, const double *k, const double *v,
                    const double *beta_logits, const double *gate_logits, double *o,
                    const int64_t *cu_seqlens, int N, int H, int dk, int dv, double scale,
                    unsigned flags, const double *init_S, double *final_S, int nthreads) {
    if (!q || !k || !v || !beta_logits || !o || !cu_seqlens || N < 1 || H < 1 || dk < 1 || dv < 1)
        return 1;
    for (int n = 0; n < N; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n]) return 1;
    delta_ctx c = {q, k, v, beta_logits, gate_logits, o, cu_seqlens, H, dk, dv,
                   scale, flags, init_S, final_S};
    for_each_pair((int64_t)N * H, nthreads, delta_pair, &c);
    return 0;
}

/* One recurrent decode step for N sequences (one new token each), state
 * updated in place: the same definition as la_oracle_delta with every
 * sequence one token long and the state as both the initial and the final
 * state (section DeltaNet (Fast Weight Programmers): forward(x, cache) with
 * t = 1 returns the new cache). */
int la_oracle_decode(const double *q, const double *k, const double *v,
                     const double *beta_logits, const double *gate_logits, double *o,
                     int N, int H, int dk, int dv, double scale, unsigned flags,
                     double *state, int nthreads) {
    if (!state || N < 1) return 1;
    int64_t *cu = (int64_t *)malloc(sizeof(int64_t) * (size_t)(N + 1));
    for (int n = 0; n <= N; ++n) cu[n] = n;
    int rc = la_oracle_delta(q, k, v, beta_logits, gate_logits, o, cu, N, H, dk, dv, scale,
                             flags, state, state, nthreads);
    free(cu);
    return rc;
}
