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
 * a read is o = S^T q (the listings' row vector q times S), a write adds
 * k u^T (the listings add the outer product of k and u to S).
 *
 * Packed layouts (tokens of all sequences back to back, as cu_seqlens says):
 *   q, k         [ntok][H][dk]
 *   v, o         [ntok][H][dv]
 *   beta_logits  [ntok][H]          (unused, may be NULL, with ORACLE_ADDITIVE)
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
#define ORACLE_ADDITIVE 16u

/* ---------------------------------------------------------------- prologue */

/* phi(x) = elu(x) + 1, the positive feature map applied to q and k
 * separately ("From GPT-2 to Kimi K3, explained", section Linear attention,
 * the forward() that replaces the KV cache: k = F.elu(k)+1, q = F.elu(q)+1). */
static double elu_plus_one(double x) { return x > 0.0 ? x + 1.0 : exp(x); }

/* silu(x) = x * sigmoid(x) (section DeltaNet (Fast Weight Programmers):
 * the layer applies silu, then L2 normalisation, to q and k). */
static double sigmoid(double x) {
    if (x >= 0.0) return 1.0 / (1.0 + exp(-x));
    double e = exp(x);
    return e / (1.0 + e);
}

/* softplus(x) = log(1 + e^x), written so that neither branch overflows. */
static double softplus(double x) {
    return (x > 0.0 ? x : 0.0) + log1p(exp(-fabs(x)));
}

/* x / max(||x||_2, 1e-12): PyTorch's default floor for the L2
 * normalisation the page's layer applies. */
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
 *     (Mamba-2's decayed state, S = alpha S + k v^T; alpha = 1 gives the pure
 *     delta rule, alpha = 0 clears the memory);
 *   - one decay per key channel: section KDA / Kimi Linear (alpha laid out
 *     as one d-vector per token of each chunk).
 * beta_t = sigmoid(beta_logit) (the page: a sigmoid of a projection), one value per
 * token and head; alpha_t = exp(-softplus(gate_logit)) per key channel.
 * With the decay first, the step equals the Householder form of the
 * chunkwise section, S_t = S_{t-1} Diag(alpha)(I - beta k k^T) + beta v k^T
 * in the column convention.
 * ORACLE_ADDITIVE turns the delta off: u_t = v_t (no read of the old value,
 * no beta), the decayed additive state of section Gated DeltaNet
 * (Mamba-2: S_t = alpha_t S_{t-1} + k_t v_t^T, the new association added at full
 * strength). */
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
        const int additive = (c->flags & ORACLE_ADDITIVE) != 0;
        const double beta = additive ? 1.0 : sigmoid(c->beta_logits[t * H + h]);
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
        /* u = beta (v - S'^T k); the additive rule writes v at full strength
         * with no read (section Gated DeltaNet: Mamba-2's
         * S_t = alpha_t S_{t-1} + k_t v_t^T) */
        for (int j = 0; j < dv; ++j) {
            double old = 0.0;
            for (int i = 0; i < dk; ++i) old += kk[i] * S[i * dv + j];
            u[j] = additive ? vt[j] : beta * (vt[j] - old);
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
    if (!q || !k || !v || !o || !cu_seqlens || N < 1 || H < 1 || dk < 1 || dv < 1) return 1;
    if (!beta_logits && !(flags & ORACLE_ADDITIVE)) return 1;
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

/* ------------------------------------------- delta rule: reverse mode */

/* Derivative of prep_qk: given x (raw), y = prep(x) and dy, writes dx.
 * L2 step y = s / max(||s||, 1e-12): ds = (dy - y (y.dy)) / ||s|| while the
 * norm is above the floor, dy / 1e-12 below it (the floor is a constant).
 * silu step s = x sigmoid(x): ds/dx = sigmoid(x) (1 + x (1 - sigmoid(x))). */
static void prep_qk_backward(const double *x, const double *y, const double *dy, double *dx,
                             int n, int do_silu, int do_norm) {
    double *ds = (double *)malloc(sizeof(double) * (size_t)n);
    if (do_norm) {
        double ss = 0.0, ydy = 0.0;
        for (int i = 0; i < n; ++i) {
            const double s = do_silu ? x[i] * sigmoid(x[i]) : x[i];
            ss += s * s;
            ydy += y[i] * dy[i];
        }
        const double nrm = sqrt(ss);
        for (int i = 0; i < n; ++i)
            ds[i] = nrm > 1e-12 ? (dy[i] - y[i] * ydy) / nrm : dy[i] / 1e-12;
    } else {
        for (int i = 0; i < n; ++i) ds[i] = dy[i];
    }
    for (int i = 0; i < n; ++i) {
        if (do_silu) {
            const double sg = sigmoid(x[i]);
            dx[i] = ds[i] * sg * (1.0 + x[i] * (1.0 - sg));
        } else {
            dx[i] = ds[i];
        }
    }
    free(ds);
}

typedef struct {
    const double *q, *k, *v, *beta_logits, *gate_logits;
    const int64_t *cu;
    int H, dk, dv;
    double scale;
    unsigned flags;
    const double *init_S, *d_o, *d_final_S;
    double *dq, *dk_out, *dv_out, *d_beta_logits, *d_gate_logits, *d_init_S;
} delta_bwd_ctx;

/* Gradients of the gated delta rule of delta_pair, one (sequence, head), by
 * reverse-mode differentiation of its token loop.  The page gives only the
 * forward pass (section DeltaNet (Parallelizing Linear Transformers with
 * Delta Rule) motivates the chunked form by training); the backward pass
 * here is the chain rule applied to each statement of delta_pair in reverse
 * order, with every intermediate state kept from a first forward sweep:
 *   o_t = scale S_t^T q_t      -> dq_t = scale S_t do_t,  dS_t += scale q_t do_t^T
 *   S_t = S' + k_t u_t^T       -> dk_t += dS_t u_t,  du_t = dS_t^T k_t,  dS' = dS_t
 *   u_t = beta (v_t - S'^T k)  -> dbeta = du.(v_t - S'^T k),  dv_t = beta du,
 *                                 dS' -= beta k du^T,  dk_t -= beta S' du
 *   S' = Diag(alpha) S_{t-1}   -> dalpha_i = sum_j dS'_ij S_{t-1,ij},
 *                                 dS_{t-1} = Diag(alpha) dS'
 * then through the prologue: beta = sigmoid(b) gives db = dbeta beta (1-beta);
 * log alpha = -softplus(g) gives dg = -dalpha alpha sigmoid(g) (summed over
 * the key channels for a scalar gate); q, k through prep_qk_backward.
 * d_o is the gradient of the outputs, d_final_S (optional) that of the
 * final state; d_init_S receives the gradient of the initial state. */
static void delta_backward_pair(void *vctx, int64_t pair) {
    const delta_bwd_ctx *c = (const delta_bwd_ctx *)vctx;
    const int H = c->H, dk = c->dk, dv = c->dv;
    const int64_t n = pair / H, h = pair % H;
    const int64_t t0 = c->cu[n], L = c->cu[n + 1] - c->cu[n];
    const size_t DD = (size_t)dk * dv;
    const int silu = (c->flags & ORACLE_SILU_QK) != 0;
    const int norm_q = (c->flags & ORACLE_L2NORM_Q) != 0, norm_k = (c->flags & ORACLE_L2NORM_K) != 0;
    const int scalar_gate = (c->flags & ORACLE_SCALAR_GATE) != 0;
    const int additive = (c->flags & ORACLE_ADDITIVE) != 0;
    const int64_t sbase = (n * H + h) * (int64_t)DD;

    /* forward sweep, keeping the state before each token (index t) and after
     * the last one (index L) */
    double *Sh = (double *)calloc((size_t)(L + 1) * DD, sizeof(double));
    double *qh = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * dk);
    double *kh = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * dk);
    double *ah = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * dk);
    double *uh = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * dv);
    double *bh = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
    if (c->init_S) memcpy(Sh, c->init_S + sbase, sizeof(double) * DD);
    for (int64_t s = 0; s < L; ++s) {
        const int64_t t = t0 + s;
        double *qq = qh + s * dk, *kk = kh + s * dk, *al = ah + s * dk, *u = uh + s * dv;
        prep_qk(c->q + (t * H + h) * dk, qq, dk, silu, norm_q);
        prep_qk(c->k + (t * H + h) * dk, kk, dk, silu, norm_k);
        bh[s] = additive ? 1.0 : sigmoid(c->beta_logits[t * H + h]);
        for (int i = 0; i < dk; ++i)
            al[i] = !c->gate_logits ? 1.0
                    : exp(-softplus(scalar_gate ? c->gate_logits[t * H + h]
                                                : c->gate_logits[(t * H + h) * dk + i]));
        const double *Sp = Sh + s * DD;
        double *Sn = Sh + (s + 1) * DD;
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j) Sn[i * dv + j] = al[i] * Sp[i * dv + j];
        const double *vt = c->v + (t * H + h) * dv;
        for (int j = 0; j < dv; ++j) {
            double old = 0.0;
            for (int i = 0; i < dk; ++i) old += kk[i] * Sn[i * dv + j];
            u[j] = additive ? vt[j] : bh[s] * (vt[j] - old);
        }
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j) Sn[i * dv + j] += kk[i] * u[j];
    }

    /* reverse sweep */
    double *dS = (double *)calloc(DD, sizeof(double));
    double *Sd = (double *)malloc(sizeof(double) * DD);   /* S' of the token */
    double *dqh = (double *)malloc(sizeof(double) * (size_t)dk);
    double *dkh = (double *)malloc(sizeof(double) * (size_t)dk);
    double *da = (double *)malloc(sizeof(double) * (size_t)dk);
    double *du = (double *)malloc(sizeof(double) * (size_t)dv);
    if (c->d_final_S) memcpy(dS, c->d_final_S + sbase, sizeof(double) * DD);
    for (int64_t s = L - 1; s >= 0; --s) {
        const int64_t t = t0 + s;
        const double *qq = qh + s * dk, *kk = kh + s * dk, *al = ah + s * dk, *u = uh + s * dv;
        const double beta = bh[s];
        const double *Sp = Sh + s * DD, *St = Sh + (s + 1) * DD;
        const double *dot = c->d_o + (t * H + h) * dv;
        const double *vt = c->v + (t * H + h) * dv;
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j) Sd[i * dv + j] = al[i] * Sp[i * dv + j];
        /* o_t = scale S_t^T q_t */
        for (int i = 0; i < dk; ++i) {
            double acc = 0.0;
            for (int j = 0; j < dv; ++j) acc += St[i * dv + j] * dot[j];
            dqh[i] = c->scale * acc;
        }
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j) dS[i * dv + j] += c->scale * qq[i] * dot[j];
        /* S_t = S' + k u^T */
        for (int i = 0; i < dk; ++i) {
            double acc = 0.0;
            for (int j = 0; j < dv; ++j) acc += dS[i * dv + j] * u[j];
            dkh[i] = acc;
        }
        for (int j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int i = 0; i < dk; ++i) acc += dS[i * dv + j] * kk[i];
            du[j] = acc;
        }
        /* u = beta (v - S'^T k), or u = v for the additive rule; dS
         * currently holds dS' */
        double dbeta = 0.0;
        for (int j = 0; j < dv; ++j) {
            double old = 0.0;
            for (int i = 0; i < dk; ++i) old += kk[i] * Sd[i * dv + j];
            dbeta += du[j] * (vt[j] - old);
            c->dv_out[(t * H + h) * dv + j] = beta * du[j];
        }
        if (!additive) {
            for (int i = 0; i < dk; ++i) {
                double acc = 0.0;
                for (int j = 0; j < dv; ++j) acc += Sd[i * dv + j] * du[j];
                dkh[i] -= beta * acc;
            }
            for (int i = 0; i < dk; ++i)
                for (int j = 0; j < dv; ++j) dS[i * dv + j] -= beta * kk[i] * du[j];
        }
        /* S' = Diag(alpha) S_{t-1} */
        for (int i = 0; i < dk; ++i) {
            double acc = 0.0;
            for (int j = 0; j < dv; ++j) acc += dS[i * dv + j] * Sp[i * dv + j];
            da[i] = acc;
            for (int j = 0; j < dv; ++j) dS[i * dv + j] *= al[i];
        }
        /* prologue (the additive rule has no beta: its gradient is 0) */
        c->d_beta_logits[t * H + h] = additive ? 0.0 : dbeta * beta * (1.0 - beta);
        if (c->gate_logits) {
            if (scalar_gate) {
                const double g = c->gate_logits[t * H + h];
                double acc = 0.0;
                for (int i = 0; i < dk; ++i) acc += da[i];
                c->d_gate_logits[t * H + h] = -acc * al[0] * sigmoid(g);
            } else {
                for (int i = 0; i < dk; ++i) {
                    const double g = c->gate_logits[(t * H + h) * dk + i];
                    c->d_gate_logits[(t * H + h) * dk + i] = -da[i] * al[i] * sigmoid(g);
                }
            }
        }
        prep_qk_backward(c->q + (t * H + h) * dk, qq, dqh, c->dq + (t * H + h) * dk, dk, silu,
                         norm_q);
        prep_qk_backward(c->k + (t * H + h) * dk, kk, dkh, c->dk_out + (t * H + h) * dk, dk, silu,
                         norm_k);
    }
    if (c->d_init_S) memcpy(c->d_init_S + sbase, dS, sizeof(double) * DD);
    free(Sh); free(qh); free(kh); free(ah); free(uh); free(bh);
    free(dS); free(Sd); free(dqh); free(dkh); free(da); free(du);
}

/* Gradients of la_oracle_delta's outputs (o, and final_S when d_final_S is
 * given) with respect to every input: see delta_backward_pair.  Layouts as
 * la_oracle_delta; dq, dk like q, k; dv like v; d_beta_logits like
 * beta_logits; d_gate_logits like gate_logits (ignored when there is no
 * gate); d_init_S [N][H][dk][dv] (optional).  Rows of tokens outside every
 * sequence are not written. */
int la_oracle_delta_backward(const double *q, const double *k, const double *v,
                             const double *beta_logits, const double *gate_logits,
                             const int64_t *cu_seqlens, int N, int H, int dk, int dv,
                             double scale, unsigned flags, const double *init_S,
                             const double *d_o, const double *d_final_S, double *dq,
                             double *dk_out, double *dv_out, double *d_beta_logits,
                             double *d_gate_logits, double *d_init_S, int nthreads) {
    if (!q || !k || !v || !cu_seqlens || !d_o || !dq || !dk_out || !dv_out || !d_beta_logits ||
        N < 1 || H < 1 || dk < 1 || dv < 1)
        return 1;
    if (!beta_logits && !(flags & ORACLE_ADDITIVE)) return 1;
    if (gate_logits && !d_gate_logits) return 1;
    for (int n = 0; n < N; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n]) return 1;
    delta_bwd_ctx c = {q, k, v, beta_logits, gate_logits, cu_seqlens, H, dk, dv, scale, flags,
                       init_S, d_o, d_final_S, dq, dk_out, dv_out, d_beta_logits, d_gate_logits,
                       d_init_S};
    for_each_pair((int64_t)N * H, nthreads, delta_backward_pair, &c);
    return 0;
}
