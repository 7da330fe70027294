/*
 * gdn_oracle.c -- fp64 CPU oracle for the gated delta rule.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library
 * and its Python binding) may include, link or call this file.  It shares no
 * code, header, table or constant with the CUDA sources.
 *
 * Sources (page title, then section / equation):
 *   [paper]    "Gated Delta Networks: Improving Mamba2 with Delta Rule"
 *              (translated page): §2.1 (Mamba2, decay mask Gamma),
 *              §2.2 eqs. 6-9 (DeltaNet UT transform and chunk recurrence),
 *              §3.1 eq. 10 (gated delta rule), §3.3 (gated chunkwise form).
 *   [blog]     "【论文解读】Gated Delta Network": §二(一)2 "Hardware-Efficient
 *              Chunkwise Training", parts (3) matrix form and (4) summary,
 *              which also fixes the output mask to the decay mask Gamma.
 *   [deepdive] "Gated DeltaNet：先忘一点，再按误差更新记忆": section
 *              "为什么再加一个遗忘门？" (decay first, then correct the
 *              decayed prediction) and "Decode 递归" (state carry).
 *
 * Layouts (all row-major, fp64):
 *   q, k        [B, T, H, dk]      token-major
 *   v, out      [B, T, H, dv]
 *   g, beta     [B, T, H]          g = log(alpha)
 *   states      [N, H, dv, dk]     S in R^{dv x dk}, read as o = S q
 *   cu_seqlens  int32 [N+1]        optional; then B == 1 and sequence n is
 *                                  tokens [cu[n], cu[n+1]) of the T axis.
 *
 * Readings where the pages are silent (restated in the design notes):
 *   - L2 norm: x / sqrt(sum x^2 + 1e-6), applied to q and k when requested.
 *   - scale multiplies q after the optional normalisation.
 *   - The recurrence is applied in the decay-then-correct order.
 *
 * Functions:
 *   oracle_recurrent_fwd   token-by-token eq. 10 (the definition).
 *   oracle_decode_step     one token of eq. 10 per (sequence, head), in place.
 *   oracle_chunked_fwd     the chunkwise WY/UT form of [paper] §3.3 and
 *                          [blog] §二(一)2(4), for any chunk size C; a second,
 *                          independent algorithm used to cross-check the
 *                          definition and to debug stage by stage.
 *   oracle_ut_transform    the per-chunk UT transform alone (W and U~).
 *   oracle_recurrent_bwd   gradients of eq. 10 with respect to q, k, v, g,
 *                          beta and the initial state, by reverse-mode
 *                          differentiation of the token recurrence (the
 *                          states are recomputed forward and kept).
 *   oracle_short_conv_silu the block prologue of q, k, v: short causal
 *                          depthwise convolution then SiLU ([paper] §3.4
 *                          "Token mixing block" and Fig. 1).
 *   oracle_gate_activations alpha in Mamba2's parameterisation and beta by a
 *                          sigmoid, from their linear projections (same
 *                          section).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORACLE_L2_EPS 1e-6

/* ------------------------------------------------------------------ */
/* small helpers                                                       */
/* ------------------------------------------------------------------ */

static int resolve_threads(int32_t nthreads)
{
    if (nthreads > 0) return nthreads;
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

/* Copy one token-head vector, optionally L2-normalised and scaled. */
static void load_vec(const double *src, double *dst, int d, int l2, double scale)
{
    double ss = 0.0;
    if (l2) {
        for (int i = 0; i < d; ++i) ss += src[i] * src[i];
        double r = 1.0 / sqrt(ss + ORACLE_L2_EPS);
        for (int i = 0; i < d; ++i) dst[i] = src[i] * r * scale;
    } else {
        for (int i = 0; i < d; ++i) dst[i] = src[i] * scale;
    }
}

/* Sequence geometry: start token (along T of batch row b) and length. */
typedef struct {
    int32_t B, T, H, dk, dv, N;
    const int32_t *cu;
} geom_t;

static void seq_span(const geom_t *gm, int n, int64_t *row0, int64_t *len)
{
    /* row0 = index of the first token in the flattened [B*T] token axis */
    if (gm->cu) {
        *row0 = gm->cu[n];
        *len = (int64_t)gm->cu[n + 1] - gm->cu[n];
    } else {
        *row0 = (int64_t)n * gm->T;
        *len = gm->T;
    }
}

/* ------------------------------------------------------------------ */
/* The gated delta rule, one token (the definition)                    */
/* ------------------------------------------------------------------ */

/*
 * One step of [paper] §3.1 eq. 10 in the decay-then-correct form of
 * [deepdive] "为什么再加一个遗忘门？":
 *   Sbar = alpha S;   S <- Sbar + beta (v - Sbar k) k^T;   o = S q.
 * S is dv x dk row-major; kk, qq already normalised/scaled.
 */
static void gdr_step(double *S, const double *qq, const double *kk, const double *vv,
                     double alpha, double beta, double *o, int dk, int dv)
{
    for (int j = 0; j < dv; ++j) {
        double *row = S + (int64_t)j * dk;
        for (int d = 0; d < dk; ++d) row[d] *= alpha;             /* Sbar = alpha S   */
        double pred = 0.0;
        for (int d = 0; d < dk; ++d) pred += row[d] * kk[d];      /* (Sbar k)_j       */
        double err = beta * (vv[j] - pred);
        for (int d = 0; d < dk; ++d) row[d] += err * kk[d];       /* + beta(v-Sbar k)k^T */
        if (o) {
            double acc = 0.0;
            for (int d = 0; d < dk; ++d) acc += row[d] * qq[d];   /* o = S_t q_t      */
            o[j] = acc;
        }
    }
}

/* ------------------------------------------------------------------ */
/* thread pool over (sequence, head) units                             */
/* ------------------------------------------------------------------ */

typedef void (*unit_fn)(void *ctx, int64_t unit, double *scratch);

typedef struct {
    unit_fn fn;
    void *ctx;
    int64_t n_units;
    int64_t next;
    size_t scratch_doubles;
    pthread_mutex_t mu;
    int failed;
} pool_t;

static void *pool_worker(void *arg)
{
    pool_t *p = (pool_t *)arg;
    double *scratch = (double *)malloc(sizeof(double) * (p->scratch_doubles ? p->scratch_doubles : 1));
    if (!scratch) {
        pthread_mutex_lock(&p->mu);
        p->failed = 1;
        pthread_mutex_unlock(&p->mu);
        return NULL;
    }
    for (;;) {
        pthread_mutex_lock(&p->mu);
        int64_t u = p->next++;
        pthread_mutex_unlock(&p->mu);
        if (u >= p->n_units) break;
        p->fn(p->ctx, u, scratch);
    }
    free(scratch);
    return NULL;
}

static int run_pool(unit_fn fn, void *ctx, int64_t n_units, size_t scratch_doubles, int32_t nthreads)
{
    pool_t p;
    p.fn = fn; p.ctx = ctx; p.n_units = n_units; p.next = 0;
    p.scratch_doubles = scratch_doubles; p.failed = 0;
    pthread_mutex_init(&p.mu, NULL);
    int nt = resolve_threads(nthreads);
    if (nt > n_units) nt = (int)(n_units > 0 ? n_units : 1);
    if (nt <= 1) {
        pool_worker(&p);
    } else {
        pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nt);
        if (!th) { pthread_mutex_destroy(&p.mu); return -3; }
        int started = 0;
        for (int i = 0; i < nt; ++i) {
            if (pthread_create(&th[i], NULL, pool_worker, &p) == 0) ++started;
        }
        if (started == 0) pool_worker(&p);
        for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
        free(th);
    }
    pthread_mutex_destroy(&p.mu);
    return p.failed ? -3 : 0;
}

/* ------------------------------------------------------------------ */
/* oracle_recurrent_fwd                                                */
/* ------------------------------------------------------------------ */

typedef struct {
    geom_t gm;
    const double *q, *k, *v, *g, *beta, *s0;
    double *out, *sf;
    double scale;
    int l2;
} rec_ctx_t;

static void rec_unit(void *vctx, int64_t unit, double *scratch)
{
    rec_ctx_t *c = (rec_ctx_t *)vctx;
    const geom_t *gm = &c->gm;
    int H = gm->H, dk = gm->dk, dv = gm->dv;
    int n = (int)(unit / H), h = (int)(unit % H);
    double *S = scratch;                 /* dv*dk */
    double *qq = S + (int64_t)dv * dk;   /* dk    */
    double *kk = qq + dk;                /* dk    */
    const int64_t sz = (int64_t)dv * dk;
    if (c->s0) memcpy(S, c->s0 + ((int64_t)n * H + h) * sz, sizeof(double) * (size_t)sz);
    else memset(S, 0, sizeof(double) * (size_t)sz);
    int64_t row0, len;
    seq_span(gm, n, &row0, &len);
    for (int64_t t = 0; t < len; ++t) {
        int64_t th = (row0 + t) * H + h;      /* token-head index */
        load_vec(c->q + th * dk, qq, dk, c->l2, c->scale);
        load_vec(c->k + th * dk, kk, dk, c->l2, 1.0);
        double alpha = exp(c->g[th]);
        gdr_step(S, qq, kk, c->v + th * dv, alpha, c->beta[th], c->out + th * dv, dk, dv);
    }
    if (c->sf) memcpy(c->sf + ((int64_t)n * H + h) * sz, S, sizeof(double) * (size_t)sz);
}

static int check_geom(const geom_t *gm)
{
    if (gm->B < 1 || gm->T < 0 || gm->H < 1 || gm->dk < 1 || gm->dv < 1) return -1;
    if (gm->cu) {
        if (gm->B != 1 || gm->N < 1) return -1;
        if (gm->cu[0] != 0 || gm->cu[gm->N] != gm->T) return -1;
        for (int n = 0; n < gm->N; ++n)
            if (gm->cu[n + 1] < gm->cu[n]) return -1;
    }
    return 0;
}

int oracle_recurrent_fwd(const double *q, const double *k, const double *v,
                         const double *g, const double *beta,
                         const double *init_state, const int32_t *cu_seqlens, int32_t num_seqs,
                         double *out, double *final_state,
                         int32_t B, int32_t T, int32_t H, int32_t dk, int32_t dv,
                         double scale, int32_t use_qk_l2norm, int32_t nthreads)
{
    rec_ctx_t c;
    c.gm.B = B; c.gm.T = T; c.gm.H = H; c.gm.dk = dk; c.gm.dv = dv;
    c.gm.cu = cu_seqlens; c.gm.N = cu_seqlens ? num_seqs : B;
    if (check_geom(&c.gm)) return -1;
    c.q = q; c.k = k; c.v = v; c.g = g; c.beta = beta; c.s0 = init_state;
    c.out = out; c.sf = final_state; c.scale = scale; c.l2 = use_qk_l2norm;
    size_t scratch = (size_t)dv * dk + 2 * (size_t)dk;
    return run_pool(rec_unit, &c, (int64_t)c.gm.N * H, scratch, nthreads);
}

/* ------------------------------------------------------------------ */
/* oracle_decode_step: one token per (sequence, head), state in place   */
/* ------------------------------------------------------------------ */

typedef struct {
    double *state;
    const double *q, *k, *v, *g, *beta;
    double *out;
    int32_t H, dk, dv;
    double scale;
    int l2;
} dec_ctx_t;

static void dec_unit(void *vctx, int64_t unit, double *scratch)
{
    dec_ctx_t *c = (dec_ctx_t *)vctx;
    int dk = c->dk, dv = c->dv;
    double *qq = scratch, *kk = scratch + dk;
    load_vec(c->q + unit * dk, qq, dk, c->l2, c->scale);
    load_vec(c->k + unit * dk, kk, dk, c->l2, 1.0);
    gdr_step(c->state + unit * (int64_t)dv * dk, qq, kk, c->v + unit * dv,
             exp(c->g[unit]), c->beta[unit], c->out ? c->out + unit * dv : NULL, dk, dv);
}

int oracle_decode_step(double *state, const double *q, const double *k, const double *v,
                       const double *g, const double *beta, double *out,
                       int32_t N, int32_t H, int32_t dk, int32_t dv,
                       double scale, int32_t use_qk_l2norm, int32_t nthreads)
{
    if (N < 0 || H < 1 || dk < 1 || dv < 1 || !state) return -1;
    dec_ctx_t c;
    c.state = state; c.q = q; c.k = k; c.v = v; c.g = g; c.beta = beta; c.out = out;
    c.H = H; c.dk = dk; c.dv = dv; c.scale = scale; c.l2 = use_qk_l2norm;
    return run_pool(dec_unit, &c, (int64_t)N * H, 2 * (size_t)dk, nthreads);
}

/* ------------------------------------------------------------------ */
/* Chunkwise form                                                      */
/* ------------------------------------------------------------------ */

/*
 * Forward substitution with a unit lower-triangular matrix L (C x C, the
 * diagonal is implicitly 1 and only the strictly lower part is read):
 * solves L X = R in place for X (C x m).
 */
static void unit_lower_solve(const double *L, double *X, int C, int m)
{
    for (int r = 0; r < C; ++r)
        for (int i = 0; i < r; ++i) {
            double a = L[(int64_t)r * C + i];
            if (a == 0.0) continue;
            for (int c = 0; c < m; ++c) X[(int64_t)r * m + c] -= a * X[(int64_t)i * m + c];
        }
}

/*
 * UT transform of one chunk ([paper] §3.3; [blog] §二(一)2(3)-(4)).
 * Inputs are the chunk's rows: K (Cn x dk), V (Cn x dv), alpha, beta (Cn),
 * with the cumulative decay gamma^r = prod_{i<=r} alpha_i re-based at the
 * chunk start.
 *   U~ = [I + strictLower(diag(beta)(Gamma o K K^T))]^{-1} diag(beta) V
 *   w_form 0: W<- = [I + strictLower(diag(beta)(Gamma o K K^T))]^{-1} diag(beta gamma) K
 *   w_form 1: W   = [I + strictLower(diag(beta) K K^T)]^{-1} diag(beta) K  (eq. 6-7),
 *             then W<- = diag(gamma) W  ([blog] §二(一)2(4))
 * W_out receives W<- (Cn x dk) and U_out receives U~ (Cn x dv).
 * scratch: Cn*Cn doubles.
 */
static void ut_transform(const double *K, const double *V, const double *gamma,
                         const double *beta, int Cn, int dk, int dv, int w_form,
                         double *W_out, double *U_out, double *L)
{
    /* Gamma-masked system matrix: L_ri = beta_r (gamma_r/gamma_i) k_i^T k_r, i < r */
    for (int r = 0; r < Cn; ++r)
        for (int i = 0; i < Cn; ++i) {
            double val = 0.0;
            if (i < r) {
                double kk = 0.0;
                for (int d = 0; d < dk; ++d) kk += K[(int64_t)i * dk + d] * K[(int64_t)r * dk + d];
                val = beta[r] * (gamma[r] / gamma[i]) * kk;
            }
            L[(int64_t)r * Cn + i] = val;
        }
    for (int r = 0; r < Cn; ++r)
        for (int c = 0; c < dv; ++c) U_out[(int64_t)r * dv + c] = beta[r] * V[(int64_t)r * dv + c];
    unit_lower_solve(L, U_out, Cn, dv);

    if (w_form == 0) {
        for (int r = 0; r < Cn; ++r)
            for (int d = 0; d < dk; ++d)
                W_out[(int64_t)r * dk + d] = beta[r] * gamma[r] * K[(int64_t)r * dk + d];
        unit_lower_solve(L, W_out, Cn, dk);
    } else {
        /* ungated system of eq. 6 */
        for (int r = 0; r < Cn; ++r)
            for (int i = 0; i < Cn; ++i) {
                double val = 0.0;
                if (i < r) {
                    double kk = 0.0;
                    for (int d = 0; d < dk; ++d) kk += K[(int64_t)i * dk + d] * K[(int64_t)r * dk + d];
                    val = beta[r] * kk;
                }
                L[(int64_t)r * Cn + i] = val;
            }
        for (int r = 0; r < Cn; ++r)
            for (int d = 0; d < dk; ++d)
                W_out[(int64_t)r * dk + d] = beta[r] * K[(int64_t)r * dk + d];
        unit_lower_solve(L, W_out, Cn, dk);
        for (int r = 0; r < Cn; ++r)
            for (int d = 0; d < dk; ++d) W_out[(int64_t)r * dk + d] *= gamma[r];
    }
}

int oracle_ut_transform(const double *K, const double *V, const double *alpha, const double *beta,
                        int32_t Cn, int32_t dk, int32_t dv, int32_t w_form,
                        double *W_out, double *U_out)
{
    if (Cn < 1 || dk < 1 || dv < 1) return -1;
    double *gamma = (double *)malloc(sizeof(double) * (size_t)Cn);
    double *L = (double *)malloc(sizeof(double) * (size_t)Cn * (size_t)Cn);
    if (!gamma || !L) { free(gamma); free(L); return -3; }
    double acc = 1.0;
    for (int r = 0; r < Cn; ++r) { acc *= alpha[r]; gamma[r] = acc; }
    ut_transform(K, V, gamma, beta, Cn, dk, dv, w_form, W_out, U_out, L);
    free(gamma); free(L);
    return 0;
}

typedef struct {
    geom_t gm;
    const double *q, *k, *v, *g, *beta, *s0;
    double *out, *sf;
    double scale;
    int l2, C, w_form;
} chk_ctx_t;

/*
 * Chunk recurrence of [paper] §3.3 with the output mask Gamma of
 * [blog] §二(一)2(3)-(4):
 *   S_[t+1] = gamma^C S_[t] + (U~ - W<- S_[t]^T)^T K->
 *   O_[t]   = Q<- S_[t]^T + (Q K^T o Gamma)(U~ - W<- S_[t]^T)
 * with Q<- = diag(gamma) Q, K-> = diag(gamma^C / gamma) K.
 */
static void chk_unit(void *vctx, int64_t unit, double *scratch)
{
    chk_ctx_t *c = (chk_ctx_t *)vctx;
    const geom_t *gm = &c->gm;
    int H = gm->H, dk = gm->dk, dv = gm->dv, C = c->C;
    int n = (int)(unit / H), h = (int)(unit % H);
    const int64_t sz = (int64_t)dv * dk;
    double *S = scratch;
    double *Q = S + sz;                       /* C x dk */
    double *K = Q + (int64_t)C * dk;          /* C x dk */
    double *V = K + (int64_t)C * dk;          /* C x dv */
    double *W = V + (int64_t)C * dv;          /* C x dk */
    double *U = W + (int64_t)C * dk;          /* C x dv */
    double *Vn = U + (int64_t)C * dv;         /* C x dv : U~ - W<- S^T */
    double *gam = Vn + (int64_t)C * dv;       /* C */
    double *bet = gam + C;                    /* C */
    double *L = bet + C;                      /* C x C */
    double *Snew = L + (int64_t)C * C;        /* dv x dk */

    if (c->s0) memcpy(S, c->s0 + ((int64_t)n * H + h) * sz, sizeof(double) * (size_t)sz);
    else memset(S, 0, sizeof(double) * (size_t)sz);
    int64_t row0, len;
    seq_span(gm, n, &row0, &len);
    for (int64_t t0 = 0; t0 < len; t0 += C) {
        int Cn = (int)((len - t0) < C ? (len - t0) : C);   /* partial last chunk */
        double acc = 1.0;
        for (int r = 0; r < Cn; ++r) {
            int64_t th = (row0 + t0 + r) * H + h;
            load_vec(c->q + th * dk, Q + (int64_t)r * dk, dk, c->l2, c->scale);
            load_vec(c->k + th * dk, K + (int64_t)r * dk, dk, c->l2, 1.0);
            memcpy(V + (int64_t)r * dv, c->v + th * dv, sizeof(double) * (size_t)dv);
            acc *= exp(c->g[th]);
            gam[r] = acc;                         /* gamma^r_[t] */
            bet[r] = c->beta[th];
        }
        ut_transform(K, V, gam, bet, Cn, dk, dv, c->w_form, W, U, L);
        /* effective values U~ - W<- S^T */
        for (int r = 0; r < Cn; ++r)
            for (int j = 0; j < dv; ++j) {
                double ws = 0.0;
                for (int d = 0; d < dk; ++d) ws += W[(int64_t)r * dk + d] * S[(int64_t)j * dk + d];
                Vn[(int64_t)r * dv + j] = U[(int64_t)r * dv + j] - ws;
            }
        /* outputs */
        for (int r = 0; r < Cn; ++r) {
            int64_t th = (row0 + t0 + r) * H + h;
            for (int j = 0; j < dv; ++j) {
                double qs = 0.0;
                for (int d = 0; d < dk; ++d) qs += Q[(int64_t)r * dk + d] * S[(int64_t)j * dk + d];
                double o = gam[r] * qs;
                for (int i = 0; i <= r; ++i) {
                    double qk = 0.0;
                    for (int d = 0; d < dk; ++d) qk += Q[(int64_t)r * dk + d] * K[(int64_t)i * dk + d];
                    o += qk * (gam[r] / gam[i]) * Vn[(int64_t)i * dv + j];
                }
                c->out[th * dv + j] = o;
            }
        }
        /* state */
        double gC = gam[Cn - 1];
        for (int j = 0; j < dv; ++j)
            for (int d = 0; d < dk; ++d) {
                double s = gC * S[(int64_t)j * dk + d];
                for (int r = 0; r < Cn; ++r)
                    s += Vn[(int64_t)r * dv + j] * (gC / gam[r]) * K[(int64_t)r * dk + d];
                Snew[(int64_t)j * dk + d] = s;
            }
        memcpy(S, Snew, sizeof(double) * (size_t)sz);
    }
    if (c->sf) memcpy(c->sf + ((int64_t)n * H + h) * sz, S, sizeof(double) * (size_t)sz);
}

int oracle_chunked_fwd(const double *q, const double *k, const double *v,
                       const double *g, const double *beta,
                       const double *init_state, const int32_t *cu_seqlens, int32_t num_seqs,
                       double *out, double *final_state,
                       int32_t B, int32_t T, int32_t H, int32_t dk, int32_t dv,
                       double scale, int32_t use_qk_l2norm, int32_t chunk_size, int32_t w_form,
                       int32_t nthreads)
{
    chk_ctx_t c;
    c.gm.B = B; c.gm.T = T; c.gm.H = H; c.gm.dk = dk; c.gm.dv = dv;
    c.gm.cu = cu_seqlens; c.gm.N = cu_seqlens ? num_seqs : B;
    if (check_geom(&c.gm) || chunk_size < 1 || (w_form != 0 && w_form != 1)) return -1;
    c.q = q; c.k = k; c.v = v; c.g = g; c.beta = beta; c.s0 = init_state;
    c.out = out; c.sf = final_state; c.scale = scale; c.l2 = use_qk_l2norm;
    c.C = chunk_size; c.w_form = w_form;
    size_t C = (size_t)chunk_size;
    size_t scratch = 2 * (size_t)dv * dk + C * (3 * (size_t)dk + 3 * (size_t)dv + 2 + C);
    return run_pool(chk_unit, &c, (int64_t)c.gm.N * H, scratch, nthreads);
}

int oracle_num_threads(void) { return resolve_threads(0); }


/* ------------------------------------------------------------------ */
/* Block prologue ([paper] §3.4 "Token mixing block", Fig. 1)          */
/* ------------------------------------------------------------------ */

/*
 * q, k, v are produced from their linear projections x by a short causal
 * convolution (depthwise: one filter of K taps per channel) followed by SiLU.
 * Readings (the page gives neither): tap j of the filter multiplies
 * x_{t-K+1+j}, so tap K-1 is the current token; no bias.  Before the first
 * token of a sequence the history comes from state_in (the K-1 most recent
 * earlier inputs, oldest first) or is zero.  state_out receives the K-1 most
 * recent inputs of each sequence in the same layout.
 *
 *   x          [B, T, H, d]        raw projections of one of q, k, v
 *   w          [H, d, K]
 *   state_in   [N, K-1, H, d] or NULL;  state_out [N, K-1, H, d] or NULL
 *   y          [B, T, H, d]        silu(conv(x))
 */
static double silu(double z) { return z / (1.0 + exp(-z)); }

int oracle_short_conv_silu(const double *x, const double *w, const double *state_in, const int32_t *cu,
                           int32_t N, int32_t B, int32_t T, int32_t H, int32_t d, int32_t K,
                           double *y, double *state_out)
{
    if (B < 1 || T < 0 || H < 1 || d < 1 || K < 1) return -1;
    if (cu && B != 1) return -1;
    if (!cu) N = B;
    geom_t gm = {B, T, H, d, d, N, cu};
    if (cu && check_geom(&gm) != 0) return -1;
    const int64_t HD = (int64_t)H * d;
    for (int n = 0; n < N; ++n) {
        int64_t row0, len;
        seq_span(&gm, n, &row0, &len);
        for (int64_t hc = 0; hc < HD; ++hc) {
            /* value of the input at position p (relative to the sequence start) */
#define XAT(p) ((p) >= 0 ? x[(row0 + (p)) * HD + hc]                                              \
                         : (state_in ? state_in[((int64_t)n * (K - 1) + (K - 1) + (p)) * HD + hc] : 0.0))
            for (int64_t t = 0; t < len; ++t) {
                double z = 0.0;
                for (int j = 0; j < K; ++j) z += w[hc * K + j] * XAT(t - (K - 1) + j);
                y[(row0 + t) * HD + hc] = silu(z);
            }
            if (state_out)
                for (int m = 0; m < K - 1; ++m)
                    state_out[((int64_t)n * (K - 1) + m) * HD + hc] = XAT(len - (K - 1) + m);
#undef XAT
        }
    }
    return 0;
}

/*
 * alpha in Mamba2's parameterisation and beta by a sigmoid ([paper] §3.4: alpha
 * and beta come from linear projections only, alpha "with Mamba2's
 * parameterisation"):  g = log alpha = -exp(A_log[h]) * softplus(a + dt_bias[h]),
 * beta = sigmoid(b).   a, b, g, beta [B, T, H];  A_log, dt_bias [H].
 */
static double softplus(double z) { return z > 30.0 ? z : log1p(exp(z)); }

int oracle_gate_activations(const double *a, const double *b, const double *A_log, const double *dt_bias,
                            int64_t BT, int32_t H, double *g, double *beta)
{
    for (int64_t t = 0; t < BT; ++t)
        for (int h = 0; h < H; ++h) {
            const int64_t i = t * H + h;
            g[i] = -exp(A_log[h]) * softplus(a[i] + dt_bias[h]);
            beta[i] = 1.0 / (1.0 + exp(-b[i]));
        }
    return 0;
}


/* ------------------------------------------------------------------ */
/* Backward of the token recurrence (reverse mode)                     */
/* ------------------------------------------------------------------ */

/*
 * With q^ = scale q r_q, k^ = k r_k (r = (|x|^2 + eps)^{-1/2} when use_qk_l2norm,
 * else 1), one step of eq. 10 in the decay-then-correct form is
 *     Sbar = alpha S_{t-1},  e = beta (v - Sbar k^),  S_t = Sbar + e k^T,  o_t = S_t q^.
 * Given D = dL/dS_t (after adding dO_t q^T for the output), the step's adjoint is
 *     de = D k^,  dv = beta de,  dbeta = de . (v - Sbar k^),
 *     dk^ = D^T e - beta Sbar^T de,   dq^ = S_t^T dO_t,
 *     dSbar = D - beta de k^T,  dg = <dSbar, Sbar>,  dS_{t-1} = alpha dSbar,
 * then the normalisations: dx = r dx^ - r^3 (x . dx^) x (times scale for q).
 * dout [B,T,H,dv] and dfinal [N,H,dv,dk] (or NULL) are the loss gradients of the
 * outputs; results dq, dk [B,T,H,dk], dv [B,T,H,dv], dg, dbeta [B,T,H],
 * dinit [N,H,dv,dk] (or NULL).
 */
typedef struct {
    geom_t gm;
    const double *q, *k, *v, *g, *beta, *s0, *dout, *dsf;
    double *dq, *dk, *dv, *dg, *dbeta, *ds0;
    double scale;
    int l2;
    int err;
} bwd_ctx_t;

static void bwd_unit(void *vctx, int64_t unit, double *scratch)
{
    bwd_ctx_t *c = (bwd_ctx_t *)vctx;
    const geom_t *gm = &c->gm;
    const int H = gm->H, dk = gm->dk, dv = gm->dv;
    const int n = (int)(unit / H), h = (int)(unit % H);
    const int64_t sz = (int64_t)dv * dk;
    int64_t row0, len;
    seq_span(gm, n, &row0, &len);
    double *St = (double *)malloc(sizeof(double) * (size_t)((len + 1) * sz));   /* S_0 .. S_len */
    double *qh = (double *)malloc(sizeof(double) * (size_t)(len > 0 ? len * dk : 1));
    double *kh = (double *)malloc(sizeof(double) * (size_t)(len > 0 ? len * dk : 1));
    if (!St || !qh || !kh) { c->err = 1; free(St); free(qh); free(kh); return; }
    double *D = scratch, *dSb = D + sz, *Sb = dSb + sz, *p = Sb + sz, *e = p + dv, *de = e + dv;
    double *dqh = de + dv, *dkh = dqh + dk;

    /* forward, keeping every state */
    if (c->s0) memcpy(St, c->s0 + ((int64_t)n * H + h) * sz, sizeof(double) * (size_t)sz);
    else memset(St, 0, sizeof(double) * (size_t)sz);
    for (int64_t t = 0; t < len; ++t) {
        const int64_t th = (row0 + t) * H + h;
        load_vec(c->q + th * dk, qh + t * dk, dk, c->l2, c->scale);
        load_vec(c->k + th * dk, kh + t * dk, dk, c->l2, 1.0);
        memcpy(St + (t + 1) * sz, St + t * sz, sizeof(double) * (size_t)sz);
        gdr_step(St + (t + 1) * sz, qh + t * dk, kh + t * dk, c->v + th * dv, exp(c->g[th]), c->beta[th],
                 NULL, dk, dv);
    }

    /* reverse */
    if (c->dsf) memcpy(D, c->dsf + ((int64_t)n * H + h) * sz, sizeof(double) * (size_t)sz);
    else memset(D, 0, sizeof(double) * (size_t)sz);
    for (int64_t t = len - 1; t >= 0; --t) {
        const int64_t th = (row0 + t) * H + h;
        const double *S1 = St + (t + 1) * sz, *S0 = St + t * sz;
        const double *qq = qh + t * dk, *kk = kh + t * dk, *vv = c->v + th * dv, *dO = c->dout + th * dv;
        const double alpha = exp(c->g[th]), b = c->beta[th];
        for (int j = 0; j < dv; ++j)
            for (int d = 0; d < dk; ++d) D[j * dk + d] += dO[j] * qq[d];
        for (int d = 0; d < dk; ++d) {
            double acc = 0.0;
            for (int j = 0; j < dv; ++j) acc += S1[j * dk + d] * dO[j];
            dqh[d] = acc;
        }
        for (int64_t i = 0; i < sz; ++i) Sb[i] = alpha * S0[i];
        double dbeta = 0.0;
        for (int j = 0; j < dv; ++j) {
            double pj = 0.0, dej = 0.0;
            for (int d = 0; d < dk; ++d) { pj += Sb[j * dk + d] * kk[d]; dej += D[j * dk + d] * kk[d]; }
            p[j] = pj;
            e[j] = b * (vv[j] - pj);
            de[j] = dej;
            dbeta += dej * (vv[j] - pj);
            c->dv[th * dv + j] = b * dej;
        }
        for (int d = 0; d < dk; ++d) {
            double acc = 0.0;
            for (int j = 0; j < dv; ++j) acc += D[j * dk + d] * e[j] - b * Sb[j * dk + d] * de[j];
            dkh[d] = acc;
        }
        double dg = 0.0;
        for (int j = 0; j < dv; ++j)
            for (int d = 0; d < dk; ++d) {
                const double x = D[j * dk + d] - b * de[j] * kk[d];
                dSb[j * dk + d] = x;
                dg += x * Sb[j * dk + d];
            }
        for (int64_t i = 0; i < sz; ++i) D[i] = alpha * dSb[i];
        c->dbeta[th] = dbeta;
        c->dg[th] = dg;
        /* through the normalisations (and scale on q) */
        const double *qr = c->q + th * dk, *kr = c->k + th * dk;
        if (c->l2) {
            double sq = 0.0, sk = 0.0, qd = 0.0, kd = 0.0;
            for (int d = 0; d < dk; ++d) { sq += qr[d] * qr[d]; sk += kr[d] * kr[d]; qd += qr[d] * dqh[d]; kd += kr[d] * dkh[d]; }
            const double rq = 1.0 / sqrt(sq + ORACLE_L2_EPS), rk = 1.0 / sqrt(sk + ORACLE_L2_EPS);
            for (int d = 0; d < dk; ++d) {
                c->dq[th * dk + d] = c->scale * (rq * dqh[d] - rq * rq * rq * qd * qr[d]);
                c->dk[th * dk + d] = rk * dkh[d] - rk * rk * rk * kd * kr[d];
            }
        } else {
            for (int d = 0; d < dk; ++d) {
                c->dq[th * dk + d] = c->scale * dqh[d];
                c->dk[th * dk + d] = dkh[d];
            }
        }
        (void)p;
    }
    if (c->ds0) memcpy(c->ds0 + ((int64_t)n * H + h) * sz, D, sizeof(double) * (size_t)sz);
    free(St);
    free(qh);
    free(kh);
}

int oracle_recurrent_bwd(const double *q, const double *k, const double *v, const double *g, const double *beta,
                         const double *init_state, const int32_t *cu_seqlens, int32_t num_seqs,
                         const double *dout, const double *dfinal,
                         double *dq, double *dk, double *dv, double *dg, double *dbeta, double *dinit,
                         int32_t B, int32_t T, int32_t H, int32_t dkk, int32_t dvv,
                         double scale, int32_t use_qk_l2norm, int32_t nthreads)
{
    bwd_ctx_t c;
    c.gm.B = B; c.gm.T = T; c.gm.H = H; c.gm.dk = dkk; c.gm.dv = dvv;
    c.gm.cu = cu_seqlens; c.gm.N = cu_seqlens ? num_seqs : B;
    if (check_geom(&c.gm)) return -1;
    c.q = q; c.k = k; c.v = v; c.g = g; c.beta = beta; c.s0 = init_state; c.dout = dout; c.dsf = dfinal;
    c.dq = dq; c.dk = dk; c.dv = dv; c.dg = dg; c.dbeta = dbeta; c.ds0 = dinit;
    c.scale = scale; c.l2 = use_qk_l2norm; c.err = 0;
    /* tokens outside every sequence get zero gradients */
    memset(dq, 0, sizeof(double) * (size_t)B * T * H * dkk);
    memset(dk, 0, sizeof(double) * (size_t)B * T * H * dkk);
    memset(dv, 0, sizeof(double) * (size_t)B * T * H * dvv);
    memset(dg, 0, sizeof(double) * (size_t)B * T * H);
    memset(dbeta, 0, sizeof(double) * (size_t)B * T * H);
    size_t scratch = 3 * (size_t)dvv * dkk + 3 * (size_t)dvv + 2 * (size_t)dkk;
    int rc = run_pool(bwd_unit, &c, (int64_t)c.gm.N * H, scratch, nthreads);
    return rc ? rc : (c.err ? -2 : 0);
}
