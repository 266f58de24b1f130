/*
 * kda_oracle.c -- fp64 CPU oracle for the Kimi Delta Attention (KDA) serving hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls this file; only the
 * test suite, the smoke check and the benchmark's CPU-baseline / reference leg do.  It shares no code,
 * header, table or constant with the CUDA library.
 *
 * What it computes, per sequence n and head h, token by token (the plain definition, no blocking):
 *
 *   The pages ("A Preview of Production-Scale Kimi K3 Support on vLLM", section "The Hardest Part:
 *   Prefix Caching for KDA") say each KDA layer advances a matrix-like recurrent state together with a
 *   short convolution state; section "KDA prefill and decode" says decode fuses the short convolution,
 *   the state update, the output gate and the normalisation.  The recurrence itself is the gated delta
 *   rule with channel-wise decay (Kimi Linear):
 *
 *       S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T ,   o_t = scale * S_t^T q_t
 *
 *   Steps for one token (channels c of q | k | v, conv width W):
 *     1. causal conv:  x^_c = sum_{j=0}^{W-1} w[h][c][j] * window[j],  window = [W-1 stored raw inputs
 *        (oldest first), current raw input];  then SiLU when conv_silu != 0;  the stored window shifts
 *        by one (it keeps raw, pre-conv inputs).
 *     2. q^ = q / sqrt(|q|^2 + l2_eps),  k^ likewise;  v^ is the conv output unchanged.
 *     3. alpha_i = sigmoid(a_i) per key channel;  beta = sigmoid(b) per head.
 *     4. S' = Diag(alpha) S;  S = S' - beta k^ (k^T S') + beta k^ v^T     (the formula above, expanded)
 *     5. o = scale * S^T q^
 *     6. y = o / sqrt(mean(o^2) + rms_eps) * norm_w * sigmoid(z)   (gate factor 1 when z is absent)
 *   Checkpoints ("vLLM Kimi K3 Support", section "Agentic Cache Retention Policies": interval
 *   retention; "Kimi-K3" recipe: prefix-match unit 128): after the token at absolute position p-1,
 *   if p is a multiple of the interval and p > start_pos, the (S, conv window) pair is recorded.
 *
 * A second entry point evaluates the same recurrence in the chunked WY/UT form (chunks aligned to
 * absolute positions), in fp64 with direct exponentials.  It exists only so that the tests can check
 * the chunked algebra against the recurrent definition.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    int32_t H, dk, dv, W;   /* heads, key dim, value dim, conv width */
    int32_t conv_silu;      /* 1: SiLU after the conv, 0: none */
    double l2_eps, rms_eps, scale;
} ora_cfg;

typedef struct {
    const double *q, *k, *v;   /* [T][H][dk], [T][H][dk], [T][H][dv] raw (pre-conv) inputs */
    const double *a, *b, *z;   /* [T][H][dk] decay logits, [T][H] beta logits, [T][H][dv] gate or NULL */
    const double *conv_w;      /* [H][2dk+dv][W] */
    const double *norm_w;      /* [dv] */
} ora_inputs;

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* Number of checkpoint boundaries p (p % interval == 0) with start < p <= start + len. */
int64_t ora_ckpt_count(int64_t start, int64_t len, int64_t interval)
{
    if (interval <= 0 || len <= 0) return 0;
    return (start + len) / interval - start / interval;
}

int32_t ora_num_threads(void)
{
#ifdef _OPENMP
    return (int32_t)omp_get_max_threads();
#else
    return 1;
#endif
}

void ora_set_threads(int32_t n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* Steps 1-3 for token t of head h: conv (advancing the window), norms, gates.
 * cs: [(W-1)][Cc] raw window of this (sequence, head), updated in place.
 * Outputs: qh[dk], kh[dk], vh[dv], alpha[dk], *beta. */
static void token_preprocess(const ora_cfg *c, const ora_inputs *in, int64_t t, int h, double *cs,
                             double *qh, double *kh, double *vh, double *alpha, double *beta)
{
    const int dk = c->dk, dv = c->dv, W = c->W, H = c->H;
    const int Cc = 2 * dk + dv;
    for (int ch = 0; ch < Cc; ++ch) {
        double x;
        if (ch < dk)
            x = in->q[(t * H + h) * dk + ch];
        else if (ch < 2 * dk)
            x = in->k[(t * H + h) * dk + (ch - dk)];
        else
            x = in->v[(t * H + h) * dv + (ch - 2 * dk)];
        const double *w = in->conv_w + ((int64_t)h * Cc + ch) * W;
        double acc = w[W - 1] * x;
        for (int j = 0; j < W - 1; ++j) acc += w[j] * cs[(int64_t)j * Cc + ch];
        if (c->conv_silu) acc = acc * sigmoid(acc);
        /* shift the raw window: drop the oldest, append x */
        for (int j = 0; j + 1 < W - 1; ++j) cs[(int64_t)j * Cc + ch] = cs[(int64_t)(j + 1) * Cc + ch];
        if (W > 1) cs[(int64_t)(W - 2) * Cc + ch] = x;
        if (ch < dk)
            qh[ch] = acc;
        else if (ch < 2 * dk)
            kh[ch - dk] = acc;
        else
            vh[ch - 2 * dk] = acc;
    }
    double nq = 0.0, nk = 0.0;
    for (int i = 0; i < dk; ++i) { nq += qh[i] * qh[i]; nk += kh[i] * kh[i]; }
    const double rq = 1.0 / sqrt(nq + c->l2_eps), rk = 1.0 / sqrt(nk + c->l2_eps);
    for (int i = 0; i < dk; ++i) { qh[i] *= rq; kh[i] *= rk; }
    for (int i = 0; i < dk; ++i) alpha[i] = sigmoid(in->a[(t * H + h) * dk + i]);
    *beta = sigmoid(in->b[t * H + h]);
}

/* Step 6 for one token. */
static void gated_rmsnorm(const ora_cfg *c, const ora_inputs *in, int64_t t, int h, const double *o, double *y)
{
    const int dv = c->dv;
    double ms = 0.0;
    for (int j = 0; j < dv; ++j) ms += o[j] * o[j];
    ms /= dv;
    const double r = 1.0 / sqrt(ms + c->rms_eps);
    for (int j = 0; j < dv; ++j) {
        double g = in->z ? sigmoid(in->z[(t * c->H + h) * dv + j]) : 1.0;
        y[j] = o[j] * r * in->norm_w[j] * g;
    }
}

/* Token-by-token recurrence for one (sequence, head). */
static void seq_head_recurrent(const ora_cfg *c, const ora_inputs *in, int64_t t0, int64_t len, int64_t start,
                               int h, double *S, double *cs, double *o_out, double *y_out, int64_t interval,
                               double *ck_S, double *ck_conv, int64_t ck_base, int64_t ck_stride_S,
                               int64_t ck_stride_conv)
{
    const int dk = c->dk, dv = c->dv, H = c->H;
    const int Cc = 2 * dk + dv;
    double *qh = malloc(sizeof(double) * dk), *kh = malloc(sizeof(double) * dk);
    double *vh = malloc(sizeof(double) * dv), *al = malloc(sizeof(double) * dk);
    double *kS = malloc(sizeof(double) * dv), *o = malloc(sizeof(double) * dv), *y = malloc(sizeof(double) * dv);
    int64_t ck = ck_base;
    for (int64_t i = 0; i < len; ++i) {
        const int64_t t = t0 + i;
        double beta;
        token_preprocess(c, in, t, h, cs, qh, kh, vh, al, &beta);
        /* S' = Diag(alpha) S */
        for (int r = 0; r < dk; ++r)
            for (int j = 0; j < dv; ++j) S[(int64_t)r * dv + j] *= al[r];
        /* kS = k^T S' */
        for (int j = 0; j < dv; ++j) kS[j] = 0.0;
        for (int r = 0; r < dk; ++r)
            for (int j = 0; j < dv; ++j) kS[j] += kh[r] * S[(int64_t)r * dv + j];
        /* S = S' - beta k (k^T S') + beta k v^T */
        for (int r = 0; r < dk; ++r)
            for (int j = 0; j < dv; ++j) S[(int64_t)r * dv + j] += beta * kh[r] * (vh[j] - kS[j]);
        /* o = scale * S^T q */
        for (int j = 0; j < dv; ++j) o[j] = 0.0;
        for (int r = 0; r < dk; ++r)
            for (int j = 0; j < dv; ++j) o[j] += S[(int64_t)r * dv + j] * qh[r];
        for (int j = 0; j < dv; ++j) o[j] *= c->scale;
        gated_rmsnorm(c, in, t, h, o, y);
        if (o_out) memcpy(o_out + (t * H + h) * dv, o, sizeof(double) * dv);
        if (y_out) memcpy(y_out + (t * H + h) * dv, y, sizeof(double) * dv);
        const int64_t p = start + i + 1; /* prefix length after this token */
        if (interval > 0 && p % interval == 0) {
            if (ck_S) memcpy(ck_S + ck * ck_stride_S + (int64_t)h * dk * dv, S, sizeof(double) * dk * dv);
            if (ck_conv)
                memcpy(ck_conv + ck * ck_stride_conv + (int64_t)h * (c->W - 1) * Cc, cs,
                       sizeof(double) * (c->W - 1) * Cc);
            ++ck;
        }
    }
    free(qh); free(kh); free(vh); free(al); free(kS); free(o); free(y);
}

/* Forward substitution: X = (I + diag(beta) A)^{-1} diag(beta) Y, A strictly lower (n x n, row stride ld).
 * Y, X: [n][m]. */
static void unit_lower_solve(int n, int m, const double *A, int ld, const double *beta, const double *Y, double *X)
{
    for (int r = 0; r < n; ++r) {
        for (int j = 0; j < m; ++j) {
            double acc = Y[(int64_t)r * m + j];
            double s = 0.0;
            for (int u = 0; u < r; ++u) s += A[(int64_t)r * ld + u] * X[(int64_t)u * m + j];
            X[(int64_t)r * m + j] = beta[r] * (acc - s);
        }
    }
}

/* The same recurrence in chunked WY/UT form, fp64, chunks aligned to absolute positions. */
static void seq_head_chunked(const ora_cfg *c, const ora_inputs *in, int64_t t0, int64_t len, int64_t start,
                             int h, double *S, double *cs, double *o_out, double *y_out, int64_t interval,
                             double *ck_S, double *ck_conv, int64_t ck_base, int64_t ck_stride_S,
                             int64_t ck_stride_conv, int C)
{
    const int dk = c->dk, dv = c->dv, H = c->H;
    const int Cc = 2 * dk + dv;
    double *Q = malloc(sizeof(double) * C * dk), *K = malloc(sizeof(double) * C * dk);
    double *V = malloc(sizeof(double) * C * dv), *G = malloc(sizeof(double) * C * dk);
    double *B = malloc(sizeof(double) * C), *A = malloc(sizeof(double) * C * C), *Qk = malloc(sizeof(double) * C * C);
    double *Kp = malloc(sizeof(double) * C * dk), *Wm = malloc(sizeof(double) * C * dk);
    double *Up = malloc(sizeof(double) * C * dv), *U = malloc(sizeof(double) * C * dv);
    double *al = malloc(sizeof(double) * dk), *o = malloc(sizeof(double) * dv), *y = malloc(sizeof(double) * dv);
    double *Sn = malloc(sizeof(double) * dk * dv);
    int64_t ck = ck_base;
    int64_t i = 0;
    while (i < len) {
        const int64_t p0 = start + i;                       /* absolute position of the chunk's first token */
        int64_t n = (p0 / C + 1) * C - p0;                  /* up to the next multiple of C */
        if (n > len - i) n = len - i;
        for (int64_t r = 0; r < n; ++r) {
            double beta;
            token_preprocess(c, in, t0 + i + r, h, cs, Q + r * dk, K + r * dk, V + r * dv, al, &beta);
            B[r] = beta;
            for (int e = 0; e < dk; ++e) G[r * dk + e] = (r ? G[(r - 1) * dk + e] : 0.0) + log(al[e]);
        }
        /* A_rs = sum_e k_re k_se exp(G_re - G_se) (s < r);  Qk_rs likewise with q_r (s <= r) */
        for (int64_t r = 0; r < n; ++r)
            for (int64_t s = 0; s < n; ++s) {
                double a_ = 0.0, q_ = 0.0;
                if (s <= r)
                    for (int e = 0; e < dk; ++e) {
                        double d = exp(G[r * dk + e] - G[s * dk + e]);
                        a_ += K[r * dk + e] * K[s * dk + e] * d;
                        q_ += Q[r * dk + e] * K[s * dk + e] * d;
                    }
                A[r * C + s] = (s < r) ? a_ : 0.0;
                Qk[r * C + s] = (s <= r) ? q_ : 0.0;
            }
        for (int64_t r = 0; r < n; ++r)
            for (int e = 0; e < dk; ++e) Kp[r * dk + e] = K[r * dk + e] * exp(G[r * dk + e]);
        unit_lower_solve((int)n, dk, A, C, B, Kp, Wm); /* W  = T K+ */
        unit_lower_solve((int)n, dv, A, C, B, V, Up);  /* U' = T V  */
        /* U = U' - W S0 */
        for (int64_t r = 0; r < n; ++r)
            for (int j = 0; j < dv; ++j) {
                double s = 0.0;
                for (int e = 0; e < dk; ++e) s += Wm[r * dk + e] * S[(int64_t)e * dv + j];
                U[r * dv + j] = Up[r * dv + j] - s;
            }
        /* o_r = scale * ( S0^T (q_r * exp(G_r)) + sum_{s<=r} Qk_rs U_s ) */
        for (int64_t r = 0; r < n; ++r) {
            for (int j = 0; j < dv; ++j) {
                double s = 0.0;
                for (int e = 0; e < dk; ++e) s += Q[r * dk + e] * exp(G[r * dk + e]) * S[(int64_t)e * dv + j];
                for (int64_t u = 0; u <= r; ++u) s += Qk[r * C + u] * U[u * dv + j];
                o[j] = c->scale * s;
            }
            gated_rmsnorm(c, in, t0 + i + r, h, o, y);
            if (o_out) memcpy(o_out + ((t0 + i + r) * H + h) * dv, o, sizeof(double) * dv);
            if (y_out) memcpy(y_out + ((t0 + i + r) * H + h) * dv, y, sizeof(double) * dv);
        }
        /* S_next = Diag(exp(G_last)) S0 + sum_s (k_s * exp(G_last - G_s)) U_s^T */
        const double *GL = G + (n - 1) * dk;
        for (int e = 0; e < dk; ++e)
            for (int j = 0; j < dv; ++j) {
                double s = exp(GL[e]) * S[(int64_t)e * dv + j];
                for (int64_t u = 0; u < n; ++u) s += K[u * dk + e] * exp(GL[e] - G[u * dk + e]) * U[u * dv + j];
                Sn[(int64_t)e * dv + j] = s;
            }
        memcpy(S, Sn, sizeof(double) * dk * dv);
        i += n;
        const int64_t p = start + i;
        if (interval > 0 && p % interval == 0) {
            if (ck_S) memcpy(ck_S + ck * ck_stride_S + (int64_t)h * dk * dv, S, sizeof(double) * dk * dv);
            if (ck_conv)
                memcpy(ck_conv + ck * ck_stride_conv + (int64_t)h * (c->W - 1) * Cc, cs,
                       sizeof(double) * (c->W - 1) * Cc);
            ++ck;
        }
    }
    free(Q); free(K); free(V); free(G); free(B); free(A); free(Qk); free(Kp); free(Wm); free(Up); free(U);
    free(al); free(o); free(y); free(Sn);
}

/*
 * Runs nseq sequences (tokens cu_seqlens[n] .. cu_seqlens[n+1]-1, absolute positions start_pos[n] + i).
 *   S:    in/out [nseq][H][dk][dv]        initial state, replaced by the final state
 *   conv: in/out [nseq][H][W-1][2dk+dv]   initial raw window, replaced by the final window
 *   o, y: out [T][H][dv] (either may be NULL)
 *   ck_S, ck_conv: out [n_ckpt][H][dk][dv] and [n_ckpt][H][W-1][2dk+dv], checkpoints in sequence order
 *     then position order (either may be NULL; interval 0 emits none)
 *   chunk: 0 = token-by-token definition; > 0 = chunked WY/UT form with that chunk size (the interval
 *     must then be a multiple of it).
 * Returns 0, or -1 for invalid arguments.
 */
int ora_kda_forward(const ora_cfg *cfg, int32_t nseq, const int64_t *cu_seqlens, const int64_t *start_pos,
                    const double *q, const double *k, const double *v, const double *a, const double *b,
                    const double *z, const double *conv_w, const double *norm_w, double *S, double *conv,
                    double *o, double *y, int64_t interval, double *ck_S, double *ck_conv, int32_t chunk)
{
    if (!cfg || nseq < 0 || cfg->H <= 0 || cfg->dk <= 0 || cfg->dv <= 0 || cfg->W < 1) return -1;
    if (chunk < 0 || (chunk > 0 && interval > 0 && interval % chunk != 0)) return -1;
    for (int32_t n = 0; n < nseq; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n] || start_pos[n] < 0) return -1;
    ora_inputs in = {q, k, v, a, b, z, conv_w, norm_w};
    const int H = cfg->H, dk = cfg->dk, dv = cfg->dv, W = cfg->W;
    const int Cc = 2 * dk + dv;
    int64_t *ck_base = malloc(sizeof(int64_t) * (nseq + 1));
    ck_base[0] = 0;
    for (int32_t n = 0; n < nseq; ++n)
        ck_base[n + 1] = ck_base[n] + ora_ckpt_count(start_pos[n], cu_seqlens[n + 1] - cu_seqlens[n], interval);
    const int64_t units = (int64_t)nseq * H;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t u = 0; u < units; ++u) {
        const int32_t n = (int32_t)(u / H);
        const int h = (int)(u % H);
        double *Sn = S + ((int64_t)n * H + h) * dk * dv;
        double *cs = conv + ((int64_t)n * H + h) * (W - 1) * Cc;
        const int64_t t0 = cu_seqlens[n], len = cu_seqlens[n + 1] - cu_seqlens[n];
        if (chunk == 0)
            seq_head_recurrent(cfg, &in, t0, len, start_pos[n], h, Sn, cs, o, y, interval, ck_S, ck_conv,
                               ck_base[n], (int64_t)H * dk * dv, (int64_t)H * (W - 1) * Cc);
        else
            seq_head_chunked(cfg, &in, t0, len, start_pos[n], h, Sn, cs, o, y, interval, ck_S, ck_conv,
                             ck_base[n], (int64_t)H * dk * dv, (int64_t)H * (W - 1) * Cc, chunk);
    }
    free(ck_base);
    return 0;
}
