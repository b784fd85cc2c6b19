/*
 * kda_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 CPU statement of what the Kimi Delta Attention (KDA)
 * layer computes.  Only the test-suite, the smoke check and the CPU-baseline
 * leg of the benchmark may load this file's library.  It shares no code,
 * header, table or constant with the CUDA library, and the CUDA library never
 * calls it.
 *
 * Sources (web pages; cited by title and section):
 *   [ORT-2843]  ONNX Runtime GenAI PR #2843, "Add BailingMoeV3 (Ling-3.0-tiny)
 *               KDA + MLA + MoE model builder and CUDA plugin EP fallback",
 *               section "Summary of Changes" (the KDA ops: causal conv with
 *               state, GatedDeltaNet with per-key-dim decay and a sigmoid
 *               gate activation, GatedRMSNorm(activation='sigmoid'),
 *               gate_lower_bound, separate decay and beta shapes) and the
 *               author's review reply ("validates its bound only in safe
 *               mode").
 *   [TF-850]    TensorFold issue #850, "Ling-3.1-flash on CUDA: a shared KDA
 *               kernel first, then the family at TP=1 and TP=2 (EXL3)",
 *               comment of Oct 15 (the per-row step order: conv window, safe
 *               or softplus gate, beta, q/k L2 norms, delta rule, gated
 *               output norm; prompt rows in chunks from a segment's first
 *               row; a float64 reference).
 *
 * The recurrence (gated delta rule with a per-key-dim decay, one dk x dv
 * state per head):
 *     S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *     o_t = scale * S_t^T q_t
 * written here in the equivalent rank-1 form
 *     S' = Diag(alpha) S ;  u = beta (v - S'^T k) ;  S = S' + k u^T.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - safe gate:      log alpha_i = lb * sigmoid(exp(A_log_h) (f_i + dt_bias_hi))
 *   - softplus gate:  log alpha_i = -exp(A_log_h) * softplus(f_i + dt_bias_hi)
 *   - conv:           depthwise over the concatenated q|k|v channels, no bias,
 *                     tap K-1 multiplies the current row; the carried state
 *                     holds the K-1 previous raw rows, oldest first; SiLU on
 *                     every channel.
 *   - L2 norm:        x * (sum x^2 + eps)^(-1/2)
 *   - output norm:    y = o * (mean o^2 + eps)^(-1/2) * w * sigmoid(g), per head.
 *
 * Parity status: every function below is pinned by the CPU tests against
 * closed forms, invariants, special cases or brute force, except the choice
 * of the two gate formulas themselves (the pages name the gates but never
 * print them): that choice is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int32_t H;            /* heads                                   */
    int32_t dk;           /* key width per head                      */
    int32_t dv;           /* value width per head                    */
    int32_t K;            /* conv taps                               */
    int32_t gate_mode;    /* 0 = softplus gate, 1 = safe gate        */
    int32_t has_out_gate; /* 1 = apply the sigmoid-gated RMSNorm     */
    int32_t chunk;        /* 0 = serial recurrence, C > 0 = chunked  */
    int32_t reserved;
    double lower_bound;   /* safe-gate bound, < 0                    */
    double l2_eps;
    double norm_eps;
    double scale;
} kda_ref_cfg;

/* ---------------------------------------------------------------- scalars */

double kda_ref_sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

double kda_ref_silu(double x) { return x * kda_ref_sigmoid(x); }

/* softplus(x) = log(1 + e^x), written so that it neither overflows nor
 * loses the small tail: max(x, 0) + log1p(e^-|x|). */
double kda_ref_softplus(double x)
{
    double ax = fabs(x);
    return (x > 0.0 ? x : 0.0) + log1p(exp(-ax));
}

/* Per-key-dim log-decay of one key dimension ([ORT-2843] "per-key-dim
 * decay", gate_lower_bound; [TF-850] "the safe or softplus gate"). */
double kda_ref_log_alpha(int32_t gate_mode, double lower_bound, double A_log_h,
                         double f, double dt_bias)
{
    double a = exp(A_log_h);
    double x = f + dt_bias;
    if (gate_mode == 1) return lower_bound * kda_ref_sigmoid(a * x);
    return -a * kda_ref_softplus(x);
}

/* ------------------------------------------------------------- vector ops */

/* y = x * (sum x^2 + eps)^(-1/2)   ([TF-850] "the q/k L2 norms") */
void kda_ref_l2norm(int32_t n, const double* x, double eps, double* y)
{
    double ss = 0.0;
    for (int32_t i = 0; i < n; ++i) ss += x[i] * x[i];
    double r = 1.0 / sqrt(ss + eps);
    for (int32_t i = 0; i < n; ++i) y[i] = x[i] * r;
}

/* y = o * (mean o^2 + eps)^(-1/2) * w * sigmoid(g)
 * ([ORT-2843] GatedRMSNorm(activation='sigmoid')).  w may be NULL (unit). */
void kda_ref_gated_rmsnorm(int32_t n, const double* o, const double* g,
                           const double* w, double eps, double* y)
{
    double ss = 0.0;
    for (int32_t j = 0; j < n; ++j) ss += o[j] * o[j];
    double r = 1.0 / sqrt(ss / (double)n + eps);
    for (int32_t j = 0; j < n; ++j)
        y[j] = o[j] * r * (w ? w[j] : 1.0) * kda_ref_sigmoid(g[j]);
}

/* Causal depthwise conv1d with a carried history ([ORT-2843]
 * CausalConvWithState).  x: [T][C] rows, hist: [K-1][C] previous raw rows
 * (oldest first), w: [C][K].  y[t][c] = sum_j w[c][j] * x_{t-K+1+j}[c], where
 * rows before t = 0 come from hist.  No activation. */
void kda_ref_conv1d(int32_t T, int32_t C, int32_t K, const double* x,
                    const double* hist, const double* w, double* y)
{
    for (int32_t t = 0; t < T; ++t) {
        for (int32_t c = 0; c < C; ++c) {
            double acc = 0.0;
            for (int32_t j = 0; j < K; ++j) {
                int32_t src = t - (K - 1) + j; /* row index, may be < 0 */
                double xv = src >= 0 ? x[(size_t)src * C + c]
                                     : hist[(size_t)(src + K - 1) * C + c];
                acc += w[(size_t)c * K + j] * xv;
            }
            y[(size_t)t * C + c] = acc;
        }
    }
}

/* New carried history after T rows: the last K-1 rows of [hist ; x]. */
void kda_ref_conv_history(int32_t T, int32_t C, int32_t K, const double* x,
                          const double* hist, double* new_hist)
{
    for (int32_t r = 0; r < K - 1; ++r) {
        int32_t src = T - (K - 1) + r; /* row of x, or < 0 -> hist */
        for (int32_t c = 0; c < C; ++c)
            new_hist[(size_t)r * C + c] =
                src >= 0 ? x[(size_t)src * C + c]
                         : hist[(size_t)(src + K - 1) * C + c];
    }
}

/* One token of the gated delta rule on a dk x dv state S (row i = key dim).
 * S' = Diag(alpha) S ; u = beta (v - S'^T k) ; S = S' + k u^T ; o = scale S^T q.
 * u_out (dv) may be NULL.  ([TF-850] "the delta rule"; [ORT-2843]
 * GatedDeltaNet with per-key-dim decay.) */
void kda_ref_delta_step(int32_t dk, int32_t dv, double* S, const double* alpha,
                        double beta, const double* k, const double* v,
                        const double* q, double scale, double* o, double* u_out)
{
    for (int32_t i = 0; i < dk; ++i)
        for (int32_t j = 0; j < dv; ++j) S[(size_t)i * dv + j] *= alpha[i];
    for (int32_t j = 0; j < dv; ++j) {
        double kv = 0.0;
        for (int32_t i = 0; i < dk; ++i) kv += S[(size_t)i * dv + j] * k[i];
        double u = beta * (v[j] - kv);
        if (u_out) u_out[j] = u;
        for (int32_t i = 0; i < dk; ++i) S[(size_t)i * dv + j] += k[i] * u;
    }
    for (int32_t j = 0; j < dv; ++j) {
        double acc = 0.0;
        for (int32_t i = 0; i < dk; ++i) acc += S[(size_t)i * dv + j] * q[i];
        o[j] = scale * acc;
    }
}

/* ------------------------------------------------ chunked (WY / UT) form */

/* Forward substitution: T = (I + A)^{-1} for a strictly lower-triangular
 * n x n matrix A (row-major), by solving (I + A) t_c = e_c column by column. */
static void unit_lower_inverse(int32_t n, const double* A, double* Tm)
{
    for (int32_t c = 0; c < n; ++c) {
        for (int32_t r = 0; r < n; ++r) {
            double acc = (r == c) ? 1.0 : 0.0;
            for (int32_t s = 0; s < r; ++s) acc -= A[(size_t)r * n + s] * Tm[(size_t)s * n + c];
            Tm[(size_t)r * n + c] = acc;
        }
    }
}

/* One chunk of n rows on state S (dk x dv), in the chunked form of the same
 * recurrence.  With G_r = sum_{t<=r} log alpha_t (per key dim):
 *   A_rs = beta_r sum_i k_ri k_si e^{G_ri - G_si}  (s < r)
 *   P_rs =        sum_i q_ri k_si e^{G_ri - G_si}  (s <= r)
 *   T    = (I + A)^{-1}
 *   W    = T Diag(beta) (K o e^G) ;  U' = T Diag(beta) V
 *   U    = U' - W S
 *   O    = scale [ (Q o e^G) S + P U ]
 *   S   <- Diag(e^{G_last}) S + (K o e^{G_last - G})^T U
 * Row-major inputs: kq/kk [n][dk], vv [n][dv], la [n][dk] (log alpha),
 * beta [n].  Output o [n][dv]. */
static void chunk_step(int32_t n, int32_t dk, int32_t dv, double* S,
                       const double* qq, const double* kk, const double* vv,
                       const double* la, const double* beta, double scale,
                       double* o)
{
    double* G = (double*)malloc(sizeof(double) * n * dk);
    double* A = (double*)calloc((size_t)n * n, sizeof(double));
    double* P = (double*)calloc((size_t)n * n, sizeof(double));
    double* Tm = (double*)malloc(sizeof(double) * n * n);
    double* X = (double*)malloc(sizeof(double) * n * dk);  /* Diag(beta)(K o e^G) */
    double* Y = (double*)malloc(sizeof(double) * n * dv);  /* Diag(beta) V        */
    double* W = (double*)malloc(sizeof(double) * n * dk);
    double* U = (double*)malloc(sizeof(double) * n * dv);

    for (int32_t i = 0; i < dk; ++i) {
        double run = 0.0;
        for (int32_t r = 0; r < n; ++r) {
            run += la[(size_t)r * dk + i];
            G[(size_t)r * dk + i] = run;
        }
    }
    for (int32_t r = 0; r < n; ++r) {
        for (int32_t s = 0; s <= r; ++s) {
            double a = 0.0, p = 0.0;
            for (int32_t i = 0; i < dk; ++i) {
                double e = exp(G[(size_t)r * dk + i] - G[(size_t)s * dk + i]);
                a += kk[(size_t)r * dk + i] * kk[(size_t)s * dk + i] * e;
                p += qq[(size_t)r * dk + i] * kk[(size_t)s * dk + i] * e;
            }
            if (s < r) A[(size_t)r * n + s] = beta[r] * a;
            P[(size_t)r * n + s] = p;
        }
    }
    unit_lower_inverse(n, A, Tm);
    for (int32_t s = 0; s < n; ++s) {
        for (int32_t i = 0; i < dk; ++i)
            X[(size_t)s * dk + i] = beta[s] * kk[(size_t)s * dk + i] * exp(G[(size_t)s * dk + i]);
        for (int32_t j = 0; j < dv; ++j) Y[(size_t)s * dv + j] = beta[s] * vv[(size_t)s * dv + j];
    }
    for (int32_t r = 0; r < n; ++r) {
        for (int32_t i = 0; i < dk; ++i) {
            double acc = 0.0;
            for (int32_t s = 0; s < n; ++s) acc += Tm[(size_t)r * n + s] * X[(size_t)s * dk + i];
            W[(size_t)r * dk + i] = acc;
        }
        for (int32_t j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int32_t s = 0; s < n; ++s) acc += Tm[(size_t)r * n + s] * Y[(size_t)s * dv + j];
            U[(size_t)r * dv + j] = acc; /* U' for now */
        }
    }
    /* U = U' - W S  (uses the state at the chunk start) */
    for (int32_t r = 0; r < n; ++r)
        for (int32_t j = 0; j < dv; ++j) {
            double ws = 0.0;
            for (int32_t i = 0; i < dk; ++i) ws += W[(size_t)r * dk + i] * S[(size_t)i * dv + j];
            U[(size_t)r * dv + j] -= ws;
        }
    /* O = (Q o e^G) S + P U */
    for (int32_t r = 0; r < n; ++r)
        for (int32_t j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int32_t i = 0; i < dk; ++i)
                acc += qq[(size_t)r * dk + i] * exp(G[(size_t)r * dk + i]) * S[(size_t)i * dv + j];
            for (int32_t s = 0; s <= r; ++s) acc += P[(size_t)r * n + s] * U[(size_t)s * dv + j];
            o[(size_t)r * dv + j] = scale * acc;
        }
    /* S <- Diag(e^{G_last}) S + (K o e^{G_last - G})^T U */
    for (int32_t i = 0; i < dk; ++i) {
        double gl = G[(size_t)(n - 1) * dk + i];
        double decay = exp(gl);
        for (int32_t j = 0; j < dv; ++j) {
            double acc = decay * S[(size_t)i * dv + j];
            for (int32_t s = 0; s < n; ++s)
                acc += kk[(size_t)s * dk + i] * exp(gl - G[(size_t)s * dk + i]) * U[(size_t)s * dv + j];
            S[(size_t)i * dv + j] = acc;
        }
    }
    free(G); free(A); free(P); free(Tm); free(X); free(Y); free(W); free(U);
}

/* ------------------------------------------------------------ full layer */

/*
 * Forward over a batch of variable-length sequences (segments of cu_seqlens,
 * [ORT-2843] VarlenCausalConvWithState), for the (sequence, head) units
 * unit_begin <= u < unit_end, u = seq * H + head.  Units write disjoint parts
 * of every output, so callers may run unit ranges on separate threads.
 *
 * Layouts (row-major, fp64):
 *   q, k, f: [T][H][dk]   v, g, out: [T][H][dv]   b: [T][H]
 *   A_log: [H]   dt_bias: [H][dk]   conv_w: [conv_dim][K]   norm_w: [dv] or NULL
 *   conv_state: [N][K-1][conv_dim]  (conv_dim = H (2 dk + dv); channel order
 *               q heads, then k heads, then v heads)          -- in/out
 *   S: [N][H][dk][dv]                                          -- in/out
 *   g may be NULL when cfg->has_out_gate == 0.
 * Per row: conv + SiLU, L2-normalised q and k, beta = sigmoid(b), log alpha
 * from the gate, then the delta rule (serially, or in chunks of cfg->chunk
 * rows starting at each segment's first row, [TF-850]), then optionally the
 * gated RMSNorm.  Returns 0, or -1 on a malformed argument.
 */
int kda_ref_forward(const kda_ref_cfg* cfg, int32_t N, const int32_t* cu_seqlens,
                    const double* q, const double* k, const double* v,
                    const double* f, const double* b, const double* g,
                    const double* A_log, const double* dt_bias,
                    const double* conv_w, const double* norm_w,
                    double* conv_state, double* S, double* out,
                    int32_t unit_begin, int32_t unit_end)
{
    const int32_t H = cfg->H, dk = cfg->dk, dv = cfg->dv, K = cfg->K;
    const int32_t conv_dim = H * (2 * dk + dv);
    const int32_t CH = 2 * dk + dv; /* this head's channels: q | k | v */
    if (H <= 0 || dk <= 0 || dv <= 0 || K < 1 || N < 0) return -1;
    if (cfg->has_out_gate && !g) return -1;
    if (CH > 2048 || dk > 1024 || dv > 1024) return -1;

    for (int32_t u = unit_begin; u < unit_end && u < N * H; ++u) {
        const int32_t s = u / H, h = u % H;
        const int32_t t0 = cu_seqlens[s], L = cu_seqlens[s + 1] - cu_seqlens[s];
        if (L < 0) return -1; /* nothing allocated yet for this unit */
        /* gather this head's raw channels: x [L][CH], hist [K-1][CH], w [CH][K] */
        double* x = (double*)malloc(sizeof(double) * ((size_t)L * CH + 1));
        double* y = (double*)malloc(sizeof(double) * ((size_t)L * CH + 1));
        double* hist = (double*)malloc(sizeof(double) * ((size_t)(K - 1) * CH + 1));
        double* nhist = (double*)malloc(sizeof(double) * ((size_t)(K - 1) * CH + 1));
        double* w = (double*)malloc(sizeof(double) * (size_t)CH * K);
        int32_t chan[2048];
        for (int32_t c = 0; c < dk; ++c) chan[c] = h * dk + c;
        for (int32_t c = 0; c < dk; ++c) chan[dk + c] = H * dk + h * dk + c;
        for (int32_t c = 0; c < dv; ++c) chan[2 * dk + c] = 2 * H * dk + h * dv + c;
        for (int32_t t = 0; t < L; ++t) {
            const size_t row = (size_t)(t0 + t) * H + h;
            for (int32_t c = 0; c < dk; ++c) x[(size_t)t * CH + c] = q[row * dk + c];
            for (int32_t c = 0; c < dk; ++c) x[(size_t)t * CH + dk + c] = k[row * dk + c];
            for (int32_t c = 0; c < dv; ++c) x[(size_t)t * CH + 2 * dk + c] = v[row * dv + c];
        }
        double* cs = conv_state + (size_t)s * (K - 1) * conv_dim;
        for (int32_t r = 0; r < K - 1; ++r)
            for (int32_t c = 0; c < CH; ++c) hist[(size_t)r * CH + c] = cs[(size_t)r * conv_dim + chan[c]];
        for (int32_t c = 0; c < CH; ++c)
            for (int32_t j = 0; j < K; ++j) w[(size_t)c * K + j] = conv_w[(size_t)chan[c] * K + j];

        kda_ref_conv1d(L, CH, K, x, hist, w, y);
        kda_ref_conv_history(L, CH, K, x, hist, nhist);
        for (int32_t r = 0; r < K - 1; ++r)
            for (int32_t c = 0; c < CH; ++c) cs[(size_t)r * conv_dim + chan[c]] = nhist[(size_t)r * CH + c];

        /* per-row activations */
        double* qh = (double*)malloc(sizeof(double) * ((size_t)L * dk + 1));
        double* kh = (double*)malloc(sizeof(double) * ((size_t)L * dk + 1));
        double* vv = (double*)malloc(sizeof(double) * ((size_t)L * dv + 1));
        double* la = (double*)malloc(sizeof(double) * ((size_t)L * dk + 1));
        double* bt = (double*)malloc(sizeof(double) * ((size_t)L + 1));
        double* oo = (double*)malloc(sizeof(double) * ((size_t)L * dv + 1));
        double tmp[1024];
        for (int32_t t = 0; t < L; ++t) {
            const size_t row = (size_t)(t0 + t) * H + h;
            for (int32_t c = 0; c < dk; ++c) tmp[c] = kda_ref_silu(y[(size_t)t * CH + c]);
            kda_ref_l2norm(dk, tmp, cfg->l2_eps, qh + (size_t)t * dk);
            for (int32_t c = 0; c < dk; ++c) tmp[c] = kda_ref_silu(y[(size_t)t * CH + dk + c]);
            kda_ref_l2norm(dk, tmp, cfg->l2_eps, kh + (size_t)t * dk);
            for (int32_t c = 0; c < dv; ++c) vv[(size_t)t * dv + c] = kda_ref_silu(y[(size_t)t * CH + 2 * dk + c]);
            bt[t] = kda_ref_sigmoid(b[row]);
            for (int32_t i = 0; i < dk; ++i)
                la[(size_t)t * dk + i] = kda_ref_log_alpha(cfg->gate_mode, cfg->lower_bound, A_log[h],
                                                           f[row * dk + i], dt_bias[(size_t)h * dk + i]);
        }

        double* Sh = S + ((size_t)s * H + h) * dk * dv;
        if (cfg->chunk <= 0) {
            double alpha[1024];
            for (int32_t t = 0; t < L; ++t) {
                for (int32_t i = 0; i < dk; ++i) alpha[i] = exp(la[(size_t)t * dk + i]);
                kda_ref_delta_step(dk, dv, Sh, alpha, bt[t], kh + (size_t)t * dk,
                                   vv + (size_t)t * dv, qh + (size_t)t * dk, cfg->scale,
                                   oo + (size_t)t * dv, NULL);
            }
        } else {
            for (int32_t c0 = 0; c0 < L; c0 += cfg->chunk) {
                int32_t n = L - c0 < cfg->chunk ? L - c0 : cfg->chunk;
                chunk_step(n, dk, dv, Sh, qh + (size_t)c0 * dk, kh + (size_t)c0 * dk,
                           vv + (size_t)c0 * dv, la + (size_t)c0 * dk, bt + c0, cfg->scale,
                           oo + (size_t)c0 * dv);
            }
        }
        for (int32_t t = 0; t < L; ++t) {
            const size_t row = (size_t)(t0 + t) * H + h;
            if (cfg->has_out_gate)
                kda_ref_gated_rmsnorm(dv, oo + (size_t)t * dv, g + row * dv, norm_w, cfg->norm_eps,
                                      out + row * dv);
            else
                for (int32_t j = 0; j < dv; ++j) out[row * dv + j] = oo[(size_t)t * dv + j];
        }
        free(x); free(y); free(hist); free(nhist); free(w);
        free(qh); free(kh); free(vv); free(la); free(bt); free(oo);
    }
    return 0;
}
