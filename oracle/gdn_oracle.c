/*
 * gdn_oracle.c -- plain fp64 CPU statement of the Gated Delta Rule (GDN) layer.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the oracle that the CUDA library is
 * checked against.  Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg may load it.  It shares no code, header, table or helper
 * with the CUDA library (gated_deltanet_linear_rule_gb300/csrc), and the
 * library never calls it.
 *
 * What it computes (one GDN linear-attention layer over a batch of sequences,
 * each sequence carrying a causal-conv buffer and a recurrent state S):
 *
 *   The steps are the ones the "System Design" page (SYSTEM_DESIGN.md of the
 *   BI-V100 vLLM patch set) lists under "Runtime Data Flow" for a GatedDeltaNet
 *   layer and under "GDN Kernel Dispatch Detail": projections (done by the
 *   caller), depthwise causal conv1d, L2-normalise q and k, the recurrent
 *   update ("temporal_state decay + delta write", then "Query @ state"), and a
 *   gated RMSNorm before out_proj.  The qLLM README ("What this is") describes
 *   the fixed-size per-sequence state the layer carries.
 *
 *   Written out (all arithmetic in double):
 *     conv:   xt[c] = silu( sum_{j=0}^{W-1} w[c][j] * x_{t-W+1+j}[c] )
 *             with x_{p}, p < 0, taken from the sequence's conv buffer
 *             (buffer row W-1+p), tap W-1 multiplying the current token.
 *             The buffer afterwards holds the last W-1 raw inputs.
 *     L2:     qh = q / sqrt(|q|^2 + eps_l2) * dk^-1/2,  kh = k / sqrt(|k|^2 + eps_l2)
 *     gates:  g = -exp(A_log[h]) * softplus(a + dt_bias[h]),
 *             alpha = exp(g),  beta = sigmoid(b)
 *     delta:  S <- alpha*S;  u = S kh;  S <- S + beta (v - u) kh^T;  o = S qh
 *     norm:   y = o / sqrt(mean_i o_i^2 + eps_n) * w_n  (.)  silu(z)
 *   v-head h reads q/k head floor(h / (Hv/Hqk)).
 *
 * The chunked (WY / UT-transform) form of the delta step is also written out
 * here, only so that the tests can check it against the recurrent definition;
 * the recurrent definition is the oracle for both decode and prefill.
 *
 * Layouts (row-major, contiguous):
 *   q, k   [T][Hqk*dk]     v, z  [T][Hv*dv]     a, b  [T][Hv]
 *   conv_w [C][W] with C = 2*Hqk*dk + Hv*dv, channels ordered [q | k | v]
 *   S      [n][Hv][dv][dk]  (row i of a head's S is the d_v index)
 *   convbuf[n][W-1][C]
 *   out    [T][Hv*dv]
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    int hqk, hv, dk, dv, conv_w;
    double l2_eps, norm_eps;
} gdn_oracle_shape;

static double silu_d(double x) { return x / (1.0 + exp(-x)); }

static double softplus_d(double x)
{
    /* log(1 + e^x), evaluated without overflowing e^x */
    return (x > 0.0 ? x : 0.0) + log1p(exp(-fabs(x)));
}

static double sigmoid_d(double x) { return 1.0 / (1.0 + exp(-x)); }

/* ---------------------------------------------------------------- conv ---- */

/* Depthwise causal conv1d + SiLU over L tokens of C channels.
 * x [L][C] raw inputs, w [C][W], buf [W-1][C] (in: the W-1 inputs preceding
 * x; out: the last W-1 inputs of buf ++ x), y [L][C]. */
void gdn_oracle_conv_silu(int C, int W, int L, const double* x, const double* w,
                          double* buf, double* y)
{
    for (int t = 0; t < L; ++t) {
        for (int c = 0; c < C; ++c) {
            double acc = 0.0;
            for (int j = 0; j < W; ++j) {
                int p = t - (W - 1) + j; /* input position this tap reads */
                double xv = (p >= 0) ? x[(size_t)p * C + c] : buf[(size_t)(W - 1 + p) * C + c];
                acc += w[(size_t)c * W + j] * xv;
            }
            y[(size_t)t * C + c] = silu_d(acc);
        }
    }
    /* new buffer row i holds input position L-(W-1)+i of (old buffer ++ x) */
    if (W > 1) {
        double* nb = (double*)malloc(sizeof(double) * (size_t)(W - 1) * C);
        for (int i = 0; i < W - 1; ++i) {
            int p = L - (W - 1) + i;
            for (int c = 0; c < C; ++c)
                nb[(size_t)i * C + c] = (p >= 0) ? x[(size_t)p * C + c] : buf[(size_t)(W - 1 + p) * C + c];
        }
        memcpy(buf, nb, sizeof(double) * (size_t)(W - 1) * C);
        free(nb);
    }
}

/* ------------------------------------------------------------------ L2 ---- */

/* n vectors of length d: y = x / sqrt(sum x^2 + eps) */
void gdn_oracle_l2norm(int n, int d, double eps, const double* x, double* y)
{
    for (int i = 0; i < n; ++i) {
        double ss = 0.0;
        for (int j = 0; j < d; ++j) ss += x[(size_t)i * d + j] * x[(size_t)i * d + j];
        double inv = 1.0 / sqrt(ss + eps);
        for (int j = 0; j < d; ++j) y[(size_t)i * d + j] = x[(size_t)i * d + j] * inv;
    }
}

/* --------------------------------------------------------------- gates ---- */

/* n tokens of one v-head: g = -exp(A_log)*softplus(a + dt_bias), beta = sigmoid(b).
 * g is the log of the decay alpha = exp(g). */
void gdn_oracle_gates(int n, double A_log, double dt_bias, const double* a, const double* b,
                      double* g, double* beta)
{
    for (int t = 0; t < n; ++t) {
        g[t] = -exp(A_log) * softplus_d(a[t] + dt_bias);
        beta[t] = sigmoid_d(b[t]);
    }
}

/* ------------------------------------------------- delta rule, recurrent ---- */

/* The recurrent definition for one head over L tokens.
 * q [L][dk] (already normalised and scaled), k [L][dk] (normalised),
 * v [L][dv], g [L] (log decay), beta [L], S [dv][dk] in/out, o [L][dv]. */
void gdn_oracle_delta_recurrent(int L, int dk, int dv, const double* q, const double* k,
                                const double* v, const double* g, const double* beta,
                                double* S, double* o)
{
    double* u = (double*)malloc(sizeof(double) * (size_t)dv);
    for (int t = 0; t < L; ++t) {
        const double* kt = k + (size_t)t * dk;
        const double* qt = q + (size_t)t * dk;
        const double* vt = v + (size_t)t * dv;
        double alpha = exp(g[t]);
        /* S <- alpha * S */
        for (int i = 0; i < dv * dk; ++i) S[i] *= alpha;
        /* u = S k */
        for (int i = 0; i < dv; ++i) {
            double acc = 0.0;
            for (int j = 0; j < dk; ++j) acc += S[(size_t)i * dk + j] * kt[j];
            u[i] = acc;
        }
        /* S <- S + beta (v - u) k^T */
        for (int i = 0; i < dv; ++i) {
            double c = beta[t] * (vt[i] - u[i]);
            for (int j = 0; j < dk; ++j) S[(size_t)i * dk + j] += c * kt[j];
        }
        /* o = S q */
        for (int i = 0; i < dv; ++i) {
            double acc = 0.0;
            for (int j = 0; j < dk; ++j) acc += S[(size_t)i * dk + j] * qt[j];
            o[(size_t)t * dv + i] = acc;
        }
    }
    free(u);
}

/* ---------------------------------------------------- delta rule, chunked ---- */

/* The chunked WY (UT-transform) form of the same recurrence, for the self-check.
 * Within a chunk of n tokens (local indices i, j), with G_i = sum_{t<=i} g_t:
 *   D_ij  = exp(G_i - G_j) for i >= j, evaluated as exp(sum_{t=j+1..i} g_t)
 *   A_ij  = beta_i D_ij (k_i . k_j) for i > j, else 0
 *   T     = (I + A)^-1                      (unit lower triangular)
 *   W     = T diag(beta e^G) K,   U = T diag(beta) V
 *   Delta = U - W S0^T
 *   o_i   = e^{G_i} S0 q_i + sum_{j<=i} D_ij (q_i . k_j) Delta_j
 *   S_end = e^{G_{n-1}} S0 + sum_j D_{n-1,j} Delta_j k_j^T
 * Same arguments as the recurrent form plus the chunk length. */
void gdn_oracle_delta_chunked(int L, int dk, int dv, int chunk, const double* q, const double* k,
                              const double* v, const double* g, const double* beta, double* S,
                              double* o)
{
    size_t C = (size_t)chunk;
    double* D = (double*)malloc(sizeof(double) * C * C);
    double* A = (double*)malloc(sizeof(double) * C * C);
    double* T = (double*)malloc(sizeof(double) * C * C);
    double* eG = (double*)malloc(sizeof(double) * C);
    double* Wm = (double*)malloc(sizeof(double) * C * (size_t)dk);
    double* U = (double*)malloc(sizeof(double) * C * (size_t)dv);
    double* Dl = (double*)malloc(sizeof(double) * C * (size_t)dv);
    double* S0 = (double*)malloc(sizeof(double) * (size_t)dv * dk);

    for (int c0 = 0; c0 < L; c0 += chunk) {
        int n = (L - c0 < chunk) ? (L - c0) : chunk;
        const double* K = k + (size_t)c0 * dk;
        const double* Q = q + (size_t)c0 * dk;
        const double* V = v + (size_t)c0 * dv;
        const double* gc = g + c0;
        const double* bc = beta + c0;
        memcpy(S0, S, sizeof(double) * (size_t)dv * dk);

        for (int i = 0; i < n; ++i) {
            double s = 0.0;
            for (int t = 0; t <= i; ++t) s += gc[t];
            eG[i] = exp(s);
            for (int j = 0; j <= i; ++j) {
                double sj = 0.0;
                for (int t = j + 1; t <= i; ++t) sj += gc[t];
                D[(size_t)i * C + j] = exp(sj);
            }
        }
        for (int i = 0; i < n; ++i)
            for (int j = 0; j < n; ++j) {
                double a = 0.0;
                if (i > j) {
                    double kk = 0.0;
                    for (int x = 0; x < dk; ++x) kk += K[(size_t)i * dk + x] * K[(size_t)j * dk + x];
                    a = bc[i] * D[(size_t)i * C + j] * kk;
                }
                A[(size_t)i * C + j] = a;
            }
        /* (I + A) T = I by forward substitution, row by row */
        for (int i = 0; i < n; ++i)
            for (int j = 0; j < n; ++j) {
                double s = (i == j) ? 1.0 : 0.0;
                for (int x = 0; x < i; ++x) s -= A[(size_t)i * C + x] * T[(size_t)x * C + j];
                T[(size_t)i * C + j] = s;
            }
        for (int i = 0; i < n; ++i) {
            for (int x = 0; x < dk; ++x) {
                double s = 0.0;
                for (int j = 0; j < n; ++j) s += T[(size_t)i * C + j] * bc[j] * eG[j] * K[(size_t)j * dk + x];
                Wm[(size_t)i * dk + x] = s;
            }
            for (int x = 0; x < dv; ++x) {
                double s = 0.0;
                for (int j = 0; j < n; ++j) s += T[(size_t)i * C + j] * bc[j] * V[(size_t)j * dv + x];
                U[(size_t)i * dv + x] = s;
            }
        }
        /* Delta = U - W S0^T */
        for (int i = 0; i < n; ++i)
            for (int r = 0; r < dv; ++r) {
                double s = 0.0;
                for (int x = 0; x < dk; ++x) s += Wm[(size_t)i * dk + x] * S0[(size_t)r * dk + x];
                Dl[(size_t)i * dv + r] = U[(size_t)i * dv + r] - s;
            }
        /* outputs */
        for (int i = 0; i < n; ++i) {
            const double* qi = Q + (size_t)i * dk;
            for (int r = 0; r < dv; ++r) {
                double s = 0.0;
                for (int x = 0; x < dk; ++x) s += S0[(size_t)r * dk + x] * qi[x];
                o[(size_t)(c0 + i) * dv + r] = eG[i] * s;
            }
            for (int j = 0; j <= i; ++j) {
                double qk = 0.0;
                for (int x = 0; x < dk; ++x) qk += qi[x] * K[(size_t)j * dk + x];
                double f = D[(size_t)i * C + j] * qk;
                for (int r = 0; r < dv; ++r) o[(size_t)(c0 + i) * dv + r] += f * Dl[(size_t)j * dv + r];
            }
        }
        /* state at the end of the chunk */
        int e = n - 1;
        for (int r = 0; r < dv; ++r)
            for (int x = 0; x < dk; ++x) {
                double s = eG[e] * S0[(size_t)r * dk + x];
                for (int j = 0; j < n; ++j)
                    s += D[(size_t)e * C + j] * Dl[(size_t)j * dv + r] * K[(size_t)j * dk + x];
                S[(size_t)r * dk + x] = s;
            }
    }
    free(D); free(A); free(T); free(eG); free(Wm); free(U); free(Dl); free(S0);
}

/* ---------------------------------------------------- gated RMSNorm ---- */

/* n rows of length dv: y = o / sqrt(mean(o^2) + eps) * w (.) silu(z) */
void gdn_oracle_gated_rmsnorm(int n, int dv, double eps, const double* o, const double* z,
                              const double* w, double* y)
{
    for (int t = 0; t < n; ++t) {
        double ss = 0.0;
        for (int i = 0; i < dv; ++i) ss += o[(size_t)t * dv + i] * o[(size_t)t * dv + i];
        double inv = 1.0 / sqrt(ss / dv + eps);
        for (int i = 0; i < dv; ++i)
            y[(size_t)t * dv + i] = o[(size_t)t * dv + i] * inv * w[i] * silu_d(z[(size_t)t * dv + i]);
    }
}

/* -------------------------------------------------------- whole layer ---- */

/* One GDN layer over n sequences packed along T with cu_seqlens[n+1].
 * chunk == 0 runs the recurrent definition; chunk > 0 runs the chunked form
 * (self-check only).  head_mask[Hv] (nullable) limits the delta/norm steps to
 * the v-heads whose entry is non-zero; S and out of the other heads are left
 * untouched (conv buffers are always advanced).  o_pre (nullable) receives
 * the delta-rule output o before the norm, [T][Hv*dv].  threads <= 0 uses the
 * OpenMP default.  Returns 0, or -1 on a bad argument. */
int gdn_oracle_layer(const gdn_oracle_shape* sh, int n, const int64_t* cu_seqlens,
                     const double* q, const double* k, const double* v, const double* a,
                     const double* b, const double* z, const double* conv_w, const double* A_log,
                     const double* dt_bias, const double* norm_w, double* S, double* convbuf,
                     double* out, double* o_pre, const int* head_mask, int chunk, int threads)
{
    if (!sh || n < 0 || !cu_seqlens) return -1;
    const int hqk = sh->hqk, hv = sh->hv, dk = sh->dk, dv = sh->dv, W = sh->conv_w;
    if (hqk <= 0 || hv <= 0 || dk <= 0 || dv <= 0 || W <= 0 || hv % hqk != 0 || chunk < 0) return -1;
    const int r = hv / hqk;
    const int Cq = hqk * dk, Cv = hv * dv, C = 2 * Cq + Cv;
    const double qscale = 1.0 / sqrt((double)dk);
    for (int s = 0; s < n; ++s)
        if (cu_seqlens[s + 1] < cu_seqlens[s]) return -1;

    /* per-token preprocessing, sequence by sequence: conv + SiLU, L2, gates */
    int64_t T = cu_seqlens[n] - cu_seqlens[0];
    int64_t t_base = cu_seqlens[0];
    double* qh = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1) * Cq);
    double* kh = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1) * Cq);
    double* vc = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1) * Cv);
    double* gg = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1) * hv);
    double* bb = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1) * hv);

    for (int s = 0; s < n; ++s) {
        int64_t t0 = cu_seqlens[s] - t_base;
        int L = (int)(cu_seqlens[s + 1] - cu_seqlens[s]);
        double* x = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * C);
        double* y = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * C);
        for (int t = 0; t < L; ++t) {
            memcpy(x + (size_t)t * C, q + (size_t)(t0 + t) * Cq, sizeof(double) * Cq);
            memcpy(x + (size_t)t * C + Cq, k + (size_t)(t0 + t) * Cq, sizeof(double) * Cq);
            memcpy(x + (size_t)t * C + 2 * Cq, v + (size_t)(t0 + t) * Cv, sizeof(double) * Cv);
        }
        gdn_oracle_conv_silu(C, W, L, x, conv_w, convbuf + (size_t)s * (W - 1) * C, y);
        for (int t = 0; t < L; ++t) {
            gdn_oracle_l2norm(hqk, dk, sh->l2_eps, y + (size_t)t * C, qh + (size_t)(t0 + t) * Cq);
            for (int i = 0; i < Cq; ++i) qh[(size_t)(t0 + t) * Cq + i] *= qscale;
            gdn_oracle_l2norm(hqk, dk, sh->l2_eps, y + (size_t)t * C + Cq, kh + (size_t)(t0 + t) * Cq);
            memcpy(vc + (size_t)(t0 + t) * Cv, y + (size_t)t * C + 2 * Cq, sizeof(double) * Cv);
        }
        free(x);
        free(y);
    }
    for (int h = 0; h < hv; ++h) {
        for (int64_t t = 0; t < T; ++t) {
            double at = a[(size_t)t * hv + h], bt = b[(size_t)t * hv + h];
            gdn_oracle_gates(1, A_log[h], dt_bias[h], &at, &bt, &gg[(size_t)t * hv + h],
                             &bb[(size_t)t * hv + h]);
        }
    }

    /* delta rule + gated RMSNorm, independently per (sequence, v-head) */
    int units = n * hv;
#ifdef _OPENMP
    if (threads > 0) omp_set_num_threads(threads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int unit = 0; unit < units; ++unit) {
        int s = unit / hv, h = unit % hv;
        if (head_mask && !head_mask[h]) continue;
        int hk = h / r;
        int64_t t0 = cu_seqlens[s] - t_base;
        int L = (int)(cu_seqlens[s + 1] - cu_seqlens[s]);
        if (L == 0) continue;
        double* Qh = (double*)malloc(sizeof(double) * (size_t)L * dk);
        double* Kh = (double*)malloc(sizeof(double) * (size_t)L * dk);
        double* Vh = (double*)malloc(sizeof(double) * (size_t)L * dv);
        double* Zh = (double*)malloc(sizeof(double) * (size_t)L * dv);
        double* Gh = (double*)malloc(sizeof(double) * (size_t)L);
        double* Bh = (double*)malloc(sizeof(double) * (size_t)L);
        double* Oh = (double*)malloc(sizeof(double) * (size_t)L * dv);
        double* Yh = (double*)malloc(sizeof(double) * (size_t)L * dv);
        for (int t = 0; t < L; ++t) {
            memcpy(Qh + (size_t)t * dk, qh + (size_t)(t0 + t) * Cq + (size_t)hk * dk, sizeof(double) * dk);
            memcpy(Kh + (size_t)t * dk, kh + (size_t)(t0 + t) * Cq + (size_t)hk * dk, sizeof(double) * dk);
            memcpy(Vh + (size_t)t * dv, vc + (size_t)(t0 + t) * Cv + (size_t)h * dv, sizeof(double) * dv);
            memcpy(Zh + (size_t)t * dv, z + (size_t)(t0 + t) * Cv + (size_t)h * dv, sizeof(double) * dv);
            Gh[t] = gg[(size_t)(t0 + t) * hv + h];
            Bh[t] = bb[(size_t)(t0 + t) * hv + h];
        }
        double* Sh = S + ((size_t)s * hv + h) * (size_t)dv * dk;
        if (chunk == 0)
            gdn_oracle_delta_recurrent(L, dk, dv, Qh, Kh, Vh, Gh, Bh, Sh, Oh);
        else
            gdn_oracle_delta_chunked(L, dk, dv, chunk, Qh, Kh, Vh, Gh, Bh, Sh, Oh);
        gdn_oracle_gated_rmsnorm(L, dv, sh->norm_eps, Oh, Zh, norm_w, Yh);
        for (int t = 0; t < L; ++t) {
            memcpy(out + (size_t)(t0 + t) * Cv + (size_t)h * dv, Yh + (size_t)t * dv, sizeof(double) * dv);
            if (o_pre)
                memcpy(o_pre + (size_t)(t0 + t) * Cv + (size_t)h * dv, Oh + (size_t)t * dv, sizeof(double) * dv);
        }
        free(Qh); free(Kh); free(Vh); free(Zh); free(Gh); free(Bh); free(Oh); free(Yh);
    }
    free(qh); free(kh); free(vc); free(gg); free(bb);
    return 0;
}

/* number of OpenMP threads the layer call would use (1 without OpenMP) */
int gdn_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
