/*
 * kda_oracle.c -- plain, slow, f64 CPU oracle of the Kimi Delta Attention (KDA) mixer and its
 * scalar-gate special case, Gated DeltaNet (GDN).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the numeric truth that the CUDA library is checked
 * against.  Nothing in the product path may link, load or call it: only the test suite, the
 * smoke check and the benchmark's CPU-baseline leg do.  It shares no code, header, table or
 * constant with the CUDA sources.
 *
 * Every routine is written straight from the definition, in f64, one token at a time, with no
 * blocking, fusion or reordering beyond what the definition states.  Sources (page titles are the
 * docs.rs pages the method is taken from):
 *   [KDA]  "memra_engine/kda.rs" (memra-engine 0.125.0): module doc, `kda_core_gated` stages 2-6,
 *          `Engine::kda_conv_silu` / `kda_conv_ring_roll` / `kda_gate` / `kda_scan` /
 *          `kda_gated_rmsnorm`.
 *   [GDN]  "aprender-serve 0.70.2 src/cuda/executor/gdn_ops.rs": `gdn_causal_conv1d_silu_into`,
 *          `gdn_per_head_l2_norm_into`, `gdn_gates_into`, `gdn_delta_rule_into`,
 *          `gdn_gated_rmsnorm_into`.
 *
 * Layouts (all row-major, C order):
 *   token-major activations  x[t][c], c = h*D + i  (channel c IS the (head, dim) pair: [KDA]
 *                            module doc, "Geometry")
 *   conv weights             w[c][j], j = 0..K-1, j = K-1 multiplies the current token
 *   conv ring                ring[c][s], s = 0..K-2, slot 0 the oldest raw sample
 *   recurrent state          M[h][j][i] = S_h[i][j]: S is the math matrix with rows i = key dim
 *                            and columns j = value dim; the buffer stores it transposed
 *                            ("M[col][i]" in [KDA] `kda_core` doc).
 *
 * Pinned by tests/test_oracle_pins.py (hand-derived recurrence, invariants, brute force, state
 * carry); see the header of that file for which pin covers which routine.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------------------------ */
/* scalar helpers                                                                              */
/* ------------------------------------------------------------------------------------------ */

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

static double silu(double x) { return x * sigmoid(x); }

/* softplus(x) = log(1 + e^x), computed exactly in f64 without a cutoff:
 * max(x, 0) + log1p(exp(-|x|)).                                                               */
static double softplus(double x) { return (x > 0.0 ? x : 0.0) + log1p(exp(-fabs(x))); }

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------------------------ */
/* a1 + a2: causal depthwise short conv + SiLU, and the ring roll                               */
/* ------------------------------------------------------------------------------------------ */

/*
 * One plane (or any set of independent channels) of one sequence.
 * [KDA] `kda_core_gated` stage 2 and `Engine::kda_conv_silu` / `kda_conv_ring_roll`; ring
 * orientation (shift left, new sample appended) from [GDN] `gdn_causal_conv1d_silu_into`.
 *
 * For channel c define the window sequence xt[] of length (K-1)+T:
 *     xt[s]       = ring_in[c][s]     for s = 0..K-2   (older history, oldest first)
 *     xt[K-1+t]   = x[t][c]           for t = 0..T-1   (this call's raw rows)
 * Then
 *     y[t][c]        = silu( sum_{j=0}^{K-1} w[c][j] * xt[t+j] )     (taps summed j ascending)
 *     ring_out[c][s] = xt[T+s]                                        (the last K-1 raw samples)
 * ring_out may alias ring_in (every old slot of a channel is read before any is written).
 * If w == NULL the conv and SiLU are skipped: y = x and the ring is not touched.
 */
void orc_conv_silu(const double* x, long x_stride, const double* w, const double* ring_in,
                   double* y, long y_stride, double* ring_out, int T, int Cch, int K) {
    if (w == NULL) {
        for (int t = 0; t < T; ++t)
            for (int c = 0; c < Cch; ++c) y[(long)t * y_stride + c] = x[(long)t * x_stride + c];
        return;
    }
    const int R = K - 1;
    double* xt = (double*)malloc(sizeof(double) * (size_t)(R + T > 0 ? R + T : 1));
    for (int c = 0; c < Cch; ++c) {
        for (int s = 0; s < R; ++s) xt[s] = ring_in[(long)c * R + s];
        for (int t = 0; t < T; ++t) xt[R + t] = x[(long)t * x_stride + c];
        for (int t = 0; t < T; ++t) {
            double acc = 0.0;
            for (int j = 0; j < K; ++j) acc += w[(long)c * K + j] * xt[t + j];
            y[(long)t * y_stride + c] = silu(acc);
        }
        for (int s = 0; s < R; ++s) ring_out[(long)c * R + s] = xt[T + s];
    }
    free(xt);
}

/* ------------------------------------------------------------------------------------------ */
/* a3: l2 norm over head_dim                                                                    */
/* ------------------------------------------------------------------------------------------ */

/*
 * y = x / sqrt( sum_i x_i^2 + eps ), row by row over rows of length D.
 * eps is added to the SUM of squares, inside the sqrt: [KDA] constant `KDA_L2_EPS` doc and
 * stage 3; [GDN] `gdn_per_head_l2_norm_into` doc.
 */
void orc_l2norm(const double* x, double* y, long rows, int D, double eps) {
    for (long r = 0; r < rows; ++r) {
        double ss = 0.0;
        for (int i = 0; i < D; ++i) ss += x[r * D + i] * x[r * D + i];
        const double inv = 1.0 / sqrt(ss + eps);
        for (int i = 0; i < D; ++i) y[r * D + i] = x[r * D + i] * inv;
    }
}

/* ------------------------------------------------------------------------------------------ */
/* a4: gates                                                                                    */
/* ------------------------------------------------------------------------------------------ */

/*
 * KDA per-channel forget gate, emitted as the raw log-decay ([KDA] stage 4, `Engine::kda_gate`):
 *     g[r][h*D+i] = lb * sigmoid( exp(a_log[h]) * (f[r][h*D+i] + dt_bias[h*D+i]) )
 * dt_bias is per CHANNEL ([KDA] `KdaAttnLayer::dt_bias` doc); lb is the lower bound (-5.0).
 */
void orc_gate_kda(const double* f, const double* dt_bias, const double* a_log, double lb,
                  double* g, long rows, int H, int D) {
    const int C = H * D;
    for (long r = 0; r < rows; ++r)
        for (int h = 0; h < H; ++h)
            for (int i = 0; i < D; ++i) {
                const int c = h * D + i;
                g[r * C + c] = lb * sigmoid(exp(a_log[h]) * (f[r * C + c] + dt_bias[c]));
            }
}

/*
 * GDN per-head scalar log-decay ([GDN] `gdn_gates_into`: dt = softplus(alpha + dt_bias) * a,
 * with the decay rate a = -exp(A_log)):
 *     g[r][h] = -exp(a_log[h]) * softplus( alpha[r][h] + dt_bias[h] )
 */
void orc_gate_gdn(const double* alpha, const double* dt_bias, const double* a_log, double* g,
                  long rows, int H) {
    for (long r = 0; r < rows; ++r)
        for (int h = 0; h < H; ++h)
            g[r * H + h] = -exp(a_log[h]) * softplus(alpha[r * H + h] + dt_bias[h]);
}

/* beta = sigmoid(beta_raw), one per (token, head): [KDA] stage 4; [GDN] `gdn_gates_into`.   */
void orc_sigmoid(const double* x, double* y, long n) {
    for (long i = 0; i < n; ++i) y[i] = sigmoid(x[i]);
}

/* ------------------------------------------------------------------------------------------ */
/* a5: the per-channel gated delta rule (KDA)                                                   */
/* ------------------------------------------------------------------------------------------ */

/*
 * One (sequence, head) unit, T tokens, generic D.  [KDA] module doc and stage 5
 * (`Engine::kda_scan`: "the per-channel-decay delta-rule scan"), in this order per token t:
 *     S   <- Diag(exp(g_t)) S            decay on the key dim i (rows of S)
 *     u   =  v_t - S^T k_t               (with the decayed S)
 *     S   <- S + beta_t * k_t u^T
 *     o_t =  scale * S^T q_t             (readout from the updated S; q only feeds the readout)
 * q, k, v, g point at this head's first row; consecutive tokens are row_stride apart.
 * beta points at this head's first token; consecutive tokens are beta_stride apart.
 * m_in / m_out hold M[j][i] = S[i][j] for this head (D*D each); they may not alias.
 */
static void scan_kda_unit(const double* q, const double* k, const double* v, const double* g,
                          long row_stride, const double* beta, long beta_stride,
                          const double* m_in, double* m_out, double* o, long o_stride, int T,
                          int D, double scale) {
    double* S = (double*)malloc(sizeof(double) * (size_t)D * D); /* S[i*D + j] */
    double* u = (double*)malloc(sizeof(double) * (size_t)D);
    for (int i = 0; i < D; ++i)
        for (int j = 0; j < D; ++j) S[i * D + j] = m_in[(long)j * D + i];

    for (int t = 0; t < T; ++t) {
        const double* qt = q + (long)t * row_stride;
        const double* kt = k + (long)t * row_stride;
        const double* vt = v + (long)t * row_stride;
        const double* gt = g + (long)t * row_stride;
        const double bt = beta[(long)t * beta_stride];
        /* decay */
        for (int i = 0; i < D; ++i) {
            const double a = exp(gt[i]);
            for (int j = 0; j < D; ++j) S[i * D + j] *= a;
        }
        /* u = v - S^T k */
        for (int j = 0; j < D; ++j) {
            double acc = 0.0;
            for (int i = 0; i < D; ++i) acc += S[i * D + j] * kt[i];
            u[j] = vt[j] - acc;
        }
        /* rank-1 update */
        for (int i = 0; i < D; ++i)
            for (int j = 0; j < D; ++j) S[i * D + j] += bt * kt[i] * u[j];
        /* readout */
        for (int j = 0; j < D; ++j) {
            double acc = 0.0;
            for (int i = 0; i < D; ++i) acc += S[i * D + j] * qt[i];
            o[(long)t * o_stride + j] = scale * acc;
        }
    }
    for (int i = 0; i < D; ++i)
        for (int j = 0; j < D; ++j) m_out[(long)j * D + i] = S[i * D + j];
    free(u);
    free(S);
}

/*
 * Batched KDA scan over N packed sequences.  Rows of sequence n are cu[n] .. cu[n+1]-1 of the
 * token-major arrays q, k, v, g ([rows][H][D]), beta ([rows][H]) and o ([rows][H][D]).
 * state_in / state_out: [N][H][D][D] in the M[j][i] layout.  OpenMP over (n, h): the units are
 * independent, and each unit's arithmetic is the serial definition above.
 */
void orc_scan_kda(const double* q, const double* k, const double* v, const double* g,
                  const double* beta, const int64_t* cu, int N, int H, int D,
                  const double* state_in, double* state_out, double* o, double scale) {
    const long C = (long)H * D;
    const long DD = (long)D * D;
    long units = (long)N * H;
#pragma omp parallel for schedule(dynamic, 1)
    for (long u = 0; u < units; ++u) {
        const int n = (int)(u / H), h = (int)(u % H);
        const long r0 = cu[n];
        const int T = (int)(cu[n + 1] - cu[n]);
        const long off = r0 * C + (long)h * D;
        scan_kda_unit(q + off, k + off, v + off, g + off, C, beta + r0 * H + h, H,
                      state_in + ((long)n * H + h) * DD, state_out + ((long)n * H + h) * DD,
                      o + off, C, T, D, scale);
    }
}

/*
 * The same recurrence with a key width Dk and a value width Dv of their own ([GDN]
 * `gdn_delta_rule_into` doc: q and k are num_k_heads * head_k_dim wide, v and the output
 * num_v_heads * head_v_dim, the state num_v_heads * head_v_dim * head_k_dim).  S is Dk x Dv
 * (rows i = key dim, columns j = value dim); the buffer stores M[j][i] = S[i][j], Dv rows of Dk.
 * q, k, g: [rows][H][Dk]; v, o: [rows][H][Dv]; beta: [rows][H]; state [N][H][Dv][Dk].
 * Written out on its own (not through the square routine), token by token, in the same order:
 * decay, u = v - S^T k, rank-1 update, readout.
 */
void orc_scan_kda_rect(const double* q, const double* k, const double* v, const double* g,
                       const double* beta, const int64_t* cu, int N, int H, int Dk, int Dv,
                       const double* state_in, double* state_out, double* o, double scale) {
    const long Ck = (long)H * Dk, Cv = (long)H * Dv;
    const long SS = (long)Dk * Dv;
    long units = (long)N * H;
#pragma omp parallel for schedule(dynamic, 1)
    for (long un = 0; un < units; ++un) {
        const int n = (int)(un / H), h = (int)(un % H);
        const long r0 = cu[n];
        const int T = (int)(cu[n + 1] - cu[n]);
        const double* min = state_in + ((long)n * H + h) * SS;
        double* mout = state_out + ((long)n * H + h) * SS;
        double* S = (double*)malloc(sizeof(double) * (size_t)SS);   /* S[i*Dv + j] */
        double* uu = (double*)malloc(sizeof(double) * (size_t)Dv);
        for (int i = 0; i < Dk; ++i)
            for (int j = 0; j < Dv; ++j) S[(long)i * Dv + j] = min[(long)j * Dk + i];
        for (int t = 0; t < T; ++t) {
            const double* qt = q + (r0 + t) * Ck + (long)h * Dk;
            const double* kt = k + (r0 + t) * Ck + (long)h * Dk;
            const double* gt = g + (r0 + t) * Ck + (long)h * Dk;
            const double* vt = v + (r0 + t) * Cv + (long)h * Dv;
            const double bt = beta[(r0 + t) * H + h];
            for (int i = 0; i < Dk; ++i) {
                const double decay = exp(gt[i]);
                for (int j = 0; j < Dv; ++j) S[(long)i * Dv + j] *= decay;
            }
            for (int j = 0; j < Dv; ++j) {
                double sk = 0.0;
                for (int i = 0; i < Dk; ++i) sk += S[(long)i * Dv + j] * kt[i];
                uu[j] = vt[j] - sk;
            }
            for (int i = 0; i < Dk; ++i)
                for (int j = 0; j < Dv; ++j) S[(long)i * Dv + j] += bt * kt[i] * uu[j];
            for (int j = 0; j < Dv; ++j) {
                double sq = 0.0;
                for (int i = 0; i < Dk; ++i) sq += S[(long)i * Dv + j] * qt[i];
                o[(r0 + t) * Cv + (long)h * Dv + j] = scale * sq;
            }
        }
        for (int i = 0; i < Dk; ++i)
            for (int j = 0; j < Dv; ++j) mout[(long)j * Dk + i] = S[(long)i * Dv + j];
        free(uu);
        free(S);
    }
}

/* ------------------------------------------------------------------------------------------ */
/* a5 (GDN): the scalar-gate delta rule, written separately                                     */
/* ------------------------------------------------------------------------------------------ */

/*
 * [GDN] `gdn_delta_rule_into` (one token per call there; here the token loop is explicit):
 * per token, with one scalar decay alpha_t = exp(g_t) for the whole head,
 *     S <- alpha_t S;  u = v - S^T k;  S <- S + beta k u^T;  o = scale S^T q.
 * Written column by column of S (value dim j), which is how the scalar gate lets the state
 * decompose: each column is an independent D-vector recurrence.
 * g: [rows][H] (one scalar per token and head).  Other layouts as orc_scan_kda.
 */
void orc_scan_gdn(const double* q, const double* k, const double* v, const double* g,
                  const double* beta, const int64_t* cu, int N, int H, int D,
                  const double* state_in, double* state_out, double* o, double scale) {
    const long C = (long)H * D;
    const long DD = (long)D * D;
    long units = (long)N * H;
#pragma omp parallel for schedule(dynamic, 1)
    for (long u = 0; u < units; ++u) {
        const int n = (int)(u / H), h = (int)(u % H);
        const long r0 = cu[n];
        const int T = (int)(cu[n + 1] - cu[n]);
        const double* min = state_in + ((long)n * H + h) * DD;
        double* mout = state_out + ((long)n * H + h) * DD;
        double* col = (double*)malloc(sizeof(double) * (size_t)D);
        for (int j = 0; j < D; ++j) {
            /* column j of S: col[i] = S[i][j] = M[j][i] */
            for (int i = 0; i < D; ++i) col[i] = min[(long)j * D + i];
            for (int t = 0; t < T; ++t) {
                const long row = (r0 + t) * C + (long)h * D;
                const double alpha = exp(g[(r0 + t) * H + h]);
                const double b = beta[(r0 + t) * H + h];
                double sk = 0.0;
                for (int i = 0; i < D; ++i) {
                    col[i] = alpha * col[i];
                    sk += col[i] * k[row + i];
                }
                const double uj = v[row + j] - sk;
                double sq = 0.0;
                for (int i = 0; i < D; ++i) {
                    col[i] = col[i] + b * k[row + i] * uj;
                    sq += col[i] * q[row + i];
                }
                o[row + j] = scale * sq;
            }
            for (int i = 0; i < D; ++i) mout[(long)j * D + i] = col[i];
        }
        free(col);
    }
}

/* ------------------------------------------------------------------------------------------ */
/* a6: gated RMSNorm over head_dim                                                              */
/* ------------------------------------------------------------------------------------------ */

/*
 * [KDA] stage 6 and `Engine::kda_gated_rmsnorm` (the gate itself is not normalised, [GDN]
 * `gdn_gated_rmsnorm_into` doc), per row of length D:
 *     y_i = o_i / sqrt( (1/D) sum_i o_i^2 + eps ) * w_i * gate(z_i)
 * w is [D], shared by all heads.  gate = sigmoid (KDA, silu_gate = 0) or SiLU, z * sigmoid(z)
 * (GDN's `gated_rmsnorm`, silu_gate = 1; the `Engine::kda_gated_rmsnorm` doc contrasts the two).
 */
void orc_gated_rmsnorm(const double* o, const double* w, const double* z, double* y, long rows,
                       int D, double eps, int silu_gate) {
    for (long r = 0; r < rows; ++r) {
        double ss = 0.0;
        for (int i = 0; i < D; ++i) ss += o[r * D + i] * o[r * D + i];
        const double inv = 1.0 / sqrt(ss / D + eps);
        for (int i = 0; i < D; ++i) {
            const double zi = z[r * D + i];
            y[r * D + i] = o[r * D + i] * inv * w[i] * (silu_gate ? silu(zi) : sigmoid(zi));
        }
    }
}

/* ------------------------------------------------------------------------------------------ */
/* stage 1: the projections that read the layer input x                                        */
/* ------------------------------------------------------------------------------------------ */

/*
 * One projection of t token rows: out[s][r] = sum_{k=0}^{in_f-1} w[r][k] * x[s][k], the terms
 * added k ascending from 0, in f64.  w is [rows][in_f] (the layer's `[out, hidden]` weight
 * layout), x is [t][in_f], out is [t][rows].
 * [KDA] `kda_core_gated` stage 1: the six projections q, k, v, forget-down, gate-down and beta
 * each read x this way (`KdaAttnLayer` field docs give the shapes: wq/wk/wv [qkv, hidden],
 * f_a/g_a [head_dim, hidden], b_proj [heads, hidden]); `Engine::kda_proj_fused6` computes the six
 * in one launch with the same result per row.
 */
void orc_matvec_rows(const double* w, const double* x, double* out, long rows, long in_f, int t) {
    for (int s = 0; s < t; ++s) {
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
        for (long r = 0; r < rows; ++r) {
            double acc = 0.0;
            for (long k = 0; k < in_f; ++k) acc += w[r * in_f + k] * x[(long)s * in_f + k];
            out[(long)s * rows + r] = acc;
        }
    }
}
