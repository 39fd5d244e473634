/*
 * Gated delta-net core: fp64 CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the slow, obviously-correct
 * restatement that the CUDA path is checked against. Only the test suite,
 * the smoke check and the benchmark's CPU-baseline leg may load it; the
 * library's product path never calls it and shares no code with it.
 *
 * Everything is plain scalar loops in double precision (long double for the
 * brute-force check), single-threaded, in the order the method is stated:
 *
 *   O1  causal depthwise conv (kernel 4, 3-wide rolling state) + SiLU
 *       -- page "ferrum-kernels gated_delta_attention_tests.rs" (the Metal
 *          conformance tests), section `cpu_segment`: the conv and the
 *          conv-state update; page "libmir-metal decode/mod.rs", section
 *          `convolve`: history concatenated before the input, depthwise
 *          conv1d, the last kernel-1 inputs kept.
 *   O2  per-head l2 normalisation of q and k
 *       -- gated_delta_attention_tests.rs `cpu_segment` / `normalize_rows`:
 *          x * (sum x^2 + eps)^(-1/2);  ferrox-core gdn.rs `l2_normalize`:
 *          x / max(||x||, eps) (the clamped form, kept as a cross-check).
 *   O3  gates: rate = -exp(A_log) (log-rate) or the given negative rate;
 *       g = rate * softplus(a + dt_bias); beta = sigmoid(b)
 *       -- gated_delta_attention_tests.rs `cpu_segment` gate lines and its
 *          `sigmoid` / `softplus` helpers (two-branch sigmoid, softplus
 *          linear above 20 and exp below -20).
 *   O4  the token recurrence (the definition), per V head h reading K head kh:
 *       S *= exp(g); pred = S k; d = beta (v - pred); S += d k^T;
 *       o = S q / sqrt(Dk)
 *       -- ferrox-core gdn.rs module docs (the six-line formula) and
 *          `delta_step`; gated_delta_attention_tests.rs `cpu_segment` and
 *          `recurrent_chunk_oracle`. Head map: Grouped kh = h / (Hv/Hk),
 *          Tiled kh = h % Hk (gdn.rs `HeadMap::k_head`).
 *   O5  gated RMSNorm: y = o (mean o^2 + eps)^(-1/2) w_j silu(z_j)
 *       -- gated_delta_attention_tests.rs `cpu_segment` output loop.
 *   O6  a whole segment: O1 -> split q|k|v -> O2 -> O3 -> O4 (-> O5).
 *   O7  the same recurrence summed chunk-wise (UT/WY form, chunk length C),
 *       written from the derivation S_t = G_t S_0 + sum_{s<=t} e^{g_t-g_s}
 *       d_s k_s^T; gdn.rs states the chunked kernel is "the same recurrence
 *       in a different summation order". Exists to check O4, not the GPU.
 *   O8  brute force for small D: S_t = a_t S_{t-1} (I - b_t k_t k_t^T)
 *       + b_t v_t k_t^T as explicit matrix products in long double.
 *
 * Layouts (row-major, innermost last):
 *   mixed_qkv/x [T][C]  with C = 2*Hk*D + Hv*D, columns [q | k | v]
 *   conv weight [C][4]  (tap 3 multiplies the current token)
 *   conv state  [C][3]  (oldest first; raw inputs, not convolved)
 *   q, k        [T][Hk][D];  v, o, z [T][Hv][D];  g, beta, a, b [T][Hv]
 *   delta state [Hv][Dv][Dk] = S[h][j][i], key index i innermost.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define GDN_ORACLE_CONV_WIDTH 4
#define GDN_ORACLE_CONV_STATE 3

/* ---------------------------------------------------------------- helpers */

double gdn_oracle_sigmoid(double x) {
    /* two branches so exp never overflows */
    if (x >= 0.0) {
        return 1.0 / (1.0 + exp(-x));
    }
    double e = exp(x);
    return e / (1.0 + e);
}

double gdn_oracle_silu(double x) { return x * gdn_oracle_sigmoid(x); }

double gdn_oracle_softplus(double x) {
    if (x > 20.0) return x;
    if (x < -20.0) return exp(x);
    return log1p(exp(x));
}

int gdn_oracle_k_head(int map, int h, int n_k_heads, int n_v_heads) {
    /* map 0 = Grouped, 1 = Tiled */
    if (map == 1) return h % n_k_heads;
    return h / (n_v_heads / n_k_heads);
}

/* ------------------------------------------------------------------- O1 */

/* One sequence of T tokens. x [T][C], w [C][4], state [C][3] in/out,
 * y [T][C] = silu(conv). Written from the definition: per channel, the
 * input sequence is the three kept inputs followed by the T new ones,
 * u = [state | x] (3 + T values); output t is the SiLU of the 4-tap window
 * of u that ends at the current token, sum_j w[j] u[t + j] (tap 3 on x_t),
 * and the new state is the last three entries of u. */
void gdn_oracle_conv(int64_t T, int32_t C, const double* x, const double* w, double* state,
                     double* y) {
    const int64_t n = GDN_ORACLE_CONV_STATE + T;
    double* u = (double*)malloc((size_t)n * sizeof(double));
    if (u == NULL) abort();
    for (int32_t c = 0; c < C; ++c) {
        for (int p = 0; p < GDN_ORACLE_CONV_STATE; ++p)
            u[p] = state[(int64_t)c * GDN_ORACLE_CONV_STATE + p];
        for (int64_t t = 0; t < T; ++t) u[GDN_ORACLE_CONV_STATE + t] = x[t * C + c];
        const double* wc = w + (int64_t)c * GDN_ORACLE_CONV_WIDTH;
        for (int64_t t = 0; t < T; ++t) {
            double acc = 0.0;
            for (int j = 0; j < GDN_ORACLE_CONV_WIDTH; ++j) acc += wc[j] * u[t + j];
            y[t * C + c] = gdn_oracle_silu(acc);
        }
        for (int p = 0; p < GDN_ORACLE_CONV_STATE; ++p)
            state[(int64_t)c * GDN_ORACLE_CONV_STATE + p] = u[n - GDN_ORACLE_CONV_STATE + p];
    }
    free(u);
}

/* ------------------------------------------------------------------- O2 */

/* rows of `width`: x *= (sum x^2 + eps)^(-1/2)  (the form the Metal test's CPU
 * oracle uses). */
void gdn_oracle_l2norm_rows(int64_t rows, int32_t width, double eps, double* x) {
    for (int64_t r = 0; r < rows; ++r) {
        double* row = x + r * width;
        double ss = 0.0;
        for (int32_t i = 0; i < width; ++i) ss += row[i] * row[i];
        double inv = 1.0 / sqrt(ss + eps);
        for (int32_t i = 0; i < width; ++i) row[i] *= inv;
    }
}

/* rows of `width`: x /= max(||x||, eps)  (ggml's form, as ferrox-core gdn.rs
 * `l2_normalize` states it). */
void gdn_oracle_l2norm_rows_clamped(int64_t rows, int32_t width, double eps, double* x) {
    for (int64_t r = 0; r < rows; ++r) {
        double* row = x + r * width;
        double ss = 0.0;
        for (int32_t i = 0; i < width; ++i) ss += row[i] * row[i];
        double n = sqrt(ss);
        double div = n > eps ? n : eps;
        for (int32_t i = 0; i < width; ++i) row[i] /= div;
    }
}

/* ------------------------------------------------------------------- O3 */

/* a, b [T][Hv] raw inputs -> g, beta [T][Hv].
 * decay 0 = log-rate (param = A_log, rate = -exp(A_log));
 * decay 1 = negative rate (param is the rate itself, already negative). */
void gdn_oracle_gates(int64_t T, int32_t Hv, int decay, const double* param,
                      const double* dt_bias, const double* a, const double* b, double* g,
                      double* beta) {
    for (int64_t t = 0; t < T; ++t) {
        for (int32_t h = 0; h < Hv; ++h) {
            double rate = decay == 0 ? -exp(param[h]) : param[h];
            g[t * Hv + h] = rate * gdn_oracle_softplus(a[t * Hv + h] + dt_bias[h]);
            beta[t * Hv + h] = gdn_oracle_sigmoid(b[t * Hv + h]);
        }
    }
}

/* ------------------------------------------------------------------- O4 */

/* T tokens of one sequence. q, k [T][Hk][D] (already normalised, NOT yet
 * scaled); v [T][Hv][D]; g, beta [T][Hv]; S [Hv][D][D] in/out; o [T][Hv][D]. */
void gdn_oracle_delta(int32_t Hk, int32_t Hv, int32_t D, int map, int64_t T, const double* q,
                      const double* k, const double* v, const double* g, const double* beta,
                      double* S, double* o) {
    const double scale = 1.0 / sqrt((double)D);
    for (int64_t t = 0; t < T; ++t) {
        for (int32_t h = 0; h < Hv; ++h) {
            const int32_t kh = gdn_oracle_k_head(map, h, Hk, Hv);
            const double* qt = q + (t * Hk + kh) * D;
            const double* kt = k + (t * Hk + kh) * D;
            const double* vt = v + (t * Hv + h) * D;
            const double alpha = exp(g[t * Hv + h]);
            const double bt = beta[t * Hv + h];
            for (int32_t j = 0; j < D; ++j) {
                double* row = S + ((int64_t)h * D + j) * D;
                /* decay the row, then the state's prediction of v_j */
                double pred = 0.0;
                for (int32_t i = 0; i < D; ++i) {
                    row[i] *= alpha;
                    pred += row[i] * kt[i];
                }
                const double d = bt * (vt[j] - pred);
                /* rank-one correction, then the read-out */
                double acc = 0.0;
                for (int32_t i = 0; i < D; ++i) {
                    row[i] += d * kt[i];
                    acc += row[i] * qt[i];
                }
                o[(t * Hv + h) * D + j] = scale * acc;
            }
        }
    }
}

/* ------------------------------------------------------------------- O5 */

/* rows of D: y = o * (mean o^2 + eps)^(-1/2) * w[j] * silu(z). */
void gdn_oracle_gated_rmsnorm(int64_t rows, int32_t D, double eps, const double* o,
                              const double* z, const double* w, double* y) {
    for (int64_t r = 0; r < rows; ++r) {
        const double* orow = o + r * D;
        double ss = 0.0;
        for (int32_t j = 0; j < D; ++j) ss += orow[j] * orow[j];
        const double inv = 1.0 / sqrt(ss / D + eps);
        for (int32_t j = 0; j < D; ++j)
            y[r * D + j] = orow[j] * inv * w[j] * gdn_oracle_silu(z[r * D + j]);
    }
}

/* ------------------------------------------------------------------- O6 */

/* One sequence: conv (O1) over mixed_qkv [T][C], split into q|k|v, l2norm q
 * and k per K head (O2, eps l2_eps; clamped form when l2_mode == 1), gates
 * (O3), recurrence (O4) and, when z != NULL, gated RMSNorm (O5) into y.
 * conv_state [C][3] and S [Hv][D][D] are updated in place. core [T][Hv][D]. */
void gdn_oracle_segment(int32_t Hk, int32_t Hv, int32_t D, int map, int decay, double l2_eps,
                        int l2_mode, double rms_eps, int64_t T, const double* mixed_qkv,
                        const double* a, const double* b, const double* z,
                        const double* conv_w, const double* decay_param,
                        const double* dt_bias, const double* norm_w, double* conv_state,
                        double* S, double* core, double* y) {
    const int32_t qkf = Hk * D, vf = Hv * D, C = 2 * qkf + vf;
    double* mixed = (double*)malloc(sizeof(double) * (size_t)(T * C + 1));
    double* q = (double*)malloc(sizeof(double) * (size_t)(T * qkf + 1));
    double* k = (double*)malloc(sizeof(double) * (size_t)(T * qkf + 1));
    double* v = (double*)malloc(sizeof(double) * (size_t)(T * vf + 1));
    double* g = (double*)malloc(sizeof(double) * (size_t)(T * Hv + 1));
    double* beta = (double*)malloc(sizeof(double) * (size_t)(T * Hv + 1));
    gdn_oracle_conv(T, C, mixed_qkv, conv_w, conv_state, mixed);
    for (int64_t t = 0; t < T; ++t) {
        memcpy(q + t * qkf, mixed + t * C, sizeof(double) * qkf);
        memcpy(k + t * qkf, mixed + t * C + qkf, sizeof(double) * qkf);
        memcpy(v + t * vf, mixed + t * C + 2 * qkf, sizeof(double) * vf);
    }
    if (l2_mode == 1) {
        gdn_oracle_l2norm_rows_clamped(T * Hk, D, l2_eps, q);
        gdn_oracle_l2norm_rows_clamped(T * Hk, D, l2_eps, k);
    } else {
        gdn_oracle_l2norm_rows(T * Hk, D, l2_eps, q);
        gdn_oracle_l2norm_rows(T * Hk, D, l2_eps, k);
    }
    gdn_oracle_gates(T, Hv, decay, decay_param, dt_bias, a, b, g, beta);
    gdn_oracle_delta(Hk, Hv, D, map, T, q, k, v, g, beta, S, core);
    if (z != NULL && y != NULL) gdn_oracle_gated_rmsnorm(T * Hv, D, rms_eps, core, z, norm_w, y);
    free(mixed);
    free(q);
    free(k);
    free(v);
    free(g);
    free(beta);
}

/* ------------------------------------------------------------------- O7 */

/* The recurrence of O4 summed chunk-wise with chunk length Cn (the last chunk
 * of a sequence may be shorter). Same arguments as gdn_oracle_delta.
 *
 * Within a chunk of L tokens starting from state S0, with c_t = sum_{s<=t} g_s
 * (inclusive, chunk-local):
 *   A[t][s] = beta_t e^{c_t - c_s} (k_t . k_s)      for s < t, else 0
 *   Tm      = (I + A)^{-1}                           (unit lower triangular)
 *   U       = Tm diag(beta) V,   W = Tm diag(beta e^{c}) K
 *   Dl      = U - W S0^T                             (rows d_t)
 *   o_t     = scale [ e^{c_t} S0 q_t + sum_{s<=t} e^{c_t-c_s} (q_t . k_s) d_s ]
 *   S_L     = e^{c_L} S0 + sum_s e^{c_L - c_s} d_s k_s^T
 */
void gdn_oracle_delta_chunked(int32_t Hk, int32_t Hv, int32_t D, int map, int64_t T,
                              int32_t Cn, const double* q, const double* k, const double* v,
                              const double* g, const double* beta, double* S, double* o) {
    const double scale = 1.0 / sqrt((double)D);
    double* cg = (double*)malloc(sizeof(double) * Cn);
    double* A = (double*)malloc(sizeof(double) * Cn * Cn);
    double* Tm = (double*)malloc(sizeof(double) * Cn * Cn);
    double* U = (double*)malloc(sizeof(double) * Cn * D);
    double* W = (double*)malloc(sizeof(double) * Cn * D);
    double* Dl = (double*)malloc(sizeof(double) * Cn * D);
    double* S0 = (double*)malloc(sizeof(double) * D * D);
    for (int32_t h = 0; h < Hv; ++h) {
        const int32_t kh = gdn_oracle_k_head(map, h, Hk, Hv);
        double* Sh = S + (int64_t)h * D * D;
        for (int64_t t0 = 0; t0 < T; t0 += Cn) {
            const int32_t L = (int32_t)((T - t0) < Cn ? (T - t0) : Cn);
#define KV(t) (k + ((t0 + (t)) * Hk + kh) * D)
#define QV(t) (q + ((t0 + (t)) * Hk + kh) * D)
#define VV(t) (v + ((t0 + (t)) * Hv + h) * D)
#define GI(t) ((t0 + (t)) * Hv + h)
            double run = 0.0;
            for (int32_t t = 0; t < L; ++t) {
                run += g[GI(t)];
                cg[t] = run;
            }
            memcpy(S0, Sh, sizeof(double) * D * D);
            /* A */
            for (int32_t t = 0; t < L; ++t)
                for (int32_t s = 0; s < L; ++s) {
                    double val = 0.0;
                    if (s < t) {
                        double kk = 0.0;
                        for (int32_t i = 0; i < D; ++i) kk += KV(t)[i] * KV(s)[i];
                        val = beta[GI(t)] * exp(cg[t] - cg[s]) * kk;
                    }
                    A[t * Cn + s] = val;
                }
            /* Tm = (I + A)^{-1} by forward substitution, column by column */
            for (int32_t s = 0; s < L; ++s) {
                for (int32_t t = 0; t < L; ++t) {
                    if (t < s) {
                        Tm[t * Cn + s] = 0.0;
                        continue;
                    }
                    double val = (t == s) ? 1.0 : 0.0;
                    for (int32_t r = s; r < t; ++r) val -= A[t * Cn + r] * Tm[r * Cn + s];
                    Tm[t * Cn + s] = val;
                }
            }
            /* U, W */
            for (int32_t t = 0; t < L; ++t)
                for (int32_t c = 0; c < D; ++c) {
                    double u = 0.0, w = 0.0;
                    for (int32_t s = 0; s <= t; ++s) {
                        u += Tm[t * Cn + s] * beta[GI(s)] * VV(s)[c];
                        w += Tm[t * Cn + s] * beta[GI(s)] * exp(cg[s]) * KV(s)[c];
                    }
                    U[t * D + c] = u;
                    W[t * D + c] = w;
                }
            /* Dl = U - W S0^T:  (W S0^T)[t][j] = sum_i W[t][i] S0[j][i] */
            for (int32_t t = 0; t < L; ++t)
                for (int32_t j = 0; j < D; ++j) {
                    double ws = 0.0;
                    for (int32_t i = 0; i < D; ++i) ws += W[t * D + i] * S0[j * D + i];
                    Dl[t * D + j] = U[t * D + j] - ws;
                }
            /* outputs */
            for (int32_t t = 0; t < L; ++t)
                for (int32_t j = 0; j < D; ++j) {
                    double sq = 0.0;
                    for (int32_t i = 0; i < D; ++i) sq += S0[j * D + i] * QV(t)[i];
                    double acc = exp(cg[t]) * sq;
                    for (int32_t s = 0; s <= t; ++s) {
                        double qk = 0.0;
                        for (int32_t i = 0; i < D; ++i) qk += QV(t)[i] * KV(s)[i];
                        acc += exp(cg[t] - cg[s]) * qk * Dl[s * D + j];
                    }
                    o[((t0 + t) * Hv + h) * D + j] = scale * acc;
                }
            /* state at the end of the chunk */
            for (int32_t j = 0; j < D; ++j)
                for (int32_t i = 0; i < D; ++i) {
                    double acc = exp(cg[L - 1]) * S0[j * D + i];
                    for (int32_t s = 0; s < L; ++s)
                        acc += exp(cg[L - 1] - cg[s]) * Dl[s * D + j] * KV(s)[i];
                    Sh[j * D + i] = acc;
                }
#undef KV
#undef QV
#undef VV
#undef GI
        }
    }
    free(cg);
    free(A);
    free(Tm);
    free(U);
    free(W);
    free(Dl);
    free(S0);
}

/* ------------------------------------------------------------------- O9 */

/* One chunk of the O7 summation written as an affine map of its start state
 * (our derivation from the chunk form above; the pages name the carry stage of
 * the chunked kernel, gated_delta_attention_tests.rs `run_chunked_core`, and
 * print no formula for it). With U, W, c as in O7, E = diag(e^{c_L - c_s}) and
 * P[t][s] = e^{c_t - c_s} (q_t . k_s) for s <= t:
 *   S_L = S0 M + N,   M = e^{c_L} I - W^T E K   (D x D, key by key)
 *                     N = U^T E K                 (D x D, value by key)
 *   o   = X S0^T + Y, X = scale (diag(e^{c}) Q - P W)   (L x D)
 *                     Y = scale P U                     (L x D)
 * None of M, N, X, Y depends on S0. This function computes them for the L
 * tokens starting at token t0 of V head h (q, k, v, g, beta laid out as for
 * gdn_oracle_delta); M, N are D*D, X, Y are L*D, row-major. */
void gdn_oracle_chunk_factors(int32_t Hk, int32_t Hv, int32_t D, int map, int64_t t0,
                              int32_t L, int32_t h, const double* q, const double* k,
                              const double* v, const double* g, const double* beta, double* M,
                              double* N, double* X, double* Y) {
    const double scale = 1.0 / sqrt((double)D);
    const int32_t kh = gdn_oracle_k_head(map, h, Hk, Hv);
    double* cg = (double*)malloc(sizeof(double) * L);
    double* A = (double*)malloc(sizeof(double) * L * L);
    double* Tm = (double*)malloc(sizeof(double) * L * L);
    double* P = (double*)malloc(sizeof(double) * L * L);
    double* U = (double*)malloc(sizeof(double) * L * D);
    double* W = (double*)malloc(sizeof(double) * L * D);
#define KV(t) (k + ((t0 + (t)) * Hk + kh) * D)
#define QV(t) (q + ((t0 + (t)) * Hk + kh) * D)
#define VV(t) (v + ((t0 + (t)) * Hv + h) * D)
#define GI(t) ((t0 + (t)) * Hv + h)
    double run = 0.0;
    for (int32_t t = 0; t < L; ++t) {
        run += g[GI(t)];
        cg[t] = run;
    }
    for (int32_t t = 0; t < L; ++t)
        for (int32_t s = 0; s < L; ++s) {
            double kk = 0.0, qk = 0.0;
            for (int32_t i = 0; i < D; ++i) {
                kk += KV(t)[i] * KV(s)[i];
                qk += QV(t)[i] * KV(s)[i];
            }
            A[t * L + s] = s < t ? beta[GI(t)] * exp(cg[t] - cg[s]) * kk : 0.0;
            P[t * L + s] = s <= t ? exp(cg[t] - cg[s]) * qk : 0.0;
        }
    for (int32_t s = 0; s < L; ++s)
        for (int32_t t = 0; t < L; ++t) {
            if (t < s) {
                Tm[t * L + s] = 0.0;
                continue;
            }
            double val = (t == s) ? 1.0 : 0.0;
            for (int32_t r = s; r < t; ++r) val -= A[t * L + r] * Tm[r * L + s];
            Tm[t * L + s] = val;
        }
    for (int32_t t = 0; t < L; ++t)
        for (int32_t c = 0; c < D; ++c) {
            double u = 0.0, w = 0.0;
            for (int32_t s = 0; s <= t; ++s) {
                u += Tm[t * L + s] * beta[GI(s)] * VV(s)[c];
                w += Tm[t * L + s] * beta[GI(s)] * exp(cg[s]) * KV(s)[c];
            }
            U[t * D + c] = u;
            W[t * D + c] = w;
        }
    /* M[a][i] = e^{c_L} [a == i] - sum_s W[s][a] e^{c_L - c_s} k_s[i];
     * N[j][i] = sum_s U[s][j] e^{c_L - c_s} k_s[i] */
    for (int32_t a = 0; a < D; ++a)
        for (int32_t i = 0; i < D; ++i) {
            double m = (a == i) ? exp(cg[L - 1]) : 0.0, n = 0.0;
            for (int32_t s = 0; s < L; ++s) {
                const double e = exp(cg[L - 1] - cg[s]) * KV(s)[i];
                m -= W[s * D + a] * e;
                n += U[s * D + a] * e;
            }
            M[a * D + i] = m;
            N[a * D + i] = n;
        }
    /* X[t][i] = scale (e^{c_t} q_t[i] - sum_s P[t][s] W[s][i]);
     * Y[t][j] = scale sum_s P[t][s] U[s][j] */
    for (int32_t t = 0; t < L; ++t)
        for (int32_t i = 0; i < D; ++i) {
            double x = exp(cg[t]) * QV(t)[i], y = 0.0;
            for (int32_t s = 0; s <= t; ++s) {
                x -= P[t * L + s] * W[s * D + i];
                y += P[t * L + s] * U[s * D + i];
            }
            X[t * D + i] = scale * x;
            Y[t * D + i] = scale * y;
        }
#undef KV
#undef QV
#undef VV
#undef GI
    free(cg);
    free(A);
    free(Tm);
    free(P);
    free(U);
    free(W);
}

/* The recurrence of O4 carried chunk by chunk through the affine maps of
 * gdn_oracle_chunk_factors: per chunk o = X S^T + Y, then S <- S M + N. Same
 * arguments as gdn_oracle_delta_chunked. */
void gdn_oracle_delta_affine(int32_t Hk, int32_t Hv, int32_t D, int map, int64_t T, int32_t Cn,
                             const double* q, const double* k, const double* v, const double* g,
                             const double* beta, double* S, double* o) {
    double* M = (double*)malloc(sizeof(double) * D * D);
    double* N = (double*)malloc(sizeof(double) * D * D);
    double* X = (double*)malloc(sizeof(double) * Cn * D);
    double* Y = (double*)malloc(sizeof(double) * Cn * D);
    double* S0 = (double*)malloc(sizeof(double) * D * D);
    for (int32_t h = 0; h < Hv; ++h) {
        double* Sh = S + (int64_t)h * D * D;
        for (int64_t t0 = 0; t0 < T; t0 += Cn) {
            const int32_t L = (int32_t)((T - t0) < Cn ? (T - t0) : Cn);
            gdn_oracle_chunk_factors(Hk, Hv, D, map, t0, L, h, q, k, v, g, beta, M, N, X, Y);
            memcpy(S0, Sh, sizeof(double) * D * D);
            for (int32_t t = 0; t < L; ++t)
                for (int32_t j = 0; j < D; ++j) {
                    double acc = Y[t * D + j];
                    for (int32_t i = 0; i < D; ++i) acc += X[t * D + i] * S0[j * D + i];
                    o[((t0 + t) * Hv + h) * D + j] = acc;
                }
            for (int32_t j = 0; j < D; ++j)
                for (int32_t i = 0; i < D; ++i) {
                    double acc = N[j * D + i];
                    for (int32_t a = 0; a < D; ++a) acc += S0[j * D + a] * M[a * D + i];
                    Sh[j * D + i] = acc;
                }
        }
    }
    free(M);
    free(N);
    free(X);
    free(Y);
    free(S0);
}

/* ------------------------------------------------------------------- O8 */

#define GDN_ORACLE_BF_MAXD 8

/* Brute force for D <= 8, long double: per token and V head
 *   M = I - beta k k^T;  S = alpha S M + beta v k^T;  o = scale S q.
 * Same arguments as gdn_oracle_delta. Returns -1 if D is too large. */
int gdn_oracle_delta_bruteforce(int32_t Hk, int32_t Hv, int32_t D, int map, int64_t T,
                                const double* q, const double* k, const double* v,
                                const double* g, const double* beta, double* S, double* o) {
    if (D > GDN_ORACLE_BF_MAXD) return -1;
    const long double scale = 1.0L / sqrtl((long double)D);
    long double St[GDN_ORACLE_BF_MAXD][GDN_ORACLE_BF_MAXD];
    long double M[GDN_ORACLE_BF_MAXD][GDN_ORACLE_BF_MAXD];
    long double P[GDN_ORACLE_BF_MAXD][GDN_ORACLE_BF_MAXD];
    for (int32_t h = 0; h < Hv; ++h) {
        const int32_t kh = gdn_oracle_k_head(map, h, Hk, Hv);
        for (int32_t j = 0; j < D; ++j)
            for (int32_t i = 0; i < D; ++i) St[j][i] = S[((int64_t)h * D + j) * D + i];
        for (int64_t t = 0; t < T; ++t) {
            const double* kt = k + (t * Hk + kh) * D;
            const double* qt = q + (t * Hk + kh) * D;
            const double* vt = v + (t * Hv + h) * D;
            const long double alpha = expl((long double)g[t * Hv + h]);
            const long double bt = beta[t * Hv + h];
            for (int32_t r = 0; r < D; ++r)
                for (int32_t c = 0; c < D; ++c)
                    M[r][c] = (r == c ? 1.0L : 0.0L) - bt * (long double)kt[r] * kt[c];
            /* P = alpha * St * M */
            for (int32_t r = 0; r < D; ++r)
                for (int32_t c = 0; c < D; ++c) {
                    long double acc = 0.0L;
                    for (int32_t m = 0; m < D; ++m) acc += St[r][m] * M[m][c];
                    P[r][c] = alpha * acc;
                }
            /* St = P + beta v k^T */
            for (int32_t r = 0; r < D; ++r)
                for (int32_t c = 0; c < D; ++c) St[r][c] = P[r][c] + bt * (long double)vt[r] * kt[c];
            for (int32_t r = 0; r < D; ++r) {
                long double acc = 0.0L;
                for (int32_t c = 0; c < D; ++c) acc += St[r][c] * qt[c];
                o[(t * Hv + h) * D + r] = (double)(scale * acc);
            }
        }
        for (int32_t j = 0; j < D; ++j)
            for (int32_t i = 0; i < D; ++i) S[((int64_t)h * D + j) * D + i] = (double)St[j][i];
    }
    return 0;
}
