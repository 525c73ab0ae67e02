/*
 * retention_oracle.c -- TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT PATH.
 *
 * A plain, slow, fp64 CPU statement of RetNet retention, written so that each
 * loop can be checked by eye against the formulas it restates.  Only the test
 * suite, the smoke check and the benchmark's CPU-baseline leg may load this
 * code; the CUDA library never links, includes or calls it, and it shares no
 * code, header or table with the CUDA library.
 *
 * Sources (web pages on RetNet; cited by page title and section):
 *   [G] "RetNet Guide: Retentive Networks & The Impossible Triangle"
 *       - section "3. Multi-Scale Retention (MSR)": per-head decay
 *         gamma = 1 - 2^(-5-h).
 *       - section "1. The Parallel Representation for High-Throughput
 *         Pretraining": causal decay matrix D_nm = gamma^(n-m) for n >= m and
 *         0 otherwise; output R = ((Q K^T) (.) D) V.
 *       - section "2. The Recurrent Representation for Constant-Memory O(1)
 *         Decoding": S_n = gamma S_{n-1} + K_n^T V_n, R_n = Q_n S_n.
 *       - section "3. The Chunkwise Recurrent Representation for Ultra-Long
 *         Sequence Prefill": per chunk i, the state is carried as
 *         S_[i] = gamma^B S_[i-1] + K_[i]^T V_[i] and the output is
 *         R_[i] = ((Q_[i] K_[i]^T) (.) D) V_[i] + (Q_[i] S_[i-1]) (.) zeta with
 *         zeta_j = gamma^(j+1).
 *       - section "1. PyTorch Implementation of MultiScaleRetention": the decay
 *         list runs over range(num_heads) (0-based heads); the parallel scores
 *         are divided by sqrt(d); the recurrent query is divided by sqrt(d)
 *         before it reads the post-update state.
 *
 * Readings taken where the pages are silent or garbled:
 *   R1  the head index h in gamma_h is 0-based (the executable statement on
 *       [G] iterates range(num_heads)).
 *   R2  the factor d_k^(-1/2) multiplies q only; the state holds unscaled
 *       k^T v sums, so a state handed from one form to another composes.
 *   R3  the printed chunk state update omits the decay inside the chunk; the
 *       update used here weights token j of a chunk of length L by
 *       gamma^(L-1-j), which is what equality with the recurrent form forces.
 *   R4  zeta_j = gamma^(j+1) with j the 0-based row inside the chunk.
 *   R5  the recurrent output reads the state after the update.
 *   R6  a last chunk shorter than C (N not a multiple of C) uses its own length
 *       L in gamma^L and in the in-chunk weights.
 *   R7  the phase rotation turns pairs (2j, 2j+1) of the real dimensions as
 *       one complex coordinate with frequency theta_j, and query and key alike
 *       by the angle (n0 + n) theta_j (see oracle_rotate).
 *
 * Layout: q, k are [B][H][N][dk], v and out are [B][H][N][dv], state is
 * [B][H][dk][dv], gamma is [H]; all row-major, all double.  The loops over
 * (b, h) are split across OpenMP threads; nothing inside a head is reordered.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* [G] "3. Multi-Scale Retention (MSR)", with reading R1 (0-based h). */
double oracle_gamma(int h)
{
    return 1.0 - pow(2.0, -5.0 - (double)h);
}

int oracle_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

static double dot(const double *a, const double *b, int n)
{
    double s = 0.0;
    for (int i = 0; i < n; ++i) s += a[i] * b[i];
    return s;
}

/*
 * Parallel form, [G] "1. The Parallel Representation ...":
 *   out[n] = sum_{m} D[n][m] * (q_n . k_m / sqrt(dk)) * v_m,
 *   D[n][m] = gamma^(n-m) if n >= m, else 0.
 * One row of (QK^T/sqrt(dk)) (.) D is formed at a time and multiplied by V.
 */
void oracle_parallel(const double *q, const double *k, const double *v,
                     const double *gamma, double *out,
                     int B, int H, int N, int dk, int dv)
{
    const double scale = 1.0 / sqrt((double)dk);
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < H; ++h) {
            const size_t head = (size_t)b * H + h;
            const double *Q = q + head * (size_t)N * dk;
            const double *K = k + head * (size_t)N * dk;
            const double *V = v + head * (size_t)N * dv;
            double *O = out + head * (size_t)N * dv;
            const double g = gamma[h];
            double *row = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
            for (int n = 0; n < N; ++n) {
                for (int m = 0; m < N; ++m) {
                    /* D[n][m] is zero above the diagonal, so the product is too */
                    row[m] = (n >= m) ? pow(g, (double)(n - m)) *
                                            dot(Q + (size_t)n * dk, K + (size_t)m * dk, dk) * scale
                                      : 0.0;
                }
                for (int j = 0; j < dv; ++j) {
                    double s = 0.0;
                    for (int m = 0; m < N; ++m) s += row[m] * V[(size_t)m * dv + j];
                    O[(size_t)n * dv + j] = s;
                }
            }
            free(row);
        }
    }
}

/*
 * The same parallel-form definition evaluated for selected rows of ONE head
 * (used to check single outputs of workloads too large for the full oracle).
 *   q_head, k_head: [N][dk]; v_head: [N][dv]; rows: the n of each wanted row;
 *   out: [count][dv].
 */
void oracle_parallel_rows(const double *q_head, const double *k_head,
                          const double *v_head, double g, int N, int dk, int dv,
                          const int *rows, int count, double *out)
{
    const double scale = 1.0 / sqrt((double)dk);
#pragma omp parallel for schedule(dynamic, 1)
    for (int r = 0; r < count; ++r) {
        const int n = rows[r];
        double *o = out + (size_t)r * dv;
        for (int j = 0; j < dv; ++j) o[j] = 0.0;
        if (n < 0 || n >= N) continue;
        for (int m = 0; m <= n; ++m) {
            double w = pow(g, (double)(n - m)) *
                       dot(q_head + (size_t)n * dk, k_head + (size_t)m * dk, dk) * scale;
            for (int j = 0; j < dv; ++j) o[j] += w * v_head[(size_t)m * dv + j];
        }
    }
}

/*
 * Recurrent form, [G] "2. The Recurrent Representation ...", readings R2, R5:
 *   S_n = gamma S_{n-1} + k_n^T v_n;   out_n = (q_n / sqrt(dk)) S_n.
 * state: [B][H][dk][dv]; if non-NULL it holds the starting state on entry and
 * the state after the last token on return; if NULL the start is zero.
 */
void oracle_recurrent(const double *q, const double *k, const double *v,
                      const double *gamma, double *state, double *out,
                      int B, int H, int N, int dk, int dv)
{
    const double scale = 1.0 / sqrt((double)dk);
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < H; ++h) {
            const size_t head = (size_t)b * H + h;
            const double *Q = q + head * (size_t)N * dk;
            const double *K = k + head * (size_t)N * dk;
            const double *V = v + head * (size_t)N * dv;
            double *O = out + head * (size_t)N * dv;
            const double g = gamma[h];
            double *S = (double *)calloc((size_t)dk * dv, sizeof(double));
            if (state) memcpy(S, state + head * (size_t)dk * dv, sizeof(double) * (size_t)dk * dv);
            for (int n = 0; n < N; ++n) {
                const double *kn = K + (size_t)n * dk;
                const double *vn = V + (size_t)n * dv;
                const double *qn = Q + (size_t)n * dk;
                for (int i = 0; i < dk; ++i)
                    for (int j = 0; j < dv; ++j)
                        S[(size_t)i * dv + j] = g * S[(size_t)i * dv + j] + kn[i] * vn[j];
                for (int j = 0; j < dv; ++j) {
                    double s = 0.0;
                    for (int i = 0; i < dk; ++i) s += qn[i] * scale * S[(size_t)i * dv + j];
                    O[(size_t)n * dv + j] = s;
                }
            }
            if (state) memcpy(state + head * (size_t)dk * dv, S, sizeof(double) * (size_t)dk * dv);
            free(S);
        }
    }
}

/*
 * Chunkwise recurrent form, [G] "3. The Chunkwise Recurrent Representation
 * ...", readings R2, R3, R4, R6.  For each chunk of L (= C, or fewer for the
 * last one) tokens starting at position s:
 *   inner:  out[s+j] = sum_{l<=j} gamma^(j-l) (q_{s+j} . k_{s+l} / sqrt(dk)) v_{s+l}
 *   cross:  out[s+j] += gamma^(j+1) (q_{s+j} / sqrt(dk)) S_prev
 *   carry:  S = gamma^L S_prev + sum_{l<L} gamma^(L-1-l) k_{s+l}^T v_{s+l}
 * state_in (nullable: zero start) and state_out (nullable) are [B][H][dk][dv].
 */
void oracle_chunkwise(const double *q, const double *k, const double *v,
                      const double *gamma, const double *state_in,
                      double *out, double *state_out,
                      int B, int H, int N, int dk, int dv, int C)
{
    const double scale = 1.0 / sqrt((double)dk);
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < H; ++h) {
            const size_t head = (size_t)b * H + h;
            const double *Q = q + head * (size_t)N * dk;
            const double *K = k + head * (size_t)N * dk;
            const double *V = v + head * (size_t)N * dv;
            double *O = out + head * (size_t)N * dv;
            const double g = gamma[h];
            double *S = (double *)calloc((size_t)dk * dv, sizeof(double));
            double *T = (double *)calloc((size_t)dk * dv, sizeof(double));
            if (state_in) memcpy(S, state_in + head * (size_t)dk * dv, sizeof(double) * (size_t)dk * dv);
            for (int s = 0; s < N; s += C) {
                const int L = (N - s < C) ? (N - s) : C;
                for (int j = 0; j < L; ++j) {
                    const double *qj = Q + (size_t)(s + j) * dk;
                    double *oj = O + (size_t)(s + j) * dv;
                    /* inner: ((Q K^T / sqrt(dk)) (.) D) V over the chunk */
                    for (int c = 0; c < dv; ++c) oj[c] = 0.0;
                    for (int l = 0; l <= j; ++l) {
                        double w = pow(g, (double)(j - l)) *
                                   dot(qj, K + (size_t)(s + l) * dk, dk) * scale;
                        for (int c = 0; c < dv; ++c) oj[c] += w * V[(size_t)(s + l) * dv + c];
                    }
                    /* cross: zeta_j (q_j / sqrt(dk)) S_prev, zeta_j = gamma^(j+1) */
                    const double zeta = pow(g, (double)(j + 1));
                    for (int c = 0; c < dv; ++c) {
                        double t = 0.0;
                        for (int i = 0; i < dk; ++i) t += qj[i] * S[(size_t)i * dv + c];
                        oj[c] += zeta * scale * t;
                    }
                }
                /* carry: S = gamma^L S + sum_l gamma^(L-1-l) k_l^T v_l
                 * (T accumulates the sum over l in order l = 0, 1, ..., L-1) */
                for (size_t e = 0; e < (size_t)dk * dv; ++e) T[e] = 0.0;
                for (int l = 0; l < L; ++l) {
                    const double w = pow(g, (double)(L - 1 - l));
                    const double *kl = K + (size_t)(s + l) * dk;
                    const double *vl = V + (size_t)(s + l) * dv;
                    for (int i = 0; i < dk; ++i)
                        for (int c = 0; c < dv; ++c) T[(size_t)i * dv + c] += w * kl[i] * vl[c];
                }
                const double gL = pow(g, (double)L);
                for (size_t e = 0; e < (size_t)dk * dv; ++e) S[e] = gL * S[e] + T[e];
            }
            if (state_out) memcpy(state_out + head * (size_t)dk * dv, S, sizeof(double) * (size_t)dk * dv);
            free(T);
            free(S);
        }
    }
}

/*
 * [G] "1. The Parallel Representation for High-Throughput Pretraining":
 * MSR(X) = GroupNorm(Concat(R_1, ..., R_H)) W_O, and [G] "1. PyTorch
 * Implementation of MultiScaleRetention": the normalisation has one group per
 * head over the concatenated channels (num_groups = H, num_channels = H dv,
 * eps = 1e-6 there; eps is an argument here), i.e. for every token n and head
 * h, over the dv channels c of R_h:
 *
 *   mu = (1/dv) sum_c R[h][n][c]      var = (1/dv) sum_c (R[h][n][c] - mu)^2
 *   Y[n][h][c] = (R[h][n][c] - mu) / sqrt(var + eps) * weight[h dv + c] + bias[h dv + c]
 *
 * r is [B][H][N][dv]; y is written with the heads concatenated per token,
 * [B][N][H][dv].  weight and bias may be NULL (one and zero).
 */
void oracle_groupnorm(const double *r, const double *weight, const double *bias,
                      double *y, int B, int H, int N, int dv, double eps)
{
  for (int b = 0; b < B; ++b)
    for (int h = 0; h < H; ++h)
      for (int n = 0; n < N; ++n) {
        const double *x = r + (((size_t)b * H + h) * N + n) * dv;
        double *out = y + (((size_t)b * N + n) * H + h) * dv;
        double mu = 0.0;
        for (int c = 0; c < dv; ++c) mu += x[c];
        mu /= dv;
        double var = 0.0;
        for (int c = 0; c < dv; ++c) var += (x[c] - mu) * (x[c] - mu);
        var /= dv;
        const double inv = 1.0 / sqrt(var + eps);
        for (int c = 0; c < dv; ++c) {
          const double w = weight ? weight[h * dv + c] : 1.0;
          const double bb = bias ? bias[h * dv + c] : 0.0;
          out[c] = (x[c] - mu) * inv * w + bb;
        }
      }
}

/*
 * [G] "2. Relative Position via Complex Exponential Phase Rotations": the
 * query and key at position n are multiplied by the phase e^(i n theta), so
 * that their product depends on n - m only.  Reading R7 (above): pairs
 * (2j, 2j+1) of the d real dimensions are the real and imaginary parts of one
 * complex coordinate with frequency theta_j, and with the real dot product the
 * kernels use, query and key are both rotated by the angle (n0 + n) theta_j,
 * which makes q_n . k_m depend on n - m only.  x, y: [B][H][N][d] (d even),
 * theta: [d/2]; n0 is the position of token 0.
 */
void oracle_rotate(const double *x, const double *theta, double *y, int B, int H, int N, int d,
                   long n0)
{
  for (int b = 0; b < B; ++b)
    for (int h = 0; h < H; ++h)
      for (int n = 0; n < N; ++n) {
        const double *xr = x + (((size_t)b * H + h) * N + n) * d;
        double *yr = y + (((size_t)b * H + h) * N + n) * d;
        for (int j = 0; j < d / 2; ++j) {
          const double a = (double)(n0 + n) * theta[j];
          const double c = cos(a), s = sin(a);
          yr[2 * j] = xr[2 * j] * c - xr[2 * j + 1] * s;
          yr[2 * j + 1] = xr[2 * j] * s + xr[2 * j + 1] * c;
        }
      }
}

/*
 * Backward pass.  The pages say the chunkwise form exists so that long
 * sequences can be trained ([G] "3. The Chunkwise Recurrent Representation
 * ..."), but print no gradient; the oracle therefore differentiates the
 * definition, written with a starting state S0 (readings R2, R5):
 *
 *   out_n = s sum_{m<=n} g^(n-m) (q_n . k_m) v_m  +  s g^(n+1) q_n S0
 *   S_N   = g^N S0 + sum_m g^(N-1-m) k_m^T v_m          (s = 1/sqrt(dk))
 *
 * For the loss sum_n dout_n . out_n + <dS, S_N> (dout: [N][dv], dS: [dk][dv])
 * the partial derivatives are
 *
 *   dq_n  = s sum_{m<=n} g^(n-m) (dout_n . v_m) k_m   +  s g^(n+1) S0 dout_n
 *   dk_m  = s sum_{n>=m} g^(n-m) (dout_n . v_m) q_n   +  g^(N-1-m) dS v_m
 *   dv_m  = s sum_{n>=m} g^(n-m) (q_n . k_m) dout_n   +  g^(N-1-m) k_m dS
 *   dS0   = s sum_n g^(n+1) q_n^T dout_n              +  g^N dS
 *
 * (S0 dout_n and dS v_m are [dk][dv] x [dv] products; k_m dS is [dk] x
 * [dk][dv].)  state_in (S0), dstate (dS) and dstate_in (dS0) are
 * [B][H][dk][dv] and may be NULL: a NULL S0 or dS is zero, a NULL dstate_in is
 * not written.  dq, dk: [B][H][N][dk]; dv_out: [B][H][N][dv].
 */
void oracle_backward(const double *q, const double *k, const double *v,
                     const double *gamma, const double *state_in,
                     const double *dout, const double *dstate,
                     double *dq, double *dk_out, double *dv_out, double *dstate_in,
                     int B, int H, int N, int dk, int dv)
{
    const double scale = 1.0 / sqrt((double)dk);
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < H; ++h) {
            const size_t head = (size_t)b * H + h;
            const double *Q = q + head * (size_t)N * dk;
            const double *K = k + head * (size_t)N * dk;
            const double *V = v + head * (size_t)N * dv;
            const double *dO = dout + head * (size_t)N * dv;
            const double *S0 = state_in ? state_in + head * (size_t)dk * dv : NULL;
            const double *dS = dstate ? dstate + head * (size_t)dk * dv : NULL;
            double *dQ = dq + head * (size_t)N * dk;
            double *dK = dk_out + head * (size_t)N * dk;
            double *dV = dv_out + head * (size_t)N * dv;
            const double g = gamma[h];

            /* dq_n: causal sum over m <= n, then the starting-state term */
            for (int n = 0; n < N; ++n) {
                double *r = dQ + (size_t)n * dk;
                for (int i = 0; i < dk; ++i) r[i] = 0.0;
                for (int m = 0; m <= n; ++m) {
                    const double w = scale * pow(g, (double)(n - m)) *
                                     dot(dO + (size_t)n * dv, V + (size_t)m * dv, dv);
                    for (int i = 0; i < dk; ++i) r[i] += w * K[(size_t)m * dk + i];
                }
                if (S0) {
                    const double z = scale * pow(g, (double)(n + 1));
                    for (int i = 0; i < dk; ++i)
                        r[i] += z * dot(S0 + (size_t)i * dv, dO + (size_t)n * dv, dv);
                }
            }
            /* dk_m and dv_m: anti-causal sums over n >= m, then the final-state term */
            for (int m = 0; m < N; ++m) {
                double *rk = dK + (size_t)m * dk;
                double *rv = dV + (size_t)m * dv;
                for (int i = 0; i < dk; ++i) rk[i] = 0.0;
                for (int c = 0; c < dv; ++c) rv[c] = 0.0;
                for (int n = m; n < N; ++n) {
                    const double d = scale * pow(g, (double)(n - m));
                    const double wk = d * dot(dO + (size_t)n * dv, V + (size_t)m * dv, dv);
                    const double wv = d * dot(Q + (size_t)n * dk, K + (size_t)m * dk, dk);
                    for (int i = 0; i < dk; ++i) rk[i] += wk * Q[(size_t)n * dk + i];
                    for (int c = 0; c < dv; ++c) rv[c] += wv * dO[(size_t)n * dv + c];
                }
                if (dS) {
                    const double xi = pow(g, (double)(N - 1 - m));
                    for (int i = 0; i < dk; ++i)
                        rk[i] += xi * dot(dS + (size_t)i * dv, V + (size_t)m * dv, dv);
                    for (int c = 0; c < dv; ++c) {
                        double t = 0.0;
                        for (int i = 0; i < dk; ++i) t += K[(size_t)m * dk + i] * dS[(size_t)i * dv + c];
                        rv[c] += xi * t;
                    }
                }
            }
            /* dS0 = s sum_n g^(n+1) q_n^T dout_n + g^N dS */
            if (dstate_in) {
                double *r = dstate_in + head * (size_t)dk * dv;
                for (int i = 0; i < dk; ++i)
                    for (int c = 0; c < dv; ++c) {
                        double t = dS ? pow(g, (double)N) * dS[(size_t)i * dv + c] : 0.0;
                        for (int n = 0; n < N; ++n)
                            t += scale * pow(g, (double)(n + 1)) * Q[(size_t)n * dk + i] *
                                 dO[(size_t)n * dv + c];
                        r[(size_t)i * dv + c] = t;
                    }
            }
        }
    }
}
