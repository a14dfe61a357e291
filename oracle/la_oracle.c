/*
 * la_oracle.c -- plain fp64 CPU oracle for causal linear attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library links, includes or calls
 * this file; only the tests, the package's smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header or constant with the CUDA
 * path.
 *
 * Three independent statements of the same quantity, each written from the
 * pages' definitions in fp64 with no blocking, fusion or reordering beyond what
 * the definition states:
 *
 *   oracle_recurrent  the token-by-token recurrence (the definition)
 *       "Linear / Sparse Attention - minimal runnable implementation",
 *           linear_attn_recurrent: S += k_t v_t^T, then o_t = q_t^T S
 *           (self-inclusive: update before read);
 *       "CS336 lecture 4, code 1: linear attention",
 *           gated_linear_attention_recurrent: S_t = gamma_t S_{t-1} + k_t v_t^T,
 *           y_t = q_t^T S_t;
 *       "adv13 - Linear Attention / SSM" section 3.2 / 4.2: the feature map
 *           phi is applied to q and k (never to v) before the recurrence.
 *
 *   oracle_parallel   the O(L^2) masked form
 *       "CS336 lecture 4, code 1", causal_linear_attention_parallel:
 *           Y = ((Q K^T) .* M) V with M lower triangular (diagonal included);
 *       same page, gated_linear_attention_parallel:
 *           D[t,s] = prod_{r=s+1..t} gamma_r = exp(cum[t] - cum[s]) for s <= t,
 *           cum = cumsum(log gamma), taken in log space to avoid underflow.
 *       The initial-state term exp(cum[t]) q_t^T S0 and the closed form of the
 *       final state follow from unrolling the recurrence above; the pages fix
 *       S0 = 0, where both terms vanish.
 *
 *   oracle_chunkwise  the chunkwise form, for the chunk-invariance pins
 *       "Linear / Sparse Attention - minimal runnable implementation",
 *           linear_attn_chunkwise: per chunk, inter = Q_c S, intra =
 *           ((Q_c K_c^T) .* tril) V_c, O_c = inter + intra, S += K_c^T V_c,
 *           ragged last chunk uses the top-left corner of the mask;
 *       "Linear / sparse attention tutorial" section 6.2: with a gate the
 *           state and the in-chunk mask carry the cumulative decay.  The
 *           factors used here (intra exp(Lam_i - Lam_j), inter exp(Lam_i),
 *           state exp(Lam_end) and exp(Lam_end - Lam_j)) are the plain
 *           expansion of the gated recurrence over one chunk.
 *
 *   oracle_noncausal  the non-causal matrix form (no mask, no decay, no S0)
 *       "adv13 - Linear Attention / SSM" section 4.3, linear_attention_matrix:
 *           S = phi(K)^T V over the whole sequence, then O = phi(Q) S;
 *       "CS336 lecture 4, code 1", demo_associativity: (Q K^T) V = Q (K^T V).
 *       Every token reads the same S, the state after the last token.
 *
 *   oracle_normalised  the normalised form, a "next" row
 *       "Linear / sparse attention tutorial" Q11: o_t = phi(q_t)^T S_t /
 *           (phi(q_t)^T z_t), z_t the running sum of phi(k_j); section 2.2:
 *           z_t is the state of one extra value column of ones, so it decays
 *           with S: z_t = a_t z_{t-1} + phi(k_t).
 *
 *   oracle_channel_gate  the per-channel (diagonal) gate, a "next" row
 *       "Linear / sparse attention tutorial" Q21 (GLA):
 *           S_t = diag(alpha_t) S_{t-1} + phi(k_t) v_t^T, alpha_t in (0,1]^dk.
 *
 *   oracle_delta  the (gated) delta rule, a "next" row
 *       "Linear / Sparse Attention - minimal runnable implementation",
 *           delta_rule_recurrent: S_t = S_{t-1}(I - beta_t k_t k_t^T) +
 *           beta_t v_t k_t^T (S as [d_v, d_k]: erase along k, then write);
 *       "Linear / sparse attention tutorial" Q21: the gated version also
 *           multiplies the old state by alpha_t.  Here the state is kept as
 *           its transpose, [d_k, d_v] like the others:
 *           S_t = alpha_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T,
 *           o_t = phi(q_t)^T S_t, with k_t = phi(k_t) as given (the page
 *           assumes unit-norm keys; the caller normalises).
 *
 *   oracle_delta_chunkwise  the same rule, a chunk at a time (WY form)
 *       The pages give the delta rule only token by token.  Unrolling it over
 *       a chunk of n tokens with state S before the chunk and Lam_t the
 *       inclusive prefix of log alpha gives
 *           u_t = beta_t (v_t - e^{Lam_t} S^T k_t
 *                         - sum_{j<t} e^{Lam_t - Lam_j} (k_t.k_j) u_j),
 *           S_t = e^{Lam_t} S + sum_{j<=t} e^{Lam_t - Lam_j} k_j u_j^T,
 *       so each u_t is one row of a unit lower-triangular solve, o_t = q_t^T S_t
 *       and the chunk ends at S_{n-1}.  C = 1 is the recurrence itself; the
 *       pins check every C against oracle_delta.
 *
 * Decay is given per token in log space, lambda_t = log(decay factor):
 *   kind 0  none                  lambda_t = 0
 *   kind 1  per head  [H]         lambda_t = log_gamma[h]          (RetNet)
 *   kind 2  per token [B,H,L]     lambda_t = log_alpha[b,h,t]
 *   kind 3  per token [B,H,L]     lambda_t = -softplus(g[b,h,t])   (gate logits,
 *           alpha_t = exp(-softplus(g_t)))
 *
 * Layouts (all row-major, contiguous): q,k [B,H,L,dk]; v,O [B,H,L,dv];
 * S0, S_final [B,H,dk,dv].  S0 may be NULL (zero initial state).
 * Return value: 0 on success, -1 on a bad argument, -2 on allocation failure.
 */
#include <math.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>

/* phi: 0 = identity; 1 = elu(x) + 1 with the torch default alpha = 1.
 * elu(x) = x for x > 0 and exp(x) - 1 otherwise, so elu(x) + 1 = x + 1 for
 * x > 0 and exp(x) for x <= 0 (page "adv13", Q1; tutorial section 2.1). */
static double feature(int phi, double x)
{
    if (phi == 1)
        return x > 0.0 ? x + 1.0 : exp(x);
    return x;
}

/* softplus(x) = log(1 + exp(x)), written so that neither branch overflows. */
static double softplus(double x)
{
    return x > 0.0 ? x + log1p(exp(-x)) : log1p(exp(x));
}

/* lambda_t for sequence (b,h); see the kind table above. */
static double log_decay(int kind, const double *decay, int H, int L,
                        int b, int h, int t)
{
    switch (kind) {
    case 1: return decay[h];
    case 2: return decay[((size_t)b * H + h) * L + t];
    case 3: return -softplus(decay[((size_t)b * H + h) * L + t]);
    default: return 0.0;
    }
}

static int check_args(int B, int H, int L, int dk, int dv, int phi, int kind,
                      const double *decay)
{
    if (B < 0 || H < 0 || L < 0 || dk <= 0 || dv <= 0) return -1;
    if (phi != 0 && phi != 1) return -1;
    if (kind < 0 || kind > 3) return -1;
    if (kind != 0 && decay == NULL) return -1;
    return 0;
}

/* The recurrence, token by token:
 *     S <- exp(lambda_t) * S + phi(k_t) v_t^T
 *     o_t = phi(q_t)^T S
 * Sequences (b,h) are independent and are spread over OpenMP threads. */
int oracle_recurrent(int B, int H, int L, int dk, int dv,
                     const double *q, const double *k, const double *v,
                     int phi, int kind, const double *decay,
                     const double *S0, double *O, double *S_final)
{
    if (check_args(B, H, L, dk, dv, phi, kind, decay)) return -1;
    int err = 0;
    long nseq = (long)B * H;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
    for (long bh = 0; bh < nseq; ++bh) {
        int b = (int)(bh / H), h = (int)(bh % H);
        double *S = malloc(sizeof(double) * (size_t)dk * dv);
        double *kf = malloc(sizeof(double) * (size_t)dk);
        double *qf = malloc(sizeof(double) * (size_t)dk);
        if (!S || !kf || !qf) { free(S); free(kf); free(qf); err |= 1; continue; }
        if (S0) memcpy(S, S0 + (size_t)bh * dk * dv, sizeof(double) * (size_t)dk * dv);
        else memset(S, 0, sizeof(double) * (size_t)dk * dv);
        for (int t = 0; t < L; ++t) {
            const double *qt = q + ((size_t)bh * L + t) * dk;
            const double *kt = k + ((size_t)bh * L + t) * dk;
            const double *vt = v + ((size_t)bh * L + t) * dv;
            double a = exp(log_decay(kind, decay, H, L, b, h, t));
            for (int i = 0; i < dk; ++i) kf[i] = feature(phi, kt[i]);
            for (int i = 0; i < dk; ++i)
                for (int j = 0; j < dv; ++j)
                    S[(size_t)i * dv + j] = a * S[(size_t)i * dv + j] + kf[i] * vt[j];
            for (int i = 0; i < dk; ++i) qf[i] = feature(phi, qt[i]);
            double *ot = O + ((size_t)bh * L + t) * dv;
            for (int j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (int i = 0; i < dk; ++i) acc += qf[i] * S[(size_t)i * dv + j];
                ot[j] = acc;
            }
        }
        if (S_final) memcpy(S_final + (size_t)bh * dk * dv, S, sizeof(double) * (size_t)dk * dv);
        free(S); free(kf); free(qf);
    }
    return err ? -2 : 0;
}

/* The O(L^2) form:
 *     cum_t = sum_{r<=t} lambda_r
 *     o_t   = sum_{s<=t} exp(cum_t - cum_s) (phi(q_t).phi(k_s)) v_s
 *             + exp(cum_t) phi(q_t)^T S0
 *     S_L   = exp(cum_{L-1}) S0 + sum_s exp(cum_{L-1} - cum_s) phi(k_s) v_s^T
 * For L = 0 the final state is S0 (or zero). */
int oracle_parallel(int B, int H, int L, int dk, int dv,
                    const double *q, const double *k, const double *v,
                    int phi, int kind, const double *decay,
                    const double *S0, double *O, double *S_final)
{
    if (check_args(B, H, L, dk, dv, phi, kind, decay)) return -1;
    int err = 0;
    long nseq = (long)B * H;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
    for (long bh = 0; bh < nseq; ++bh) {
        int b = (int)(bh / H), h = (int)(bh % H);
        double *cum = malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
        double *qf = malloc(sizeof(double) * (size_t)L * dk + 1);
        double *kf = malloc(sizeof(double) * (size_t)L * dk + 1);
        if (!cum || !qf || !kf) { free(cum); free(qf); free(kf); err |= 1; continue; }
        double run = 0.0;
        for (int t = 0; t < L; ++t) {
            run += log_decay(kind, decay, H, L, b, h, t);
            cum[t] = run;
        }
        for (size_t i = 0; i < (size_t)L * dk; ++i) {
            qf[i] = feature(phi, q[(size_t)bh * L * dk + i]);
            kf[i] = feature(phi, k[(size_t)bh * L * dk + i]);
        }
        const double *s0 = S0 ? S0 + (size_t)bh * dk * dv : NULL;
        const double *vb = v + (size_t)bh * L * dv;
        for (int t = 0; t < L; ++t) {
            double *ot = O + ((size_t)bh * L + t) * dv;
            for (int j = 0; j < dv; ++j) ot[j] = 0.0;
            for (int s = 0; s <= t; ++s) {
                double dot = 0.0;
                for (int i = 0; i < dk; ++i) dot += qf[(size_t)t * dk + i] * kf[(size_t)s * dk + i];
                double w = exp(cum[t] - cum[s]) * dot;
                for (int j = 0; j < dv; ++j) ot[j] += w * vb[(size_t)s * dv + j];
            }
            if (s0) {
                double e = exp(cum[t]);
                for (int j = 0; j < dv; ++j) {
                    double acc = 0.0;
                    for (int i = 0; i < dk; ++i) acc += qf[(size_t)t * dk + i] * s0[(size_t)i * dv + j];
                    ot[j] += e * acc;
                }
            }
        }
        if (S_final) {
            double *sf = S_final + (size_t)bh * dk * dv;
            double eL = L > 0 ? exp(cum[L - 1]) : 1.0;
            for (int i = 0; i < dk; ++i)
                for (int j = 0; j < dv; ++j)
                    sf[(size_t)i * dv + j] = s0 ? eL * s0[(size_t)i * dv + j] : 0.0;
            for (int s = 0; s < L; ++s) {
                double w = exp(cum[L - 1] - cum[s]);
                for (int i = 0; i < dk; ++i)
                    for (int j = 0; j < dv; ++j)
                        sf[(size_t)i * dv + j] += w * kf[(size_t)s * dk + i] * vb[(size_t)s * dv + j];
            }
        }
        free(cum); free(qf); free(kf);
    }
    return err ? -2 : 0;
}

/* The chunkwise form with chunk size C >= 1.  For chunk [s0, s0 + n):
 *     Lam_i = sum_{r=s0}^{s0+i} lambda_r                  (inclusive prefix)
 *     o_i   = exp(Lam_i) phi(q_i)^T S                                (inter)
 *             + sum_{j<=i} exp(Lam_i - Lam_j) (phi(q_i).phi(k_j)) v_j (intra)
 *     S    <- exp(Lam_{n-1}) S + sum_j exp(Lam_{n-1} - Lam_j) phi(k_j) v_j^T */
int oracle_chunkwise(int B, int H, int L, int dk, int dv, int C,
                     const double *q, const double *k, const double *v,
                     int phi, int kind, const double *decay,
                     const double *S0, double *O, double *S_final)
{
    if (check_args(B, H, L, dk, dv, phi, kind, decay) || C < 1) return -1;
    int err = 0;
    long nseq = (long)B * H;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
    for (long bh = 0; bh < nseq; ++bh) {
        int b = (int)(bh / H), h = (int)(bh % H);
        double *S = malloc(sizeof(double) * (size_t)dk * dv);
        double *lam = malloc(sizeof(double) * (size_t)C);
        double *qf = malloc(sizeof(double) * (size_t)C * dk);
        double *kf = malloc(sizeof(double) * (size_t)C * dk);
        if (!S || !lam || !qf || !kf) { free(S); free(lam); free(qf); free(kf); err |= 1; continue; }
        if (S0) memcpy(S, S0 + (size_t)bh * dk * dv, sizeof(double) * (size_t)dk * dv);
        else memset(S, 0, sizeof(double) * (size_t)dk * dv);
        const double *vb = v + (size_t)bh * L * dv;
        for (int s0 = 0; s0 < L; s0 += C) {
            int n = L - s0 < C ? L - s0 : C;
            double run = 0.0;
            for (int i = 0; i < n; ++i) {
                run += log_decay(kind, decay, H, L, b, h, s0 + i);
                lam[i] = run;
                for (int c = 0; c < dk; ++c) {
                    qf[(size_t)i * dk + c] = feature(phi, q[((size_t)bh * L + s0 + i) * dk + c]);
                    kf[(size_t)i * dk + c] = feature(phi, k[((size_t)bh * L + s0 + i) * dk + c]);
                }
            }
            for (int i = 0; i < n; ++i) {
                double *oi = O + ((size_t)bh * L + s0 + i) * dv;
                double e = exp(lam[i]);
                for (int j = 0; j < dv; ++j) {
                    double acc = 0.0;
                    for (int c = 0; c < dk; ++c) acc += qf[(size_t)i * dk + c] * S[(size_t)c * dv + j];
                    oi[j] = e * acc;
                }
                for (int jj = 0; jj <= i; ++jj) {
                    double dot = 0.0;
                    for (int c = 0; c < dk; ++c) dot += qf[(size_t)i * dk + c] * kf[(size_t)jj * dk + c];
                    double w = exp(lam[i] - lam[jj]) * dot;
                    for (int j = 0; j < dv; ++j) oi[j] += w * vb[(size_t)(s0 + jj) * dv + j];
                }
            }
            double eEnd = exp(lam[n - 1]);
            for (size_t x = 0; x < (size_t)dk * dv; ++x) S[x] *= eEnd;
            for (int jj = 0; jj < n; ++jj) {
                double w = exp(lam[n - 1] - lam[jj]);
                for (int c = 0; c < dk; ++c)
                    for (int j = 0; j < dv; ++j)
                        S[(size_t)c * dv + j] += w * kf[(size_t)jj * dk + c] * vb[(size_t)(s0 + jj) * dv + j];
            }
        }
        if (S_final) memcpy(S_final + (size_t)bh * dk * dv, S, sizeof(double) * (size_t)dk * dv);
        free(S); free(lam); free(qf); free(kf);
    }
    return err ? -2 : 0;
}

/* Number of threads an OpenMP parallel region in this library would use (1
 * when built without OpenMP); reported beside the CPU timings. */
/* The non-causal form: S = sum_t phi(k_t) v_t^T over all L tokens of (b,h),
 * then o_t = phi(q_t)^T S for every t.  kind must be 0 and S0 NULL (the form
 * has neither); S_final receives S. */
int oracle_noncausal(int B, int H, int L, int dk, int dv,
                     const double *q, const double *k, const double *v,
                     int phi, int kind, const double *decay,
                     const double *S0, double *O, double *S_final)
{
    if (check_args(B, H, L, dk, dv, phi, kind, decay) || kind != 0 || S0 != NULL) return -1;
    int err = 0;
    long nseq = (long)B * H;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
    for (long bh = 0; bh < nseq; ++bh) {
        double *S = calloc((size_t)dk * dv, sizeof(double));
        double *f = malloc(sizeof(double) * (size_t)dk);
        if (!S || !f) { free(S); free(f); err |= 1; continue; }
        for (int t = 0; t < L; ++t) {  /* S = phi(K)^T V */
            const double *kt = k + ((size_t)bh * L + t) * dk;
            const double *vt = v + ((size_t)bh * L + t) * dv;
            for (int i = 0; i < dk; ++i) f[i] = feature(phi, kt[i]);
            for (int i = 0; i < dk; ++i)
                for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] += f[i] * vt[j];
        }
        for (int t = 0; t < L; ++t) {  /* O = phi(Q) S */
            const double *qt = q + ((size_t)bh * L + t) * dk;
            double *ot = O + ((size_t)bh * L + t) * dv;
            for (int i = 0; i < dk; ++i) f[i] = feature(phi, qt[i]);
            for (int j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (int i = 0; i < dk; ++i) acc += f[i] * S[(size_t)i * dv + j];
                ot[j] = acc;
            }
        }
        if (S_final) memcpy(S_final + (size_t)bh * dk * dv, S, sizeof(double) * (size_t)dk * dv);
        free(S); free(f);
    }
    return err ? -2 : 0;
}

/* The normalised form, token by token:
 *     S <- a_t S + phi(k_t) v_t^T ;  z <- a_t z + phi(k_t)
 *     o_t = phi(q_t)^T S / (phi(q_t)^T z)
 * z0 [B,H,dk] may be NULL (zero); z_final [B,H,dk] may be NULL.  A zero
 * denominator gives inf or NaN, as the formula does. */
int oracle_normalised(int B, int H, int L, int dk, int dv,
                      const double *q, const double *k, const double *v,
                      int phi, int kind, const double *decay,
                      const double *S0, const double *z0,
                      double *O, double *S_final, double *z_final)
{
    if (check_args(B, H, L, dk, dv, phi, kind, decay)) return -1;
    int err = 0;
    long nseq = (long)B * H;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
    for (long bh = 0; bh < nseq; ++bh) {
        int b = (int)(bh / H), h = (int)(bh % H);
        double *S = malloc(sizeof(double) * (size_t)dk * dv);
        double *z = malloc(sizeof(double) * (size_t)dk);
        double *kf = malloc(sizeof(double) * (size_t)dk);
        double *qf = malloc(sizeof(double) * (size_t)dk);
        if (!S || !z || !kf || !qf) { free(S); free(z); free(kf); free(qf); err |= 1; continue; }
        if (S0) memcpy(S, S0 + (size_t)bh * dk * dv, sizeof(double) * (size_t)dk * dv);
        else memset(S, 0, sizeof(double) * (size_t)dk * dv);
        if (z0) memcpy(z, z0 + (size_t)bh * dk, sizeof(double) * (size_t)dk);
        else memset(z, 0, sizeof(double) * (size_t)dk);
        for (int t = 0; t < L; ++t) {
            const double *qt = q + ((size_t)bh * L + t) * dk;
            const double *kt = k + ((size_t)bh * L + t) * dk;
            const double *vt = v + ((size_t)bh * L + t) * dv;
            double a = exp(log_decay(kind, decay, H, L, b, h, t));
            for (int i = 0; i < dk; ++i) kf[i] = feature(phi, kt[i]);
            for (int i = 0; i < dk; ++i) {
                for (int j = 0; j < dv; ++j)
                    S[(size_t)i * dv + j] = a * S[(size_t)i * dv + j] + kf[i] * vt[j];
                z[i] = a * z[i] + kf[i];
            }
            for (int i = 0; i < dk; ++i) qf[i] = feature(phi, qt[i]);
            double den = 0.0;
            for (int i = 0; i < dk; ++i) den += qf[i] * z[i];
            double *ot = O + ((size_t)bh * L + t) * dv;
            for (int j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (int i = 0; i < dk; ++i) acc += qf[i] * S[(size_t)i * dv + j];
                ot[j] = acc / den;
            }
        }
        if (S_final) memcpy(S_final + (size_t)bh * dk * dv, S, sizeof(double) * (size_t)dk * dv);
        if (z_final) memcpy(z_final + (size_t)bh * dk, z, sizeof(double) * (size_t)dk);
        free(S); free(z); free(kf); free(qf);
    }
    return err ? -2 : 0;
}

/* The per-channel gate, token by token:
 *     S[i,:] <- alpha_t[i] S[i,:] + phi(k_t)[i] v_t^T ;   o_t = phi(q_t)^T S
 * log_alpha [B,H,L,dk] holds log alpha_t[i] (<= 0). */
int oracle_channel_gate(int B, int H, int L, int dk, int dv,
                        const double *q, const double *k, const double *v,
                        int phi, const double *log_alpha,
                        const double *S0, double *O, double *S_final)
{
    if (check_args(B, H, L, dk, dv, phi, 0, NULL) || !log_alpha) return -1;
    int err = 0;
    long nseq = (long)B * H;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
    for (long bh = 0; bh < nseq; ++bh) {
        double *S = malloc(sizeof(double) * (size_t)dk * dv);
        double *kf = malloc(sizeof(double) * (size_t)dk);
        double *qf = malloc(sizeof(double) * (size_t)dk);
        if (!S || !kf || !qf) { free(S); free(kf); free(qf); err |= 1; continue; }
        if (S0) memcpy(S, S0 + (size_t)bh * dk * dv, sizeof(double) * (size_t)dk * dv);
        else memset(S, 0, sizeof(double) * (size_t)dk * dv);
        for (int t = 0; t < L; ++t) {
            const double *qt = q + ((size_t)bh * L + t) * dk;
            const double *kt = k + ((size_t)bh * L + t) * dk;
            const double *vt = v + ((size_t)bh * L + t) * dv;
            const double *la = log_alpha + ((size_t)bh * L + t) * dk;
            for (int i = 0; i < dk; ++i) kf[i] = feature(phi, kt[i]);
            for (int i = 0; i < dk; ++i) {
                const double a = exp(la[i]);
                for (int j = 0; j < dv; ++j)
                    S[(size_t)i * dv + j] = a * S[(size_t)i * dv + j] + kf[i] * vt[j];
            }
            for (int i = 0; i < dk; ++i) qf[i] = feature(phi, qt[i]);
            double *ot = O + ((size_t)bh * L + t) * dv;
            for (int j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (int i = 0; i < dk; ++i) acc += qf[i] * S[(size_t)i * dv + j];
                ot[j] = acc;
            }
        }
        if (S_final) memcpy(S_final + (size_t)bh * dk * dv, S, sizeof(double) * (size_t)dk * dv);
        free(S); free(kf); free(qf);
    }
    return err ? -2 : 0;
}

/* The gated delta rule, token by token, with the state as [d_k, d_v]:
 *     S <- alpha_t (S - beta_t k (k^T S)) + beta_t k v_t^T ;  o_t = q^T S
 * with k = phi(k_t), q = phi(q_t).  beta [B,H,L]; log_alpha [B,H,L] or NULL
 * (alpha = 1). */
int oracle_delta(int B, int H, int L, int dk, int dv,
                 const double *q, const double *k, const double *v,
                 int phi, const double *beta, const double *log_alpha,
                 const double *S0, double *O, double *S_final)
{
    if (check_args(B, H, L, dk, dv, phi, 0, NULL) || !beta) return -1;
    int err = 0;
    long nseq = (long)B * H;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
    for (long bh = 0; bh < nseq; ++bh) {
        double *S = malloc(sizeof(double) * (size_t)dk * dv);
        double *kf = malloc(sizeof(double) * (size_t)dk);
        double *qf = malloc(sizeof(double) * (size_t)dk);
        double *ks = malloc(sizeof(double) * (size_t)dv);
        if (!S || !kf || !qf || !ks) { free(S); free(kf); free(qf); free(ks); err |= 1; continue; }
        if (S0) memcpy(S, S0 + (size_t)bh * dk * dv, sizeof(double) * (size_t)dk * dv);
        else memset(S, 0, sizeof(double) * (size_t)dk * dv);
        for (int t = 0; t < L; ++t) {
            const double *qt = q + ((size_t)bh * L + t) * dk;
            const double *kt = k + ((size_t)bh * L + t) * dk;
            const double *vt = v + ((size_t)bh * L + t) * dv;
            const double bt = beta[(size_t)bh * L + t];
            const double a = log_alpha ? exp(log_alpha[(size_t)bh * L + t]) : 1.0;
            for (int i = 0; i < dk; ++i) kf[i] = feature(phi, kt[i]);
            for (int j = 0; j < dv; ++j) {  /* k^T S, a row of d_v values */
                double acc = 0.0;
                for (int i = 0; i < dk; ++i) acc += kf[i] * S[(size_t)i * dv + j];
                ks[j] = acc;
            }
            for (int i = 0; i < dk; ++i)
                for (int j = 0; j < dv; ++j)
                    S[(size_t)i * dv + j] = a * (S[(size_t)i * dv + j] - bt * kf[i] * ks[j]) +
                                            bt * kf[i] * vt[j];
            for (int i = 0; i < dk; ++i) qf[i] = feature(phi, qt[i]);
            double *ot = O + ((size_t)bh * L + t) * dv;
            for (int j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (int i = 0; i < dk; ++i) acc += qf[i] * S[(size_t)i * dv + j];
                ot[j] = acc;
            }
        }
        if (S_final) memcpy(S_final + (size_t)bh * dk * dv, S, sizeof(double) * (size_t)dk * dv);
        free(S); free(kf); free(qf); free(ks);
    }
    return err ? -2 : 0;
}

/* The delta rule chunk by chunk (see the header): per chunk, the u_t by
 * forward substitution, then every output and the state at the chunk end. */
int oracle_delta_chunkwise(int B, int H, int L, int dk, int dv, int C,
                           const double *q, const double *k, const double *v,
                           int phi, const double *beta, const double *log_alpha,
                           const double *S0, double *O, double *S_final)
{
    if (check_args(B, H, L, dk, dv, phi, 0, NULL) || !beta || C < 1) return -1;
    int err = 0;
    long nseq = (long)B * H;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
    for (long bh = 0; bh < nseq; ++bh) {
        double *S = malloc(sizeof(double) * (size_t)dk * dv);
        double *lam = malloc(sizeof(double) * (size_t)C);
        double *qf = malloc(sizeof(double) * (size_t)C * dk);
        double *kf = malloc(sizeof(double) * (size_t)C * dk);
        double *U = malloc(sizeof(double) * (size_t)C * dv);
        if (!S || !lam || !qf || !kf || !U) {
            free(S); free(lam); free(qf); free(kf); free(U); err |= 1; continue;
        }
        if (S0) memcpy(S, S0 + (size_t)bh * dk * dv, sizeof(double) * (size_t)dk * dv);
        else memset(S, 0, sizeof(double) * (size_t)dk * dv);
        for (int s0 = 0; s0 < L; s0 += C) {
            int n = L - s0 < C ? L - s0 : C;
            double run = 0.0;
            for (int t = 0; t < n; ++t) {
                size_t row = (size_t)bh * L + s0 + t;
                run += log_alpha ? log_alpha[row] : 0.0;
                lam[t] = run;
                for (int c = 0; c < dk; ++c) {
                    qf[(size_t)t * dk + c] = feature(phi, q[row * dk + c]);
                    kf[(size_t)t * dk + c] = feature(phi, k[row * dk + c]);
                }
            }
            for (int t = 0; t < n; ++t) {  /* forward substitution, row by row */
                size_t row = (size_t)bh * L + s0 + t;
                double bt = beta[row], et = exp(lam[t]);
                for (int j = 0; j < dv; ++j) {
                    double kS = 0.0;
                    for (int c = 0; c < dk; ++c) kS += kf[(size_t)t * dk + c] * S[(size_t)c * dv + j];
                    double acc = v[row * dv + j] - et * kS;
                    for (int i = 0; i < t; ++i) {
                        double kk = 0.0;
                        for (int c = 0; c < dk; ++c)
                            kk += kf[(size_t)t * dk + c] * kf[(size_t)i * dk + c];
                        acc -= exp(lam[t] - lam[i]) * kk * U[(size_t)i * dv + j];
                    }
                    U[(size_t)t * dv + j] = bt * acc;
                }
            }
            for (int t = 0; t < n; ++t) {  /* o_t = q_t^T S_t */
                double *ot = O + ((size_t)bh * L + s0 + t) * dv;
                double et = exp(lam[t]);
                for (int j = 0; j < dv; ++j) {
                    double acc = 0.0;
                    for (int c = 0; c < dk; ++c) acc += qf[(size_t)t * dk + c] * S[(size_t)c * dv + j];
                    acc *= et;
                    for (int i = 0; i <= t; ++i) {
                        double qk = 0.0;
                        for (int c = 0; c < dk; ++c)
                            qk += qf[(size_t)t * dk + c] * kf[(size_t)i * dk + c];
                        acc += exp(lam[t] - lam[i]) * qk * U[(size_t)i * dv + j];
                    }
                    ot[j] = acc;
                }
            }
            double eEnd = exp(lam[n - 1]);  /* S <- S_{n-1} */
            for (size_t x = 0; x < (size_t)dk * dv; ++x) S[x] *= eEnd;
            for (int i = 0; i < n; ++i) {
                double w = exp(lam[n - 1] - lam[i]);
                for (int c = 0; c < dk; ++c)
                    for (int j = 0; j < dv; ++j)
                        S[(size_t)c * dv + j] += w * kf[(size_t)i * dk + c] * U[(size_t)i * dv + j];
            }
        }
        if (S_final) memcpy(S_final + (size_t)bh * dk * dv, S, sizeof(double) * (size_t)dk * dv);
        free(S); free(lam); free(qf); free(kf); free(U);
    }
    return err ? -2 : 0;
}

#ifdef _OPENMP
#include <omp.h>
int oracle_num_threads(void) { return omp_get_max_threads(); }
#else
int oracle_num_threads(void) { return 1; }
#endif
