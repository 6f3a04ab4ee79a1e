/*
 * gla_oracle.c -- fp64 CPU oracle of causal gated linear attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code with
 * the CUDA path and is deliberately plain: one token at a time, in float64,
 * in the order the pages write the method.
 *
 * Sources (page title, section):
 *  [GLA]  "Gated Linear Attention" (garden note), "GLA / Recurrent Form":
 *         S_t = Diag(alpha_t) S_{t-1} + (outer product of k_t and v_t),
 *         with alpha_t in (0,1)^{d_k}; the flowchart multiplies q_t with the
 *         *updated* state S_t to give o_t.
 *  [LA]   "linear-attention" blog, "Linear attention" and "Gated linear
 *         attention": o_n depends on (S_{n-1}, q_n, k_n, v_n); the state
 *         update is S_n = S_{n-1} + k_n^T v_n (row-vector convention, so the
 *         state is d_k x d_v), gated by alpha_n.
 *  [RNN]  "Transformers are RNNs" notes, kernel derivation: normalised form
 *         V'_i = sum_j sim(Q_i,K_j) V_j / sum_j sim(Q_i,K_j) with
 *         sim = phi(Q_i)^T phi(K_j), made causal (j <= i).
 *  [CHK]  "Gated Linear Attention", "Summary" / "Chunk-Wise Block-Parallel":
 *         the chunk-wise form that interpolates between the parallel and the
 *         recurrent form (used only by oracle_gla_fwd_chunked).
 *  [DLT]  "linear-attention" blog, "Delta attention": before writing, ask
 *         what the memory already predicts for the key and write only the
 *         error, with a write strength beta_n; the gated variant decays the
 *         state first (used only by oracle_delta_fwd).
 *
 * Readings taken where the pages are silent or garbled:
 *  - state S is d_k x d_v, the update is k_t v_t^T, the decay scales the d_k
 *    rows, and o_t = S_t^T q_t (inclusive: S_t already holds token t);
 *  - phi(x) = elu(x) + 1 (x + 1 for x > 0, e^x otherwise) when requested;
 *  - the normaliser z_t is carried like one extra all-ones value column of
 *    the state, so it decays with the same Diag(alpha_t) when a gate is
 *    present; no epsilon is added (phi > 0 keeps the denominator positive).
 *
 *  - delta rule: p_n = S_{n-1}^T k_n (the memory's prediction for k_n),
 *    u_n = beta_n (v_n - p_n) (the error, written with strength beta_n),
 *    S_n = S_{n-1} + k_n u_n^T, o_n = S_n^T q_n; with a gate the decay
 *    Diag(alpha_n) is applied to S_{n-1} before the prediction.
 *
 *  - backward: reverse mode through the recurrence with every state kept
 *    (dL/dS_t = Diag(alpha_{t+1}) dL/dS_{t+1} + q_t dout_t^T), pinned by
 *    finite differences of the forward oracle.
 *
 * Planted mistakes: compiling with -DORACLE_PLANT=n (n >= 1) builds a
 * deliberately wrong variant that the pinning tests must reject.  The normal
 * build has ORACLE_PLANT = 0 and none of those branches.
 */
#include <math.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifndef ORACLE_PLANT
#define ORACLE_PLANT 0
#endif

#define ORACLE_FEATURE_ELU1 1
#define ORACLE_NORMALIZE 2

static double phi_elu1(double x) { return x > 0.0 ? x + 1.0 : exp(x); }

static void set_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* One token of the recurrence for one (batch, head) pair.
 *   S  [dk][dv] in/out, z [dk] in/out (normalised mode only)
 *   q, k [dk], v [dv], la [dk] (log alpha; NULL means alpha == 1)
 *   o  [dv] out
 */
static void recur_token(double *S, double *z, const double *q, const double *k,
                        const double *v, const double *la, double *o,
                        long dk, long dv, int flags, double *qf, double *kf) {
    const int elu1 = flags & ORACLE_FEATURE_ELU1;
    const int norm = flags & ORACLE_NORMALIZE;
    for (long i = 0; i < dk; i++) {
        qf[i] = elu1 ? phi_elu1(q[i]) : q[i];
        kf[i] = elu1 ? phi_elu1(k[i]) : k[i];
    }
    /* S_t = Diag(alpha_t) S_{t-1} + k_t v_t^T   [GLA Recurrent Form] */
    for (long i = 0; i < dk; i++) {
        double a = la ? exp(la[i]) : 1.0;
#if ORACLE_PLANT == 1
        /* planted: decay applied after the write (write decays at its own step) */
        for (long j = 0; j < dv; j++) S[i * dv + j] = a * (S[i * dv + j] + kf[i] * v[j]);
        if (norm) z[i] = a * (z[i] + kf[i]);
        continue;
#endif
        for (long j = 0; j < dv; j++) S[i * dv + j] = a * S[i * dv + j] + kf[i] * v[j];
        if (norm) z[i] = a * z[i] + kf[i];
    }
    /* o_t = S_t^T q_t  (q multiplies the updated state)   [GLA flowchart] */
    for (long j = 0; j < dv; j++) {
        double acc = 0.0;
#if ORACLE_PLANT == 2
        /* planted: transposed contraction (only meaningful when dk == dv) */
        for (long i = 0; i < dk; i++) acc += qf[i] * S[j * dv + i];
#else
        for (long i = 0; i < dk; i++) acc += qf[i] * S[i * dv + j];
#endif
        o[j] = acc;
    }
    if (norm) {
        double den = 0.0;
        for (long i = 0; i < dk; i++) den += qf[i] * z[i];
#if ORACLE_PLANT == 3
        den = 1.0; /* planted: normaliser dropped */
#endif
        for (long j = 0; j < dv; j++) o[j] /= den;
    }
}

#if ORACLE_PLANT == 4
/* planted: output taken from S_{t-1} (exclusive) instead of S_t */
#define PLANT_EXCLUSIVE 1
#endif

/*
 * Prefill: every (b, h) runs the recurrence over t = 0 .. L-1.
 * Layouts (row-major): q, k, log_alpha [B][H][L][dk]; v, out [B][H][L][dv];
 * init_state, final_state [B][H][dk][dv]; init_z, final_z [B][H][dk].
 * log_alpha, init_state, init_z, final_state, final_z may be NULL.
 */
int oracle_gla_fwd(const double *q, const double *k, const double *v,
                   const double *log_alpha, const double *init_state,
                   const double *init_z, double *out, double *final_state,
                   double *final_z, long B, long H, long L, long dk, long dv,
                   int flags, int nthreads) {
    if (B < 0 || H < 0 || L < 0 || dk <= 0 || dv <= 0) return 1;
    set_threads(nthreads);
    long BH = B * H;
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (long bh = 0; bh < BH; bh++) {
        double *S = (double *)calloc((size_t)(dk * dv), sizeof(double));
        double *z = (double *)calloc((size_t)dk, sizeof(double));
        double *qf = (double *)malloc((size_t)dk * sizeof(double));
        double *kf = (double *)malloc((size_t)dk * sizeof(double));
        double *prev = (double *)malloc((size_t)(dk * dv) * sizeof(double));
        if (!S || !z || !qf || !kf || !prev) {
#pragma omp atomic write
            err = 2;
            free(S); free(z); free(qf); free(kf); free(prev);
            continue;
        }
        if (init_state) memcpy(S, init_state + bh * dk * dv, (size_t)(dk * dv) * sizeof(double));
        if (init_z) memcpy(z, init_z + bh * dk, (size_t)dk * sizeof(double));
        for (long t = 0; t < L; t++) {
            const double *qt = q + (bh * L + t) * dk;
            const double *kt = k + (bh * L + t) * dk;
            const double *vt = v + (bh * L + t) * dv;
            const double *lat = log_alpha ? log_alpha + (bh * L + t) * dk : NULL;
            double *ot = out + (bh * L + t) * dv;
#ifdef PLANT_EXCLUSIVE
            memcpy(prev, S, (size_t)(dk * dv) * sizeof(double));
            recur_token(S, z, qt, kt, vt, lat, ot, dk, dv, flags, qf, kf);
            for (long j = 0; j < dv; j++) {
                double acc = 0.0;
                for (long i = 0; i < dk; i++) acc += qf[i] * prev[i * dv + j];
                ot[j] = acc;
            }
#else
            recur_token(S, z, qt, kt, vt, lat, ot, dk, dv, flags, qf, kf);
#endif
        }
        if (final_state) memcpy(final_state + bh * dk * dv, S, (size_t)(dk * dv) * sizeof(double));
        if (final_z) memcpy(final_z + bh * dk, z, (size_t)dk * sizeof(double));
        free(S); free(z); free(qf); free(kf); free(prev);
    }
    return err;
}

/*
 * Decode: one token per (sequence, head); the state is updated in place.
 * q, k, log_alpha [NS][H][dk]; v, out [NS][H][dv]; state [NS][H][dk][dv].
 */
int oracle_gla_decode_step(const double *q, const double *k, const double *v,
                           const double *log_alpha, double *state, double *out,
                           long NS, long H, long dk, long dv, int nthreads) {
    if (NS < 0 || H < 0 || dk <= 0 || dv <= 0) return 1;
    set_threads(nthreads);
    long n = NS * H;
    int err = 0;
#pragma omp parallel for schedule(static)
    for (long s = 0; s < n; s++) {
        double *qf = (double *)malloc((size_t)dk * sizeof(double));
        double *kf = (double *)malloc((size_t)dk * sizeof(double));
        if (!qf || !kf) {
#pragma omp atomic write
            err = 2;
            free(qf); free(kf);
            continue;
        }
        recur_token(state + s * dk * dv, NULL, q + s * dk, k + s * dk, v + s * dv,
                    log_alpha ? log_alpha + s * dk : NULL, out + s * dv, dk, dv, 0, qf, kf);
        free(qf); free(kf);
    }
    return err;
}

/*
 * Chunk-wise restatement [CHK], in fp64, for chunk size C >= 1.  It is the
 * same function of the inputs as oracle_gla_fwd (an exact refactoring of the
 * recurrence); tests compare the two.  With b_t the inclusive cumulative sum
 * of log alpha from the chunk start and b_C its value at the chunk's last
 * token, unrolling the gated recurrence over one chunk gives
 *   o_t = (q_t * e^{b_t})^T S_prev
 *         + sum_{i in chunk, i <= t} [(q_t * e^{b_t}) . (k_i * e^{-b_i})] v_i
 *   S   = Diag(e^{b_C}) S_prev + sum_{i in chunk} (k_i * e^{b_C - b_i}) v_i^T
 * (no feature map or normaliser here).
 */
int oracle_gla_fwd_chunked(const double *q, const double *k, const double *v,
                           const double *log_alpha, const double *init_state,
                           double *out, double *final_state, long B, long H,
                           long L, long dk, long dv, long C, int nthreads) {
    if (B < 0 || H < 0 || L < 0 || dk <= 0 || dv <= 0 || C <= 0) return 1;
    set_threads(nthreads);
    long BH = B * H;
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (long bh = 0; bh < BH; bh++) {
        double *S = (double *)calloc((size_t)(dk * dv), sizeof(double));
        double *b = (double *)malloc((size_t)(C * dk) * sizeof(double));
        if (!S || !b) {
#pragma omp atomic write
            err = 2;
            free(S); free(b);
            continue;
        }
        if (init_state) memcpy(S, init_state + bh * dk * dv, (size_t)(dk * dv) * sizeof(double));
        for (long c0 = 0; c0 < L; c0 += C) {
            long n = (L - c0) < C ? (L - c0) : C;
            for (long d = 0; d < dk; d++) {
                double run = 0.0;
                for (long t = 0; t < n; t++) {
                    if (log_alpha) run += log_alpha[(bh * L + c0 + t) * dk + d];
                    b[t * dk + d] = run;
                }
            }
            const double *bC = b + (n - 1) * dk;
            for (long t = 0; t < n; t++) {
                const double *qt = q + (bh * L + c0 + t) * dk;
                double *ot = out + (bh * L + c0 + t) * dv;
                for (long j = 0; j < dv; j++) {
                    double acc = 0.0;
                    for (long d = 0; d < dk; d++) acc += qt[d] * exp(b[t * dk + d]) * S[d * dv + j];
                    ot[j] = acc;
                }
                for (long i = 0; i <= t; i++) {
                    const double *ki = k + (bh * L + c0 + i) * dk;
                    const double *vi = v + (bh * L + c0 + i) * dv;
                    double a = 0.0;
                    for (long d = 0; d < dk; d++)
                        a += (qt[d] * exp(b[t * dk + d])) * (ki[d] * exp(-b[i * dk + d]));
                    for (long j = 0; j < dv; j++) ot[j] += a * vi[j];
                }
            }
            for (long d = 0; d < dk; d++) {
                double g = exp(bC[d]);
                for (long j = 0; j < dv; j++) S[d * dv + j] *= g;
            }
            for (long i = 0; i < n; i++) {
                const double *ki = k + (bh * L + c0 + i) * dk;
                const double *vi = v + (bh * L + c0 + i) * dv;
                for (long d = 0; d < dk; d++) {
                    double kh = ki[d] * exp(bC[d] - b[i * dk + d]);
                    for (long j = 0; j < dv; j++) S[d * dv + j] += kh * vi[j];
                }
            }
        }
        if (final_state) memcpy(final_state + bh * dk * dv, S, (size_t)(dk * dv) * sizeof(double));
        free(S); free(b);
    }
    return err;
}

/*
 * Delta rule [DLT], token by token, for every (b, h):
 *   S <- Diag(alpha_n) S            (gated variant; log_alpha may be NULL)
 *   p  = S^T k_n                    (what the memory predicts for k_n)
 *   u  = beta_n (v_n - p)           (the error, written with strength beta_n)
 *   S <- S + k_n u^T
 *   o_n = S^T q_n
 * Layouts: q, k, log_alpha [BH][L][dk]; v, out [BH][L][dv]; beta [BH][L];
 * init_state, final_state [BH][dk][dv] (init_state may be NULL: zero).
 */
int oracle_delta_fwd(const double *q, const double *k, const double *v, const double *beta,
                     const double *log_alpha, const double *init_state, double *out,
                     double *final_state, long BH, long L, long dk, long dv, int nthreads) {
    set_threads(nthreads);
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (long h = 0; h < BH; h++) {
        double *S = malloc(sizeof(double) * dk * dv);
        double *p = malloc(sizeof(double) * dv);
        double *u = malloc(sizeof(double) * dv);
        if (!S || !p || !u) {
#pragma omp atomic write
            err = 1;
            free(S);
            free(p);
            free(u);
            continue;
        }
        for (long i = 0; i < dk * dv; i++) S[i] = init_state ? init_state[h * dk * dv + i] : 0.0;
        for (long t = 0; t < L; t++) {
            const double *qt = q + (h * L + t) * dk, *kt = k + (h * L + t) * dk;
            const double *vt = v + (h * L + t) * dv;
            const double bt = beta[h * L + t];
            if (log_alpha)
                for (long i = 0; i < dk; i++) {
                    const double a = exp(log_alpha[(h * L + t) * dk + i]);
                    for (long j = 0; j < dv; j++) S[i * dv + j] *= a;
                }
            for (long j = 0; j < dv; j++) {
                double acc = 0.0;
                for (long i = 0; i < dk; i++) acc += S[i * dv + j] * kt[i];
                p[j] = acc;
            }
            for (long j = 0; j < dv; j++) {
#if ORACLE_PLANT == 5
                u[j] = bt * vt[j]; /* planted: prediction dropped (plain linear attention) */
#else
                u[j] = bt * (vt[j] - p[j]);
#endif
            }
            double *ot = out + (h * L + t) * dv;
#if ORACLE_PLANT == 6
            /* planted: output read before the write */
            for (long j = 0; j < dv; j++) {
                double acc = 0.0;
                for (long i = 0; i < dk; i++) acc += S[i * dv + j] * qt[i];
                ot[j] = acc;
            }
#endif
            for (long i = 0; i < dk; i++)
                for (long j = 0; j < dv; j++) S[i * dv + j] += kt[i] * u[j];
#if ORACLE_PLANT != 6
            for (long j = 0; j < dv; j++) {
                double acc = 0.0;
                for (long i = 0; i < dk; i++) acc += S[i * dv + j] * qt[i];
                ot[j] = acc;
            }
#endif
        }
        if (final_state)
            for (long i = 0; i < dk * dv; i++) final_state[h * dk * dv + i] = S[i];
        free(S);
        free(p);
        free(u);
    }
    return err;
}

/*
 * Backward of the recurrence [GLA Recurrent Form], reverse mode, for every
 * (b, h), given dout = dL/do_t and dfinal = dL/dS_{L-1} (may be NULL):
 *   forward:  S_t = Diag(alpha_t) S_{t-1} + k_t v_t^T  (every S_t kept),
 *             dq_t = S_t dout_t
 *   reverse:  H = dfinal (or 0); for t = L-1 .. 0:
 *               G   = H + q_t dout_t^T              (dL/dS_t, total)
 *               dk_t = G v_t,  dv_t = G^T k_t
 *               dlog_alpha_t[i] = alpha_t[i] sum_j G[i][j] S_{t-1}[i][j]
 *               H   = Diag(alpha_t) G               (dL/dS_{t-1} so far)
 *             dinit = H.
 * Layouts as oracle_gla_fwd; dout [BH][L][dv]; dq, dk, dla [BH][L][dk];
 * dv [BH][L][dv]; dfinal, dinit [BH][dk][dv].  dla and dinit may be NULL.
 */
int oracle_gla_bwd(const double *q, const double *k, const double *v, const double *log_alpha,
                   const double *init_state, const double *dout, const double *dfinal, double *dq,
                   double *dk_out, double *dv_out, double *dla, double *dinit, long BH, long L, long dk,
                   long dv, int nthreads) {
    set_threads(nthreads);
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (long h = 0; h < BH; h++) {
        /* states[t + 1] = S_t, states[0] = S_{-1} */
        double *states = malloc(sizeof(double) * (size_t)(L + 1) * dk * dv);
        double *G = malloc(sizeof(double) * dk * dv);
        double *Hs = malloc(sizeof(double) * dk * dv);
        if (!states || !G || !Hs) {
#pragma omp atomic write
            err = 1;
            free(states);
            free(G);
            free(Hs);
            continue;
        }
        for (long i = 0; i < dk * dv; i++) states[i] = init_state ? init_state[h * dk * dv + i] : 0.0;
        for (long t = 0; t < L; t++) {
            const double *Sp = states + (size_t)t * dk * dv;
            double *S = states + (size_t)(t + 1) * dk * dv;
            const double *kt = k + (h * L + t) * dk, *vt = v + (h * L + t) * dv;
            const double *dot = dout + (h * L + t) * dv;
            for (long i = 0; i < dk; i++) {
                const double a = log_alpha ? exp(log_alpha[(h * L + t) * dk + i]) : 1.0;
                for (long j = 0; j < dv; j++) S[i * dv + j] = a * Sp[i * dv + j] + kt[i] * vt[j];
            }
            for (long i = 0; i < dk; i++) {
                double acc = 0.0;
                for (long j = 0; j < dv; j++) acc += S[i * dv + j] * dot[j];
                dq[(h * L + t) * dk + i] = acc;
            }
        }
        for (long i = 0; i < dk * dv; i++) Hs[i] = dfinal ? dfinal[h * dk * dv + i] : 0.0;
        for (long t = L - 1; t >= 0; t--) {
            const double *Sp = states + (size_t)t * dk * dv;
            const double *qt = q + (h * L + t) * dk, *kt = k + (h * L + t) * dk, *vt = v + (h * L + t) * dv;
            const double *dot = dout + (h * L + t) * dv;
            for (long i = 0; i < dk; i++)
                for (long j = 0; j < dv; j++) G[i * dv + j] = Hs[i * dv + j] + qt[i] * dot[j];
            for (long i = 0; i < dk; i++) {
                double acc = 0.0;
                for (long j = 0; j < dv; j++) acc += G[i * dv + j] * vt[j];
                dk_out[(h * L + t) * dk + i] = acc;
            }
            for (long j = 0; j < dv; j++) {
                double acc = 0.0;
                for (long i = 0; i < dk; i++) acc += G[i * dv + j] * kt[i];
                dv_out[(h * L + t) * dv + j] = acc;
            }
            for (long i = 0; i < dk; i++) {
                const double a = log_alpha ? exp(log_alpha[(h * L + t) * dk + i]) : 1.0;
                if (dla) {
                    double acc = 0.0;
#if ORACLE_PLANT == 7
                    /* planted: gate gradient paired with S_t instead of S_{t-1} */
                    for (long j = 0; j < dv; j++) acc += G[i * dv + j] * Sp[dk * dv + i * dv + j];
#else
                    for (long j = 0; j < dv; j++) acc += G[i * dv + j] * Sp[i * dv + j];
#endif
                    dla[(h * L + t) * dk + i] = a * acc;
                }
#if ORACLE_PLANT == 8
                /* planted: state gradient carried back without the decay */
                for (long j = 0; j < dv; j++) Hs[i * dv + j] = G[i * dv + j];
#else
                for (long j = 0; j < dv; j++) Hs[i * dv + j] = a * G[i * dv + j];
#endif
            }
        }
        if (dinit)
            for (long i = 0; i < dk * dv; i++) dinit[h * dk * dv + i] = Hs[i];
        free(states);
        free(G);
        free(Hs);
    }
    return err;
}
