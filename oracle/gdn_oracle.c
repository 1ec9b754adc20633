/*
 * gdn_oracle.c -- fp64 CPU oracle for the gated delta-rule recurrence.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file: only the tests, the smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header or constant with the CUDA library.
 *
 * Every routine works on one unit: one batch row b and one value head h.
 * Arrays are the caller's, in fp64, in these layouts (token-major, dk or dv
 * fastest):
 *   q, k   [total_T, Hk, dk]     (query and key heads; Hq == Hk)
 *   v, o   [total_T, Hv, dv]
 *   alpha, beta [total_T, Hv]
 *   S      [dv, dk]              (one state matrix; S[i][j], j fastest)
 *   state_update  [capacity, Hv + Hk*dk + Hv*dv] for this row: per slot the
 *                 decay of every value head, then the key of every key head,
 *                 then the delta of every value head.
 * A row's tokens are tok0 .. tok0+T_b-1.  Value head h reads key/query head
 * hk = h / (Hv / Hk)  (inverse-GQA sharing, contiguous groups).
 *
 * Sources:
 *  - The per-token gated delta rule of Gated DeltaNet: decay the state by
 *    alpha_t, form delta_t = beta_t (v_t - S k_t) with the decayed state, add
 *    the rank-1 term delta_t k_t^T, read out o_t = S q_t with the updated state.
 *  - "[WebGPU EP] adds state update capacity support for GatedDeltaNet"
 *    (onnxruntime PR 32767), section "Changes": capture of the clamped
 *    per-row prefix of decay, shared-key and delta factors, which replay
 *    S = decay * S + outer(key, delta); inverse-GQA key sharing.
 *  - "Enable the native Kev example on NVIDIA GPUs through ExecuTorch's AOTI
 *    CUDA backend" (executorch issue 23097), work list: a chunked GDN prefill
 *    with explicit initial and final state and an FP32 recurrence.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------------- */
/* Recurrent form: the definition, one token at a time.                    */
/* ---------------------------------------------------------------------- */

/*
 * Runs the per-token recurrence for unit (row, value head h).
 * S is read as the initial state and overwritten with the final one.
 * If state_update is non-NULL, tokens t < n_capture store their factors in
 * slot t; the key of key head hk is stored by the first value head of its
 * group (h % G == 0) so that every slot field has exactly one writer.
 */
void gdn_oracle_recurrent_unit(const double *q, const double *k, const double *v,
                               const double *alpha, const double *beta,
                               long tok0, int T_b, int Hk, int Hv, int dk, int dv,
                               int h, double scale, double *S, double *o,
                               int n_capture, double *state_update)
{
    const int G = Hv / Hk;
    const int hk = h / G;
    const long slot = (long)Hv + (long)Hk * dk + (long)Hv * dv;
    double *Sk = (double *)malloc(sizeof(double) * dv);
    double *delta = (double *)malloc(sizeof(double) * dv);

    for (int t = 0; t < T_b; ++t) {
        const long tok = tok0 + t;
        const double *kt = k + (tok * Hk + hk) * dk;
        const double *qt = q + (tok * Hk + hk) * dk;
        const double *vt = v + (tok * Hv + h) * dv;
        const double a = alpha[tok * Hv + h];
        const double b = beta[tok * Hv + h];

        /* step 1: S <- alpha_t S */
        for (int i = 0; i < dv; ++i)
            for (int j = 0; j < dk; ++j)
                S[(long)i * dk + j] *= a;

        /* step 2: delta_t = beta_t (v_t - S k_t), S already decayed */
        for (int i = 0; i < dv; ++i) {
            double acc = 0.0;
            for (int j = 0; j < dk; ++j)
                acc += S[(long)i * dk + j] * kt[j];
            Sk[i] = acc;
        }
        for (int i = 0; i < dv; ++i)
            delta[i] = b * (vt[i] - Sk[i]);

        /* step 3: S <- S + delta_t k_t^T */
        for (int i = 0; i < dv; ++i)
            for (int j = 0; j < dk; ++j)
                S[(long)i * dk + j] += delta[i] * kt[j];

        /* step 4: o_t = S (scale q_t), S updated */
        double *ot = o + (tok * Hv + h) * dv;
        for (int i = 0; i < dv; ++i) {
            double acc = 0.0;
            for (int j = 0; j < dk; ++j)
                acc += S[(long)i * dk + j] * (scale * qt[j]);
            ot[i] = acc;
        }

        /* capture of token t's factors (decay, shared key, delta) */
        if (state_update != NULL && t < n_capture) {
            double *s = state_update + (long)t * slot;
            s[h] = a;
            if (h % G == 0)
                for (int j = 0; j < dk; ++j)
                    s[Hv + (long)hk * dk + j] = kt[j];
            for (int i = 0; i < dv; ++i)
                s[Hv + (long)Hk * dk + (long)h * dv + i] = delta[i];
        }
    }
    free(Sk);
    free(delta);
}

/* ---------------------------------------------------------------------- */
/* Replay: S <- decay * S + outer(delta, key) for the first m slots.        */
/* ---------------------------------------------------------------------- */

/*
 * The replay identity of the capture contract.  With S stored [dv, dk] the
 * outer product's (i, j) entry is delta[i] * key[j].
 */
void gdn_oracle_replay_unit(double *S, const double *state_update, int m,
                            int Hk, int Hv, int dk, int dv, int h)
{
    const int G = Hv / Hk;
    const int hk = h / G;
    const long slot = (long)Hv + (long)Hk * dk + (long)Hv * dv;
    for (int t = 0; t < m; ++t) {
        const double *s = state_update + (long)t * slot;
        const double decay = s[h];
        const double *key = s + Hv + (long)hk * dk;
        const double *delta = s + Hv + (long)Hk * dk + (long)h * dv;
        for (int i = 0; i < dv; ++i)
            for (int j = 0; j < dk; ++j)
                S[(long)i * dk + j] = decay * S[(long)i * dk + j] + delta[i] * key[j];
    }
}

/* ---------------------------------------------------------------------- */
/* Chunked form (UT / WY), written independently of the recurrent form.     */
/* ---------------------------------------------------------------------- */

/*
 * Chunk-parallel restatement of the same recurrence.  Inside a chunk of n
 * tokens with start state S0 and local log-decay sums g_t = sum_{s<=t} log
 * alpha_s (gamma_t = exp(g_t)), unrolling the recurrence gives
 *   S_t = gamma_t S0 + sum_{i<=t} (gamma_t / gamma_i) delta_i k_i^T,
 * hence, for the n x dv matrix Delta whose rows are delta_t,
 *   (I + A) Delta = diag(beta) V - diag(beta gamma) K S0^T,
 *   A[t][i] = beta_t (gamma_t / gamma_i) (k_t . k_i)   for i < t, else 0,
 * i.e. Delta = U - W S0^T with U = T diag(beta) V, W = T diag(beta gamma) K,
 * T = (I + A)^{-1};  the outputs and the end-of-chunk state are
 *   o_t   = gamma_t S0 q_t + sum_{i<=t} (gamma_t/gamma_i)(k_i . q_t) delta_i,
 *   S_end = gamma_n S0 + sum_i (gamma_n / gamma_i) delta_i k_i^T.
 * The last chunk of a row simply has fewer tokens.  Every alpha must be > 0
 * (the log-decay needs it).  T is formed explicitly by forward substitution.
 */
void gdn_oracle_chunked_unit(const double *q, const double *k, const double *v,
                             const double *alpha, const double *beta,
                             long tok0, int T_b, int Hk, int Hv, int dk, int dv,
                             int h, double scale, int chunk, double *S, double *o)
{
    const int G = Hv / Hk;
    const int hk = h / G;
    const int C = chunk;
    double *g = (double *)malloc(sizeof(double) * C);
    double *A = (double *)malloc(sizeof(double) * C * C);
    double *Tinv = (double *)malloc(sizeof(double) * C * C);
    double *U = (double *)malloc(sizeof(double) * C * dv);
    double *W = (double *)malloc(sizeof(double) * C * dk);
    double *Delta = (double *)malloc(sizeof(double) * C * dv);
    double *Snew = (double *)malloc(sizeof(double) * dv * dk);

    for (int c0 = 0; c0 < T_b; c0 += C) {
        const int n = (T_b - c0 < C) ? (T_b - c0) : C;
#define KROW(t) (k + ((tok0 + c0 + (t)) * Hk + hk) * dk)
#define QROW(t) (q + ((tok0 + c0 + (t)) * Hk + hk) * dk)
#define VROW(t) (v + ((tok0 + c0 + (t)) * Hv + h) * dv)
#define ALPHA(t) (alpha[(tok0 + c0 + (t)) * Hv + h])
#define BETA(t) (beta[(tok0 + c0 + (t)) * Hv + h])

        /* cumulative log decay */
        double run = 0.0;
        for (int t = 0; t < n; ++t) {
            run += log(ALPHA(t));
            g[t] = run;
        }

        /* A, strictly lower triangular */
        for (int t = 0; t < n; ++t)
            for (int i = 0; i < n; ++i) {
                double val = 0.0;
                if (i < t) {
                    double kk = 0.0;
                    for (int j = 0; j < dk; ++j)
                        kk += KROW(t)[j] * KROW(i)[j];
                    val = BETA(t) * exp(g[t] - g[i]) * kk;
                }
                A[t * C + i] = val;
            }

        /* Tinv = (I + A)^{-1} by forward substitution, column by column:
           row t of (I + A) X = I reads X[t] = e_t - sum_{i<t} A[t][i] X[i]. */
        for (int col = 0; col < n; ++col)
            for (int t = 0; t < n; ++t) {
                double x = (t == col) ? 1.0 : 0.0;
                for (int i = 0; i < t; ++i)
                    x -= A[t * C + i] * Tinv[i * C + col];
                Tinv[t * C + col] = x;
            }

        /* U = Tinv diag(beta) V,  W = Tinv diag(beta gamma) K */
        for (int t = 0; t < n; ++t) {
            for (int i = 0; i < dv; ++i) {
                double acc = 0.0;
                for (int s = 0; s < n; ++s)
                    acc += Tinv[t * C + s] * BETA(s) * VROW(s)[i];
                U[t * dv + i] = acc;
            }
            for (int j = 0; j < dk; ++j) {
                double acc = 0.0;
                for (int s = 0; s < n; ++s)
                    acc += Tinv[t * C + s] * BETA(s) * exp(g[s]) * KROW(s)[j];
                W[t * dk + j] = acc;
            }
        }

        /* Delta = U - W S0^T */
        for (int t = 0; t < n; ++t)
            for (int i = 0; i < dv; ++i) {
                double ws = 0.0;
                for (int j = 0; j < dk; ++j)
                    ws += W[t * dk + j] * S[(long)i * dk + j];
                Delta[t * dv + i] = U[t * dv + i] - ws;
            }

        /* outputs of the chunk (q scaled by `scale`) */
        for (int t = 0; t < n; ++t) {
            double *ot = o + ((tok0 + c0 + t) * Hv + h) * dv;
            for (int i = 0; i < dv; ++i) {
                double inter = 0.0;
                for (int j = 0; j < dk; ++j)
                    inter += S[(long)i * dk + j] * QROW(t)[j];
                double intra = 0.0;
                for (int s = 0; s <= t; ++s) {
                    double kq = 0.0;
                    for (int j = 0; j < dk; ++j)
                        kq += KROW(s)[j] * QROW(t)[j];
                    intra += exp(g[t] - g[s]) * kq * Delta[s * dv + i];
                }
                ot[i] = scale * (exp(g[t]) * inter + intra);
            }
        }

        /* state at the end of the chunk */
        for (int i = 0; i < dv; ++i)
            for (int j = 0; j < dk; ++j) {
                double acc = exp(g[n - 1]) * S[(long)i * dk + j];
                for (int s = 0; s < n; ++s)
                    acc += exp(g[n - 1] - g[s]) * Delta[s * dv + i] * KROW(s)[j];
                Snew[(long)i * dk + j] = acc;
            }
        memcpy(S, Snew, sizeof(double) * dv * dk);
#undef KROW
#undef QROW
#undef VROW
#undef ALPHA
#undef BETA
    }
    free(g);
    free(A);
    free(Tinv);
    free(U);
    free(W);
    free(Delta);
    free(Snew);
}
