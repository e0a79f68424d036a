/*
 * fp64 CPU oracle for the linear-attention memory S_t (d_v x d_k) under the
 * gated delta rule and its special cases.
 *
 * TEST INFRASTRUCTURE ONLY.  This file defines what the GPU library must
 * compute; it is never part of the product path.  Only tests/, the smoke
 * check in __graft_entry__.py and the cpu_baseline leg of bench.py may load
 * it.  It shares no code, header or constant with the CUDA library.
 *
 * What it computes (the plain sequential definition, one token at a time):
 *
 *   mode 0  LINEAR       S_t = S_{t-1} + v_t k_t^T
 *           "Scrivere meglio nella memoria: gate e delta rule", opening
 *           equation (linear-attention accumulation) and the summary table.
 *   mode 1  DECAY        S_t = alpha_t S_{t-1} + v_t k_t^T
 *           same page, section "Dimenticare: i gate", scalar-decay equation
 *           (RetNet with a fixed gamma, Mamba-2 with a data-dependent alpha).
 *   mode 2  DELTA        S_t = S_{t-1} + beta_t (v_t - S_{t-1} k_t) k_t^T
 *           same page, section "Correggere: la delta rule", Widrow-Hoff form.
 *   mode 3  GATED_DELTA  S_t = S_{t-1} [alpha_t (I - beta_t k_t k_t^T)]
 *                              + beta_t v_t k_t^T
 *           same page, section "Unire oblio e correzione: Gated DeltaNet".
 *   mode 4  DIAG_DECAY   S_t = S_{t-1} Diag(alpha_t) + v_t k_t^T,
 *                        alpha_t in (0,1)^dk, one gate per key channel
 *           same page, section "Dimenticare: i gate", the GLA equation:
 *           the diagonal multiplies from the right, so column c of S (key
 *           channel c) decays by alpha_t[c].
 *
 * and the read-out o_t = S_t q_t with the state AFTER the update of token t
 * (opening section of the same page: "o_t = S_t q_t", S_t being the memory
 * after the first t tokens).
 *
 * The GATED_DELTA product S[alpha(I - beta k k^T)] is evaluated as
 *   alpha S - alpha beta (S k) k^T
 * i.e. the matrix S (k k^T) is formed as the outer product (S k) k^T, which
 * is the same matrix by associativity; nothing else is rearranged.
 *
 * Layouts (row-major, contiguous, all double):
 *   q, k   [B][H][T][dk]     v, o  [B][H][T][dv]
 *   alpha, beta  [B][H][T]   (ignored, and may be NULL, where the mode has
 *                             no such parameter: LINEAR ignores both, DECAY
 *                             and DIAG_DECAY ignore beta, DELTA ignores alpha)
 *   alpha for DIAG_DECAY     [B][H][T][dk]
 *   S0, ST [B][H][dv][dk]    rows are value channels, columns key channels
 *                             (o = S q); S0 == NULL means S_0 = 0.
 *
 * Every (b, h) pair is an independent sequence; OpenMP runs them in
 * parallel.  Within a sequence the loop over t is strictly sequential.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_LINEAR = 0, OR_DECAY = 1, OR_DELTA = 2, OR_GATED_DELTA = 3, OR_DIAG_DECAY = 4 };

/* One sequence: T tokens of the chosen recurrence.  Scratch w has dv slots. */
static void run_sequence(int mode, int T, int dk, int dv,
                         const double *q, const double *k, const double *v,
                         const double *alpha, const double *beta,
                         double *S, double *o, double *w)
{
    for (int t = 0; t < T; ++t) {
        const double *kt = k + (size_t)t * dk;
        const double *qt = q + (size_t)t * dk;
        const double *vt = v + (size_t)t * dv;
        const double a = (mode == OR_DECAY || mode == OR_GATED_DELTA) ? alpha[t] : 1.0;
        const double *at = mode == OR_DIAG_DECAY ? alpha + (size_t)t * dk : NULL;
        const double b = (mode == OR_DELTA || mode == OR_GATED_DELTA) ? beta[t] : 1.0;

        /* w = S_{t-1} k_t : what the memory currently returns for k_t */
        for (int r = 0; r < dv; ++r) {
            double acc = 0.0;
            for (int c = 0; c < dk; ++c) acc += S[(size_t)r * dk + c] * kt[c];
            w[r] = acc;
        }

        for (int r = 0; r < dv; ++r) {
            double *row = S + (size_t)r * dk;
            for (int c = 0; c < dk; ++c) {
                switch (mode) {
                case OR_LINEAR:       /* S + v k^T */
                    row[c] = row[c] + vt[r] * kt[c];
                    break;
                case OR_DECAY:        /* alpha S + v k^T */
                    row[c] = a * row[c] + vt[r] * kt[c];
                    break;
                case OR_DELTA:        /* S + beta (v - S k) k^T */
                    row[c] = row[c] + b * (vt[r] - w[r]) * kt[c];
                    break;
                case OR_DIAG_DECAY:   /* S Diag(alpha) + v k^T: column c scaled by alpha[c] */
                    row[c] = row[c] * at[c] + vt[r] * kt[c];
                    break;
                default:              /* alpha S - alpha beta (S k) k^T + beta v k^T */
                    row[c] = a * row[c] - a * b * w[r] * kt[c] + b * vt[r] * kt[c];
                    break;
                }
            }
        }

        /* o_t = S_t q_t, with the state that already holds token t */
        double *ot = o + (size_t)t * dv;
        for (int r = 0; r < dv; ++r) {
            double acc = 0.0;
            for (int c = 0; c < dk; ++c) acc += S[(size_t)r * dk + c] * qt[c];
            ot[r] = acc;
        }
    }
}

/*
 * Returns 0 on success, 1 on a bad argument (unknown mode, non-positive
 * size, NULL where the mode needs a pointer), 2 if scratch allocation fails.
 * ST may alias S0.
 */
int gdr_oracle_recurrent(int mode, int B, int H, int T, int dk, int dv,
                         const double *q, const double *k, const double *v,
                         const double *alpha, const double *beta,
                         const double *S0, double *o, double *ST,
                         int num_threads)
{
    if (mode < OR_LINEAR || mode > OR_DIAG_DECAY) return 1;
    if (B <= 0 || H <= 0 || T < 0 || dk <= 0 || dv <= 0) return 1;
    if (!q || !k || !v || !o || !ST) return 1;
    if ((mode == OR_DECAY || mode == OR_GATED_DELTA || mode == OR_DIAG_DECAY) && !alpha) return 1;
    if ((mode == OR_DELTA || mode == OR_GATED_DELTA) && !beta) return 1;

    const int BH = B * H;
    const size_t sz = (size_t)dv * dk;
    int failed = 0;

#ifdef _OPENMP
    if (num_threads <= 0) num_threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads) reduction(| : failed)
#endif
    for (int bh = 0; bh < BH; ++bh) {
        double *S = (double *)malloc(sz * sizeof(double));
        double *w = (double *)malloc((size_t)dv * sizeof(double));
        if (!S || !w) {
            free(S);
            free(w);
            failed |= 1;
            continue;
        }
        if (S0) memcpy(S, S0 + (size_t)bh * sz, sz * sizeof(double));
        else memset(S, 0, sz * sizeof(double));

        run_sequence(mode, T, dk, dv,
                     q + (size_t)bh * T * dk, k + (size_t)bh * T * dk,
                     v + (size_t)bh * T * dv,
                     alpha ? alpha + (size_t)bh * T * (mode == OR_DIAG_DECAY ? dk : 1) : NULL,
                     beta ? beta + (size_t)bh * T : NULL,
                     S, o + (size_t)bh * T * dv, w);

        memcpy(ST + (size_t)bh * sz, S, sz * sizeof(double));
        free(S);
        free(w);
    }
    (void)num_threads;
    return failed ? 2 : 0;
}

/*
 * mLSTM (page "Le architetture lineari: RetNet, RWKV, xLSTM", section on
 * xLSTM, the matrix-memory cell): the scalar-gate row with a write factor
 * i_t = exp(igate_t) and a normaliser,
 *
 *     C_t = f_t C_{t-1} + i_t v_t k_t^T,   n_t = f_t n_{t-1} + i_t k_t,
 *     h_t = C_t q_t / max(|n_t^T q_t|, 1),
 *
 * evaluated in the stabilised form the page takes from the authors' appendix:
 * a log-space state m_t = max(log f_t + m_{t-1}, igate_t) is subtracted
 * before exponentiating, so the stored memory is C~ = e^{-m} C, n~ = e^{-m} n,
 * and the threshold carries the same factor: h_t = C~_t q_t /
 * max(|n~_t^T q_t|, e^{-m_t}).  (The plain form lives in oracle/mlstm.py; the
 * tests pin the two against each other.)
 *
 * Layouts: q, k [B][H][T][dk]; v, h [B][H][T][dv]; logf, igate [B][H][T]
 * (log of the forget gate, <= 0, and the input-gate pre-activation);
 * C0, CT [B][H][dv][dk]; n0, nT [B][H][dk]; m0, mT [B][H].  C0, n0, m0 may
 * all be NULL for the empty memory (C = 0, n = 0, m = -inf, so that the first
 * step gives m = igate).  Returns 0, 1 on a bad argument, 2 on allocation
 * failure.
 */
int gdr_oracle_mlstm(int B, int H, int T, int dk, int dv,
                     const double *q, const double *k, const double *v,
                     const double *logf, const double *igate,
                     const double *C0, const double *n0, const double *m0,
                     double *h, double *CT, double *nT, double *mT, int num_threads)
{
    if (B <= 0 || H <= 0 || T < 0 || dk <= 0 || dv <= 0) return 1;
    if (!q || !k || !v || !logf || !igate || !h || !CT || !nT || !mT) return 1;
    if ((C0 || n0 || m0) && !(C0 && n0 && m0)) return 1;
    const int BH = B * H;
    const size_t sz = (size_t)dv * dk;
    int failed = 0;
#ifdef _OPENMP
    if (num_threads <= 0) num_threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads) reduction(| : failed)
#endif
    for (int bh = 0; bh < BH; ++bh) {
        double *C = (double *)malloc(sz * sizeof(double));
        double *n = (double *)malloc((size_t)dk * sizeof(double));
        if (!C || !n) {
            free(C);
            free(n);
            failed |= 1;
            continue;
        }
        double m;
        if (C0) {
            memcpy(C, C0 + (size_t)bh * sz, sz * sizeof(double));
            memcpy(n, n0 + (size_t)bh * dk, (size_t)dk * sizeof(double));
            m = m0[bh];
        } else {
            memset(C, 0, sz * sizeof(double));
            memset(n, 0, (size_t)dk * sizeof(double));
            m = -1.0 / 0.0;
        }
        for (int t = 0; t < T; ++t) {
            const size_t it = (size_t)bh * T + t;
            const double *qt = q + it * dk, *kt = k + it * dk, *vt = v + it * dv;
            const double lf = logf[it], ig = igate[it];
            const double m_new = (lf + m > ig) ? lf + m : ig;
            const double a = exp(lf + m - m_new), b = exp(ig - m_new);
            for (int r = 0; r < dv; ++r)
                for (int c = 0; c < dk; ++c)
                    C[(size_t)r * dk + c] = a * C[(size_t)r * dk + c] + b * vt[r] * kt[c];
            double nq = 0.0;
            for (int c = 0; c < dk; ++c) {
                n[c] = a * n[c] + b * kt[c];
                nq += n[c] * qt[c];
            }
            const double den = fabs(nq) > exp(-m_new) ? fabs(nq) : exp(-m_new);
            for (int r = 0; r < dv; ++r) {
                double acc = 0.0;
                for (int c = 0; c < dk; ++c) acc += C[(size_t)r * dk + c] * qt[c];
                h[it * dv + r] = acc / den;
            }
            m = m_new;
        }
        memcpy(CT + (size_t)bh * sz, C, sz * sizeof(double));
        memcpy(nT + (size_t)bh * dk, n, (size_t)dk * sizeof(double));
        mT[bh] = m;
        free(C);
        free(n);
    }
    (void)num_threads;
    return failed ? 2 : 0;
}

/*
 * Generalised delta rule of RWKV-7 (page "Le architetture lineari: RetNet,
 * RWKV, xLSTM", RWKV section).  The extracted page lost the update equation;
 * its prose fixes a per-channel decay w_t multiplying the state (near 1 keeps,
 * near 0 forgets), a normalised removal key kappa_t decoupled from the write
 * key kw_t, a per-channel in-context learning rate a_t, a transition that is
 * a diagonal decay plus a rank-one correction with eigenvalues in [-1, 1], and
 * the chapter's convention (S is d_v x d_k, transitions multiply from the
 * right).  Read as
 *
 *     S_t = S_{t-1} (Diag(w_t) - kappa_t (a_t * kappa_t)^T) + v_t kw_t^T,   o_t = S_t q_t,
 *
 * evaluated per value row r with s = S[r,:]:  u = s . kappa_t,
 * s <- s * w_t - u (a_t * kappa_t) + v_t[r] kw_t.
 *
 * Layouts: q, kw, w, kappa, a [B][H][T][dk]; v, o [B][H][T][dv];
 * S0, ST [B][H][dv][dk] (S0 NULL = zeros).  Returns 0, 1, or 2.
 */
int gdr_oracle_gen_delta(int B, int H, int T, int dk, int dv,
                         const double *q, const double *kw, const double *v,
                         const double *w, const double *kappa, const double *a,
                         const double *S0, double *o, double *ST, int num_threads)
{
    if (B <= 0 || H <= 0 || T < 0 || dk <= 0 || dv <= 0) return 1;
    if (!q || !kw || !v || !w || !kappa || !a || !o || !ST) return 1;
    const int BH = B * H;
    const size_t sz = (size_t)dv * dk;
    int failed = 0;
#ifdef _OPENMP
    if (num_threads <= 0) num_threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads) reduction(| : failed)
#endif
    for (int bh = 0; bh < BH; ++bh) {
        double *S = (double *)malloc(sz * sizeof(double));
        if (!S) {
            failed |= 1;
            continue;
        }
        if (S0) memcpy(S, S0 + (size_t)bh * sz, sz * sizeof(double));
        else memset(S, 0, sz * sizeof(double));
        for (int t = 0; t < T; ++t) {
            const size_t it = (size_t)bh * T + t;
            const double *qt = q + it * dk, *kt = kw + it * dk, *wt = w + it * dk;
            const double *ct = kappa + it * dk, *at = a + it * dk, *vt = v + it * dv;
            for (int r = 0; r < dv; ++r) {
                double *row = S + (size_t)r * dk;
                double u = 0.0;
                for (int c = 0; c < dk; ++c) u += row[c] * ct[c];
                double acc = 0.0;
                for (int c = 0; c < dk; ++c) {
                    row[c] = row[c] * wt[c] - u * at[c] * ct[c] + vt[r] * kt[c];
                    acc += row[c] * qt[c];
                }
                o[it * dv + r] = acc;
            }
        }
        memcpy(ST + (size_t)bh * sz, S, sz * sizeof(double));
        free(S);
    }
    (void)num_threads;
    return failed ? 2 : 0;
}

/* Number of threads an OpenMP region would use (1 without OpenMP). */
int gdr_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
