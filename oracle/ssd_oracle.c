/*
 * CPU oracle for the SSD forward scan -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the package's smoke check and the benchmark's CPU-baseline
 * leg may load this library.  The CUDA path never calls it, links it or
 * shares code with it.
 *
 * What it computes (plain fp64, one token at a time, no blocking or fusion):
 * the selective state-space recurrence of Mamba-2's SSD layer.  For every
 * sequence s and head h (group g = h / (H / G)), with state S in R^{P x N}
 * starting at initial_states[s, h] (or 0), for each token t in order
 *
 *     S      <- exp(dt_t * A_h) * S + dt_t * (x_t (outer) B_{t,g})
 *     y_t[p]  = sum_n S[p, n] * C_{t,g}[n] + D_h * x_t[p]
 *
 * and final_states[s, h] = S after the sequence's last token.
 *
 * Sources.  The selective SSM with input-dependent B, C, Delta and the
 * recurrence h_t = Abar h_{t-1} + Bbar x_t, y_t = C_t h_t: Mamba-1
 * walkthrough "Mamba: Linear-Time Sequence Modeling with Selective State
 * Spaces", section 三(二) "引入选择机制到 SSM 中".  Abar = exp(Delta * A):
 * same page, section 三 3 "选择机制中各参数的解释与扩展" (the A paragraph).
 * One scalar A per head, Bbar = dt * B (not ZOH), y read from the updated
 * state, the D skip term, and heads mapping to B/C groups contiguously are
 * the readings taken where the pages are silent (the pages' ZOH formula was
 * lost in extraction); each is listed with its reason in the design notes.
 * Packed variable-length sequences are independent and start from their own
 * initial state: QbitAI article "新架构Mamba更新二代！", section
 * "Mamba-2：更强学习能力，更快训练推理" (variable sequence length), and the
 * boundary-resetting intuition of the Mamba-1 walkthrough, section 三 2.3
 * "边界重置".
 *
 * Layouts (row-major, contiguous): x, y (batch, L, H, P); dt (batch, L, H);
 * A, D (H); B, C (batch, L, G, N); initial/final states (nseq, H, P, N).
 * Without cu_seqlens, sequence s is batch row s (nseq == batch).  With
 * cu_seqlens (int32[nseq+1], batch == 1) sequence s is tokens
 * [cu[s], cu[s+1]) of the single row.
 *
 * Parallelism: OpenMP over independent (sequence, head) units only.
 *
 * The `mutation` argument of ssd_oracle_recurrent_mut() exists so that tests
 * can plant a known mistake in the ORACLE and check that the pins catch it;
 * it is 0 in every other use.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum {
    MUT_NONE = 0,
    MUT_Y_FROM_OLD_STATE = 1,  /* y_t read from S before the update        */
    MUT_DECAY_SIGN = 2,        /* exp(-dt*A) instead of exp(dt*A)           */
    MUT_GROUP_MAP = 3,         /* group g = h % G instead of h / (H/G)      */
    MUT_DROP_D = 4,            /* D term dropped                            */
    MUT_DROP_DT_INPUT = 5,     /* input term x (outer) B without the dt     */
    MUT_NO_RESET = 6           /* state carried across packed sequences    */
};

static int oracle_impl(int64_t batch, int64_t seqlen, int nheads, int headdim,
                       int dstate, int ngroups, int nseq,
                       const int32_t *cu_seqlens, const double *x,
                       const double *dt, const double *A, const double *B,
                       const double *C, const double *D, const double *init,
                       double *y, double *final_states, const int32_t *units,
                       int nunits, int nthreads, int mutation)
{
    if (batch < 1 || seqlen < 0 || nheads < 1 || headdim < 1 || dstate < 1 ||
        ngroups < 1 || nheads % ngroups != 0 || nseq < 1)
        return 1;
    if (cu_seqlens) {
        if (batch != 1 || cu_seqlens[0] != 0 || cu_seqlens[nseq] != seqlen)
            return 1;
        for (int s = 0; s < nseq; ++s)
            if (cu_seqlens[s + 1] < cu_seqlens[s]) return 1;
    } else if (nseq != batch) {
        return 1;
    }
    const int H = nheads, P = headdim, N = dstate, G = ngroups;
    const int heads_per_group = H / G;
    const int64_t total_units = (int64_t)nseq * H;
    const int64_t nwork = units ? nunits : total_units;

#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif

    int bad = 0;
#pragma omp parallel
    {
        double *S = (double *)malloc(sizeof(double) * (size_t)P * N);
        if (!S) {
#pragma omp atomic write
            bad = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t w = 0; w < nwork; ++w) {
            if (!S) continue;
            const int64_t u = units ? units[w] : w;
            if (u < 0 || u >= total_units) {
#pragma omp atomic write
                bad = 1;
                continue;
            }
            const int s = (int)(u / H), h = (int)(u % H);
            int g = h / heads_per_group;
            if (mutation == MUT_GROUP_MAP) g = h % G;
            /* token range of this sequence inside its batch row */
            int64_t row = cu_seqlens ? 0 : s;
            int64_t t0 = cu_seqlens ? cu_seqlens[s] : 0;
            int64_t t1 = cu_seqlens ? cu_seqlens[s + 1] : seqlen;
            if (init)
                memcpy(S, init + ((int64_t)s * H + h) * P * N,
                       sizeof(double) * (size_t)P * N);
            else
                memset(S, 0, sizeof(double) * (size_t)P * N);
            for (int64_t t = t0; t < t1; ++t) {
                const int64_t tok = row * seqlen + t;
                const double *xt = x + (tok * H + h) * P;
                const double *Bt = B + (tok * G + g) * N;
                const double *Ct = C + (tok * G + g) * N;
                const double dtt = dt[tok * H + h];
                const double decay =
                    exp((mutation == MUT_DECAY_SIGN ? -1.0 : 1.0) * dtt * A[h]);
                const double dscale = (mutation == MUT_DROP_DT_INPUT) ? 1.0 : dtt;
                const double Dh = (D && mutation != MUT_DROP_D) ? D[h] : 0.0;
                double *yt = y + (tok * H + h) * P;
                for (int p = 0; p < P; ++p) {
                    double *Sp = S + (int64_t)p * N;
                    double acc = 0.0;
                    if (mutation == MUT_Y_FROM_OLD_STATE)
                        for (int n = 0; n < N; ++n) acc += Sp[n] * Ct[n];
                    const double ux = dscale * xt[p];
                    for (int n = 0; n < N; ++n) Sp[n] = decay * Sp[n] + ux * Bt[n];
                    if (mutation != MUT_Y_FROM_OLD_STATE)
                        for (int n = 0; n < N; ++n) acc += Sp[n] * Ct[n];
                    yt[p] = acc + Dh * xt[p];
                }
            }
            if (final_states)
                memcpy(final_states + ((int64_t)s * H + h) * P * N, S,
                       sizeof(double) * (size_t)P * N);
        }
        free(S);
    }
    return bad ? 2 : 0;
}

/*
 * No-reset mutation: treat the packed row as one sequence (state carried
 * across cu_seqlens boundaries, first sequence's initial state only).  Only
 * y is written; final_states is left untouched.
 */
static int oracle_no_reset(int64_t seqlen, int H, int P, int N, int G, int nseq,
                           const int32_t *cu, const double *x, const double *dt,
                           const double *A, const double *B, const double *C,
                           const double *D, const double *init, double *y,
                           double *final_states)
{
    int rc = oracle_impl(1, seqlen, H, P, N, G, 1, NULL, x, dt, A, B, C, D,
                         init, y, NULL, NULL, 0, 0, MUT_NONE);
    (void)cu; (void)nseq; (void)final_states;
    return rc;
}

int ssd_oracle_recurrent(int64_t batch, int64_t seqlen, int nheads, int headdim,
                         int dstate, int ngroups, int nseq,
                         const int32_t *cu_seqlens, const double *x,
                         const double *dt, const double *A, const double *B,
                         const double *C, const double *D, const double *init,
                         double *y, double *final_states, const int32_t *units,
                         int nunits, int nthreads)
{
    return oracle_impl(batch, seqlen, nheads, headdim, dstate, ngroups, nseq,
                       cu_seqlens, x, dt, A, B, C, D, init, y, final_states,
                       units, nunits, nthreads, MUT_NONE);
}

int ssd_oracle_recurrent_mut(int64_t batch, int64_t seqlen, int nheads,
                             int headdim, int dstate, int ngroups, int nseq,
                             const int32_t *cu_seqlens, const double *x,
                             const double *dt, const double *A, const double *B,
                             const double *C, const double *D,
                             const double *init, double *y,
                             double *final_states, int mutation)
{
    if (mutation == MUT_NO_RESET && cu_seqlens)
        return oracle_no_reset(seqlen, nheads, headdim, dstate, ngroups, nseq,
                               cu_seqlens, x, dt, A, B, C, D, init, y,
                               final_states);
    return oracle_impl(batch, seqlen, nheads, headdim, dstate, ngroups, nseq,
                       cu_seqlens, x, dt, A, B, C, D, init, y, final_states,
                       NULL, 0, 0, mutation);
}

int ssd_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
