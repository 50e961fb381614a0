/*
 * ssm_oracle.c -- plain, sequential, double-precision CPU oracle for the selective
 * state-space scan (Mamba "S6") and its single-token recurrent state update.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the benchmark's CPU
 * baseline may load this file's library. It shares no code, header, table or helper with
 * the CUDA path, and the CUDA path never calls it.
 *
 * What it computes: the definition of the discretised selective state-space model, in
 * double, one timestep after another (no blocking, no reordering, no parallel algorithm).
 * The equations, per batch row b, channel d and state n, for t = 0, 1, ..., L-1:
 *
 *   (1) step        dt_t = softplus(delta_t + bias)        input-dependent step; bias added
 *                                                           before the softplus (lmnt.cn
 *                                                           "From RNN to Mamba", section 3.3)
 *   (2) discretise  A_bar_t[n] = exp(dt_t * A[n])           A diagonal, so the matrix
 *                   B_bar_t[n] = dt_t * B_t[n]              exponential is elementwise
 *                                                           (same page, sections 2.2, 3.2)
 *   (3) recurrence  h_t[n] = A_bar_t[n] h_{t-1}[n] + B_bar_t[n] u_t,   h_{-1} = 0
 *   (4) readout     y_t = sum_n C_t[n] h_t[n] + D u_t,  then y_t * SiLU(z_t)
 *                                                           (section 3.2: output C h plus
 *                                                           the D skip term, gated by z)
 *
 * Section 5.3 of the same page: recurrent inference keeps one fixed-size fp32 state per
 * channel and advances it one token at a time -- that is oracle_state_update below, the
 * same equations (2)-(4) for one step with the (already positive) step given directly.
 *
 * Readings where the pages are silent or disagree (each also listed in the design notes):
 *   - B_bar = dt * B (the page's code) by default. The exact zero-order-hold variant of
 *     "Mamba architecture principles and industrial long-text practice" (jsqmd.com, section
 *     2.3) and of the Mamba paper notes (section 3.2), B_bar = (exp(dt*A) - 1)/A * B, is
 *     selected with zoh != 0 and computed as dt*B * phi(dt*A), phi(x) = expm1(x)/x, phi(0) = 1
 *     (the A -> 0 limit is the Euler step).
 *   - softplus is log1p(exp(v)) with the common pass-through for v > 20 (beta = 1).
 *   - y_t reads the state AFTER the update at t (the page's code updates, then reads).
 *   - A is a real diagonal (per channel, per state); B and C are shared by all channels
 *     of a batch row; the state starts at zero unless h0 is given (h0 is an oracle-only
 *     extension used to check that a split scan equals the whole scan).
 *
 * Besides y and the final state the oracle can return a "magnitude companion": the same
 * recurrence run on absolute values (hm = A_bar*hm + |B_bar*x|, s = (sum|C|*hm + |D*x|)
 * * |SiLU(z)|). It bounds every term that enters y and is the denominator of the parity
 * error metric, so that outputs that cancel to near zero are judged against the size of
 * the terms that produced them.
 */
#include <math.h>
#include <pthread.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>

static double softplus(double v) { return v > 20.0 ? v : log1p(exp(v)); }
static double silu(double v) { return v / (1.0 + exp(-v)); }
/* expm1(x)/x, the factor that turns dt*B into the zero-order-hold B_bar; 1 at x = 0 */
static double zoh_factor(double x) { return x == 0.0 ? 1.0 : expm1(x) / x; }

/* One channel: equations (1)-(4) above, one timestep after another. */
static void scan_one_channel(int64_t L, int64_t N,
                             const double *u, const double *delta, const double *A,
                             const double *B, const double *C, /* [N][L] of this batch row */
                             int has_D, double Dval, const double *z,
                             int has_bias, double bias, int use_softplus, int zoh,
                             const double *h0, double *h, double *hm,
                             double *y, double *ymag) {
    for (int64_t n = 0; n < N; ++n) {
        h[n] = h0 ? h0[n] : 0.0;
        hm[n] = h0 ? fabs(h0[n]) : 0.0;
    }
    for (int64_t t = 0; t < L; ++t) {
        double dt = delta[t] + (has_bias ? bias : 0.0);
        if (use_softplus) dt = softplus(dt);
        double x = u[t];
        double acc = 0.0, accm = 0.0;
        for (int64_t n = 0; n < N; ++n) {
            double A_bar = exp(dt * A[n]);
            double B_bar = dt * B[n * L + t];
            if (zoh) B_bar *= zoh_factor(dt * A[n]);
            h[n] = A_bar * h[n] + B_bar * x;
            hm[n] = A_bar * hm[n] + fabs(B_bar * x);
            acc += h[n] * C[n * L + t];
            accm += hm[n] * fabs(C[n * L + t]);
        }
        double yt = acc + (has_D ? x * Dval : 0.0);
        double st = accm + (has_D ? fabs(x * Dval) : 0.0);
        if (z) {
            double g = silu(z[t]);
            yt *= g;
            st *= fabs(g);
        }
        y[t] = yt;
        if (ymag) ymag[t] = st;
    }
}

typedef struct {
    int64_t nchan, L, N;
    const double *u, *delta, *A, *B, *C, *Dskip, *z, *dbias, *h0;
    const int64_t *bidx;
    int softplus, zoh;
    double *y, *ymag, *hlast, *hmag;
    int tid, nthreads;
    int status;
} scan_job_t;

static void *scan_worker(void *arg) {
    scan_job_t *j = (scan_job_t *)arg;
    double *h = (double *)malloc(sizeof(double) * (size_t)j->N);
    double *hm = (double *)malloc(sizeof(double) * (size_t)j->N);
    if (!h || !hm) {
        free(h);
        free(hm);
        j->status = 2;
        return NULL;
    }
    for (int64_t c = j->tid; c < j->nchan; c += j->nthreads) {
        const int64_t b = j->bidx[c];
        const double *Bb = j->B + b * j->N * j->L;
        const double *Cb = j->C + b * j->N * j->L;
        scan_one_channel(j->L, j->N, j->u + c * j->L, j->delta + c * j->L, j->A + c * j->N,
                         Bb, Cb, j->Dskip != NULL, j->Dskip ? j->Dskip[c] : 0.0,
                         j->z ? j->z + c * j->L : NULL, j->dbias != NULL,
                         j->dbias ? j->dbias[c] : 0.0, j->softplus, j->zoh,
                         j->h0 ? j->h0 + c * j->N : NULL, h, hm, j->y + c * j->L,
                         j->ymag ? j->ymag + c * j->L : NULL);
        for (int64_t n = 0; n < j->N; ++n) {
            if (j->hlast) j->hlast[c * j->N + n] = h[n];
            if (j->hmag) j->hmag[c * j->N + n] = hm[n];
        }
    }
    free(h);
    free(hm);
    j->status = 0;
    return NULL;
}

/*
 * Scan a list of channels. Every per-channel array is packed by channel ("rows"):
 *   u, delta, z, y, ymag : [nchan][L]      A, h0, hlast, hmag : [nchan][N]
 *   Dskip, dbias         : [nchan]          (NULL = absent)
 *   B, C                 : [nbatch][N][L]   shared by the channels of one batch row;
 *   bidx                 : [nchan]          batch row of each channel.
 * Channels are independent; with nthreads > 1 they are dealt out round-robin to threads.
 * Returns 0, or nonzero on bad arguments / allocation failure.
 */
int oracle_scan_channels_disc(int64_t nchan, int64_t L, int64_t N,
                              const double *u, const double *delta, const double *A,
                              const double *B, const double *C, const int64_t *bidx,
                              const double *Dskip, const double *z, const double *dbias,
                              int use_softplus, int zoh, const double *h0,
                              double *y, double *ymag, double *hlast, double *hmag,
                              int nthreads) {
    if (nchan < 0 || L < 0 || N < 1) return 1;
    if (nchan == 0 || L == 0) {
        for (int64_t c = 0; c < nchan; ++c)
            for (int64_t n = 0; n < N; ++n) {
                if (hlast) hlast[c * N + n] = h0 ? h0[c * N + n] : 0.0;
                if (hmag) hmag[c * N + n] = h0 ? fabs(h0[c * N + n]) : 0.0;
            }
        return 0;
    }
    if (!u || !delta || !A || !B || !C || !bidx || !y) return 1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    scan_job_t jobs[256];
    pthread_t th[256];
    for (int i = 0; i < nthreads; ++i) {
        scan_job_t j = {nchan, L, N, u, delta, A, B, C, Dskip, z, dbias, h0, bidx,
                        use_softplus, zoh, y, ymag, hlast, hmag, i, nthreads, 1};
        jobs[i] = j;
    }
    if (nthreads == 1) {
        scan_worker(&jobs[0]);
        return jobs[0].status;
    }
    int started = 0;
    for (int i = 0; i < nthreads; ++i) {
        if (pthread_create(&th[i], NULL, scan_worker, &jobs[i]) != 0) break;
        ++started;
    }
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    for (int i = started; i < nthreads; ++i) scan_worker(&jobs[i]);
    int st = 0;
    for (int i = 0; i < nthreads; ++i) st |= jobs[i].status;
    return st;
}

/* The page's Euler step B_bar = dt * B (zoh = 0). */
int oracle_scan_channels(int64_t nchan, int64_t L, int64_t N,
                         const double *u, const double *delta, const double *A,
                         const double *B, const double *C, const int64_t *bidx,
                         const double *Dskip, const double *z, const double *dbias,
                         int use_softplus, const double *h0,
                         double *y, double *ymag, double *hlast, double *hmag,
                         int nthreads) {
    return oracle_scan_channels_disc(nchan, L, N, u, delta, A, B, C, bidx, Dskip, z, dbias,
                                     use_softplus, 0, h0, y, ymag, hlast, hmag, nthreads);
}

/*
 * One recurrent inference step for every (b, d): the page's loop body for a single
 * timestep, starting from the given state, with dt already the positive step (no bias,
 * no softplus). Layouts: state, smag [Bt][D][N] (in/out); x, dt, z, y, ymag [Bt][D];
 * A [D][N]; B, C [Bt][N]; Dskip [D]. smag/ymag: magnitude companion (NULL = skip).
 */
int oracle_state_update_disc(int64_t Bt, int64_t D, int64_t N, double *state, double *smag,
                             const double *x, const double *dt, const double *A,
                             const double *B, const double *C, const double *Dskip,
                             const double *z, int zoh, double *y, double *ymag) {
    if (Bt < 0 || D < 0 || N < 1) return 1;
    if (Bt == 0 || D == 0) return 0;
    if (!state || !x || !dt || !A || !B || !C || !y) return 1;
    for (int64_t b = 0; b < Bt; ++b) {
        for (int64_t d = 0; d < D; ++d) {
            const int64_t bd = b * D + d;
            double *h = state + bd * N;
            double *hm = smag ? smag + bd * N : NULL;
            double acc = 0.0, accm = 0.0;
            for (int64_t n = 0; n < N; ++n) {
                double A_bar = exp(dt[bd] * A[d * N + n]);
                double B_bar = dt[bd] * B[b * N + n];
                if (zoh) B_bar *= zoh_factor(dt[bd] * A[d * N + n]);
                h[n] = A_bar * h[n] + B_bar * x[bd];
                acc += h[n] * C[b * N + n];
                if (hm) {
                    hm[n] = A_bar * hm[n] + fabs(B_bar * x[bd]);
                    accm += hm[n] * fabs(C[b * N + n]);
                }
            }
            double yt = acc + (Dskip ? x[bd] * Dskip[d] : 0.0);
            double st = accm + (Dskip ? fabs(x[bd] * Dskip[d]) : 0.0);
            if (z) {
                double g = silu(z[bd]);
                yt *= g;
                st *= fabs(g);
            }
            y[bd] = yt;
            if (ymag) ymag[bd] = st;
        }
    }
    return 0;
}

/* The page's Euler step for the recurrent update (zoh = 0). */
int oracle_state_update(int64_t Bt, int64_t D, int64_t N, double *state, double *smag,
                        const double *x, const double *dt, const double *A,
                        const double *B, const double *C, const double *Dskip,
                        const double *z, double *y, double *ymag) {
    return oracle_state_update_disc(Bt, D, N, state, smag, x, dt, A, B, C, Dskip, z, 0, y, ymag);
}

/*
 * The conv-to-gate span in front of the scan (lmnt.cn "From RNN to Mamba", sections 3.1-3.2:
 * nn.Conv1d(d_inner, d_inner, kernel_size=d_conv, groups=d_inner, padding=d_conv-1), the
 * output cut to the first L steps, then SiLU), per channel:
 *     u[t] = SiLU(bias + sum_{k<K} w[k] * x[t - (K-1) + k]),   x[t < 0] = 0
 * i.e. a causal depthwise correlation. Layouts: x, u [nchan][L]; w [nchan][K]; cb [nchan]
 * (NULL = no bias). Returns 0, or nonzero on bad arguments.
 */
int oracle_conv_silu(int64_t nchan, int64_t L, int64_t K, const double *x, const double *w,
                     const double *cb, double *u) {
    if (nchan < 0 || L < 0 || K < 1) return 1;
    if (nchan == 0 || L == 0) return 0;
    if (!x || !w || !u) return 1;
    for (int64_t c = 0; c < nchan; ++c) {
        for (int64_t t = 0; t < L; ++t) {
            double acc = cb ? cb[c] : 0.0;
            for (int64_t k = 0; k < K; ++k) {
                const int64_t s = t - (K - 1) + k;
                if (s >= 0) acc += w[c * K + k] * x[c * L + s];
            }
            u[c * L + t] = silu(acc);
        }
    }
    return 0;
}
