/*
 * Mamba-2 SSD prefill forward: the CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the plain, slow, obviously correct
 * definition that the CUDA path is checked against. Only the test suite, the
 * package smoke check and the CPU-baseline leg of the benchmark may load it.
 * It shares no code with the CUDA library (no headers, helpers or tables).
 *
 * What it computes (fp64, token by token, one independent chain per (b, h)):
 *
 *   h_{-1}     = init state (P x N, zero when absent)
 *   dt_t       = softplus(dt_raw_t + dt_bias)
 *   h_t[p][n]  = exp(dt_t * A) * h_{t-1}[p][n] + dt_t * x_t[p] * B_t[n]
 *   y_t[p]     = sum_n C_t[n] * h_t[p][n] + D * x_t[p]
 *   final      = h_{L-1}
 *
 * Sources:
 *  - "Mamba-2 state space model compiler optimisation" (bxzpzcl.cn), section
 *    1.1: the SSM h' = Ah + Bx, y = Ch + Dx, discretised per step, with A a
 *    per-head scalar and B, C, step size input dependent.
 *  - "Mamba hardware-aware algorithms" (metaphor-xennon), section "associative
 *    scan foundations": the selective linear recurrence h_t = A_t h_{t-1} +
 *    B_t x_t, y_t = C_t h_t, which the chunked SSD reproduces exactly.
 *  - Readings where the pages disagree: the decay is exp(dt*A) with A already
 *    negative and softplus applied to dt only; the input matrix is discretised
 *    as dt*B (the form the chunked SSD's L o CB^T applied to dt*x implies).
 *
 * Parity pins (in the tests, not here): hand-worked two-token examples,
 * brute-force quadratic SSD with the segsum mask, chunked == sequential for
 * every chunk size, dt = 0 identity, A = 0 cumulative-sum closed form,
 * split-and-rerun with init states, linearity, B = 0.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* softplus(v) = log(1 + e^v), evaluated without overflow in fp64. */
static double softplus(double v) {
    double a = v > 0.0 ? v : 0.0;
    return a + log1p(exp(-fabs(v)));
}

typedef struct {
    int64_t L, P, N;
    const double *x, *dt_raw, *dt_bias, *A, *B, *C, *D, *init;
    double *y, *final_states;
    int64_t first, last; /* chains [first, last) */
} job_t;

/* One chain: x [L][P], dt_raw [L], B/C [L][N], init [P][N], y [L][P], final [P][N]. */
static void run_chain(const job_t *j, int64_t c) {
    const int64_t L = j->L, P = j->P, N = j->N;
    const double *x = j->x + c * L * P;
    const double *dtr = j->dt_raw + c * L;
    const double *B = j->B + c * L * N;
    const double *C = j->C + c * L * N;
    const double A = j->A[c], bias = j->dt_bias[c];
    const double D = j->D ? j->D[c] : 0.0;
    double *y = j->y + c * L * P;
    double *h = (double *)malloc((size_t)(P * N) * sizeof(double));
    if (!h) return;
    if (j->init)
        memcpy(h, j->init + c * P * N, (size_t)(P * N) * sizeof(double));
    else
        memset(h, 0, (size_t)(P * N) * sizeof(double));
    for (int64_t t = 0; t < L; ++t) {
        const double dt = softplus(dtr[t] + bias);
        const double decay = exp(dt * A);
        const double *xt = x + t * P, *Bt = B + t * N, *Ct = C + t * N;
        for (int64_t p = 0; p < P; ++p) {
            double *hp = h + p * N;
            const double u = dt * xt[p];
            double acc = 0.0;
            for (int64_t n = 0; n < N; ++n) {
                hp[n] = decay * hp[n] + u * Bt[n];
                acc += Ct[n] * hp[n];
            }
            y[t * P + p] = acc + D * xt[p];
        }
    }
    if (j->final_states)
        memcpy(j->final_states + c * P * N, h, (size_t)(P * N) * sizeof(double));
    free(h);
}

static void *worker(void *arg) {
    const job_t *j = (const job_t *)arg;
    for (int64_t c = j->first; c < j->last; ++c) run_chain(j, c);
    return NULL;
}

/*
 * oracle_ssd_chains: run `nchains` independent chains, each given as its own
 * contiguous slices (the caller gathers x[b, :, h, :], B[b, :, g(h), :] ...).
 *   x [nchains][L][P], dt_raw [nchains][L], dt_bias/A/D [nchains],
 *   B, C [nchains][L][N], init [nchains][P][N] (NULL = zeros), D NULL = 0.
 * Outputs y [nchains][L][P], final_states [nchains][P][N] (NULL = skip).
 * Returns 0, or -1 on a bad argument. Uses up to `nthreads` threads.
 */
int oracle_ssd_chains(int64_t nchains, int64_t L, int64_t P, int64_t N,
                      const double *x, const double *dt_raw, const double *dt_bias,
                      const double *A, const double *B, const double *C,
                      const double *D, const double *init, double *y,
                      double *final_states, int nthreads) {
    if (nchains < 0 || L < 0 || P <= 0 || N <= 0 || !x || !dt_raw || !dt_bias ||
        !A || !B || !C || !y)
        return -1;
    if (nchains == 0 || L == 0) {
        if (final_states && nchains > 0) {
            if (init)
                memcpy(final_states, init, (size_t)(nchains * P * N) * sizeof(double));
            else
                memset(final_states, 0, (size_t)(nchains * P * N) * sizeof(double));
        }
        return 0;
    }
    if (nthreads < 1) nthreads = 1;
    if (nthreads > nchains) nthreads = (int)nchains;
    job_t base = {L, P, N, x, dt_raw, dt_bias, A, B, C, D, init, y, final_states, 0, 0};
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    job_t *jobs = (job_t *)malloc(sizeof(job_t) * (size_t)nthreads);
    int *running = (int *)calloc((size_t)nthreads, sizeof(int));
    if (!tid || !jobs || !running) {
        free(tid);
        free(jobs);
        free(running);
        return -1;
    }
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = base;
        jobs[t].first = nchains * t / nthreads;
        jobs[t].last = nchains * (t + 1) / nthreads;
        running[t] = pthread_create(&tid[t], NULL, worker, &jobs[t]) == 0;
        if (!running[t]) worker(&jobs[t]); /* no thread: run it here */
    }
    for (int t = 0; t < nthreads; ++t)
        if (running[t]) pthread_join(tid[t], NULL);
    free(tid);
    free(jobs);
    free(running);
    return 0;
}
