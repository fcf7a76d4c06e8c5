/*
 * Oracle for the Mamba-2 SSD forward: the plain token-by-token recurrence in
 * fp64 on the CPU.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the checker, not the product: only
 * the tests, the smoke check and the benchmark's CPU-baseline leg may load
 * it. It shares no code with the CUDA path.
 *
 * What it computes (per batch b and head h, with group g = h / (nheads/ngroups)):
 *
 *   s_{-1}  = init_state[b,h]                 (zeros when init_state is NULL)
 *   for t = 0 .. L-1:
 *     if seq_idx given and t > 0 and seq_idx[b,t] != seq_idx[b,t-1]: s_{t-1} = 0
 *     delta_t = clamp(softplus(dt[b,t,h] + dt_bias[h]), dt_min, dt_max)
 *     s_t     = exp(delta_t * A[h]) * s_{t-1} + delta_t * x[b,t,h,:] (outer) B[b,t,g,:]
 *     y[b,t,h,:] = s_t . C[b,t,g,:] + D[h] * x[b,t,h,:]
 *   final_state[b,h] = s_{L-1}
 *
 * Sources (the pages' own statements of the method):
 *   - lrnnx "ops/selective_scan.html", selective_scan_ref: the sequential scan
 *     loop (state update first, then the C readout of the updated state, then
 *     the D skip), with delta = softplus(delta + delta_bias) and the "mamba"
 *     discretisation exp(delta*A) for the decay and delta*B*u for the input.
 *   - flash-linear-attention "fla/layers/mamba2.py", Mamba2.torch_forward,
 *     single-token branch: state*exp(dt*A) + dt*B*x, readout state.C + D*x;
 *     dt = softplus(dt + dt_bias), then torch.clamp to time_step_limit
 *     (lower bound first, then upper; the default (0, inf) changes nothing),
 *     the same clamp the naive chunked branch applies and the fused branch
 *     passes on as dt_limit.
 *   - Group map head -> group = head / (nheads/ngroups): burn-mamba
 *     "mamba2/ssd/serial.rs", ssd_serial (heads_per_group).
 *   - seq_idx (packed sequences): flash-linear-attention "fla/layers/mamba2.py"
 *     passes seq_idx to the fused chunked scan, the one place it appears; the
 *     pages never spell out what it does. Reading taken: tokens of one row
 *     whose seq_idx differ belong to different sequences, so no state crosses
 *     a change of seq_idx between consecutive tokens: the state restarts from
 *     zero there. init_state is the state before the row's first token (its
 *     first sequence); final_state is the state after the row's last token.
 *
 * Precision: inputs are fp32 arrays (bf16 inputs arrive widened, exactly);
 * every operation is done in fp64. softplus(v) = log1p(exp(v)), evaluated as
 * v + log1p(exp(-v)) for v > 0 to avoid overflow.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int64_t batch, seqlen, nheads, headdim, ngroups, dstate;
    const float *x, *dt, *dt_bias, *A, *B, *C, *D, *init_state;
    const int32_t *seq_idx; /* [batch, seqlen] or NULL */
    double dt_min, dt_max;
    int64_t nsel;
    const int64_t *sel_b, *sel_h;
    double *y_sel;      /* [nsel, seqlen, headdim] */
    double *final_sel;  /* [nsel, headdim, dstate] */
    int64_t next;       /* work counter (guarded by lock) */
    pthread_mutex_t lock;
} oracle_job;

static double softplus(double v) {
    return v > 0.0 ? v + log1p(exp(-v)) : log1p(exp(v));
}

/* One (b, h) chain, all L tokens. s is a [headdim, dstate] scratch. */
static void run_chain(const oracle_job *j, int64_t k, double *s) {
    const int64_t b = j->sel_b[k], h = j->sel_h[k];
    const int64_t L = j->seqlen, H = j->nheads, P = j->headdim, N = j->dstate, G = j->ngroups;
    const int64_t g = h / (H / G);
    const double a_h = (double)j->A[h];
    const double bias_h = (double)j->dt_bias[h];
    const double d_h = j->D ? (double)j->D[h] : 0.0;

    if (j->init_state) {
        const float *s0 = j->init_state + (b * H + h) * P * N;
        for (int64_t i = 0; i < P * N; ++i) s[i] = (double)s0[i];
    } else {
        memset(s, 0, sizeof(double) * (size_t)(P * N));
    }

    double *y = j->y_sel ? j->y_sel + k * L * P : NULL;
    const int32_t *seq = j->seq_idx ? j->seq_idx + b * L : NULL;
    for (int64_t t = 0; t < L; ++t) {
        if (seq && t > 0 && seq[t] != seq[t - 1])
            memset(s, 0, sizeof(double) * (size_t)(P * N)); /* a new sequence starts from zero */
        double delta = softplus((double)j->dt[(b * L + t) * H + h] + bias_h);
        if (delta < j->dt_min) delta = j->dt_min;
        if (delta > j->dt_max) delta = j->dt_max;
        const double decay = exp(delta * a_h);
        const float *xt = j->x + ((b * L + t) * H + h) * P;
        const float *Bt = j->B + ((b * L + t) * G + g) * N;
        const float *Ct = j->C + ((b * L + t) * G + g) * N;
        for (int64_t p = 0; p < P; ++p) {
            const double xp = (double)xt[p];
            const double u = delta * xp;
            double *sp = s + p * N;
            double acc = 0.0;
            for (int64_t n = 0; n < N; ++n) {
                sp[n] = decay * sp[n] + u * (double)Bt[n];
                acc += sp[n] * (double)Ct[n];
            }
            if (y) y[t * P + p] = acc + d_h * xp;
        }
    }
    if (j->final_sel) memcpy(j->final_sel + k * P * N, s, sizeof(double) * (size_t)(P * N));
}

static void *worker(void *arg) {
    oracle_job *j = (oracle_job *)arg;
    double *s = (double *)malloc(sizeof(double) * (size_t)(j->headdim * j->dstate));
    if (!s) return (void *)1;
    for (;;) {
        pthread_mutex_lock(&j->lock);
        const int64_t k = j->next++;
        pthread_mutex_unlock(&j->lock);
        if (k >= j->nsel) break;
        run_chain(j, k, s);
    }
    free(s);
    return NULL;
}

/*
 * Runs the recurrence for the selected (b, h) chains (every token of each),
 * with softplus(dt + dt_bias) clamped to [dt_min, dt_max] (0, INFINITY: none)
 * and, when seq_idx [batch, seqlen] is given, the state reset to zero wherever
 * seq_idx changes between consecutive tokens of a row.
 * Returns 0 on success, -1 on invalid arguments, -2 on allocation/thread failure.
 * y_sel or final_sel may be NULL to skip that output.
 */
int ssd_oracle_recurrence(int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim,
                          int64_t ngroups, int64_t dstate,
                          const float *x, const float *dt, const float *dt_bias, const float *A,
                          const float *B, const float *C, const float *D,
                          const float *init_state,
                          int64_t nsel, const int64_t *sel_b, const int64_t *sel_h,
                          double *y_sel, double *final_sel, int nthreads,
                          double dt_min, double dt_max, const int32_t *seq_idx) {
    if (batch < 1 || seqlen < 1 || nheads < 1 || headdim < 1 || ngroups < 1 || dstate < 1)
        return -1;
    if (nheads % ngroups != 0) return -1;
    if (!x || !dt || !dt_bias || !A || !B || !C || nsel < 0 || (nsel > 0 && (!sel_b || !sel_h)))
        return -1;
    for (int64_t k = 0; k < nsel; ++k)
        if (sel_b[k] < 0 || sel_b[k] >= batch || sel_h[k] < 0 || sel_h[k] >= nheads) return -1;

    oracle_job j;
    j.batch = batch; j.seqlen = seqlen; j.nheads = nheads; j.headdim = headdim;
    j.ngroups = ngroups; j.dstate = dstate;
    j.x = x; j.dt = dt; j.dt_bias = dt_bias; j.A = A; j.B = B; j.C = C; j.D = D;
    j.init_state = init_state;
    j.seq_idx = seq_idx;
    j.dt_min = dt_min; j.dt_max = dt_max;
    j.nsel = nsel; j.sel_b = sel_b; j.sel_h = sel_h;
    j.y_sel = y_sel; j.final_sel = final_sel;
    j.next = 0;
    pthread_mutex_init(&j.lock, NULL);

    if (nthreads < 1) nthreads = 1;
    if (nthreads > nsel) nthreads = nsel > 0 ? (int)nsel : 1;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    if (!th) { pthread_mutex_destroy(&j.lock); return -2; }
    int started = 0, rc = 0;
    for (int i = 0; i < nthreads; ++i) {
        if (pthread_create(&th[i], NULL, worker, &j) != 0) { rc = -2; break; }
        ++started;
    }
    for (int i = 0; i < started; ++i) {
        void *ret = NULL;
        pthread_join(th[i], &ret);
        if (ret) rc = -2;
    }
    if (started == 0) rc = -2;
    free(th);
    pthread_mutex_destroy(&j.lock);
    return rc;
}
