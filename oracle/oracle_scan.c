/*
 * fp64 CPU oracle for the selective scan (S6) and its single-token update.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the package's smoke check and
 * the benchmark's CPU-baseline leg may load or call this code.  The CUDA
 * library never links, includes or calls it, and it shares no code with it.
 *
 * What it computes (page "Mamba: linear-time sequence modeling with
 * selective state spaces", section "What they did", the S6 bullet and its two
 * sub-bullets; the recurrence, Euler input term, skip term and silu gate are
 * the S6 layer's definition as restated in the workload description):
 *
 *   s_t      = delta[b,d,t] + dt_bias[d]                  (dt_bias may be absent)
 *   Delta_t  = softplus(s_t)  if the softplus flag is set, else s_t
 *   Abar     = exp(Delta_t * A[d,n])                      (A input-independent)
 *   h[n]     = Abar * h[n] + Delta_t * B[b,n,t] * u[b,d,t]
 *   y[b,d,t] = (sum_n C[b,n,t] * h[n] + D_skip[d] * u[b,d,t]) * silu(z[b,d,t])
 *
 * with h = h0[b,d,:] (zero when h0 is absent) before the first step, the gate
 * skipped when z is absent, and the state after the last step returned in
 * final_state.
 *
 * With the zoh flag the input term Delta_t * B * u becomes the zero-order
 * hold one, w * B * u with w = (exp(Delta_t * A[d,n]) - 1) / A[d,n]: the
 * textbook exact discretisation of h' = A h + B x over a step of length
 * Delta_t with x held constant (for diagonal A the matrix formula
 * (Delta A)^-1 (exp(Delta A) - I) Delta B reduces to this per entry).  The
 * pages print only Abar = exp(Delta*A); this is the reading under which
 * Theorem 1 (page "Mamba: linear-time sequence modeling with selective
 * state spaces", "Main results") is exact.  w tends to Delta_t as A -> 0,
 * and A[d,n] == 0 takes that limit.  The single-token update is one step of the same recurrence
 * applied in place to a caller-held state, with softplus always applied (the
 * generation mode of page "Mamba: Linear-Time Sequence Modeling with
 * Selective State Spaces", section "Architecture": one state update per
 * token).
 *
 * Everything is plain fp64, one (b, d) row at a time, time-sequential inside
 * a row.  Rows are independent and are split statically over POSIX threads.
 * Layouts are dense row-major: u, delta, z, y (batch, dim, L); B, C
 * (batch, N, L); A (dim, N); dt_bias, D_skip (dim); h0, final_state
 * (batch, dim, N).  Inputs arrive already widened to double by the caller.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* softplus(s) = log(1 + e^s), evaluated without overflow or cancellation. */
double oracle_softplus_f64(double s)
{
    if (s > 0.0)
        return s + log1p(exp(-s));
    return log1p(exp(s));
}

/* Zero-order-hold input weight (exp(dt*a) - 1) / a, and its limit dt at
 * a == 0.  expm1 keeps full relative precision when dt*a is small. */
double oracle_zoh_weight_f64(double dt, double a)
{
    if (a == 0.0)
        return dt;
    return expm1(dt * a) / a;
}

/* silu(z) = z * sigmoid(z) = z / (1 + e^-z). */
double oracle_silu_f64(double z)
{
    return z / (1.0 + exp(-z));
}

typedef struct {
    int64_t batch, dim, dstate, seqlen;
    const double *u, *delta, *dt_bias, *A, *B, *C, *D_skip, *z, *h0;
    int softplus, zoh;
    double *y, *final_state;
    int64_t row_begin, row_end;
    int status;
} scan_job;

static void scan_rows(scan_job *j)
{
    const int64_t N = j->dstate, L = j->seqlen, D = j->dim;
    double *h = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    if (!h) {
        j->status = -1;
        return;
    }
    for (int64_t row = j->row_begin; row < j->row_end; ++row) {
        const int64_t b = row / D, d = row % D;
        const double *u = j->u + row * L;
        const double *dl = j->delta + row * L;
        const double *z = j->z ? j->z + row * L : NULL;
        const double *Bb = j->B + b * N * L;
        const double *Cb = j->C + b * N * L;
        const double *Ad = j->A + d * N;
        const double bias = j->dt_bias ? j->dt_bias[d] : 0.0;
        const double dsk = j->D_skip ? j->D_skip[d] : 0.0;
        double *y = j->y + row * L;

        for (int64_t n = 0; n < N; ++n)
            h[n] = j->h0 ? j->h0[row * N + n] : 0.0;

        for (int64_t t = 0; t < L; ++t) {
            const double s = dl[t] + bias;
            const double dt = j->softplus ? oracle_softplus_f64(s) : s;
            double acc = 0.0;
            for (int64_t n = 0; n < N; ++n) {
                const double abar = exp(dt * Ad[n]);
                const double w = j->zoh ? oracle_zoh_weight_f64(dt, Ad[n]) : dt;
                h[n] = abar * h[n] + w * Bb[n * L + t] * u[t];
                acc += Cb[n * L + t] * h[n];
            }
            double out = acc + dsk * u[t];
            if (z)
                out *= oracle_silu_f64(z[t]);
            y[t] = out;
        }
        if (j->final_state)
            for (int64_t n = 0; n < N; ++n)
                j->final_state[row * N + n] = h[n];
    }
    free(h);
    j->status = 0;
}

static void *scan_thread(void *p)
{
    scan_rows((scan_job *)p);
    return NULL;
}

static int pick_threads(int requested, int64_t rows)
{
    long n = requested > 0 ? requested : sysconf(_SC_NPROCESSORS_ONLN);
    if (n < 1)
        n = 1;
    if (n > 512)
        n = 512;
    if ((int64_t)n > rows)
        n = (long)(rows > 0 ? rows : 1);
    return (int)n;
}

/* Returns the number of threads used (>0) or a negative error code. */
int oracle_scan_f64(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
                    const double *u, const double *delta, const double *dt_bias,
                    const double *A, const double *B, const double *C,
                    const double *D_skip, const double *z, int softplus, int zoh,
                    const double *h0, double *y, double *final_state,
                    int nthreads)
{
    if (batch < 0 || dim < 0 || dstate < 0 || seqlen < 0)
        return -2;
    if (!u || !delta || !A || !B || !C || !y)
        return -1;
    const int64_t rows = batch * dim;
    const int nt = pick_threads(nthreads, rows);
    scan_job *jobs = (scan_job *)calloc((size_t)nt, sizeof(scan_job));
    pthread_t *th = (pthread_t *)calloc((size_t)nt, sizeof(pthread_t));
    if (!jobs || !th) {
        free(jobs);
        free(th);
        return -3;
    }
    for (int i = 0; i < nt; ++i) {
        scan_job *j = &jobs[i];
        j->batch = batch;
        j->dim = dim;
        j->dstate = dstate;
        j->seqlen = seqlen;
        j->u = u;
        j->delta = delta;
        j->dt_bias = dt_bias;
        j->A = A;
        j->B = B;
        j->C = C;
        j->D_skip = D_skip;
        j->z = z;
        j->h0 = h0;
        j->softplus = softplus;
        j->zoh = zoh;
        j->y = y;
        j->final_state = final_state;
        j->row_begin = rows * i / nt;
        j->row_end = rows * (i + 1) / nt;
    }
    int status = 0;
    if (nt == 1) {
        scan_rows(&jobs[0]);
        status = jobs[0].status;
    } else {
        int started = 0;
        for (int i = 0; i < nt; ++i) {
            if (pthread_create(&th[i], NULL, scan_thread, &jobs[i]) != 0)
                break;
            ++started;
        }
        for (int i = 0; i < started; ++i)
            pthread_join(th[i], NULL);
        for (int i = started; i < nt; ++i)
            scan_rows(&jobs[i]); /* thread creation failed: finish inline */
        for (int i = 0; i < nt; ++i)
            if (jobs[i].status)
                status = jobs[i].status;
    }
    free(jobs);
    free(th);
    return status ? status : nt;
}

/*
 * One generation step on a (batch, dim, N) state, in place:
 *   Delta = softplus(delta[b,d] + dt_bias[d])   (delta + dt_bias without softplus)
 *   h[n]  = exp(Delta*A[d,n]) * h[n] + w*B[b,n]*x[b,d]
 *   y     = (sum_n C[b,n]*h[n] + D_skip[d]*x[b,d]) * silu(z[b,d])
 * with w = Delta (Euler), or the zero-order-hold weight with the zoh flag.
 * x, delta, z, y are (batch, dim); B, C are (batch, N).
 */
int oracle_state_update_f64(int64_t batch, int64_t dim, int64_t dstate,
                            double *state, const double *x, const double *delta,
                            const double *dt_bias, const double *A,
                            const double *B, const double *C,
                            const double *D_skip, const double *z, int softplus, int zoh,
                            double *y)
{
    if (batch < 0 || dim < 0 || dstate < 0)
        return -2;
    if (!state || !x || !delta || !A || !B || !C || !y)
        return -1;
    const int64_t N = dstate;
    for (int64_t b = 0; b < batch; ++b) {
        for (int64_t d = 0; d < dim; ++d) {
            const int64_t row = b * dim + d;
            const double s = delta[row] + (dt_bias ? dt_bias[d] : 0.0);
            const double dt = softplus ? oracle_softplus_f64(s) : s;
            double *h = state + row * N;
            double acc = 0.0;
            for (int64_t n = 0; n < N; ++n) {
                const double a = A[d * N + n];
                const double w = zoh ? oracle_zoh_weight_f64(dt, a) : dt;
                h[n] = exp(dt * a) * h[n] + w * B[b * N + n] * x[row];
                acc += C[b * N + n] * h[n];
            }
            double out = acc + (D_skip ? D_skip[d] : 0.0) * x[row];
            if (z)
                out *= oracle_silu_f64(z[row]);
            y[row] = out;
        }
    }
    return 0;
}

/*
 * Reverse-mode gradient of oracle_scan_f64 (Euler input term), for the
 * backward pass that recomputes the state instead of storing it (page
 * "Mamba: linear-time sequence modeling with selective state spaces", "What
 * they did": the fused scan keeps the expanded state on chip and recomputes
 * it in the backward pass).  Given dy = dJ/dy and, optionally, dfinal =
 * dJ/d final_state, it returns the gradients of J with respect to every
 * input.  Written out from the chain rule on the forward loop:
 *
 *   pre_t   = sum_n C[n,t] h_t[n] + D u_t,       y_t = pre_t * silu(z_t)
 *   g_t     = dy_t * silu(z_t)                   (dy_t without z)
 *   dz_t    = dy_t * pre_t * silu'(z_t),         silu'(z) = s(z) (1 + z (1 - s(z)))
 *   dh      accumulates g_t C[:,t] at step t, then flows to step t-1 times Abar_t
 *   dB[n,t] = dh[n] Delta_t u_t   (summed over d)    dC[n,t] = g_t h_t[n]  (over d)
 *   du_t    = g_t D + sum_n dh[n] Delta_t B[n,t]
 *   dDelta  = sum_n dh[n] (A[n] Abar_t[n] h_{t-1}[n] + B[n,t] u_t)
 *   dA[n]   = sum_t dh[n] Delta_t Abar_t[n] h_{t-1}[n]   (summed over b)
 *   ddelta  = dDelta * sigmoid(s_t) with softplus (dDelta without); ddt_bias = sum of ddelta
 *   dD      = sum_t g_t u_t;   dh0 = dh after step 0
 *
 * Single-threaded; dz may be NULL when z is; dh0, dfinal, h0 nullable.
 * Accumulated outputs (dA, dB, dC, dD, ddt_bias) are zeroed first.
 */
int oracle_scan_bwd_f64(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
                        const double *u, const double *delta, const double *dt_bias,
                        const double *A, const double *B, const double *C,
                        const double *D_skip, const double *z, int softplus,
                        const double *h0, const double *dy, const double *dfinal,
                        double *du, double *ddelta, double *dA, double *dB, double *dC,
                        double *dD, double *dz, double *ddt_bias, double *dh0)
{
    if (batch < 0 || dim < 0 || dstate < 0 || seqlen < 0)
        return -2;
    if (!u || !delta || !A || !B || !C || !dy || !du || !ddelta || !dA || !dB || !dC || !dD ||
        !ddt_bias || (z && !dz))
        return -1;
    const int64_t N = dstate, L = seqlen, D = dim;
    memset(dA, 0, sizeof(double) * (size_t)(D * N));
    memset(dB, 0, sizeof(double) * (size_t)(batch * N * L));
    memset(dC, 0, sizeof(double) * (size_t)(batch * N * L));
    memset(dD, 0, sizeof(double) * (size_t)D);
    memset(ddt_bias, 0, sizeof(double) * (size_t)D);
    double *hs = (double *)malloc(sizeof(double) * (size_t)((L + 1) * (N > 0 ? N : 1)));
    double *dh = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    if (!hs || !dh) {
        free(hs);
        free(dh);
        return -3;
    }
    for (int64_t row = 0; row < batch * D; ++row) {
        const int64_t b = row / D, d = row % D;
        const double *ur = u + row * L, *dl = delta + row * L, *dyr = dy + row * L;
        const double *zr = z ? z + row * L : NULL;
        const double *Bb = B + b * N * L, *Cb = C + b * N * L, *Ad = A + d * N;
        const double bias = dt_bias ? dt_bias[d] : 0.0;
        const double dsk = D_skip ? D_skip[d] : 0.0;
        /* forward, keeping every state: hs[t*N + n] is the state before step t */
        for (int64_t n = 0; n < N; ++n)
            hs[n] = h0 ? h0[row * N + n] : 0.0;
        for (int64_t t = 0; t < L; ++t) {
            const double s = dl[t] + bias;
            const double dt = softplus ? oracle_softplus_f64(s) : s;
            for (int64_t n = 0; n < N; ++n)
                hs[(t + 1) * N + n] = exp(dt * Ad[n]) * hs[t * N + n] + dt * Bb[n * L + t] * ur[t];
        }
        for (int64_t n = 0; n < N; ++n)
            dh[n] = dfinal ? dfinal[row * N + n] : 0.0;
        for (int64_t t = L - 1; t >= 0; --t) {
            const double s = dl[t] + bias;
            const double dt = softplus ? oracle_softplus_f64(s) : s;
            const double sig = softplus ? 1.0 / (1.0 + exp(-s)) : 1.0;
            const double *ht = hs + (t + 1) * N, *hp = hs + t * N;
            double pre = dsk * ur[t];
            for (int64_t n = 0; n < N; ++n)
                pre += Cb[n * L + t] * ht[n];
            double g = dyr[t];
            if (zr) {
                const double sz = 1.0 / (1.0 + exp(-zr[t]));
                g = dyr[t] * zr[t] * sz;
                dz[row * L + t] = dyr[t] * pre * sz * (1.0 + zr[t] * (1.0 - sz));
            }
            dD[d] += g * ur[t];
            double dut = g * dsk, ddt = 0.0;
            for (int64_t n = 0; n < N; ++n) {
                const double abar = exp(dt * Ad[n]);
                dh[n] += g * Cb[n * L + t];
                dC[b * N * L + n * L + t] += g * ht[n];
                dB[b * N * L + n * L + t] += dh[n] * dt * ur[t];
                dut += dh[n] * dt * Bb[n * L + t];
                ddt += dh[n] * (Ad[n] * abar * hp[n] + Bb[n * L + t] * ur[t]);
                dA[d * N + n] += dh[n] * dt * abar * hp[n];
                dh[n] *= abar;
            }
            du[row * L + t] = dut;
            ddelta[row * L + t] = ddt * sig;
            ddt_bias[d] += ddt * sig;
        }
        if (dh0)
            for (int64_t n = 0; n < N; ++n)
                dh0[row * N + n] = dh[n];
    }
    free(hs);
    free(dh);
    return 0;
}

/*
 * Causal depthwise convolution over time with an optional SiLU: the short
 * convolution of the Mamba block's H3-derived branch, in front of the scan
 * (page "Mamba: linear-time sequence modeling with selective state spaces",
 * "What they did", Architecture bullet: the block merges the H3 block and a
 * gated MLP; the pages print no formula for it, so this is the plain
 * reading: one width-W filter per channel, causal, bias, then SiLU).
 *
 *   xp(t)      = x[b,d,t] for t >= 0, state[b,d,W-1+t] for -(W-1) <= t < 0
 *                (zero without a state)
 *   out[b,d,t] = act( bias[d] + sum_{k=0}^{W-1} w[d,k] * xp(t - (W-1) + k) )
 *
 * state (batch, dim, W-1) holds the last W-1 inputs before t = 0, oldest
 * first; state_out receives the last W-1 inputs of xp up to t = L-1.
 * Layouts: x, out (batch, dim, L); w (dim, W); bias (dim).
 */
int oracle_conv1d_f64(int64_t batch, int64_t dim, int64_t seqlen, int64_t width,
                      const double *x, const double *w, const double *bias,
                      const double *state, int silu, double *out, double *state_out)
{
    if (batch < 0 || dim < 0 || seqlen < 0 || width < 1)
        return -2;
    if (!x || !w || !out)
        return -1;
    const int64_t L = seqlen, W = width, S = width - 1;
    for (int64_t row = 0; row < batch * dim; ++row) {
        const int64_t d = row % dim;
        const double *xr = x + row * L;
        for (int64_t t = 0; t < L; ++t) {
            double acc = bias ? bias[d] : 0.0;
            for (int64_t k = 0; k < W; ++k) {
                const int64_t s = t - (W - 1) + k;
                double v;
                if (s >= 0)
                    v = xr[s];
                else
                    v = state ? state[row * S + (S + s)] : 0.0;
                acc += w[d * W + k] * v;
            }
            out[row * L + t] = silu ? oracle_silu_f64(acc) : acc;
        }
        if (state_out) {
            for (int64_t j = 0; j < S; ++j) {
                const int64_t s = L - S + j;   /* position of the j-th kept input */
                state_out[row * S + j] = s >= 0 ? xr[s] : (state ? state[row * S + (S + s)] : 0.0);
            }
        }
    }
    return 0;
}
