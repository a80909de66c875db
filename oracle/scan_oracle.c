/*
 * Reference oracle for the Mamba selective scan -- TEST INFRASTRUCTURE ONLY.
 *
 * This file is a plain, slow, sequential fp64 CPU restatement of the selective
 * state-space recurrence.  It exists so that the CUDA library can be checked
 * against something obviously correct.  Only the test-suite, the smoke check
 * and the benchmark's CPU-baseline leg may load it; the product path never
 * does, and it shares no code, header or constant with the CUDA sources.
 *
 * What it computes (sources are the pages' section names):
 *   - "Selective SSM" Keras layer (highthink.cn page, "Mamba 的核心创新" and the
 *     SelectiveSSM listing): A = -exp(A_log) diagonal, Abar = exp(A*dt),
 *     Bbar = B*dt, state = Abar*state + Bbar*u, y = sum_n C*state + D*u,
 *     initial state zero.
 *   - Zero-order-hold formulas and the small-step simplification Bbar ~ dt*B
 *     (luzhipeng.com tutorial, "数学基础" and step 1 "discrete_bilinear").
 *   - Input-dependent step dt = softplus(Linear(x)) with a bias on the dt
 *     projection (codechina.net overview, section 2.1; highthink.cn dt_proj
 *     with use_bias=True).
 *   - SiLU output gate on the z branch (highthink.cn "Mamba 整体架构" block
 *     diagram: the SiLU branch multiplies the SSM output).
 *   - The causal depthwise convolution (+ SiLU) in front of the scan
 *     (luzhipeng.com tutorial, step 2 nn.Conv1d with groups = d_model;
 *     highthink.cn "Mamba 整体架构": causal Conv1D then SiLU), at the end of
 *     this file.
 *   - The complex-state variant: S4D-Lin initialisation A = -0.5 + i*n and a
 *     complex state that keeps phase (codechina.net overview, section 4.1 and
 *     section 5.3), at the end of this file.
 *   - Document boundaries: Mamba isolates documents by resetting its hidden
 *     state (codechina.net overview, section 3.2, point 2 "边界控制"), and a
 *     given starting state lets a long sequence be processed block by block
 *     (the same page's deployment notes on sequences beyond 1M tokens).
 *
 * Readings taken where the pages are silent or disagree:
 *   - Bbar is the Euler form dt*B (not the exact ZOH inverse form).
 *   - dt is per (batch, channel, time).
 *   - y_t reads the state after the update at step t.
 *   - out = (sum_n C h + D u) * SiLU(z); z, D and the bias are optional.
 *   - softplus_flag == 0 uses dt = delta + bias as given.
 *   - reset[b][t] != 0 marks token t as the first of a new document: every
 *     state of every channel of batch b restarts from zero before step t.
 *     h0 (optional) is the state before step 0.
 *
 * Layouts (row-major, contiguous):
 *   u, delta, z, y : [batch][dim][seqlen]
 *   B, C           : [batch][seqlen][dstate]   (shared by all channels)
 *   A_log          : [dim][dstate]
 *   D, delta_bias  : [dim]
 *   h0, last_state : [batch][dim][dstate]
 *   reset          : [batch][seqlen] bytes (optional)
 * Every other array is double precision.  The caller widens bf16 or fp32 values.
 *
 * Parallelism: the (batch, channel) chains are independent; they are split
 * over POSIX threads.  That changes no arithmetic: every chain is evaluated in
 * exactly the order written below.
 */
#include <complex.h>
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <unistd.h>

/* softplus(x) = log(1 + e^x), written so that neither branch overflows. */
static double oracle_softplus(double x) {
    if (x > 0.0) return x + log1p(exp(-x));
    return log1p(exp(x));
}

/* SiLU(z) = z * sigmoid(z) = z / (1 + e^-z). */
static double oracle_silu(double z) { return z / (1.0 + exp(-z)); }

typedef struct {
    const double *u, *delta, *A_log, *B, *C, *D, *z, *delta_bias, *h0;
    const unsigned char *reset;
    double *y, *last_state;
    int64_t batch, dim, seqlen, dstate;
    int softplus_flag;
    int64_t chain_begin, chain_end; /* chains are b*dim + d */
} scan_job;

/* One (b, d) chain: the recurrence of the Keras listing, step by step. */
static void scan_one_chain(const scan_job *j, int64_t chain, double *h, double *A) {
    const int64_t b = chain / j->dim, d = chain % j->dim;
    const int64_t L = j->seqlen, N = j->dstate;
    const double *u = j->u + chain * L;
    const double *dl = j->delta + chain * L;
    const double *zz = j->z ? j->z + chain * L : NULL;
    const double *Bb = j->B + b * L * N;
    const double *Cb = j->C + b * L * N;
    const unsigned char *rs = j->reset ? j->reset + b * L : NULL;
    double *y = j->y + chain * L;
    const double Dd = j->D ? j->D[d] : 0.0;
    const double bias = j->delta_bias ? j->delta_bias[d] : 0.0;

    for (int64_t n = 0; n < N; ++n) {
        A[n] = -exp(j->A_log[d * N + n]);          /* A = -exp(A_log) */
        h[n] = j->h0 ? j->h0[chain * N + n] : 0.0;  /* zero initial state */
    }
    for (int64_t t = 0; t < L; ++t) {
        if (rs && rs[t])                                /* new document:      */
            for (int64_t n = 0; n < N; ++n) h[n] = 0.0; /* state restarts     */
        const double raw = dl[t] + bias;
        const double dt = j->softplus_flag ? oracle_softplus(raw) : raw;
        const double ut = u[t];
        double acc = 0.0;
        for (int64_t n = 0; n < N; ++n) {
            const double abar = exp(dt * A[n]);        /* Abar = exp(A*dt)   */
            const double bbar_u = dt * Bb[t * N + n] * ut; /* Bbar*u = dt*B*u */
            h[n] = abar * h[n] + bbar_u;                /* state update       */
            acc += Cb[t * N + n] * h[n];                /* C . state          */
        }
        const double yt = acc + Dd * ut;                /* + D*u skip         */
        y[t] = zz ? yt * oracle_silu(zz[t]) : yt;       /* SiLU(z) gate       */
    }
    if (j->last_state)
        for (int64_t n = 0; n < N; ++n) j->last_state[chain * N + n] = h[n];
}

static void *scan_worker(void *arg) {
    const scan_job *j = (const scan_job *)arg;
    double *h = (double *)malloc(sizeof(double) * (size_t)j->dstate);
    double *A = (double *)malloc(sizeof(double) * (size_t)j->dstate);
    if (h && A)
        for (int64_t c = j->chain_begin; c < j->chain_end; ++c) scan_one_chain(j, c, h, A);
    free(h);
    free(A);
    return NULL;
}

/* Number of hardware threads this process may use. */
int oracle_hw_threads(void) {
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

/*
 * Full selective scan.  h0 may be NULL (zero initial state, as on the pages);
 * reset may be NULL (one document per row).  nthreads <= 0 means all hardware
 * threads.  Returns the number of threads used, or a negative value on a bad
 * argument.
 */
int oracle_selective_scan_f64(const double *u, const double *delta, const double *A_log,
                              const double *B, const double *C, const double *D,
                              const double *z, const double *delta_bias, int softplus_flag,
                              const double *h0, const unsigned char *reset, double *y,
                              double *last_state,
                              int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate,
                              int nthreads) {
    if (!u || !delta || !A_log || !B || !C || !y) return -1;
    if (batch < 0 || dim < 0 || seqlen < 0 || dstate < 0) return -2;
    const int64_t chains = batch * dim;
    if (nthreads <= 0) nthreads = oracle_hw_threads();
    if (nthreads > chains) nthreads = chains > 0 ? (int)chains : 1;

    scan_job base = {u, delta, A_log, B, C, D, z, delta_bias, h0, reset, y, last_state,
                     batch, dim, seqlen, dstate, softplus_flag, 0, 0};
    scan_job *jobs = (scan_job *)malloc(sizeof(scan_job) * (size_t)nthreads);
    pthread_t *tids = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    if (!jobs || !tids) { free(jobs); free(tids); return -3; }
    for (int i = 0; i < nthreads; ++i) {
        jobs[i] = base;
        jobs[i].chain_begin = chains * i / nthreads;
        jobs[i].chain_end = chains * (i + 1) / nthreads;
    }
    if (nthreads == 1) {
        scan_worker(&jobs[0]);
    } else {
        for (int i = 0; i < nthreads; ++i) pthread_create(&tids[i], NULL, scan_worker, &jobs[i]);
        for (int i = 0; i < nthreads; ++i) pthread_join(tids[i], NULL);
    }
    free(jobs);
    free(tids);
    return nthreads;
}

/*
 * Gradients of the full selective scan (training): given dout = dLoss/dy for
 * the gated output, the gradients of every input, by the chain rule through
 * the same recurrence (the codechina.net overview, section 2.2 point 3,
 * trains by recomputing the forward states in the backward pass; here the
 * forward states of a chain are simply kept in a buffer).  Per chain:
 *   forward:  dt_t = softplus(raw_t), Abar_tn = exp(dt_t A_n),
 *             h_tn = Abar_tn h_{t-1,n} + dt_t B_tn u_t,  y_t = C_t.h_t + D u_t
 *   reverse:  dy_t = dout_t SiLU(z_t)   (dout_t without a gate)
 *             dz_t = dout_t y_t SiLU'(z_t),  SiLU'(z) = s (1 + z (1 - s)), s = sigmoid(z)
 *             g_tn = dy_t C_tn + Abar_{t+1,n} g_{t+1,n}     (adjoint of h_tn)
 *             dC_tn += dy_t h_tn,   dB_tn += g_tn dt_t u_t,   dD += dy_t u_t
 *             du_t = dy_t D + sum_n g_tn dt_t B_tn
 *             ddt_t = sum_n g_tn (A_n Abar_tn h_{t-1,n} + u_t B_tn)
 *             dA_n += g_tn dt_t Abar_tn h_{t-1,n}
 *             ddelta_t = ddt_t sigmoid(raw_t) (softplus on) or ddt_t;  dbias += ddelta_t
 *   dA_log = dA * A  (A = -exp(A_log)).
 * B, C, A_log, D and the bias are shared, so their gradients are sums over
 * chains (dB, dC over channels; dA_log, dD, dbias over batches).  Zero
 * initial state.  Outputs: du, ddelta, dz [batch][dim][seqlen] (dz only with
 * z), dB, dC [batch][seqlen][dstate], dA_log [dim][dstate], dD, ddelta_bias
 * [dim]; all are overwritten.  Single-threaded: the shared sums are formed in
 * a fixed order.  Returns 0, or a negative value on a bad argument.
 */
/* The backward with an optional starting state h0 [batch][dim][dstate], an
 * optional reset mask [batch][seqlen] (non-zero: the state restarts from zero
 * before that step, as in oracle_selective_scan_f64) and the gradient of h0
 * (dh0, same layout; written when non-NULL).  A reset makes the step's decay
 * exactly zero: h_t = 0 * h_{t-1} + dt B u, so nothing flows back across it. */
static int scan_bwd_impl(const double *u, const double *delta, const double *A_log,
                         const double *B, const double *C, const double *D, const double *z,
                         const double *delta_bias, int softplus_flag, const double *h0,
                         const unsigned char *reset, const double *dout,
                         const double *dlast, double *du, double *ddelta, double *dA_log,
                         double *dB, double *dC, double *dD, double *dz, double *ddelta_bias,
                         double *dh0, int64_t batch, int64_t dim, int64_t seqlen,
                         int64_t dstate) {
    if (!u || !delta || !A_log || !B || !C || !dout || !du || !ddelta || !dA_log || !dB || !dC)
        return -1;
    if (batch < 0 || dim < 0 || seqlen < 0 || dstate < 0) return -2;
    const int64_t L = seqlen, N = dstate;
    double *hs = (double *)malloc(sizeof(double) * (size_t)(L * N + 1));
    double *ab = (double *)malloc(sizeof(double) * (size_t)(L * N + 1));
    double *dts = (double *)malloc(sizeof(double) * (size_t)(L + 1));
    double *ys = (double *)malloc(sizeof(double) * (size_t)(L + 1));
    double *A = (double *)malloc(sizeof(double) * (size_t)(N + 1));
    double *g = (double *)malloc(sizeof(double) * (size_t)(N + 1));
    double *dA = (double *)malloc(sizeof(double) * (size_t)(dim * N + 1));
    if (!hs || !ab || !dts || !ys || !A || !g || !dA) {
        free(hs); free(ab); free(dts); free(ys); free(A); free(g); free(dA);
        return -3;
    }
    for (int64_t i = 0; i < batch * L * N; ++i) dB[i] = dC[i] = 0.0;
    for (int64_t i = 0; i < dim * N; ++i) dA[i] = 0.0;
    for (int64_t i = 0; i < dim; ++i) {
        if (dD) dD[i] = 0.0;
        if (ddelta_bias) ddelta_bias[i] = 0.0;
    }
    for (int64_t b = 0; b < batch; ++b) {
        for (int64_t d = 0; d < dim; ++d) {
            const int64_t chain = b * dim + d;
            const double *uc = u + chain * L, *dl = delta + chain * L, *go = dout + chain * L;
            const double *zz = z ? z + chain * L : NULL;
            const double *Bb = B + b * L * N, *Cb = C + b * L * N;
            const double Dd = D ? D[d] : 0.0, bias = delta_bias ? delta_bias[d] : 0.0;
            const double *hin = h0 ? h0 + chain * N : NULL;         /* state before step 0 */
            const unsigned char *rsb = reset ? reset + b * L : NULL;  /* document starts */
            for (int64_t n = 0; n < N; ++n) A[n] = -exp(A_log[d * N + n]);
            /* forward, keeping every state */
            for (int64_t t = 0; t < L; ++t) {
                const double xr = dl[t] + bias;
                const double dt = softplus_flag ? oracle_softplus(xr) : xr;
                dts[t] = dt;
                double acc = 0.0;
                for (int64_t n = 0; n < N; ++n) {
                    const double hp = t > 0 ? hs[(t - 1) * N + n] : (hin ? hin[n] : 0.0);
                    const double a = (rsb && rsb[t]) ? 0.0 : exp(dt * A[n]);
                    ab[t * N + n] = a;
                    hs[t * N + n] = a * hp + dt * Bb[t * N + n] * uc[t];
                    acc += Cb[t * N + n] * hs[t * N + n];
                }
                ys[t] = acc + Dd * uc[t];
            }
            /* reverse */
            /* g = what reaches the state after step t from later on: Abar_{t+1} g_{t+1};
             * after the last step, the loss's own gradient on the final state (if any) */
            for (int64_t n = 0; n < N; ++n) g[n] = dlast ? dlast[chain * N + n] : 0.0;
            for (int64_t t = L - 1; t >= 0; --t) {
                double dy = go[t];
                if (zz) {
                    const double s = 1.0 / (1.0 + exp(-zz[t]));
                    dz[chain * L + t] = go[t] * ys[t] * s * (1.0 + zz[t] * (1.0 - s));
                    dy = go[t] * zz[t] * s;
                }
                if (dD) dD[d] += dy * uc[t];
                double dut = dy * Dd, ddt = 0.0;
                const double dt = dts[t];
                for (int64_t n = 0; n < N; ++n) {
                    const double gn = dy * Cb[t * N + n] + g[n];
                    const double hp = t > 0 ? hs[(t - 1) * N + n] : (hin ? hin[n] : 0.0);
                    const double a = ab[t * N + n];
                    dC[(b * L + t) * N + n] += dy * hs[t * N + n];
                    dB[(b * L + t) * N + n] += gn * dt * uc[t];
                    dut += gn * dt * Bb[t * N + n];
                    ddt += gn * (A[n] * a * hp + uc[t] * Bb[t * N + n]);
                    dA[d * N + n] += gn * dt * a * hp;
                    g[n] = a * gn;
                }
                du[chain * L + t] = dut;
                const double xr = dl[t] + bias;
                const double dr = softplus_flag ? ddt / (1.0 + exp(-xr)) : ddt;
                ddelta[chain * L + t] = dr;
                if (ddelta_bias) ddelta_bias[d] += dr;
            }
            /* Abar_0 g_0: what flows into the state before step 0 */
            if (dh0)
                for (int64_t n = 0; n < N; ++n) dh0[chain * N + n] = g[n];
        }
    }
    for (int64_t d = 0; d < dim; ++d)
        for (int64_t n = 0; n < N; ++n) dA_log[d * N + n] = dA[d * N + n] * -exp(A_log[d * N + n]);
    free(hs); free(ab); free(dts); free(ys); free(A); free(g); free(dA);
    return 0;
}

int oracle_selective_scan_bwd_f64(const double *u, const double *delta, const double *A_log,
                                  const double *B, const double *C, const double *D,
                                  const double *z, const double *delta_bias, int softplus_flag,
                                  const double *dout, double *du, double *ddelta,
                                  double *dA_log, double *dB, double *dC, double *dD,
                                  double *dz, double *ddelta_bias, int64_t batch, int64_t dim,
                                  int64_t seqlen, int64_t dstate) {
    return scan_bwd_impl(u, delta, A_log, B, C, D, z, delta_bias, softplus_flag, NULL, NULL,
                         dout, NULL, du, ddelta, dA_log, dB, dC, dD, dz, ddelta_bias, NULL,
                         batch, dim, seqlen, dstate);
}

/* The backward of oracle_selective_scan_f64 with h0 and document resets
 * (codechina.net overview, section 3.2 point 2 and the deployment notes on
 * block-by-block processing); dh0 receives the gradient of h0.  dlast
 * [batch][dim][dstate] (optional) is the loss's gradient on last_state: a
 * sequence cut into blocks is trained by passing one block's dh0 as the
 * preceding block's dlast (its last_state is the next block's h0). */
int oracle_selective_scan_bwd_ex_f64(const double *u, const double *delta, const double *A_log,
                                     const double *B, const double *C, const double *D,
                                     const double *z, const double *delta_bias,
                                     int softplus_flag, const double *h0,
                                     const unsigned char *reset, const double *dout,
                                     const double *dlast, double *du, double *ddelta,
                                     double *dA_log, double *dB, double *dC, double *dD,
                                     double *dz, double *ddelta_bias, double *dh0, int64_t batch,
                                     int64_t dim, int64_t seqlen, int64_t dstate) {
    return scan_bwd_impl(u, delta, A_log, B, C, D, z, delta_bias, softplus_flag, h0, reset,
                         dout, dlast, du, ddelta, dA_log, dB, dC, dD, dz, ddelta_bias, dh0,
                         batch, dim, seqlen, dstate);
}

/*
 * One decode step ("inference stays RNN-like": each new token touches only the
 * previous state).  state [batch][dim][dstate] is updated in place; x, dt, z
 * and out are [batch][dim]; B, C are [batch][dstate].
 */
int oracle_selective_state_update_f64(double *state, const double *x, const double *dt,
                                      const double *A_log, const double *B, const double *C,
                                      const double *D, const double *z, const double *dt_bias,
                                      int softplus_flag, double *out,
                                      int64_t batch, int64_t dim, int64_t dstate) {
    if (!state || !x || !dt || !A_log || !B || !C || !out) return -1;
    if (batch < 0 || dim < 0 || dstate < 0) return -2;
    const int64_t N = dstate;
    for (int64_t b = 0; b < batch; ++b) {
        for (int64_t d = 0; d < dim; ++d) {
            const int64_t e = b * dim + d;
            const double raw = dt[e] + (dt_bias ? dt_bias[d] : 0.0);
            const double step = softplus_flag ? oracle_softplus(raw) : raw;
            double acc = 0.0;
            for (int64_t n = 0; n < N; ++n) {
                const double A = -exp(A_log[d * N + n]);
                const double abar = exp(step * A);
                double *h = &state[e * N + n];
                *h = abar * *h + step * B[b * N + n] * x[e];
                acc += C[b * N + n] * *h;
            }
            const double yt = acc + (D ? D[d] : 0.0) * x[e];
            out[e] = z ? yt * oracle_silu(z[e]) : yt;
        }
    }
    return 0;
}

/*
 * Causal depthwise convolution, optionally followed by SiLU: the short
 * convolution the Mamba block applies to its x branch before the scan
 * (luzhipeng.com tutorial, step 2: nn.Conv1d with kernel_size = d_conv,
 * padding = d_conv - 1, groups = d_model -- one filter per channel;
 * highthink.cn "Mamba 整体架构": Conv1D (causal) followed by SiLU).
 *
 * Readings: "causal" keeps the first seqlen outputs of the padded
 * convolution, so output t sees inputs t-width+1 .. t.  The convolution is a
 * cross-correlation as in PyTorch: weight[d][width-1] multiplies the current
 * input.  Inputs before the sequence come from init_state (the last width-1
 * inputs of a previous block, oldest first) or are zero when it is NULL;
 * final_state (optional) receives the last width-1 inputs, for the next block.
 *
 *   xin(s)  = x[b][d][s] for s >= 0;  init_state[b][d][width-1+s] (or 0) for s < 0
 *   pre     = bias[d] + sum_{k=0}^{width-1} weight[d][k] * xin(t - (width-1) + k)
 *   out[b][d][t] = silu_flag ? SiLU(pre) : pre
 *   final_state[b][d][j] = xin(seqlen - (width-1) + j),  j = 0 .. width-2
 *
 * Layouts: x, out [batch][dim][seqlen]; weight [dim][width]; bias [dim]
 * (optional); init_state, final_state [batch][dim][width-1].
 */
static double conv_input(const double *xr, const double *st, int64_t width, int64_t s) {
    if (s >= 0) return xr[s];
    return st ? st[width - 1 + s] : 0.0;
}

int oracle_causal_conv1d_f64(const double *x, const double *weight, const double *bias,
                             const double *init_state, int silu_flag, double *out,
                             double *final_state, int64_t batch, int64_t dim, int64_t seqlen,
                             int64_t width) {
    if ((!x && batch * dim * seqlen > 0) || !weight || (!out && batch * dim * seqlen > 0))
        return -1;
    if (batch < 0 || dim < 0 || seqlen < 0 || width < 1) return -2;
    for (int64_t b = 0; b < batch; ++b) {
        for (int64_t d = 0; d < dim; ++d) {
            const int64_t row = b * dim + d;
            const double *xr = x ? x + row * seqlen : NULL;
            const double *st = init_state ? init_state + row * (width - 1) : NULL;
            const double *w = weight + d * width;
            for (int64_t t = 0; t < seqlen; ++t) {
                double pre = bias ? bias[d] : 0.0;
                for (int64_t k = 0; k < width; ++k)
                    pre += w[k] * conv_input(xr, st, width, t - (width - 1) + k);
                out[row * seqlen + t] = silu_flag ? oracle_silu(pre) : pre;
            }
            if (final_state)
                for (int64_t j = 0; j < width - 1; ++j)
                    final_state[row * (width - 1) + j] =
                        conv_input(xr, st, width, seqlen - (width - 1) + j);
        }
    }
    return 0;
}

/*
 * Complex-state selective scan (codechina.net overview, section 4.1: the
 * complex version initialises A = -0.5 + i*n (S4D-Lin); section 5.3: a
 * complex state keeps phase information).  The pages give nothing else, so:
 *
 *   A[d][n]  = -exp(A_log_re[d][n]) + i * A_im[d][n]        (Re A < 0)
 *   dt       = softplus(delta + bias) (or delta + bias), real
 *   h[n]     = exp(dt * A[d][n]) * h[n] + dt * B[b][t][n] * u      (complex)
 *   out      = (Re(sum_n C[b][t][n] * h[n]) + D[d] * u) * SiLU(z)
 *
 * B and C are complex, input-dependent, stored as interleaved (re, im)
 * pairs: [batch][seqlen][dstate][2]; the state starts at zero and
 * last_state is [batch][dim][dstate][2].  Everything else is laid out as for
 * oracle_selective_scan_f64.  Chains run one after another (no threads).
 */
int oracle_selective_scan_complex_f64(const double *u, const double *delta,
                                      const double *A_log_re, const double *A_im,
                                      const double *B, const double *C, const double *D,
                                      const double *z, const double *delta_bias,
                                      int softplus_flag, double *y, double *last_state,
                                      int64_t batch, int64_t dim, int64_t seqlen,
                                      int64_t dstate) {
    if (!u || !delta || !A_log_re || !A_im || !B || !C || !y) return -1;
    if (batch < 0 || dim < 0 || seqlen < 0 || dstate < 1) return -2;
    const int64_t L = seqlen, N = dstate;
    double complex *h = malloc((size_t)N * sizeof(double complex));
    double complex *A = malloc((size_t)N * sizeof(double complex));
    if (!h || !A) {
        free(h);
        free(A);
        return -3;
    }
    for (int64_t b = 0; b < batch; ++b) {
        for (int64_t d = 0; d < dim; ++d) {
            const int64_t chain = b * dim + d;
            for (int64_t n = 0; n < N; ++n) {
                A[n] = -exp(A_log_re[d * N + n]) + I * A_im[d * N + n];
                h[n] = 0.0;
            }
            for (int64_t t = 0; t < L; ++t) {
                const double ut = u[chain * L + t];
                const double raw = delta[chain * L + t] + (delta_bias ? delta_bias[d] : 0.0);
                const double dt = softplus_flag ? oracle_softplus(raw) : raw;
                double complex acc = 0.0;
                for (int64_t n = 0; n < N; ++n) {
                    const int64_t k = ((b * L + t) * N + n) * 2;
                    const double complex Bn = B[k] + I * B[k + 1];
                    const double complex Cn = C[k] + I * C[k + 1];
                    h[n] = cexp(dt * A[n]) * h[n] + dt * Bn * ut;
                    acc += Cn * h[n];
                }
                const double yt = creal(acc) + (D ? D[d] : 0.0) * ut;
                y[chain * L + t] = z ? yt * oracle_silu(z[chain * L + t]) : yt;
            }
            if (last_state)
                for (int64_t n = 0; n < N; ++n) {
                    last_state[(chain * N + n) * 2] = creal(h[n]);
                    last_state[(chain * N + n) * 2 + 1] = cimag(h[n]);
                }
        }
    }
    free(h);
    free(A);
    return 0;
}

