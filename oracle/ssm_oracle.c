/*
 * Sequential fp64 oracle for the Mamba selective state-space scan, its
 * gradients (reverse-mode differentiation of the same recurrence) and its
 * single-token decode step.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the slow, obviously correct CPU
 * statement of what the GPU path computes. Only the test suite, the smoke
 * check and the benchmark's CPU-baseline leg may load it. It shares no code,
 * header, table or helper with the CUDA library, and the CUDA library never
 * calls it.
 *
 * What it follows (page titles and the passage on each page):
 *   [SSM]  "State Space Models and Mamba" (jonathanding.github.io, llm-learning)
 *          §1  continuous system x' = A x + B u, y = C x + D u
 *          §1.5 S4D-Real: A stored as A_log, A = -exp(A_log)
 *          §2  zero-order-hold discretisation: Abar = exp(dt A),
 *              Bbar = A^-1 (exp(dt A) - I) B; recurrence x_k = Abar x_{k-1} + Bbar u_k
 *          §4  selectivity: dt_k = softplus(Linear(u_k)), B_k, C_k per step
 *   [NOTES] "Mamba" paper notes (awesome.papernotes.org, 2023_mamba)
 *          "Design 1: Selective State Space": Bbar = (dt A)^-1 (exp(dt A) - I) dt B,
 *          and the selective_ssm sketch: y + D * x skip
 *          "Overall framework": out = y * SiLU(z)
 *   [COMP] "Mamba" concept page (compassingai.com) §3.1: the same discrete update
 *
 * Because A is diagonal, (dt A)^-1 (exp(dt A) - I) dt B is elementwise per
 * state n: Bbar_n = expm1(dt A_n) / (dt A_n) * dt * B_n. This file writes it in
 * exactly that form, with the limit expm1(x)/x -> 1 taken when dt A_n == 0.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - the scan starts from h = 0 unless an initial state is passed;
 *   - delta_bias is added before softplus; a NULL bias, D or z means 0 / 0 / no gate;
 *   - the gate multiplies after the D skip: out = (C.h + D u) * z * sigmoid(z);
 *   - softplus is exact: max(x,0) + log1p(exp(-|x|)), no cut-off.
 *
 * Layouts (row-major, contiguous):
 *   u, delta, z, out : (batch, seqlen, dim)
 *   B, C             : (batch, seqlen, dstate)
 *   A_log            : (dim, dstate)
 *   D, delta_bias    : (dim)
 *   h0, last_state   : (batch, dim, dstate)
 *   decode: u, delta, z, out : (batch, dim); B, C : (batch, dstate);
 *           state : (batch, dim, dstate), updated in place.
 *
 * The variant flag selects the input matrix: 0 = zero-order hold (the method),
 * 1 = the simplified Bbar = dt * B that the paper-notes sketch and the
 * first-order (Euler) reading of [SSM] §2 give. Variant 1 is kept for the
 * optional simplified-discretisation row only.
 */
#include <math.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#else
static int omp_get_max_threads(void) { return 1; }
#endif

#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1
/* Largest state size the oracle accepts (per-channel scratch lives on the stack). */
#define ORACLE_MAX_DSTATE 1024

/* [SSM] §4: dt = softplus(.), written as the overflow-free identity
 * log(1 + e^x) = max(x, 0) + log1p(e^-|x|). */
static double oracle_softplus(double x)
{
    return fmax(x, 0.0) + log1p(exp(-fabs(x)));
}

/* [NOTES] "Overall framework": SiLU(z) = z * sigmoid(z). */
static double oracle_silu(double z)
{
    return z / (1.0 + exp(-z));
}

/* Zero-order-hold input coefficient for one state, [NOTES] Design 1 /
 * [SSM] §2: (dt A)^-1 (exp(dt A) - 1) dt B, elementwise because A is
 * diagonal. */
static double oracle_bbar(double dt, double A_n, double B_n, int variant)
{
    if (variant == 1)
        return dt * B_n;
    double dA = dt * A_n;
    double phi = (dA == 0.0) ? 1.0 : expm1(dA) / dA;
    return phi * dt * B_n;
}

/* One channel (b, d) of the scan, sequential over t. */
static void oracle_scan_channel(long b, long d, long dim, long dstate, long seqlen,
                                const double *u, const double *delta,
                                const double *A_log, const double *B,
                                const double *C, const double *D,
                                const double *z, const double *delta_bias,
                                const double *h0, double *out,
                                double *last_state, int variant, double *h,
                                double *A)
{
    for (long n = 0; n < dstate; ++n) {
        A[n] = -exp(A_log[d * dstate + n]); /* [SSM] §1.5 */
        h[n] = h0 ? h0[(b * dim + d) * dstate + n] : 0.0;
    }
    const double bias = delta_bias ? delta_bias[d] : 0.0;
    for (long t = 0; t < seqlen; ++t) {
        const long i = (b * seqlen + t) * dim + d;   /* (b, t, d) */
        const long j = (b * seqlen + t) * dstate;    /* (b, t, 0) */
        const double dt = oracle_softplus(delta[i] + bias);
        double y = 0.0;
        for (long n = 0; n < dstate; ++n) {
            const double abar = exp(dt * A[n]);                       /* [SSM] §2 */
            const double bbar = oracle_bbar(dt, A[n], B[j + n], variant);
            h[n] = abar * h[n] + bbar * u[i];                         /* recurrence */
            y += C[j + n] * h[n];                                     /* y = C h */
        }
        if (D)
            y += D[d] * u[i];                                         /* D skip */
        if (z)
            y *= oracle_silu(z[i]);                                   /* gate */
        out[i] = y;
    }
    if (last_state)
        for (long n = 0; n < dstate; ++n)
            last_state[(b * dim + d) * dstate + n] = h[n];
}

/* Whole scan. nthreads <= 0 uses the OpenMP default; channels are
 * independent, so the parallel loop changes no arithmetic. */
int oracle_selective_scan(long batch, long dim, long dstate, long seqlen,
                          const double *u, const double *delta,
                          const double *A_log, const double *B, const double *C,
                          const double *D, const double *z,
                          const double *delta_bias, const double *h0,
                          double *out, double *last_state, int variant,
                          int nthreads)
{
    if (batch < 0 || dim < 0 || dstate <= 0 || seqlen < 0)
        return ORACLE_BAD_ARG;
    if (batch == 0 || dim == 0)
        return ORACLE_OK;
    if ((seqlen > 0 && (!u || !delta || !B || !C || !out)) || !A_log)
        return ORACLE_BAD_ARG;
    if (dstate > ORACLE_MAX_DSTATE)
        return ORACLE_BAD_ARG;
    const long nch = batch * dim;
#pragma omp parallel for schedule(static) num_threads(nthreads > 0 ? nthreads : omp_get_max_threads())
    for (long c = 0; c < nch; ++c) {
        double h[ORACLE_MAX_DSTATE], A[ORACLE_MAX_DSTATE];
        oracle_scan_channel(c / dim, c % dim, dim, dstate, seqlen, u, delta,
                            A_log, B, C, D, z, delta_bias, h0, out,
                            last_state, variant, h, A);
    }
    return ORACLE_OK;
}

/* Single-token decode step on a resident state, [SSM] §3 recurrence mode:
 * the same body as one step of the scan, starting from the given state. */
int oracle_state_update(long batch, long dim, long dstate, double *state,
                        const double *u, const double *delta,
                        const double *A_log, const double *B, const double *C,
                        const double *D, const double *z,
                        const double *delta_bias, double *out, int variant)
{
    if (batch < 0 || dim < 0 || dstate <= 0)
        return ORACLE_BAD_ARG;
    if (batch == 0 || dim == 0)
        return ORACLE_OK;
    if (!state || !u || !delta || !A_log || !B || !C || !out || dstate > ORACLE_MAX_DSTATE)
        return ORACLE_BAD_ARG;
    for (long b = 0; b < batch; ++b) {
        for (long d = 0; d < dim; ++d) {
            const long i = b * dim + d;
            const double dt = oracle_softplus(delta[i] + (delta_bias ? delta_bias[d] : 0.0));
            double y = 0.0;
            for (long n = 0; n < dstate; ++n) {
                const double A_n = -exp(A_log[d * dstate + n]);
                const double abar = exp(dt * A_n);
                const double bbar = oracle_bbar(dt, A_n, B[b * dstate + n], variant);
                double *h = &state[i * dstate + n];
                *h = abar * (*h) + bbar * u[i];
                y += C[b * dstate + n] * (*h);
            }
            if (D)
                y += D[d] * u[i];
            if (z)
                y *= oracle_silu(z[i]);
            out[i] = y;
        }
    }
    return ORACLE_OK;
}

/* Causal depthwise 1-D convolution followed by SiLU, the step in front of the
 * scan in the Mamba block ("Mamba" paper notes, Design 3; compassingai
 * "Mamba" §3.3; "State Space Models and Mamba", Mamba Block architecture):
 *   u[b,t,d] = SiLU( sum_{k=0}^{width-1} w[d,k] * x[b, t-(width-1)+k, d] + bias[d] ),
 * with x taken as zero before t = 0 (causal padding). The tap w[d, width-1]
 * multiplies the current input. Layouts: x, u (batch, seqlen, dim); w (dim,
 * width); bias (dim) or NULL. */
int oracle_causal_conv1d_silu(long batch, long dim, long seqlen, long width,
                              const double *x, const double *w,
                              const double *bias, double *u)
{
    if (batch < 0 || dim < 0 || seqlen < 0 || width < 1)
        return ORACLE_BAD_ARG;
    if (batch == 0 || dim == 0 || seqlen == 0)
        return ORACLE_OK;
    if (!x || !w || !u)
        return ORACLE_BAD_ARG;
    for (long b = 0; b < batch; ++b)
        for (long t = 0; t < seqlen; ++t)
            for (long d = 0; d < dim; ++d) {
                double acc = bias ? bias[d] : 0.0;
                for (long k = 0; k < width; ++k) {
                    const long ts = t - (width - 1) + k;
                    if (ts >= 0)
                        acc += w[d * width + k] * x[(b * seqlen + ts) * dim + d];
                }
                u[(b * seqlen + t) * dim + d] = oracle_silu(acc);
            }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------
 * Backward of the scan: the gradient of a scalar loss
 *     loss = sum_{b,t,d} dout[b,t,d] * out[b,t,d] + sum_{b,d,n} dlast[b,d,n] * last_state[b,d,n]
 * with respect to every input of oracle_selective_scan. The pages give the
 * forward recurrence only; this is the chain rule applied to it in reverse
 * time (reverse-mode differentiation of the loop above, step by step), with
 * the forward states of each channel kept in full (no recomputation).
 *
 * Derivatives used (x = delta + bias, dt = softplus(x), A = -exp(A_log),
 * abar = exp(dt A), and for zero-order hold bbar = expm1(dt A) / A * B):
 *   d softplus(x) / dx   = sigmoid(x)
 *   d abar / d dt        = A abar,           d abar / dA = dt abar
 *   d bbar / d dt        = abar B            (simplified: B)
 *   d bbar / dA          = B dt^2 phi'(dt A) (simplified: 0), where
 *                          phi(s) = expm1(s) / s and phi'(s) = (s e^s - expm1(s)) / s^2
 *   d A / d A_log        = A
 *   d SiLU(z) / dz       = sigmoid(z) (1 + z (1 - sigmoid(z)))
 *
 * Outputs (all written, none accumulated into): du, ddelta, dz like u;
 * dB, dC like B; dA_log like A_log; dD, ddelta_bias (dim); dh0 like h0.
 * dz, dD, ddelta_bias and dh0 may be NULL (not computed); dlast may be NULL
 * (zero). Sequential: the cross-channel sums (dB, dC) and the cross-batch
 * sums (dA_log, dD, ddelta_bias) are plain running sums.
 * ------------------------------------------------------------------------ */

static double oracle_sigmoid(double x)
{
    return 1.0 / (1.0 + exp(-x));
}

/* phi'(s) for phi(s) = expm1(s) / s. Below |s| = 1e-3 the closed form cancels,
 * so the Taylor series sum_k (k + 1) s^k / (k + 2)! is used (terms to s^4;
 * the next term is below 1e-17). */
static double oracle_dphi(double s)
{
    if (fabs(s) < 1e-3)
        return 0.5 + s * (1.0 / 3.0 + s * (1.0 / 8.0 + s * (1.0 / 30.0 + s * (1.0 / 144.0))));
    return (s * exp(s) - expm1(s)) / (s * s);
}

int oracle_selective_scan_bwd(long batch, long dim, long dstate, long seqlen,
                              const double *u, const double *delta,
                              const double *A_log, const double *B, const double *C,
                              const double *D, const double *z,
                              const double *delta_bias, const double *h0,
                              const double *dout, const double *dlast,
                              double *du, double *ddelta, double *dA_log,
                              double *dB, double *dC, double *dD, double *dz,
                              double *ddelta_bias, double *dh0, int variant)
{
    if (batch < 0 || dim < 0 || dstate <= 0 || seqlen < 0 || dstate > ORACLE_MAX_DSTATE)
        return ORACLE_BAD_ARG;
    if (!A_log || !dA_log)
        return ORACLE_BAD_ARG;
    if (seqlen > 0 && (!u || !delta || !B || !C || !dout || !du || !ddelta || !dB || !dC))
        return ORACLE_BAD_ARG;
    for (long k = 0; k < dim * dstate; ++k)
        dA_log[k] = 0.0;
    for (long k = 0; k < batch * seqlen * dstate; ++k)
        dB[k] = dC[k] = 0.0;
    for (long d = 0; d < dim; ++d) {
        if (dD)
            dD[d] = 0.0;
        if (ddelta_bias)
            ddelta_bias[d] = 0.0;
    }
    if (batch == 0 || dim == 0)
        return ORACLE_OK;

    /* forward record of one channel: h after each step (hs[t+1]), h0 in hs[0] */
    double *hs = malloc(sizeof(double) * (size_t)(seqlen + 1) * (size_t)dstate);
    double *dts = malloc(sizeof(double) * (size_t)(seqlen + 1));
    double *ys = malloc(sizeof(double) * (size_t)(seqlen + 1));
    if (!hs || !dts || !ys) {
        free(hs);
        free(dts);
        free(ys);
        return ORACLE_BAD_ARG;
    }
    double A[ORACLE_MAX_DSTATE], hbar[ORACLE_MAX_DSTATE], Abar_acc[ORACLE_MAX_DSTATE];

    for (long b = 0; b < batch; ++b) {
        for (long d = 0; d < dim; ++d) {
            const double bias_d = (delta_bias != NULL) ? delta_bias[d] : 0.0;
            const double *A_log_d = A_log + d * dstate;
            for (long n = 0; n < dstate; ++n) {
                A[n] = -exp(A_log_d[n]);
                hs[n] = h0 ? h0[(b * dim + d) * dstate + n] : 0.0;
            }
            /* forward, as in oracle_scan_channel, recording h_t, dt_t and the
             * pre-gate y_t */
            for (long t = 0; t < seqlen; ++t) {
                const long i = (b * seqlen + t) * dim + d;
                const long j = (b * seqlen + t) * dstate;
                const double dt = oracle_softplus(delta[i] + bias_d);
                double y = 0.0;
                for (long n = 0; n < dstate; ++n) {
                    const double B_tn = B[j + n];
                    const double abar = exp(dt * A[n]);
                    const double bbar = oracle_bbar(dt, A[n], B_tn, variant);
                    hs[(t + 1) * dstate + n] = abar * hs[t * dstate + n] + bbar * u[i];
                    y += C[j + n] * hs[(t + 1) * dstate + n];
                }
                if (D)
                    y += D[d] * u[i];
                dts[t] = dt;
                ys[t] = y;
            }
            /* reverse */
            for (long n = 0; n < dstate; ++n) {
                hbar[n] = dlast ? dlast[(b * dim + d) * dstate + n] : 0.0;
                Abar_acc[n] = 0.0;
            }
            for (long t = seqlen - 1; t >= 0; --t) {
                const long i = (b * seqlen + t) * dim + d;
                const long j = (b * seqlen + t) * dstate;
                const double dt = dts[t];
                /* out = y * SiLU(z) */
                double ybar = dout[i];
                if (z) {
                    const double sg = oracle_sigmoid(z[i]);
                    if (dz)
                        dz[i] = dout[i] * ys[t] * sg * (1.0 + z[i] * (1.0 - sg));
                    ybar = dout[i] * oracle_silu(z[i]);
                } else if (dz) {
                    dz[i] = 0.0;
                }
                /* y = sum_n C_n h_n + D u */
                double ubar = 0.0;
                if (D) {
                    ubar += ybar * D[d];
                    if (dD)
                        dD[d] += ybar * u[i];
                }
                double dtbar = 0.0;
                for (long n = 0; n < dstate; ++n) {
                    const double h_t = hs[(t + 1) * dstate + n];
                    const double h_prev = hs[t * dstate + n];
                    dC[j + n] += ybar * h_t;
                    hbar[n] += ybar * C[j + n];
                    /* h_t = abar h_prev + bbar u */
                    const double B_tn = B[j + n];
                    const double abar = exp(dt * A[n]);
                    const double bbar = oracle_bbar(dt, A[n], B_tn, variant);
                    const double abar_bar = hbar[n] * h_prev;
                    const double bbar_bar = hbar[n] * u[i];
                    ubar += hbar[n] * bbar;
                    /* abar = exp(dt A) */
                    dtbar += abar_bar * abar * A[n];
                    Abar_acc[n] += abar_bar * abar * dt;
                    /* bbar */
                    dB[j + n] += bbar_bar * oracle_bbar(dt, A[n], 1.0, variant); /* bbar is linear in B */
                    if (variant == 1) {
                        dtbar += bbar_bar * B_tn;
                    } else {
                        dtbar += bbar_bar * abar * B_tn;
                        Abar_acc[n] += bbar_bar * B_tn * dt * dt * oracle_dphi(dt * A[n]);
                    }
                    hbar[n] *= abar; /* to h_prev */
                }
                /* dt = softplus(delta + bias) */
                const double xbar = dtbar * oracle_sigmoid(delta[i] + bias_d);
                ddelta[i] = xbar;
                if (ddelta_bias)
                    ddelta_bias[d] += xbar;
                du[i] = ubar;
            }
            for (long n = 0; n < dstate; ++n) {
                dA_log[d * dstate + n] += Abar_acc[n] * A[n]; /* A = -exp(A_log) */
                if (dh0)
                    dh0[(b * dim + d) * dstate + n] = hbar[n];
            }
        }
    }
    free(hs);
    free(dts);
    free(ys);
    return ORACLE_OK;
}
