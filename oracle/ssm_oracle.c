/*
 * ssm_oracle.c -- fp64 CPU oracle for the selective state-space scan (S6).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this file's library.  The product path
 * (the CUDA library) never links, loads or calls it, and this file shares no
 * code, header, table or constant with it.
 *
 * What it computes, and where the definition comes from
 * (page titles as they appear in the source pages):
 *
 *   - State-space model, discrete form: the state equation
 *     h(t+1) = A h(t) + B x(t) and the observation y(t) = C h(t)
 *     ("Mamba: Linear-Time Sequence Modeling with Selective State Spaces",
 *     dhy1.tistory.com, section "0. State Space Models").  The time index is
 *     read so that the current token enters its own output:
 *     h_t = dA_t * h_{t-1} + dBx_t,  y_t = C_t . h_t.
 *   - Selection: Delta, B and C are given per token (per (batch, time)),
 *     B and C shared by all channels ("Mamba的三大创新" page,
 *     weblog-19d.pages.dev, section on S4 -> S6 and the gating roles of
 *     Delta, B, C).
 *   - Discretisation, stage 1 of that page (zero-order hold): the decay is
 *     dA = exp(Delta * A) exactly; the input term is taken in its first-order
 *     (Euler) form dBx = Delta * B * x.
 *   - Recurrent mode, stage 2 of that page: the linear recurrence evaluated
 *     with a plain loop over time.
 *   - Delta = softplus(delta_raw + bias), the skip term D * x added before the
 *     output gate, and the gate silu(z) = z / (1 + exp(-z)).
 *
 * Arithmetic is IEEE fp64 throughout, with libm exp/log1p, and no reordering
 * beyond the loops written here: for each (batch, channel) pair, time runs
 * forward, and for each time step the state index runs 0..dstate-1.
 *
 * Layouts (row-major, last index fastest):
 *   x, delta, z, out     : (batch, seqlen, dim)
 *   B, C                 : (batch, seqlen, dstate)
 *   A                    : (dim, dstate)
 *   D, delta_bias        : (dim)
 *   initial/last state   : (batch, dim, dstate)
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* softplus(u) = log(1 + e^u), evaluated without overflow and without the
 * cancellation of forming 1 + e^u for very negative u. */
static double oracle_softplus(double u)
{
    if (u > 0.0)
        return u + log1p(exp(-u));
    return log1p(exp(u));
}

/* silu(v) = v * sigmoid(v) = v / (1 + e^{-v}). */
static double oracle_silu(double v)
{
    return v / (1.0 + exp(-v));
}

/* Full-sequence forward scan.  Returns 0 on success, -1 on bad arguments.
 * `nthreads` <= 0 lets OpenMP choose. */
int oracle_scan_fwd(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate,
                    const double *x, const double *delta, const double *A,
                    const double *B, const double *C, const double *D,
                    const double *z, const double *delta_bias, int delta_softplus,
                    const double *initial_state, double *out, double *last_state,
                    int nthreads)
{
    if (batch < 0 || seqlen < 0 || dim < 0 || dstate <= 0 || dstate > 4096)
        return -1;
    if (!x || !delta || !A || !B || !C || !out)
        return -1;
    const int64_t nchan = batch * dim;
#ifdef _OPENMP
    if (nthreads <= 0)
        nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (int64_t ch = 0; ch < nchan; ++ch) {
        const int64_t b = ch / dim;
        const int64_t d = ch % dim;
        double h[4096];
        for (int64_t n = 0; n < dstate; ++n)
            h[n] = initial_state ? initial_state[(b * dim + d) * dstate + n] : 0.0;
        for (int64_t t = 0; t < seqlen; ++t) {
            const int64_t tok = (b * seqlen + t) * dim + d;  /* (b, t, d) */
            const int64_t row = (b * seqlen + t) * dstate;   /* (b, t, :) */
            const double xv = x[tok];
            double u = delta[tok] + (delta_bias ? delta_bias[d] : 0.0);
            const double dt = delta_softplus ? oracle_softplus(u) : u;
            double y = 0.0;
            for (int64_t n = 0; n < dstate; ++n) {
                const double dA = exp(dt * A[d * dstate + n]);
                h[n] = dA * h[n] + dt * B[row + n] * xv;
                y += C[row + n] * h[n];
            }
            if (D)
                y += D[d] * xv;
            if (z)
                y *= oracle_silu(z[tok]);
            out[tok] = y;
        }
        if (last_state)
            for (int64_t n = 0; n < dstate; ++n)
                last_state[(b * dim + d) * dstate + n] = h[n];
    }
    return 0;
}

/* One decode step: the same recurrence for a single token per sequence,
 * with the state read and written in place.
 *   state            : (batch, dim, dstate), updated in place
 *   x, delta, z, out : (batch, dim)
 *   B, C             : (batch, dstate)
 */
int oracle_state_update(int64_t batch, int64_t dim, int64_t dstate, double *state,
                        const double *x, const double *delta, const double *A,
                        const double *B, const double *C, const double *D,
                        const double *z, const double *delta_bias, int delta_softplus,
                        double *out)
{
    if (batch < 0 || dim < 0 || dstate <= 0)
        return -1;
    if (!state || !x || !delta || !A || !B || !C || !out)
        return -1;
    for (int64_t b = 0; b < batch; ++b) {
        for (int64_t d = 0; d < dim; ++d) {
            const int64_t tok = b * dim + d;
            double *h = state + tok * dstate;
            double u = delta[tok] + (delta_bias ? delta_bias[d] : 0.0);
            const double dt = delta_softplus ? oracle_softplus(u) : u;
            double y = 0.0;
            for (int64_t n = 0; n < dstate; ++n) {
                const double dA = exp(dt * A[d * dstate + n]);
                h[n] = dA * h[n] + dt * B[b * dstate + n] * x[tok];
                y += C[b * dstate + n] * h[n];
            }
            if (D)
                y += D[d] * x[tok];
            if (z)
                y *= oracle_silu(z[tok]);
            out[tok] = y;
        }
    }
    return 0;
}

/* Causal depthwise convolution over time, per channel, followed by an
 * optional SiLU: the local-context convolution the Mamba block applies to x
 * before the selective SSM ("Mamba的三大创新", section on the simplified
 * architecture, "为什么SSM前面有个卷积": each token sees its neighbours
 * before the SSM; the unite.ai overview: a causal Conv1d layer in the block).
 * Width K, taps w[d][0..K-1] with w[d][K-1] on the current token:
 *   pre[t, d] = bias[d] + sum_{k=0..K-1} w[d][k] * x[t - (K-1) + k, d]
 *   out[t, d] = activation ? silu(pre) : pre
 * Inputs before t = 0 come from conv_state_in[b][d][0..K-2] (oldest first),
 * or are zero when it is NULL.  conv_state_out receives the last K-1 inputs
 * of the sequence (oldest first), continuing the state when L < K-1.
 * Layouts: x, out (batch, seqlen, dim); w (dim, K); bias (dim);
 * states (batch, dim, K-1). */
int oracle_conv1d_fwd(int64_t batch, int64_t seqlen, int64_t dim, int64_t width,
                      int activation, const double *x, const double *w, const double *bias,
                      const double *conv_state_in, double *out, double *conv_state_out)
{
    if (batch < 0 || seqlen < 0 || dim < 0 || width < 1 || width > 64)
        return -1;
    if (!w || (seqlen > 0 && (!x || !out)))
        return -1;
    const int64_t H = width - 1;   /* history length */
    for (int64_t b = 0; b < batch; ++b) {
        for (int64_t d = 0; d < dim; ++d) {
            /* the input at time t, for t in [-H, seqlen) */
            for (int64_t t = 0; t < seqlen; ++t) {
                double acc = bias ? bias[d] : 0.0;
                for (int64_t k = 0; k < width; ++k) {
                    const int64_t tt = t - H + k;
                    double v;
                    if (tt >= 0)
                        v = x[(b * seqlen + tt) * dim + d];
                    else
                        v = conv_state_in ? conv_state_in[(b * dim + d) * H + (H + tt)] : 0.0;
                    acc += w[d * width + k] * v;
                }
                out[(b * seqlen + t) * dim + d] = activation ? oracle_silu(acc) : acc;
            }
            if (conv_state_out) {
                for (int64_t k = 0; k < H; ++k) {
                    const int64_t tt = seqlen - H + k;   /* time of state slot k */
                    double v;
                    if (tt >= 0)
                        v = x[(b * seqlen + tt) * dim + d];
                    else
                        v = conv_state_in ? conv_state_in[(b * dim + d) * H + (H + tt)] : 0.0;
                    conv_state_out[(b * dim + d) * H + k] = v;
                }
            }
        }
    }
    return 0;
}

/* The scan with the exact zero-order-hold input term ("Mamba的三大创新",
 * stage 1, zero-order hold): holding x constant over a step of length Delta,
 * the diagonal system h' = A h + B x integrates exactly to
 *   h_t = exp(Delta A) h_{t-1} + ((exp(Delta A) - 1) / A) B x_t,
 * i.e. Bbar = (Delta A)^{-1} (exp(Delta A) - I) Delta B, which tends to
 * Delta B (the first-order form of oracle_scan_fwd) as Delta A -> 0; at
 * A = 0 it is Delta B exactly.  Everything else (softplus, readout, skip,
 * gate, layouts, arguments) is that of oracle_scan_fwd. */
int oracle_scan_fwd_zoh(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate,
                        const double *x, const double *delta, const double *A,
                        const double *B, const double *C, const double *D,
                        const double *z, const double *delta_bias, int delta_softplus,
                        const double *initial_state, double *out, double *last_state,
                        int nthreads)
{
    if (batch < 0 || seqlen < 0 || dim < 0 || dstate <= 0 || dstate > 4096)
        return -1;
    if (!x || !delta || !A || !B || !C || !out)
        return -1;
    const int64_t nchan = batch * dim;
#ifdef _OPENMP
    if (nthreads <= 0)
        nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (int64_t ch = 0; ch < nchan; ++ch) {
        const int64_t bb = ch / dim;
        const int64_t dd = ch % dim;
        double st[4096];   /* the state of channel (bb, dd) */
        for (int64_t n = 0; n < dstate; ++n)
            st[n] = initial_state ? initial_state[ch * dstate + n] : 0.0;
        for (int64_t t = 0; t < seqlen; ++t) {
            const int64_t i = (bb * seqlen + t) * dim + dd;   /* (b, t, d) */
            const int64_t r = (bb * seqlen + t) * dstate;     /* (b, t, :) */
            const double step = delta_softplus
                ? oracle_softplus(delta[i] + (delta_bias ? delta_bias[dd] : 0.0))
                : delta[i] + (delta_bias ? delta_bias[dd] : 0.0);
            double acc = 0.0;
            for (int64_t n = 0; n < dstate; ++n) {
                const double a = A[dd * dstate + n];
                const double decay = exp(step * a);
                const double gain = a != 0.0 ? expm1(step * a) / a : step;   /* (e^{dt a} - 1) / a */
                st[n] = decay * st[n] + gain * B[r + n] * x[i];
                acc += C[r + n] * st[n];
            }
            acc += D ? D[dd] * x[i] : 0.0;
            out[i] = z ? acc * oracle_silu(z[i]) : acc;
        }
        for (int64_t n = 0; last_state && n < dstate; ++n)
            last_state[ch * dstate + n] = st[n];
    }
    return 0;
}

/* Convolution kernel of the time-invariant (LTI, S4) model ("Mamba的三大创新",
 * stage 3, the convolution mode): with a constant step Delta[d] and
 * per-channel B[d][n], C[d][n], unrolling the recurrence from a zero state
 * gives y = K * x with
 *   K[d][k] = sum_n C[d][n] exp(k Delta[d] A[d][n]) Bbar[d][n],   k = 0 .. L-1,
 * Bbar = Delta B (zoh = 0, the first-order form) or (exp(Delta A) - 1) / A B
 * (zoh = 1).  Layouts: delta (dim); A, B, C (dim, dstate); K (dim, L). */
int oracle_lti_kernel(int64_t dim, int64_t dstate, int64_t seqlen, const double *delta,
                      const double *A, const double *B, const double *C, int zoh, double *K)
{
    if (dim < 0 || dstate <= 0 || seqlen < 0 || !delta || !A || !B || !C || !K)
        return -1;
    for (int64_t d = 0; d < dim; ++d) {
        const double dt = delta[d];
        for (int64_t k = 0; k < seqlen; ++k) {
            double acc = 0.0;
            for (int64_t n = 0; n < dstate; ++n) {
                const double a = A[d * dstate + n];
                const double gain = zoh ? (a != 0.0 ? expm1(dt * a) / a : dt) : dt;
                acc += C[d * dstate + n] * exp((double)k * dt * a) * gain * B[d * dstate + n];
            }
            K[d * seqlen + k] = acc;
        }
    }
    return 0;
}

/* The convolution mode itself: y[b][t][d] = sum_{k=0..t} K[d][k] x[b][t-k][d]
 * + D[d] x[b][t][d], then the gate silu(z) when z is given (as in
 * oracle_scan_fwd).  x, z, out: (batch, seqlen, dim); K: (dim, seqlen). */
int oracle_lti_conv(int64_t batch, int64_t seqlen, int64_t dim, const double *K,
                    const double *x, const double *D, const double *z, double *out)
{
    if (batch < 0 || seqlen < 0 || dim < 0 || (seqlen > 0 && (!K || !x || !out)))
        return -1;
    for (int64_t b = 0; b < batch; ++b)
        for (int64_t d = 0; d < dim; ++d)
            for (int64_t t = 0; t < seqlen; ++t) {
                double y = 0.0;
                for (int64_t k = 0; k <= t; ++k)
                    y += K[d * seqlen + k] * x[(b * seqlen + (t - k)) * dim + d];
                const int64_t tok = (b * seqlen + t) * dim + d;
                if (D)
                    y += D[d] * x[tok];
                if (z)
                    y *= oracle_silu(z[tok]);
                out[tok] = y;
            }
    return 0;
}

/* Gradients of oracle_scan_fwd: the loop of that function differentiated
 * by hand in reverse mode (the backward half of training the selective SSM:
 * "Mamba的三大创新", stage 2, the parallel training of the recurrence; the
 * gradients of the same recurrence, run backwards in time).
 *
 * Given dout = dL/dout (batch, seqlen, dim) and optionally
 * dlast = dL/dlast_state (batch, dim, dstate), with, per (b, d) and time t,
 *   u_t = delta + bias,  Delta_t = softplus(u_t) (or u_t),
 *   dA_{t,n} = exp(Delta_t A_n),  h_{t,n} = dA_{t,n} h_{t-1,n} + Delta_t B_{t,n} x_t,
 *   yc_t = sum_n C_{t,n} h_{t,n} + D x_t,  out_t = yc_t silu(z_t),
 * time runs backwards carrying g_n = dL/dh_{t,n} (starting from dlast):
 *   dyc = dout_t silu(z_t);     dz_t = dout_t yc_t silu'(z_t)
 *   g_n += dyc C_{t,n};         dC_{t,n} += dyc h_{t,n};  dD += dyc x_t;  dx_t = dyc D
 *   dDelta_t = sum_n g_n (B_{t,n} x_t + A_n dA_{t,n} h_{t-1,n})
 *   dA_n += g_n Delta_t dA_{t,n} h_{t-1,n};   dB_{t,n} += g_n Delta_t x_t
 *   dx_t += Delta_t sum_n g_n B_{t,n};        g_n *= dA_{t,n}   (now dL/dh_{t-1,n})
 *   du_t = dDelta_t sigmoid(u_t) (or dDelta_t);  ddelta_t = du_t;  dbias += du_t
 * and after t = 0, dinitial_state = g.  silu'(z) = s (1 + z (1 - s)), s = sigmoid(z).
 *
 * Outputs are written, not accumulated: dx, ddelta (batch, seqlen, dim);
 * dA (dim, dstate); dB, dC (batch, seqlen, dstate); dD, ddelta_bias (dim);
 * dz (batch, seqlen, dim); dinitial_state (batch, dim, dstate).  Any output
 * pointer may be NULL (not computed); dz must be NULL when z is.
 * Sums over channels (dB, dC) and over sequences (dA, dD, ddelta_bias) are
 * formed per thread over a fixed range of channels, then added in thread order. */
int oracle_scan_bwd(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate,
                    const double *x, const double *delta, const double *A,
                    const double *B, const double *C, const double *D,
                    const double *z, const double *delta_bias, int delta_softplus,
                    const double *initial_state, const double *dout, const double *dlast,
                    double *dx, double *ddelta, double *dA, double *dB, double *dC,
                    double *dD, double *dz, double *ddelta_bias, double *dinitial_state,
                    int nthreads)
{
    if (batch < 0 || seqlen < 0 || dim < 0 || dstate <= 0 || dstate > 4096)
        return -1;
    if (!x || !delta || !A || !B || !C || !dout || (dz && !z))
        return -1;
    const int64_t nchan = batch * dim;
    const int64_t nbc = batch * seqlen * dstate;     /* elements of dB (and dC) */
    int nt = 1;
#ifdef _OPENMP
    nt = nthreads > 0 ? nthreads : omp_get_max_threads();
#endif
    if (nt < 1)
        nt = 1;
    if ((int64_t)nt > nchan && nchan > 0)
        nt = (int)nchan;
    /* per-thread partial sums: dB, dC | dA | dD | dbias */
    const int64_t per = 2 * nbc + dim * dstate + 2 * dim;
    double *part = (double *)calloc((size_t)nt * (size_t)per, sizeof(double));
    double *hist = (double *)malloc((size_t)nt * (size_t)(seqlen + 1) * (size_t)dstate * sizeof(double));
    if (!part || !hist) {
        free(part);
        free(hist);
        return -1;
    }
#ifdef _OPENMP
#pragma omp parallel num_threads(nt)
#endif
    {
        int tid = 0;
#ifdef _OPENMP
        tid = omp_get_thread_num();
#endif
        double *pB = part + (int64_t)tid * per;
        double *pC = pB + nbc;
        double *pA = pC + nbc;
        double *pD = pA + dim * dstate;
        double *pbias = pD + dim;
        /* h_{t,n} for t = -1 .. seqlen-1 at hs[(t + 1) * dstate + n] */
        double *hs = hist + (int64_t)tid * (seqlen + 1) * dstate;
        double g[4096];
        const int64_t lo = nchan * tid / nt, hi = nchan * (tid + 1) / nt;
        for (int64_t ch = lo; ch < hi; ++ch) {
            const int64_t b = ch / dim;
            const int64_t d = ch % dim;
            const double bias = delta_bias ? delta_bias[d] : 0.0;
            /* forward again, keeping every state */
            for (int64_t n = 0; n < dstate; ++n)
                hs[n] = initial_state ? initial_state[(b * dim + d) * dstate + n] : 0.0;
            for (int64_t t = 0; t < seqlen; ++t) {
                const int64_t tok = (b * seqlen + t) * dim + d;
                const int64_t row = (b * seqlen + t) * dstate;
                const double u = delta[tok] + bias;
                const double dt = delta_softplus ? oracle_softplus(u) : u;
                for (int64_t n = 0; n < dstate; ++n)
                    hs[(t + 1) * dstate + n] = exp(dt * A[d * dstate + n]) * hs[t * dstate + n]
                                               + dt * B[row + n] * x[tok];
            }
            /* backwards in time */
            for (int64_t n = 0; n < dstate; ++n)
                g[n] = dlast ? dlast[(b * dim + d) * dstate + n] : 0.0;
            for (int64_t t = seqlen - 1; t >= 0; --t) {
                const int64_t tok = (b * seqlen + t) * dim + d;
                const int64_t row = (b * seqlen + t) * dstate;
                const double *h = hs + (t + 1) * dstate;      /* h_t */
                const double *hp = hs + t * dstate;           /* h_{t-1} */
                const double xv = x[tok];
                const double u = delta[tok] + bias;
                const double dt = delta_softplus ? oracle_softplus(u) : u;
                double yc = D ? D[d] * xv : 0.0;
                for (int64_t n = 0; n < dstate; ++n)
                    yc += C[row + n] * h[n];
                double dyc = dout[tok];
                if (z) {
                    const double s = 1.0 / (1.0 + exp(-z[tok]));
                    dyc = dout[tok] * z[tok] * s;
                    if (dz)
                        dz[tok] = dout[tok] * yc * s * (1.0 + z[tok] * (1.0 - s));
                }
                pD[d] += dyc * xv;
                double dxv = dyc * (D ? D[d] : 0.0);
                double ddt = 0.0;
                for (int64_t n = 0; n < dstate; ++n) {
                    const double a = A[d * dstate + n];
                    const double dAn = exp(dt * a);
                    g[n] += dyc * C[row + n];
                    pC[row + n] += dyc * h[n];
                    ddt += g[n] * (B[row + n] * xv + a * dAn * hp[n]);
                    pA[d * dstate + n] += g[n] * dt * dAn * hp[n];
                    pB[row + n] += g[n] * dt * xv;
                    dxv += dt * g[n] * B[row + n];
                    g[n] *= dAn;
                }
                const double du = delta_softplus ? ddt / (1.0 + exp(-u)) : ddt;
                if (dx)
                    dx[tok] = dxv;
                if (ddelta)
                    ddelta[tok] = du;
                pbias[d] += du;
            }
            if (dinitial_state)
                for (int64_t n = 0; n < dstate; ++n)
                    dinitial_state[(b * dim + d) * dstate + n] = g[n];
        }
    }
    /* add the per-thread partial sums in thread order */
    for (int64_t i = 0; i < nbc; ++i) {
        double sb = 0.0, sc = 0.0;
        for (int tid = 0; tid < nt; ++tid) {
            sb += part[(int64_t)tid * per + i];
            sc += part[(int64_t)tid * per + nbc + i];
        }
        if (dB)
            dB[i] = sb;
        if (dC)
            dC[i] = sc;
    }
    for (int64_t i = 0; i < dim * dstate + 2 * dim; ++i) {
        double s = 0.0;
        for (int tid = 0; tid < nt; ++tid)
            s += part[(int64_t)tid * per + 2 * nbc + i];
        if (i < dim * dstate) {
            if (dA)
                dA[i] = s;
        } else if (i < dim * dstate + dim) {
            if (dD)
                dD[i - dim * dstate] = s;
        } else if (ddelta_bias) {
            ddelta_bias[i - dim * dstate - dim] = s;
        }
    }
    free(part);
    free(hist);
    return 0;
}

/* Scalar helpers exposed for the pins on the nonlinearities. */
double oracle_softplus_scalar(double u) { return oracle_softplus(u); }
double oracle_silu_scalar(double v) { return oracle_silu(v); }
