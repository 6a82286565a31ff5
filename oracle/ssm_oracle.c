/*
 * ssm_oracle.c — fp64 CPU oracle for the Mamba selective scan and its
 * single-token decode step.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, sequential
 * definition that the CUDA path is checked against.  It shares no code, header
 * or constant with the CUDA library; only the test suite, the smoke check and
 * the benchmark's CPU-baseline leg load it.  The product path never calls it.
 *
 * What it computes, and where the pages say so:
 *
 *   Δ_t   = softplus(Δraw_t + bias)                [Mamba and selective state
 *           spaces, from first principles — "Selection: B, C and Δ from the
 *           token"; Δ kept positive by a softplus: Mamba: Linear-Time Sequence
 *           Modeling with Selective State Spaces (erikxu.me notes) — "Mamba"]
 *   Ā_t,n = exp(Δ_t · A_n)                          [first-principles page —
 *           "Discretisation: zero-order hold" and "Selection"]
 *   B̄_t,n = Δ_t · B_t,n          (first-order form; the first-principles page,
 *           "Discretisation: zero-order hold", says this is what the reference
 *           implementation computes)
 *         = (exp(Δ_t A_n) − 1)/A_n · B_t,n   (exact zero-order hold: the
 *           integral ∫₀^Δ e^{sA} ds · B named on the same page, evaluated for
 *           one diagonal entry; Δ·B when A_n = 0)
 *   h_t,n = Ā_t,n h_{t−1},n + B̄_t,n u_t,   h_{−1} = h0 (zero by default)
 *           [erikxu.me notes — "State Space Models", the discrete system and
 *           h_{−1}=0; State space models and Mamba — "One system, two views"]
 *   y_t   = (Σ_n C_t,n h_t,n + D u_t) · silu(z_t)
 *           [D term: State space models and Mamba — "One system, two views";
 *           the SiLU gate branch multiplies the SSM output: first-principles
 *           page — "The Mamba block", erikxu.me notes — "Mamba Architecture"]
 *
 * The decode step is the same body with L = 1 on a carried state
 * [first-principles page — "A fixed state against a growing cache"; State
 * space models and Mamba — "One system, two views", streaming inference].
 *
 * Readings taken where the pages are silent:
 *   - the gate multiplies the whole SSM output including D·u;
 *   - softplus is evaluated exactly, x + log1p(e^{-x}) for x > 0 and
 *     log1p(e^x) otherwise;
 *   - the bias is one value per channel, added before the softplus.
 *
 * Parity is pinned by tests/test_oracle_pins.py (worked example, convolution
 * kernel, gated-RNN reduction, Δ limits, first output, product-form brute
 * force, continuation) and tests/test_oracle_mutants.py (planted mistakes
 * must fail a pin).
 *
 * Layouts (all row-major, fp64):
 *   u, delta, z, y : batch × dim × seqlen    (time fastest)
 *   B, C           : batch × dstate × seqlen (time fastest)
 *   A              : dim × dstate
 *   Dskip, bias    : dim
 *   h0, hL         : batch × dim × dstate
 * z, Dskip, bias, h0 and hL may be NULL (no gate, zero, zero, zero, not
 * written).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>

static double oracle_softplus(double x)
{
    return x > 0.0 ? x + log1p(exp(-x)) : log1p(exp(x));
}

static double oracle_silu(double x)
{
    return x / (1.0 + exp(-x));
}

/* The input weight B̄ for one (t, n).  zoh == 0: first order Δ·B.
 * zoh != 0: exact zero-order hold (e^{ΔA} − 1)/A · B, with the A = 0 limit. */
static double oracle_bbar(double delta, double a, double b, int zoh)
{
    if (!zoh || a == 0.0)
        return delta * b;
    return expm1(delta * a) / a * b;
}

/*
 * Full forward scan over channels [channel_begin, channel_end) of the
 * batch × dim channel grid (channel c is batch c / dim, inner channel c % dim).
 * Returns 0, or -1 if dstate < 1 or the scratch state cannot be allocated.
 */
int oracle_scan(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
                const double *u, const double *delta, const double *z,
                const double *B, const double *C, const double *A,
                const double *Dskip, const double *bias,
                int delta_softplus, int zoh, const double *h0,
                double *y, double *hL,
                int64_t channel_begin, int64_t channel_end)
{
    if (dstate < 1)
        return -1;
    double *h = (double *)malloc((size_t)dstate * sizeof(double));
    if (!h)
        return -1;
    if (channel_end > batch * dim)
        channel_end = batch * dim;

    for (int64_t c = channel_begin; c < channel_end; ++c) {
        const int64_t b = c / dim;
        const int64_t d = c % dim;
        const double *u_c = u + c * seqlen;
        const double *dt_c = delta + c * seqlen;
        const double *z_c = z ? z + c * seqlen : NULL;
        const double *B_b = B + b * dstate * seqlen;
        const double *C_b = C + b * dstate * seqlen;
        const double *A_d = A + d * dstate;
        const double skip = Dskip ? Dskip[d] : 0.0;
        const double bias_d = bias ? bias[d] : 0.0;
        double *y_c = y + c * seqlen;

        for (int64_t n = 0; n < dstate; ++n)
            h[n] = h0 ? h0[c * dstate + n] : 0.0;

        for (int64_t t = 0; t < seqlen; ++t) {
            double dt = dt_c[t] + bias_d;
            if (delta_softplus)
                dt = oracle_softplus(dt);
            double s = 0.0;
            for (int64_t n = 0; n < dstate; ++n) {
                const double abar = exp(dt * A_d[n]);
                const double bbar = oracle_bbar(dt, A_d[n], B_b[n * seqlen + t], zoh);
                h[n] = abar * h[n] + bbar * u_c[t];
                s += C_b[n * seqlen + t] * h[n];
            }
            double out = s + skip * u_c[t];
            if (z_c)
                out *= oracle_silu(z_c[t]);
            y_c[t] = out;
        }

        if (hL)
            for (int64_t n = 0; n < dstate; ++n)
                hL[c * dstate + n] = h[n];
    }
    free(h);
    return 0;
}

/*
 * One decode token for every channel: the scan body with seqlen = 1 on the
 * carried state, which is read and overwritten in place.
 *   state : batch × dim × dstate     u, delta, z, y : batch × dim
 *   B, C  : batch × dstate           A : dim × dstate; Dskip, bias : dim
 */
int oracle_step(int64_t batch, int64_t dim, int64_t dstate,
                double *state, const double *u, const double *delta,
                const double *z, const double *B, const double *C,
                const double *A, const double *Dskip, const double *bias,
                int delta_softplus, int zoh, double *y)
{
    if (dstate < 1)
        return -1;
    for (int64_t b = 0; b < batch; ++b) {
        for (int64_t d = 0; d < dim; ++d) {
            const int64_t c = b * dim + d;
            double dt = delta[c] + (bias ? bias[d] : 0.0);
            if (delta_softplus)
                dt = oracle_softplus(dt);
            double s = 0.0;
            for (int64_t n = 0; n < dstate; ++n) {
                const double a = A[d * dstate + n];
                const double abar = exp(dt * a);
                const double bbar = oracle_bbar(dt, a, B[b * dstate + n], zoh);
                double *h = &state[c * dstate + n];
                *h = abar * *h + bbar * u[c];
                s += C[b * dstate + n] * *h;
            }
            double out = s + (Dskip ? Dskip[d] : 0.0) * u[c];
            if (z)
                out *= oracle_silu(z[c]);
            y[c] = out;
        }
    }
    return 0;
}
