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
 * The short convolution in front of the SSM (oracle_conv1d, oracle_conv1d_step):
 *   u_t = silu(bias + Σ_{k=0}^{W−1} w_k · x_{t−(W−1)+k})
 *           [a causal depthwise convolution of width 4, then SiLU, feeds the
 *           SSM branch: first-principles page — "The Mamba block"; erikxu.me
 *           notes — "Mamba Architecture"; the per-channel bias and width 4
 *           follow from the per-layer weight count on the first-principles
 *           page, "The Mamba block", which only adds up with D·4 + D
 *           convolution weights]
 *   inputs before the sequence come from a carried state of the last W−1
 *   inputs, oldest first (zeros when none) [three numbers per channel in the
 *   state count of "A fixed state against a growing cache" / "What a fixed
 *   state is bad at" on the same page].
 * Reading taken: tap k = W−1 multiplies the current input (the taps are the
 * filter in time order, oldest first); SiLU is optional so the plain
 * convolution can be checked on its own.
 *
 * The backward scan (oracle_scan_bwd) is the gradient of that forward map for
 * a loss whose gradient with respect to y is dy and with respect to hL is dhL
 * [the training half of the hardware-aware scan: erikxu.me notes — "GPU Memory
 * Hierarchy"; first-principles page — "The hardware-aware scan", which
 * recomputes the intermediate states in the backward pass instead of storing
 * them].  It runs the adjoint of the recurrence backwards in time,
 *   λ_t = C_t ŷ_t + Ā_{t+1} λ_{t+1},  λ_L = dhL,  ŷ_t = dy_t · silu(z_t),
 * and reads every input's gradient off it by the chain rule; the pages give no
 * formulas, so this is calculus on the forward definition above, and it is
 * pinned to central finite differences of oracle_scan.
 *
 * The Mamba-2 layer (oracle_ssd) restricts A_t to a scalar times the identity
 * per head: a_t = exp(Δ_t A_h), heads of P channels share a_t, B_t and C_t, and
 * each head's state is an N × P matrix [first-principles page — "Mamba-2:
 * state space duality"]:
 *   S_t = a_t S_{t−1} + Δ_t B_t x_tᵀ,   y_t = S_tᵀ C_t + D_h x_t.
 * The chunked SSD algorithm on the same page reaches exactly this result (it
 * reorders the same sums), so the oracle is the recurrence itself.
 *
 * Parity is pinned by tests/test_oracle_pins.py (worked example, convolution
 * kernel, gated-RNN reduction, Δ limits, first output, product-form brute
 * force, continuation; for the short convolution: numpy's convolution, the
 * impulse response, split and decode continuation, and the printed Mamba-2.8B
 * weight and state totals) and tests/test_oracle_mutants.py (planted mistakes
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

/*
 * Causal depthwise convolution + bias + optional SiLU over a whole sequence,
 * for every channel c = (b, d).
 *   x, u      : batch × dim × seqlen (time fastest)
 *   w         : dim × width (tap width−1 multiplies the current input)
 *   bias      : dim, may be NULL (zero)
 *   state_in  : batch × dim × (width−1), the inputs just before x[.., 0],
 *               oldest first; NULL = zeros
 *   state_out : batch × dim × (width−1), the last width−1 inputs of the
 *               sequence (reaching into state_in when seqlen < width−1),
 *               oldest first; NULL = not written.  Must not overlap state_in.
 * Returns 0, or -1 if width < 1.
 */
int oracle_conv1d(int64_t batch, int64_t dim, int64_t seqlen, int64_t width,
                  const double *x, const double *w, const double *bias, int silu,
                  const double *state_in, double *u, double *state_out)
{
    if (width < 1)
        return -1;
    const int64_t hist = width - 1;
    for (int64_t c = 0; c < batch * dim; ++c) {
        const int64_t d = c % dim;
        const double *x_c = x + c * seqlen;
        const double *s_c = state_in ? state_in + c * hist : NULL;
        /* the input at time s, reaching back into the carried state for s < 0 */
#define ORACLE_X_AT(s) ((s) >= 0 ? x_c[(s)] : (s_c ? s_c[hist + (s)] : 0.0))
        for (int64_t t = 0; t < seqlen; ++t) {
            double acc = bias ? bias[d] : 0.0;
            for (int64_t k = 0; k < width; ++k) {
                const int64_t s = t - hist + k;
                acc += w[d * width + k] * ORACLE_X_AT(s);
            }
            u[c * seqlen + t] = silu ? oracle_silu(acc) : acc;
        }
        if (state_out)
            for (int64_t j = 0; j < hist; ++j) {
                const int64_t s = seqlen - hist + j;
                state_out[c * hist + j] = ORACLE_X_AT(s);
            }
#undef ORACLE_X_AT
    }
    return 0;
}

/*
 * One decode token of the same convolution: the window is the carried state
 * (width−1 inputs, oldest first) followed by this token's input; the state
 * then drops its oldest input and appends this one, in place.
 *   state : batch × dim × (width−1)     x, u : batch × dim
 */
int oracle_conv1d_step(int64_t batch, int64_t dim, int64_t width, double *state,
                       const double *x, const double *w, const double *bias, int silu,
                       double *u)
{
    if (width < 1)
        return -1;
    const int64_t hist = width - 1;
    for (int64_t c = 0; c < batch * dim; ++c) {
        const int64_t d = c % dim;
        double *s_c = state + c * hist;
        double acc = bias ? bias[d] : 0.0;
        for (int64_t k = 0; k < hist; ++k)
            acc += w[d * width + k] * s_c[k];
        acc += w[d * width + hist] * x[c];
        u[c] = silu ? oracle_silu(acc) : acc;
        for (int64_t k = 0; k + 1 < hist; ++k)
            s_c[k] = s_c[k + 1];
        if (hist > 0)
            s_c[hist - 1] = x[c];
    }
    return 0;
}

/*
 * Gradient of the forward scan over channels [channel_begin, channel_end).
 * Inputs are those of oracle_scan, plus
 *   dy  : batch × dim × seqlen, ∂loss/∂y
 *   dhL : batch × dim × dstate, ∂loss/∂hL; NULL = 0
 * Written for the channels in range (any may be NULL = not wanted):
 *   du, ddelta (∂loss/∂Δraw), dz : batch × dim × seqlen
 *   dh0                          : batch × dim × dstate
 * ADDED to (the caller zeroes them; each channel range may use its own
 * buffers, to be summed afterwards):
 *   dB, dC : batch × dstate × seqlen   (sums over the channels)
 *   dA     : dim × dstate             (sums over batch and time)
 *   dDskip, dbias : dim
 * Returns 0, or -1 if dstate < 1 or scratch cannot be allocated.
 */
int oracle_scan_bwd(int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen,
                    const double *u, const double *delta, const double *z,
                    const double *B, const double *C, const double *A,
                    const double *Dskip, const double *bias,
                    int delta_softplus, int zoh, const double *h0,
                    const double *dy, const double *dhL,
                    double *du, double *ddelta, double *dz, double *dB, double *dC,
                    double *dA, double *dDskip, double *dbias, double *dh0,
                    int64_t channel_begin, int64_t channel_end)
{
    if (dstate < 1)
        return -1;
    const int64_t N = dstate, L = seqlen;
    /* h[(t + 1) * N + n] = h_t,n for t = -1 .. L-1; dt[t] = Δ_t; pre[t] = C·h + D·u */
    double *h = (double *)malloc((size_t)(L + 1) * N * sizeof(double));
    double *dt = (double *)malloc((size_t)L * sizeof(double));
    double *pre = (double *)malloc((size_t)L * sizeof(double));
    double *lam = (double *)malloc((size_t)N * sizeof(double));
    if (!h || !dt || !pre || !lam) {
        free(h); free(dt); free(pre); free(lam);
        return -1;
    }
    if (channel_end > batch * dim)
        channel_end = batch * dim;

    for (int64_t c = channel_begin; c < channel_end; ++c) {
        const int64_t b = c / dim;
        const int64_t d = c % dim;
        const double *u_c = u + c * L;
        const double *dr_c = delta + c * L;
        const double *z_c = z ? z + c * L : NULL;
        const double *dy_c = dy + c * L;
        const double *B_b = B + b * N * L;
        const double *C_b = C + b * N * L;
        const double *A_d = A + d * N;
        const double skip = Dskip ? Dskip[d] : 0.0;
        const double bias_d = bias ? bias[d] : 0.0;

        /* forward, keeping every state */
        for (int64_t n = 0; n < N; ++n)
            h[n] = h0 ? h0[c * N + n] : 0.0;
        for (int64_t t = 0; t < L; ++t) {
            double x = dr_c[t] + bias_d;
            dt[t] = delta_softplus ? oracle_softplus(x) : x;
            double s = 0.0;
            for (int64_t n = 0; n < N; ++n) {
                const double abar = exp(dt[t] * A_d[n]);
                const double bbar = oracle_bbar(dt[t], A_d[n], B_b[n * L + t], zoh);
                h[(t + 1) * N + n] = abar * h[t * N + n] + bbar * u_c[t];
                s += C_b[n * L + t] * h[(t + 1) * N + n];
            }
            pre[t] = s + skip * u_c[t];
        }

        /* backward in time */
        for (int64_t n = 0; n < N; ++n)
            lam[n] = dhL ? dhL[c * N + n] : 0.0;
        for (int64_t t = L - 1; t >= 0; --t) {
            double gate = 1.0;
            if (z_c) {
                const double sg = 1.0 / (1.0 + exp(-z_c[t]));
                gate = z_c[t] * sg;
                /* silu'(z) = σ(z) (1 + z (1 − σ(z))) */
                if (dz)
                    dz[c * L + t] = dy_c[t] * pre[t] * sg * (1.0 + z_c[t] * (1.0 - sg));
            }
            const double yhat = dy_c[t] * gate;          /* ∂loss/∂(C·h + D·u) */
            double du_t = yhat * skip;
            double ddt = 0.0;
            if (dDskip)
                dDskip[d] += yhat * u_c[t];
            for (int64_t n = 0; n < N; ++n) {
                const double a = A_d[n];
                const double Bv = B_b[n * L + t];
                const double hprev = h[t * N + n];
                const double abar = exp(dt[t] * a);
                lam[n] += C_b[n * L + t] * yhat;         /* λ_t: readout at t joins */
                dC[b * N * L + n * L + t] += yhat * h[(t + 1) * N + n];
                /* h_t = Ā h_{t-1} + B̄ u_t */
                const double dabar = lam[n] * hprev;
                const double dbbar = lam[n] * u_c[t];
                du_t += lam[n] * oracle_bbar(dt[t], a, Bv, zoh);
                ddt += dabar * abar * a;                 /* ∂Ā/∂Δ = A Ā */
                dA[d * N + n] += dabar * abar * dt[t];   /* ∂Ā/∂A = Δ Ā */
                if (!zoh || a == 0.0) {
                    /* B̄ = Δ B (also the A → 0 limit of the exact hold) */
                    ddt += dbbar * Bv;
                    dB[b * N * L + n * L + t] += dbbar * dt[t];
                    if (zoh)                             /* ∂B̄/∂A at A = 0: Δ² B / 2 */
                        dA[d * N + n] += dbbar * Bv * dt[t] * dt[t] * 0.5;
                } else {
                    /* B̄ = (Ā − 1)/A · B */
                    ddt += dbbar * abar * Bv;                               /* ∂B̄/∂Δ = Ā B */
                    dB[b * N * L + n * L + t] += dbbar * expm1(dt[t] * a) / a;
                    dA[d * N + n] += dbbar * Bv * (dt[t] * abar * a - expm1(dt[t] * a)) / (a * a);
                }
                lam[n] *= abar;                          /* on to ∂loss/∂h_{t-1} */
            }
            if (du)
                du[c * L + t] = du_t;
            /* Δ = softplus(Δraw + bias): ∂Δ/∂Δraw = σ(Δraw + bias) */
            double dx = ddt;
            if (delta_softplus)
                dx *= 1.0 / (1.0 + exp(-(dr_c[t] + bias_d)));
            if (ddelta)
                ddelta[c * L + t] = dx;
            if (dbias)
                dbias[d] += dx;
        }
        if (dh0)
            for (int64_t n = 0; n < N; ++n)
                dh0[c * N + n] = lam[n];
    }
    free(h); free(dt); free(pre); free(lam);
    return 0;
}

/*
 * Mamba-2 (SSD) forward for every batch element and head.
 *   x, y : batch × seqlen × nheads × headdim   (token-major, as the block's
 *          projection produces them)
 *   dt   : batch × seqlen × nheads             Δraw per head
 *   B, C : batch × seqlen × dstate             one group shared by all heads
 *   A, Dskip, dt_bias : nheads                 (Dskip, dt_bias may be NULL)
 *   h0, hL : batch × nheads × headdim × dstate (NULL = zeros / not written)
 * Δ = softplus(Δraw + dt_bias) when dt_softplus, else Δraw + dt_bias.
 * Returns 0, or -1 on bad sizes or allocation failure.
 */
int oracle_ssd(int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim, int64_t dstate,
               const double *x, const double *dt, const double *A, const double *B,
               const double *C, const double *Dskip, const double *dt_bias, int dt_softplus,
               const double *h0, double *y, double *hL)
{
    if (headdim < 1 || dstate < 1)
        return -1;
    const int64_t P = headdim, N = dstate, H = nheads, L = seqlen;
    double *S = (double *)malloc((size_t)P * N * sizeof(double));
    if (!S)
        return -1;
    for (int64_t b = 0; b < batch; ++b) {
        for (int64_t h = 0; h < H; ++h) {
            for (int64_t i = 0; i < P * N; ++i)
                S[i] = h0 ? h0[(b * H + h) * P * N + i] : 0.0;
            for (int64_t t = 0; t < L; ++t) {
                double d = dt[(b * L + t) * H + h] + (dt_bias ? dt_bias[h] : 0.0);
                if (dt_softplus)
                    d = oracle_softplus(d);
                const double a = exp(d * A[h]);
                const double *xt = x + ((b * L + t) * H + h) * P;
                const double *Bt = B + (b * L + t) * N;
                const double *Ct = C + (b * L + t) * N;
                double *yt = y + ((b * L + t) * H + h) * P;
                for (int64_t p = 0; p < P; ++p) {
                    double acc = 0.0;
                    for (int64_t n = 0; n < N; ++n) {
                        S[p * N + n] = a * S[p * N + n] + d * Bt[n] * xt[p];
                        acc += S[p * N + n] * Ct[n];
                    }
                    yt[p] = acc + (Dskip ? Dskip[h] : 0.0) * xt[p];
                }
            }
            if (hL)
                for (int64_t i = 0; i < P * N; ++i)
                    hL[(b * H + h) * P * N + i] = S[i];
        }
    }
    free(S);
    return 0;
}
