"""Pins that tie the fp64 oracle to what the pages and the mathematics fix.

Each ``pin_*`` function takes a loaded oracle library (ctypes) and raises
AssertionError when the oracle disagrees with an independently computed
expectation.  The expectations never reuse the oracle's sequential loop: they
come from printed values, the convolution view, the gated-RNN closed form,
limits, or the explicit product form of the unrolled recurrence.

tests/test_oracle_pins.py runs them on the real oracle; tests/test_oracle_mutants.py
runs them on deliberately broken copies of it and requires each copy to fail
at least one pin.
"""

from __future__ import annotations

import os

import numpy as np
from scipy.special import expit

from oracle import oracle as orc

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _softplus(x):
    return np.logaddexp(0.0, x)


def _silu(x):
    return x * expit(x)


def _close(got, want, rtol, atol=0.0, what=""):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    err = np.abs(got - want)
    bound = atol + rtol * np.abs(want)
    assert np.all(err <= bound), f"{what}: max err {err.max():.3e} (bound {bound.max():.3e})"


def read_golden(name="worked_example.txt"):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *nums = line.split()
            vals[key] = [float(x) for x in nums]
    return vals


# --------------------------------------------------------------------------
# P1: the worked example printed on "State space models and Mamba" —
# "A worked example".  a = 0.8 is Ā = exp(Δ·A) with A = ln(0.8)/Δ; b = 0.5 is
# the first-order B̄ = Δ·B with B = 0.5/Δ; C = 1, D = 0, no gate.

def pin_worked_example(lib):
    g = read_golden()
    a, bb, u = g["a"][0], g["b"][0], np.array(g["u"])
    L = len(u)
    for dt in (1.0, 2.0, 0.37):                       # Δ must cancel out of Ā and B̄
        A = np.array([[np.log(a) / dt]])
        B = np.full((1, 1, L), bb / dt)
        C = np.ones((1, 1, L))
        delta = np.full((1, 1, L), dt)
        y, hL = orc.scan(u.reshape(1, 1, L), delta, A, B, C, delta_softplus=False, lib=lib)
        _close(y[0, 0], g["y"], 1e-12, 1e-14, "worked example outputs")
        _close(hL[0, 0], [g["y"][-1]], 1e-12, 1e-14, "worked example final state")
        imp = np.zeros((1, 1, L))
        imp[0, 0, 0] = 1.0
        k, _ = orc.scan(imp, delta, A, B, C, delta_softplus=False, lib=lib)
        _close(k[0, 0], g["kernel"], 1e-12, 1e-14, "worked example kernel")
    # the page's convolution view of the third output: kernel · reversed input
    third = sum(g["kernel"][lag] * u[2 - lag] for lag in range(3))
    _close(third, g["y"][2], 1e-12, 0, "convolution view of the third output")


# --------------------------------------------------------------------------
# P2: with Δ, B and C fixed in time the recurrence is the causal convolution
# y = u * K̄, K̄_k = C Ā^k B̄ (Mamba notes on erikxu.me — "State Space Models";
# "State space models and Mamba" — "One system, two views", whose K_0 carries
# the D term).  A nonzero initial state h_{-1} adds C Ā^{t+1} h_{-1}.

def pin_lti_convolution(lib, seed=11):
    rng = np.random.default_rng(seed)
    b, dim, N, L = 2, 3, 4, 24
    A = -rng.uniform(0.1, 2.0, (dim, N))
    Braw = rng.normal(size=(b, N))
    Craw = rng.normal(size=(b, N))
    draw = rng.normal(size=(b, dim))
    bias = rng.normal(size=dim)
    Dsk = rng.normal(size=dim)
    u = rng.normal(size=(b, dim, L))
    z = rng.normal(size=(b, dim, L))
    h0 = rng.normal(size=(b, dim, N))
    B = np.repeat(Braw[:, :, None], L, axis=2)
    C = np.repeat(Craw[:, :, None], L, axis=2)
    delta = np.repeat(draw[:, :, None], L, axis=2)
    for zoh in (False, True):
        for use_h0 in (False, True):
            y, _ = orc.scan(u, delta, A, B, C, Dskip=Dsk, z=z, bias=bias,
                            h0=h0 if use_h0 else None, zoh=zoh, lib=lib)
            want = np.zeros_like(u)
            for bi in range(b):
                for d in range(dim):
                    dt = _softplus(draw[bi, d] + bias[d])
                    abar = np.exp(dt * A[d])
                    bbar = (np.expm1(dt * A[d]) / A[d] if zoh else dt) * Braw[bi]
                    K = np.array([np.sum(Craw[bi] * abar ** k * bbar) for k in range(L)])
                    K[0] += Dsk[d]                        # K_0 = D + C B̄
                    for t in range(L):
                        acc = sum(K[k] * u[bi, d, t - k] for k in range(t + 1))
                        if use_h0:
                            acc += np.sum(Craw[bi] * abar ** (t + 1) * h0[bi, d])
                        want[bi, d, t] = acc * _silu(z[bi, d, t])
            _close(y, want, 1e-10, 1e-12, f"LTI convolution (zoh={zoh}, h0={use_h0})")


# --------------------------------------------------------------------------
# P3: with N = 1, A = -1, B = 1 and Δ = softplus(z_t), exact zero-order hold
# gives the gated RNN h_t = (1 - σ(z_t)) h_{t-1} + σ(z_t) x_t
# (first-principles page — "Discretisation: zero-order hold"; fdeinterviews
# summary: with N = 1 the model is a gated RNN).

def pin_gated_rnn(lib, seed=12):
    rng = np.random.default_rng(seed)
    L = 40
    zt = rng.normal(0, 2, L)
    x = rng.normal(size=L)
    for h_init in (0.0, 1.7):
        y, hL = orc.scan(x.reshape(1, 1, L), zt.reshape(1, 1, L), np.array([[-1.0]]),
                         np.ones((1, 1, L)), np.ones((1, 1, L)),
                         h0=np.array([[[h_init]]]), delta_softplus=True, zoh=True, lib=lib)
        h = h_init
        want = []
        for t in range(L):
            g = expit(zt[t])
            h = (1 - g) * h + g * x[t]
            want.append(h)
        _close(y[0, 0], want, 1e-12, 1e-14, "gated RNN")
        _close(hL[0, 0], [want[-1]], 1e-12, 1e-14, "gated RNN state")


# --------------------------------------------------------------------------
# P4: the Δ limits (first-principles page — "Discretisation: zero-order hold";
# fdeinterviews summary): Δ → 0 keeps the state, Δ → ∞ wipes it; with exact
# ZOH, A = -1 and B = 1 the state becomes the current input; with the
# first-order B̄ it becomes Δ·B·u.

def pin_delta_limits(lib, seed=13):
    rng = np.random.default_rng(seed)
    b, dim, N, L = 1, 2, 5, 12
    A = -np.arange(1, N + 1, dtype=np.float64)[None].repeat(dim, 0)
    u = rng.normal(size=(b, dim, L))
    z = rng.normal(size=(b, dim, L))
    B = rng.normal(size=(b, N, L))
    C = rng.normal(size=(b, N, L))
    Dsk = rng.normal(size=dim)
    h0 = rng.normal(size=(b, dim, N))
    # Δ → 0: softplus(-40) ≈ 4e-18
    y, hL = orc.scan(u, np.full((b, dim, L), -40.0), A, B, C, Dskip=Dsk, z=z, h0=h0, lib=lib)
    _close(hL, h0, 1e-15, 1e-15, "Δ→0 keeps the state")
    want = np.einsum("bnt,bdn->bdt", C, h0) + Dsk[None, :, None] * u
    _close(y, want * _silu(z), 1e-14, 1e-15, "Δ→0 output reads the kept state")
    # Δ → ∞: the previous state no longer matters
    big = np.full((b, dim, L), 1e4)
    y1, h1 = orc.scan(u, big, A, B, C, Dskip=Dsk, z=z, h0=h0, delta_softplus=False, lib=lib)
    y2, h2 = orc.scan(u, big, A, B, C, Dskip=Dsk, z=z, h0=-3 * h0, delta_softplus=False, lib=lib)
    assert np.array_equal(y1, y2) and np.array_equal(h1, h2), "Δ→∞ must forget the initial state"
    _close(y1[..., 0], (np.einsum("bn,bn->b", C[..., 0], 1e4 * B[..., 0])[:, None] * u[..., 0]
                        + Dsk[None] * u[..., 0]) * _silu(z[..., 0]), 1e-12, 1e-12,
           "Δ→∞ first-order state is Δ·B·u")
    # exact ZOH, A = -1, B = 1, C = 1: h_t = u_t
    yz, hz = orc.scan(u[:, :1], big[:, :1], np.array([[-1.0]]), np.ones((1, 1, L)),
                      np.ones((1, 1, L)), h0=np.array([[[5.0]]]), delta_softplus=False,
                      zoh=True, lib=lib)
    _close(yz[0, 0], u[0, 0], 1e-15, 0, "Δ→∞ ZOH state is the current input")


# --------------------------------------------------------------------------
# P5: from h_{-1} = 0 the first state is B̄ x_0 and the first output C B̄ x_0
# (erikxu.me notes — "State Space Models"), plus the skip and the gate.

def pin_first_output(lib, seed=14):
    rng = np.random.default_rng(seed)
    b, dim, N, L = 2, 3, 8, 5
    A = -rng.uniform(0.2, 3, (dim, N))
    u = rng.normal(size=(b, dim, L))
    dr = rng.normal(size=(b, dim, L))
    z = rng.normal(size=(b, dim, L))
    B = rng.normal(size=(b, N, L))
    C = rng.normal(size=(b, N, L))
    Dsk = rng.normal(size=dim)
    bias = rng.normal(size=dim)
    y, _ = orc.scan(u, dr, A, B, C, Dskip=Dsk, z=z, bias=bias, lib=lib)
    for bi in range(b):
        for d in range(dim):
            dt = _softplus(dr[bi, d, 0] + bias[d])
            want = (np.dot(C[bi, :, 0], dt * B[bi, :, 0]) * u[bi, d, 0] + Dsk[d] * u[bi, d, 0])
            _close(y[bi, d, 0], want * _silu(z[bi, d, 0]), 1e-13, 1e-15, "first output")


# --------------------------------------------------------------------------
# P6: the unrolled time-varying recurrence written as explicit products,
# y_t = C_t·[Σ_{k≤t} (Π_{s=k+1..t} Ā_s) B̄_k u_k + (Π_{s≤t} Ā_s) h_{-1}] + D u_t
# (the selective output of the first-principles page — "Selection", whose
# display equation was lost; rebuilt from the recurrence), gated by silu(z).

def pin_product_form(lib, seed=15):
    rng = np.random.default_rng(seed)
    b, dim, N, L = 2, 3, 6, 14
    A = -rng.uniform(0.1, 2.5, (dim, N))
    u = rng.normal(size=(b, dim, L))
    dr = rng.normal(0, 0.8, (b, dim, L))
    z = rng.normal(size=(b, dim, L))
    B = rng.normal(size=(b, N, L))
    C = rng.normal(size=(b, N, L))
    Dsk = rng.normal(size=dim)
    bias = rng.normal(0, 0.5, dim)
    h0 = rng.normal(size=(b, dim, N))
    for zoh in (False, True):
        y, hL = orc.scan(u, dr, A, B, C, Dskip=Dsk, z=z, bias=bias, h0=h0, zoh=zoh, lib=lib)
        wy = np.zeros_like(u)
        wh = np.zeros_like(h0)
        for bi in range(b):
            for d in range(dim):
                dt = _softplus(dr[bi, d] + bias[d])                      # (L,)
                abar = np.exp(dt[:, None] * A[d][None, :])               # (L, N)
                if zoh:
                    bbar = np.expm1(dt[:, None] * A[d][None, :]) / A[d][None, :] * B[bi].T
                else:
                    bbar = dt[:, None] * B[bi].T                         # (L, N)
                for t in range(L):
                    state = np.prod(abar[:t + 1], axis=0) * h0[bi, d]
                    for k in range(t + 1):
                        state = state + np.prod(abar[k + 1:t + 1], axis=0) * bbar[k] * u[bi, d, k]
                    wy[bi, d, t] = (np.dot(C[bi, :, t], state) + Dsk[d] * u[bi, d, t]) * _silu(z[bi, d, t])
                    if t == L - 1:
                        wh[bi, d] = state
        _close(y, wy, 1e-11, 1e-13, f"product form outputs (zoh={zoh})")
        _close(hL, wh, 1e-11, 1e-13, f"product form final state (zoh={zoh})")


# --------------------------------------------------------------------------
# P7: the scan is a composition of affine maps h ↦ Ā h + B̄ u, associative
# (erikxu.me notes — "Mamba"; first-principles page — "The hardware-aware
# scan"), so a scan split at any token and resumed from the carried state
# equals the whole scan; and a scan of length L equals L single-token decode
# steps on a carried state.

def pin_continuation(lib, seed=16):
    rng = np.random.default_rng(seed)
    b, dim, N, L = 2, 4, 5, 33
    A = -rng.uniform(0.1, 2.0, (dim, N))
    u = rng.normal(size=(b, dim, L))
    dr = rng.normal(size=(b, dim, L))
    z = rng.normal(size=(b, dim, L))
    B = rng.normal(size=(b, N, L))
    C = rng.normal(size=(b, N, L))
    Dsk = rng.normal(size=dim)
    bias = rng.normal(size=dim)
    h0 = rng.normal(size=(b, dim, N))
    kw = dict(Dskip=Dsk, bias=bias, lib=lib)
    y, hL = orc.scan(u, dr, A, B, C, z=z, h0=h0, **kw)
    for cut in (1, 13, 32):
        ya, ha = orc.scan(u[..., :cut], dr[..., :cut], A, B[..., :cut], C[..., :cut],
                          z=z[..., :cut], h0=h0, **kw)
        yb, hb = orc.scan(u[..., cut:], dr[..., cut:], A, B[..., cut:], C[..., cut:],
                          z=z[..., cut:], h0=ha, **kw)
        _close(np.concatenate([ya, yb], -1), y, 1e-14, 1e-15, f"split at {cut}")
        _close(hb, hL, 1e-14, 1e-15, f"state after split at {cut}")
    # the same composition in pairs (a, b) ↦ (a2 a1, a2 b1 + b2), one channel
    bi, d = 1, 2
    dt = _softplus(dr[bi, d] + bias[d])
    a = np.exp(dt[:, None] * A[d][None])
    bb = dt[:, None] * B[bi].T * u[bi, d][:, None]
    P, S = np.ones(N), np.zeros(N)
    for t in range(L):
        P, S = a[t] * P, a[t] * S + bb[t]
    _close(hL[bi, d], P * h0[bi, d] + S, 1e-12, 1e-14, "affine-pair composition")


def pin_decode_equals_scan(lib, seed=17):
    rng = np.random.default_rng(seed)
    b, dim, N, T = 3, 4, 6, 20
    A = -rng.uniform(0.1, 2.0, (dim, N))
    u = rng.normal(size=(b, dim, T))
    dr = rng.normal(size=(b, dim, T))
    z = rng.normal(size=(b, dim, T))
    B = rng.normal(size=(b, N, T))
    C = rng.normal(size=(b, N, T))
    Dsk = rng.normal(size=dim)
    bias = rng.normal(size=dim)
    h0 = rng.normal(size=(b, dim, N))
    for zoh in (False, True):
        y, hL = orc.scan(u, dr, A, B, C, Dskip=Dsk, z=z, bias=bias, h0=h0, zoh=zoh, lib=lib)
        st = h0.copy()
        for t in range(T):
            yt, st = orc.step(st, u[..., t], dr[..., t], A, B[..., t], C[..., t], Dskip=Dsk,
                              z=z[..., t], bias=bias, zoh=zoh, lib=lib)
            _close(yt, y[..., t], 1e-13, 1e-15, f"decode token {t} (zoh={zoh})")
        _close(st, hL, 1e-13, 1e-15, f"decode carried state (zoh={zoh})")


# --------------------------------------------------------------------------
# P8: the short convolution in front of the SSM (first-principles page — "The
# Mamba block"; erikxu.me notes — "Mamba Architecture") is a causal FIR filter
# per channel: with no SiLU it is numpy's full convolution of the carried
# inputs followed by the sequence with the taps in reverse, cut to the
# sequence's positions, plus the bias; with SiLU it is that value times its
# logistic sigmoid.  The final state is the last W−1 inputs.

def pin_conv_library(lib, seed=18):
    rng = np.random.default_rng(seed)
    b, dim = 2, 3
    for W in (1, 2, 3, 4):
        for L in (1, 2, 5, 17):
            x = rng.normal(size=(b, dim, L))
            w = rng.normal(size=(dim, W))
            bias = rng.normal(size=dim)
            for st0 in (None, rng.normal(size=(b, dim, W - 1))):
                hist = np.zeros((b, dim, W - 1)) if st0 is None else st0
                full = np.concatenate([hist, x], axis=2)
                want = np.zeros((b, dim, L))
                for bi in range(b):
                    for d in range(dim):
                        want[bi, d] = np.convolve(full[bi, d], w[d][::-1])[W - 1:W - 1 + L] + bias[d]
                for silu in (False, True):
                    u, st = orc.conv1d(x, w, bias=bias, state_in=st0, silu=silu, lib=lib)
                    _close(u, _silu(want) if silu else want, 1e-13, 1e-14,
                           f"conv W={W} L={L} silu={silu} state={st0 is not None}")
                    _close(st, full[..., full.shape[2] - (W - 1):], 0, 0, f"conv state W={W} L={L}")


# P9: the taps in time order, oldest first: an impulse at τ comes out as the
# taps reversed, w_{W−1} at τ, w_{W−2} at τ+1, … — and nothing before τ.

def pin_conv_impulse(lib, seed=19):
    rng = np.random.default_rng(seed)
    W, L, tau = 4, 12, 5
    w = rng.normal(size=(1, W))
    x = np.zeros((1, 1, L))
    x[0, 0, tau] = 1.0
    u, _ = orc.conv1d(x, w, silu=False, lib=lib)
    want = np.zeros(L)
    for lag in range(W):
        want[tau + lag] = w[0, W - 1 - lag]
    _close(u[0, 0], want, 0, 0, "conv impulse response")
    # an impulse carried in the state at position j (oldest first) is the
    # input at time j − (W−1)
    for j in range(W - 1):
        st = np.zeros((1, 1, W - 1))
        st[0, 0, j] = 1.0
        u, _ = orc.conv1d(np.zeros((1, 1, L)), w, state_in=st, silu=False, lib=lib)
        want = np.zeros(L)
        for t in range(L):
            k = (j - (W - 1)) - t + (W - 1)  # tap that sees time j−(W−1) at output t
            if 0 <= k < W:
                want[t] = w[0, k]
        _close(u[0, 0], want, 0, 0, f"conv state impulse {j}")


# P10: the convolution state carries across any split of the sequence, and W−1
# inputs are all it needs: the sequence form equals one decode step per token.

def pin_conv_continuation(lib, seed=20):
    rng = np.random.default_rng(seed)
    b, dim, L = 2, 3, 23
    for W in (1, 2, 4):
        x = rng.normal(size=(b, dim, L))
        w = rng.normal(size=(dim, W))
        bias = rng.normal(size=dim)
        st0 = rng.normal(size=(b, dim, W - 1))
        u, st = orc.conv1d(x, w, bias=bias, state_in=st0, lib=lib)
        for cut in (1, 2, 11):
            ua, sa = orc.conv1d(x[..., :cut], w, bias=bias, state_in=st0, lib=lib)
            ub, sb = orc.conv1d(x[..., cut:], w, bias=bias, state_in=sa, lib=lib)
            _close(np.concatenate([ua, ub], -1), u, 1e-15, 1e-15, f"conv split at {cut}, W={W}")
            _close(sb, st, 0, 0, f"conv state after split at {cut}, W={W}")
        s = st0.copy()
        for t in range(L):
            ut, s = orc.conv1d_step(s, x[..., t], w, bias=bias, lib=lib)
            _close(ut, u[..., t], 1e-15, 1e-15, f"conv decode token {t}, W={W}")
        _close(s, st, 0, 0, f"conv decode state, W={W}")


# P11: the block's shapes against the totals printed for Mamba-2.8B
# (tests/golden/mamba28b_counts.txt).  A convolution of width 4 with one bias
# per channel is what makes the per-layer weights add up to the printed model
# total, and a state of W−1 = 3 inputs per channel, next to N = 16 SSM states,
# is what makes the printed whole-state size; the state length is taken from
# the oracle's own output.

def pin_block_counts(lib):
    g = {k: int(v[0]) for k, v in read_golden("mamba28b_counts.txt").items()}
    dm, E, N, R, W = g["d_model"], g["inner"], g["dstate"], g["dt_rank"], g["conv_width"]
    ssm = E * (R + 2 * N) + (R * E + E) + E * N + E        # x_proj, dt_proj (+bias), A, D
    assert ssm == g["ssm_weights_per_layer"]
    assert E * N == g["state_entries_per_layer"]
    conv = E * W + E                                       # depthwise taps + one bias per channel
    layer = dm * 2 * E + conv + ssm + E * dm + dm          # in_proj, conv, SSM, out_proj, norm
    assert g["layers"] * layer + g["vocab"] * dm + dm == g["total_weights"]
    _, st = orc.conv1d(np.zeros((1, 1, 5)), np.ones((1, W)), silu=False, lib=lib)
    per_channel_conv_state = st.shape[2]
    assert g["layers"] * E * (N + per_channel_conv_state) == g["whole_state"]
    assert g["pythia_tokens"] * 2 * g["pythia_layers"] * dm == g["whole_state"]


# --------------------------------------------------------------------------
# P12: the backward scan is the gradient of the forward map.  For the loss
# Σ w_y·y + Σ w_h·hL its output must equal central finite differences of the
# forward oracle in every input coordinate (the forward is independent code:
# oracle_scan), with and without SiLU gate, softplus, initial state, exact
# hold, and with an A entry of zero (the exact hold's A → 0 limit).

def pin_backward_finite_differences(lib, seed=21):
    rng = np.random.default_rng(seed)
    b, dim, N, L = 2, 3, 4, 6
    base = dict(u=rng.normal(size=(b, dim, L)), delta=rng.normal(size=(b, dim, L)),
                z=rng.normal(size=(b, dim, L)), B=rng.normal(size=(b, N, L)),
                C=rng.normal(size=(b, N, L)), A=-rng.uniform(0.2, 2.0, (dim, N)),
                Dskip=rng.normal(size=dim), bias=rng.normal(size=dim),
                h0=rng.normal(size=(b, dim, N)))
    base["A"][1, 2] = 0.0
    wy = rng.normal(size=(b, dim, L))
    wh = rng.normal(size=(b, dim, N))
    cases = [dict(zoh=False, softplus=True, gate=True, h0=True),
             dict(zoh=True, softplus=True, gate=True, h0=True),
             dict(zoh=False, softplus=False, gate=False, h0=False)]
    for cs in cases:
        inp = dict(base)
        if not cs["gate"]:
            inp["z"] = None
        if not cs["h0"]:
            inp["h0"] = None
        if not cs["softplus"]:
            inp["delta"] = np.abs(inp["delta"]) + 0.1        # Δ = Δraw + bias must stay usable
            inp["bias"] = np.abs(inp["bias"])

        def loss(**over):
            a = dict(inp)
            a.update(over)
            y, hL = orc.scan(a["u"], a["delta"], a["A"], a["B"], a["C"], Dskip=a["Dskip"], z=a["z"],
                             bias=a["bias"], h0=a["h0"], delta_softplus=cs["softplus"], zoh=cs["zoh"],
                             lib=lib)
            return float((wy * y).sum() + (wh * hL).sum())

        g = orc.scan_bwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], wy, Dskip=inp["Dskip"],
                         z=inp["z"], bias=inp["bias"], h0=inp["h0"], dhL=wh,
                         delta_softplus=cs["softplus"], zoh=cs["zoh"], lib=lib)
        names = [("u", "du"), ("delta", "ddelta"), ("B", "dB"), ("C", "dC"), ("A", "dA"),
                 ("Dskip", "dDskip"), ("bias", "dbias")]
        if cs["gate"]:
            names.append(("z", "dz"))
        if cs["h0"]:
            names.append(("h0", "dh0"))
        eps = 1e-6
        for name, key in names:
            arr = inp[name]
            fd = np.zeros_like(arr)
            for idx in np.ndindex(arr.shape):
                p_, m_ = arr.copy(), arr.copy()
                p_[idx] += eps
                m_[idx] -= eps
                fd[idx] = (loss(**{name: p_}) - loss(**{name: m_})) / (2 * eps)
            _close(g[key], fd, 0, 1e-7 * (1 + np.abs(fd).max()), f"backward {key} {cs}")


# --------------------------------------------------------------------------
# P13: a Mamba-2 head is Mamba-1 with one A for every state (first-principles
# page — "Mamba-2: state space duality": A_t is a scalar times the identity,
# heads of P channels share a_t, B_t and C_t).  oracle_ssd must equal
# oracle_scan run on the head's P channels with A[d, n] = A_h, Δraw of the head,
# the shared B, C, no gate — an independent implementation of the recurrence.

def pin_ssd_is_mamba1_with_scalar_A(lib, seed=22):
    rng = np.random.default_rng(seed)
    b, L, H, P, N = 2, 19, 3, 4, 5
    x = rng.normal(size=(b, L, H, P))
    dt = rng.normal(size=(b, L, H))
    A = -rng.uniform(0.2, 2.0, H)
    B = rng.normal(size=(b, L, N))
    C = rng.normal(size=(b, L, N))
    Dh = rng.normal(size=H)
    bias = rng.normal(size=H)
    h0 = rng.normal(size=(b, H, P, N))
    for soft in (True, False):
        dtu = dt if soft else np.abs(dt) + 0.05
        y, hL = orc.ssd(x, dtu, A, B, C, Dskip=Dh, dt_bias=bias if soft else None, h0=h0,
                        dt_softplus=soft, lib=lib)
        u = x.transpose(0, 2, 3, 1).reshape(b, H * P, L)              # channel h·P + p
        delta = np.repeat(dtu.transpose(0, 2, 1), P, axis=1)           # (b, H·P, L)
        A1 = np.repeat(A, P)[:, None].repeat(N, axis=1)                # (H·P, N)
        ym, hm = orc.scan(u, delta, A1, B.transpose(0, 2, 1), C.transpose(0, 2, 1), Dskip=np.repeat(Dh, P),
                          bias=np.repeat(bias, P) if soft else None, h0=h0.reshape(b, H * P, N),
                          delta_softplus=soft, lib=lib)
        _close(y, ym.reshape(b, H, P, L).transpose(0, 3, 1, 2), 1e-12, 1e-13, "SSD = Mamba-1 with scalar A")
        _close(hL, hm.reshape(b, H, P, N), 1e-12, 1e-13, "SSD final state")


# P14: the duality — unrolled, the layer is one masked matrix product
# Y = (L ∘ C Bᵀ)(Δ·X) + D X with L[i, j] = exp(Σ_{k=j+1..i} Δ_k A_h) for i >= j
# (and 0 above the diagonal), plus the initial state read through the decay
# from the start, exp(Σ_{k<=i} Δ_k A_h)·C_i·S_0 (same section: "the whole layer
# is one matrix product", causal attention with a decay mask).

def pin_ssd_matrix_form(lib, seed=23):
    rng = np.random.default_rng(seed)
    b, L, H, P, N = 2, 23, 2, 3, 6
    x = rng.normal(size=(b, L, H, P))
    dt = rng.normal(size=(b, L, H))
    A = -rng.uniform(0.1, 1.5, H)
    B = rng.normal(size=(b, L, N))
    C = rng.normal(size=(b, L, N))
    Dh = rng.normal(size=H)
    bias = rng.normal(size=H)
    h0 = rng.normal(size=(b, H, P, N))
    y, _ = orc.ssd(x, dt, A, B, C, Dskip=Dh, dt_bias=bias, h0=h0, lib=lib)
    want = np.zeros_like(y)
    for bi in range(b):
        for h in range(H):
            delta = _softplus(dt[bi, :, h] + bias[h])
            cs = np.cumsum(delta * A[h])
            Lm = np.tril(np.exp(cs[:, None] - cs[None, :]))
            G = C[bi] @ B[bi].T
            want[bi, :, h, :] = (Lm * G) @ (delta[:, None] * x[bi, :, h, :])
            want[bi, :, h, :] += np.exp(cs)[:, None] * (C[bi] @ h0[bi, h].T)
            want[bi, :, h, :] += Dh[h] * x[bi, :, h, :]
    _close(y, want, 1e-11, 1e-12, "SSD matrix form")


# P15: the Mamba-2 2.7B shapes against the printed totals: 80 heads × 64 = 5,120
# channels, an input projection 2·5120 + 2·128 + 80 wide (one B and C group,
# one Δ per head), and 40,216,560 weights per layer with a width-4 convolution
# over x, B, C (plus bias), per-head Δ bias, A and D, and a gated norm.

def pin_mamba2_counts(lib):
    g = {k: int(v[0]) for k, v in read_golden("mamba28b_counts.txt").items()}
    dm, H, P, N, W = g["d_model"], g["m2_heads"], g["m2_headdim"], g["m2_dstate"], g["conv_width"]
    E = H * P
    assert E == g["inner"]
    proj = 2 * E + 2 * N + H
    assert proj == g["m2_in_proj_out"]
    conv = (E + 2 * N) * (W + 1)
    layer = dm * proj + conv + 3 * H + E + E * dm + dm
    assert layer == g["m2_layer_weights"]


# P16: for fixed Δraw, B, C and z the selective scan is a linear time-varying
# system in its input and its initial state (erikxu.me notes — "State Space
# Models": h_t = Ā_t h_{t−1} + B̄_t x_t, y_t = C_t h_t; datarekha.com — "One
# system, two views": the D·x skip; the gate multiplies each token's output by
# silu(z_t), a fixed scale here): superposition holds for y and h_L, in both
# discretisations and in the decode step.

def pin_superposition(lib, seed=24):
    rng = np.random.default_rng(seed)
    b, dim, N, L = 2, 3, 5, 17
    A = -rng.uniform(0.1, 2.0, (dim, N))
    dr = rng.normal(size=(b, dim, L))
    z = rng.normal(size=(b, dim, L))
    B = rng.normal(size=(b, N, L))
    C = rng.normal(size=(b, N, L))
    Dsk = rng.normal(size=dim)
    bias = rng.normal(size=dim)
    u1, u2 = rng.normal(size=(b, dim, L)), rng.normal(size=(b, dim, L))
    h1, h2 = rng.normal(size=(b, dim, N)), rng.normal(size=(b, dim, N))
    al, be = 0.7, -1.3
    for zoh in (False, True):
        kw = dict(Dskip=Dsk, z=z, bias=bias, zoh=zoh, lib=lib)
        y1, s1 = orc.scan(u1, dr, A, B, C, h0=h1, **kw)
        y2, s2 = orc.scan(u2, dr, A, B, C, h0=h2, **kw)
        y, st = orc.scan(al * u1 + be * u2, dr, A, B, C, h0=al * h1 + be * h2, **kw)
        _close(y, al * y1 + be * y2, 1e-12, 1e-13, f"superposition y (zoh={zoh})")
        _close(st, al * s1 + be * s2, 1e-12, 1e-13, f"superposition h_L (zoh={zoh})")
        t = 5
        ya, sa = orc.step(h1.copy(), u1[..., t], dr[..., t], A, B[..., t], C[..., t], Dskip=Dsk,
                          z=z[..., t], bias=bias, zoh=zoh, lib=lib)
        yb, sb = orc.step(h2.copy(), u2[..., t], dr[..., t], A, B[..., t], C[..., t], Dskip=Dsk,
                          z=z[..., t], bias=bias, zoh=zoh, lib=lib)
        yc, sc = orc.step(al * h1 + be * h2, al * u1[..., t] + be * u2[..., t], dr[..., t], A, B[..., t],
                          C[..., t], Dskip=Dsk, z=z[..., t], bias=bias, zoh=zoh, lib=lib)
        _close(yc, al * ya + be * yb, 1e-12, 1e-13, f"superposition decode y (zoh={zoh})")
        _close(sc, al * sa + be * sb, 1e-12, 1e-13, f"superposition decode state (zoh={zoh})")


ALL_PINS = [pin_worked_example, pin_lti_convolution, pin_gated_rnn, pin_delta_limits,
            pin_first_output, pin_product_form, pin_continuation, pin_decode_equals_scan,
            pin_conv_library, pin_conv_impulse, pin_conv_continuation, pin_block_counts,
            pin_backward_finite_differences, pin_ssd_is_mamba1_with_scalar_A, pin_ssd_matrix_form,
            pin_mamba2_counts, pin_superposition]
