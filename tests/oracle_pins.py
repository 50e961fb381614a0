"""Pins for the fp64 oracle: checks against what the source pages and the mathematics fix,
independent of the oracle's own code. Each ``pin_*`` takes a loaded oracle library (so the
mutation tests can run the same pins against planted-mistake builds) and raises
AssertionError on failure.

Sources: "From RNN to Mamba: state-space model principles and long-sequence modelling in
practice" (lmnt.cn) -- section 2.1 (a time-invariant SSM is a convolution), section 2.2
(the recurrence is associative, so a parallel prefix scan equals the loop; inference falls
back to a serial recurrence holding one state), section 3.2 (the per-timestep loop);
"Mamba architecture principles and industrial long-text practice" (jsqmd.com), section 2.2
(softplus(x) = log(1 + e^x)) and section 3.4 (the scan as a composition of affine maps).
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _close(a, b, rtol, atol=0.0, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    err = np.abs(a - b)
    lim = atol + rtol * np.maximum(np.abs(b), 1e-300)
    assert np.all(err <= lim), f"{what}: max err {err.max():.3e} (rtol {rtol}, atol {atol})"


# P1 -- time-invariant case equals a convolution (section 2.1 of the lmnt.cn page).
def pin_lti_convolution(lib):
    rng = _rng(11)
    L, N = 97, 5
    for dt in (0.05, 0.7):
        A = -rng.uniform(0.1, 3.0, size=N)
        Bc = rng.standard_normal(N)
        Cc = rng.standard_normal(N)
        u = rng.standard_normal(L)
        Dv = 0.8
        # kernel K_k = sum_n C_n * exp(dt*A_n)^k * dt * B_n, from numpy powers
        k = np.arange(L)[:, None]
        K = (Cc[None, :] * np.power(np.exp(dt * A)[None, :], k) * dt * Bc[None, :]).sum(1)
        y_ref = np.convolve(u, K)[:L] + Dv * u
        y, h = oracle.scan_rows(u[None], np.full((1, L), dt), A[None],
                                np.repeat(Bc[:, None], L, 1)[None], np.repeat(Cc[:, None], L, 1)[None],
                                [0], D=[Dv], delta_softplus=False, lib=lib)
        _close(y[0], y_ref, 1e-11, 1e-12, "LTI convolution")
        # final state: h_L-1,n = sum_s exp(dt A_n)^(L-1-s) dt B_n u_s
        p = np.power(np.exp(dt * A)[:, None], (L - 1 - np.arange(L))[None, :])
        h_ref = (p * dt * Bc[:, None] * u[None, :]).sum(1)
        _close(h[0], h_ref, 1e-11, 1e-12, "LTI final state")


# P2 -- step -> 0: A_bar -> 1, B_bar -> 0, so y = D*u (times the gate).
def pin_tiny_step(lib):
    rng = _rng(12)
    L, N = 40, 6
    u = rng.standard_normal((2, L))
    z = rng.standard_normal((2, L))
    A = -np.arange(1, N + 1, dtype=float)[None].repeat(2, 0)
    B = rng.standard_normal((1, N, L))
    C = rng.standard_normal((1, N, L))
    Dv = np.array([1.0, -2.5])
    y, h = oracle.scan_rows(u, np.full((2, L), 1e-30), A, B, C, [0, 0], D=Dv, delta_softplus=False, lib=lib)
    _close(y, Dv[:, None] * u, 0.0, 1e-20, "step->0 ungated")
    assert np.all(np.abs(h) < 1e-20)
    # gated: y(z) - y(-z) = z * D*u (SiLU(z) - SiLU(-z) = z); at z = 0 the gate is exactly 0
    yp, _ = oracle.scan_rows(u, np.full((2, L), 1e-30), A, B, C, [0, 0], D=Dv, z=z, delta_softplus=False, lib=lib)
    ym, _ = oracle.scan_rows(u, np.full((2, L), 1e-30), A, B, C, [0, 0], D=Dv, z=-z, delta_softplus=False, lib=lib)
    _close(yp - ym, z * Dv[:, None] * u, 1e-12, 1e-20, "step->0 gated")
    z0 = z.copy()
    z0[:, ::3] = 0.0
    y0, _ = oracle.scan_rows(u, np.full((2, L), 1e-30), A, B, C, [0, 0], D=Dv, z=z0, delta_softplus=False, lib=lib)
    assert np.all(y0[:, ::3] == 0.0), "gate at z=0 must be exactly 0"


# P3 -- A = 0, step 1: the recurrence is a prefix sum of B*u (exact on integers).
def pin_prefix_sum(lib):
    rng = _rng(13)
    L, N = 64, 3
    u = rng.integers(-8, 9, size=(1, L)).astype(float)
    B = rng.integers(-5, 6, size=(1, N, L)).astype(float)
    C = rng.integers(-3, 4, size=(1, N, L)).astype(float)
    A = np.zeros((1, N))
    y, h = oracle.scan_rows(u, np.ones((1, L)), A, B, C, [0], D=[2.0], delta_softplus=False, lib=lib)
    hs = np.cumsum(B[0] * u[0][None, :], axis=1)          # [N, L] running sums
    y_ref = (C[0] * hs).sum(0) + 2.0 * u[0]
    assert np.array_equal(y[0], y_ref), "prefix-sum case must be exact"
    assert np.array_equal(h[0], hs[:, -1]), "prefix-sum final state must be exact"
    # N=1, C=1: y is literally the prefix sum of B*u
    y1, _ = oracle.scan_rows(u, np.ones((1, L)), np.zeros((1, 1)), B[:, :1], np.ones((1, 1, L)), [0], lib=lib)
    assert np.array_equal(y1[0], np.cumsum(B[0, 0] * u[0]))


# softplus reading: softplus(v) - softplus(-v) = v; pass-through above 20.
def pin_softplus(lib):
    v = np.array([-30.0, -7.0, -1.0, -1e-3, 0.0, 0.5, 3.0, 19.0, 25.0])
    L = 1
    # A = 0, B = C = u = 1, no D: y = softplus(delta + bias) exactly
    def run(delta, bias=None):
        y, _ = oracle.scan_rows(np.ones((len(delta), L)), np.asarray(delta, float)[:, None],
                                np.zeros((len(delta), 1)), np.ones((1, 1, L)), np.ones((1, 1, L)),
                                np.zeros(len(delta), dtype=np.int64), delta_bias=bias,
                                delta_softplus=True, lib=lib)
        return y[:, 0]
    sp, sm = run(v), run(-v)
    _close(sp - sm, v, 1e-12, 1e-9, "softplus(v) - softplus(-v) = v")
    assert run([0.0])[0] == math.log(2.0) or abs(run([0.0])[0] - math.log(2.0)) < 1e-16
    assert run([25.0])[0] == 25.0, "pass-through above the threshold"
    assert np.all(sp > 0)
    # the bias is added before the softplus: f(delta, bias) = f(delta + bias, 0)
    _close(run(v - 1.25, np.full(len(v), 1.25)), run(v), 1e-15, 1e-300, "bias before softplus")


# SiLU gate identity: SiLU(z) - SiLU(-z) = z, and SiLU(z) -> z for large z.
def pin_gate(lib):
    rng = _rng(14)
    L, N = 30, 4
    u = rng.standard_normal((1, L))
    d = np.full((1, L), 0.1)
    A = -np.arange(1, N + 1, dtype=float)[None]
    B = rng.standard_normal((1, N, L))
    C = rng.standard_normal((1, N, L))
    z = rng.standard_normal((1, L)) * 3
    y0, _ = oracle.scan_rows(u, d, A, B, C, [0], D=[0.3], delta_softplus=False, lib=lib)
    yp, _ = oracle.scan_rows(u, d, A, B, C, [0], D=[0.3], z=z, delta_softplus=False, lib=lib)
    ym, _ = oracle.scan_rows(u, d, A, B, C, [0], D=[0.3], z=-z, delta_softplus=False, lib=lib)
    _close(yp - ym, z * y0, 1e-12, 1e-13, "SiLU(z) - SiLU(-z) = z")
    yb, _ = oracle.scan_rows(u, d, A, B, C, [0], D=[0.3], z=np.full((1, L), 60.0), delta_softplus=False, lib=lib)
    _close(yb, 60.0 * y0, 1e-15, 1e-300, "SiLU(60) = 60")


# P4 -- associativity: splitting the sequence and resuming from the state equals the whole
# run; and a Hillis-Steele tree over the affine maps (a, b) equals the loop.
def pin_split_resume(lib):
    rng = _rng(15)
    Bt, Dm, L, N = 2, 3, 77, 5
    u = rng.standard_normal((Bt, Dm, L))
    de = rng.standard_normal((Bt, Dm, L)) * 0.5
    A = -rng.uniform(0.2, 4, size=(Dm, N))
    B = rng.standard_normal((Bt, N, L))
    C = rng.standard_normal((Bt, N, L))
    z = rng.standard_normal((Bt, Dm, L))
    bias = rng.uniform(-4, -1, size=Dm)
    Dv = rng.standard_normal(Dm)
    y, h = oracle.selective_scan(u, de, A, B, C, D=Dv, z=z, delta_bias=bias, delta_softplus=True, lib=lib)
    for m in (1, 30, 76):
        y1, h1 = oracle.selective_scan(u[..., :m], de[..., :m], A, B[..., :m], C[..., :m], D=Dv,
                                       z=z[..., :m], delta_bias=bias, delta_softplus=True, lib=lib)
        y2, h2 = oracle.selective_scan(u[..., m:], de[..., m:], A, B[..., m:], C[..., m:], D=Dv,
                                       z=z[..., m:], delta_bias=bias, delta_softplus=True, h0=h1, lib=lib)
        assert np.array_equal(y1, y[..., :m]), "prefix must not depend on the suffix"
        _close(y2, y[..., m:], 1e-13, 1e-14, f"resume at {m}")
        _close(h2, h, 1e-13, 1e-14, f"final state after resume at {m}")


def _tree_scan(a, b):
    """Inclusive Hillis-Steele scan of affine maps h -> a*h + b (pure Python, tiny L):
    (a1, b1) then (a2, b2) composes to (a1*a2, a2*b1 + b2)."""
    L = len(a)
    A, Bv = list(a), list(b)
    off = 1
    while off < L:
        A2, B2 = list(A), list(Bv)
        for t in range(off, L):
            A2[t] = A[t - off] * A[t]
            B2[t] = A[t] * Bv[t - off] + Bv[t]
        A, Bv = A2, B2
        off *= 2
    return Bv


def pin_tree_bruteforce(lib):
    rng = _rng(16)
    for L in (1, 2, 7, 32):
        N = 3
        u = rng.standard_normal(L)
        dt = np.log1p(np.exp(rng.standard_normal(L)))
        A = -rng.uniform(0.5, 2, size=N)
        B = rng.standard_normal((N, L))
        C = rng.standard_normal((N, L))
        y_ref = np.zeros(L)
        for n in range(N):
            a = [math.exp(dt[t] * A[n]) for t in range(L)]
            b = [dt[t] * B[n, t] * u[t] for t in range(L)]
            hs = _tree_scan(a, b)
            y_ref += np.array(hs) * C[n]
        y_ref += 0.7 * u
        y, _ = oracle.scan_rows(u[None], dt[None], A[None], B[None], C[None], [0], D=[0.7],
                                delta_softplus=False, lib=lib)
        _close(y[0], y_ref, 1e-12, 1e-13, f"tree scan L={L}")


# P5 -- linear in u (step, B, C fixed) and causal.
def pin_linear_causal(lib):
    rng = _rng(17)
    Bt, Dm, L, N = 1, 4, 50, 6
    u1, u2 = rng.standard_normal((2, Bt, Dm, L))
    de = rng.standard_normal((Bt, Dm, L))
    A = -rng.uniform(0.1, 5, size=(Dm, N))
    B = rng.standard_normal((Bt, N, L))
    C = rng.standard_normal((Bt, N, L))
    Dv = rng.standard_normal(Dm)
    kw = dict(D=Dv, delta_softplus=True, lib=lib)
    ya, ha = oracle.selective_scan(u1, de, A, B, C, **kw)
    yb, hb = oracle.selective_scan(u2, de, A, B, C, **kw)
    yc, hc = oracle.selective_scan(2.5 * u1 - 0.75 * u2, de, A, B, C, **kw)
    _close(yc, 2.5 * ya - 0.75 * yb, 1e-11, 1e-12, "linearity y")
    _close(hc, 2.5 * ha - 0.75 * hb, 1e-11, 1e-12, "linearity state")
    t0 = 23
    up = u1.copy()
    up[..., t0] += 3.0
    yp, _ = oracle.selective_scan(up, de, A, B, C, **kw)
    assert np.array_equal(yp[..., :t0], ya[..., :t0]), "causality"
    assert np.all(yp[..., t0] != ya[..., t0])


# P6 -- the hand-worked scalar case (tests/golden/hand_scalar_n1_l3.json).
def pin_hand_case(lib):
    with open(os.path.join(GOLDEN, "hand_scalar_n1_l3.json")) as f:
        g = json.load(f)
    i = g["inputs"]
    L = len(i["u"])
    y, h = oracle.scan_rows(np.array([i["u"]]), np.array([i["delta"]]), np.array([[i["A"]]]),
                            np.array([[i["B"]]]), np.array([[i["C"]]]), [0], D=[i["D"]],
                            delta_softplus=False, lib=lib)
    assert L == 3
    _close(y[0], g["expected"]["y"], 1e-14, 1e-14, "hand case y")
    _close(h[0, 0], g["expected"]["last_state"], 1e-14, 1e-14, "hand case state")


# P7 -- the recurrent step, applied k times, equals the scan started from the same state.
def pin_decode_equals_scan(lib):
    rng = _rng(18)
    Bt, Dm, N, S = 3, 5, 4, 64
    A = -rng.uniform(0.1, 6, size=(Dm, N))
    st0 = rng.standard_normal((Bt, Dm, N))
    x = rng.standard_normal((S, Bt, Dm))
    dt = np.log1p(np.exp(rng.standard_normal((S, Bt, Dm)) - 2))
    B = rng.standard_normal((S, Bt, N))
    C = rng.standard_normal((S, Bt, N))
    z = rng.standard_normal((S, Bt, Dm))
    Dv = rng.standard_normal(Dm)
    st = st0
    ys = []
    for s in range(S):
        y, st = oracle.state_update(st, x[s], dt[s], A, B[s], C[s], D=Dv, z=z[s], lib=lib)
        ys.append(y)
    ys = np.stack(ys, -1)                                   # [Bt, D, S]
    yr, hr = oracle.selective_scan(np.moveaxis(x, 0, -1), np.moveaxis(dt, 0, -1), A,
                                   np.moveaxis(B, 0, -1), np.moveaxis(C, 0, -1), D=Dv,
                                   z=np.moveaxis(z, 0, -1), delta_softplus=False, h0=st0, lib=lib)
    _close(ys, yr, 1e-13, 1e-14, "decode vs scan outputs")
    _close(st, hr, 1e-13, 1e-14, "decode vs scan state")


# Magnitude companion: bounds |y| and |h|, and equals them when every term is >= 0.
def pin_magnitude(lib):
    rng = _rng(19)
    Bt, Dm, L, N = 1, 3, 40, 4
    u = rng.standard_normal((Bt, Dm, L))
    de = rng.standard_normal((Bt, Dm, L))
    A = -rng.uniform(0.1, 3, size=(Dm, N))
    B = rng.standard_normal((Bt, N, L))
    C = rng.standard_normal((Bt, N, L))
    z = rng.standard_normal((Bt, Dm, L))
    y, h, ym, hm = oracle.selective_scan(u, de, A, B, C, D=np.ones(Dm), z=z, delta_softplus=True,
                                         with_mag=True, lib=lib)
    assert np.all(np.abs(y) <= ym * (1 + 1e-12)) and np.all(np.abs(h) <= hm * (1 + 1e-12))
    y2, h2, ym2, hm2 = oracle.selective_scan(np.abs(u), de, A, np.abs(B), np.abs(C), D=np.ones(Dm),
                                             delta_softplus=True, with_mag=True, lib=lib)
    _close(ym2, y2, 1e-13, 0, "companion equals y for non-negative terms")
    _close(hm2, h2, 1e-13, 0, "companion equals state for non-negative terms")


# ---- exact zero-order hold (jsqmd.com "Mamba architecture principles ...", section 2.3) ----
# The ZOH discretisation samples the continuous system dh/dtau = A h + B u, with u and B held
# constant over each step, exactly at the step ends.

# Constant input from h = 0: h(tau) = (exp(A tau) - 1)/A * B u  (tau * B u for A = 0).
def pin_zoh_step_response(lib):
    rng = _rng(21)
    L, N, dt, uu = 60, 5, 0.13, 0.7
    A = np.array([-3.0, -0.4, -1e-3, 0.0, 0.5])
    Bc, Cc = rng.standard_normal(N), rng.standard_normal(N)
    y, h = oracle.scan_rows(np.full((1, L), uu), np.full((1, L), dt), A[None],
                            np.repeat(Bc[:, None], L, 1)[None], np.repeat(Cc[:, None], L, 1)[None],
                            [0], delta_softplus=False, lib=lib, zoh=True)
    tau = dt * (np.arange(L) + 1)
    with np.errstate(divide="ignore", invalid="ignore"):
        g = np.where(A[:, None] == 0, tau[None, :], np.expm1(A[:, None] * tau[None, :]) / A[:, None])
    h_ref = g * (Bc * uu)[:, None]                                # [N, L]
    _close(y[0], (Cc[:, None] * h_ref).sum(0), 1e-11, 1e-13, "ZOH step response y")
    _close(h[0], h_ref[:, -1], 1e-11, 1e-13, "ZOH step response state")


# Varying steps, inputs and B: each step integrated as an ODE by scipy (no closed form used).
def pin_zoh_piecewise_ode(lib):
    from scipy.integrate import solve_ivp
    rng = _rng(22)
    L, N = 12, 3
    A = np.array([-2.0, -0.3, 0.2])
    dt = rng.uniform(0.05, 0.6, L)
    u = rng.standard_normal(L)
    B = rng.standard_normal((N, L))
    C = rng.standard_normal((N, L))
    y, h = oracle.scan_rows(u[None], dt[None], A[None], B[None], C[None], [0],
                            delta_softplus=False, lib=lib, zoh=True)
    hs = np.zeros(N)
    for t in range(L):
        sol = solve_ivp(lambda _tau, x, t=t: A * x + B[:, t] * u[t], (0.0, dt[t]), hs,
                        rtol=1e-12, atol=1e-14, method="DOP853")
        hs = sol.y[:, -1]
        _close(y[0, t], (C[:, t] * hs).sum(), 1e-8, 1e-10, f"ZOH vs ODE y[{t}]")
    _close(h[0], hs, 1e-8, 1e-10, "ZOH vs ODE state")


# As the step goes to zero ZOH and the Euler step agree to first order in dt*A.
def pin_zoh_small_step_limit(lib):
    rng = _rng(23)
    L, N = 50, 4
    A = -rng.uniform(0.5, 4, N)
    u = rng.standard_normal(L)
    B = rng.standard_normal((N, L))
    C = rng.standard_normal((N, L))
    dt = np.full(L, 1e-7)
    yz, hz = oracle.scan_rows(u[None], dt[None], A[None], B[None], C[None], [0], lib=lib, zoh=True)
    ye, he = oracle.scan_rows(u[None], dt[None], A[None], B[None], C[None], [0], lib=lib, zoh=False)
    _close(hz, he, 1e-5, 0.0, "ZOH -> Euler as dt -> 0")
    assert np.max(np.abs(hz - he)) > 0.0, "ZOH flag has no effect"


# The recurrent step with ZOH equals the ZOH scan started from the same state.
def pin_zoh_decode_equals_scan(lib):
    rng = _rng(24)
    Bt, Dm, N, S = 2, 3, 4, 40
    A = -rng.uniform(0.1, 6, size=(Dm, N))
    st0 = rng.standard_normal((Bt, Dm, N))
    x = rng.standard_normal((S, Bt, Dm))
    dt = np.log1p(np.exp(rng.standard_normal((S, Bt, Dm)) - 1))
    B = rng.standard_normal((S, Bt, N))
    C = rng.standard_normal((S, Bt, N))
    st = st0
    ys = []
    for s in range(S):
        y, st = oracle.state_update(st, x[s], dt[s], A, B[s], C[s], lib=lib, zoh=True)
        ys.append(y)
    yr, hr = oracle.selective_scan(np.moveaxis(x, 0, -1), np.moveaxis(dt, 0, -1), A,
                                   np.moveaxis(B, 0, -1), np.moveaxis(C, 0, -1),
                                   delta_softplus=False, h0=st0, lib=lib, zoh=True)
    _close(np.stack(ys, -1), yr, 1e-13, 1e-14, "ZOH decode vs scan outputs")
    _close(st, hr, 1e-13, 1e-14, "ZOH decode vs scan state")


# ---- conv-to-gate span (lmnt.cn sections 3.1-3.2: depthwise Conv1d, padding d_conv-1,
# output cut to L, then SiLU) --------------------------------------------------------------
def _silu(v):
    return v / (1.0 + np.exp(-v))


# The causal correlation equals numpy's full convolution with the reversed kernel, cut to L.
def pin_conv_numpy(lib):
    rng = _rng(31)
    nch, L = 4, 37
    for K in (1, 2, 4):
        x = rng.standard_normal((nch, L))
        w = rng.standard_normal((nch, K))
        cb = rng.standard_normal(nch)
        u = oracle.conv_silu(x, w, cb, lib=lib)
        ref = np.stack([np.convolve(x[c], w[c][::-1])[:L] + cb[c] for c in range(nch)])
        _close(u, _silu(ref), 1e-13, 1e-15, f"conv K={K} vs numpy")


# The page's module itself: torch Conv1d(groups=D, padding=K-1) in fp64, cut to L, SiLU.
def pin_conv_torch_module(lib):
    import torch
    rng = _rng(32)
    Dm, L, K = 6, 29, 4
    x = rng.standard_normal((2, Dm, L))
    conv = torch.nn.Conv1d(Dm, Dm, kernel_size=K, groups=Dm, padding=K - 1, dtype=torch.float64)
    with torch.no_grad():
        conv.weight.copy_(torch.from_numpy(rng.standard_normal((Dm, 1, K))))
        conv.bias.copy_(torch.from_numpy(rng.standard_normal(Dm)))
        ref = torch.nn.functional.silu(conv(torch.from_numpy(x))[:, :, :L]).numpy()
    w = conv.weight.detach().numpy()[:, 0, :]
    cb = conv.bias.detach().numpy()
    u = oracle.conv_silu(x, np.broadcast_to(w, (2, Dm, K)), np.broadcast_to(cb, (2, Dm)), lib=lib)
    _close(u, ref, 1e-13, 1e-15, "conv vs torch Conv1d module")


# ---- backward (gradients of the loop, by PyTorch autograd in float64) ----------------------
# The autograd forward equals the C oracle, and every gradient equals a central finite
# difference of the C oracle's forward (an independent derivative of the pinned loop).
def pin_backward_finite_differences(lib):
    import torch

    from oracle import backward as bwd
    rng = _rng(41)
    Bt, Dm, L, N = 1, 2, 9, 3
    ins = {"u": rng.standard_normal((Bt, Dm, L)), "delta": rng.standard_normal((Bt, Dm, L)) * 0.5,
           "A": -rng.uniform(0.3, 2.0, (Dm, N)), "B": rng.standard_normal((Bt, N, L)),
           "C": rng.standard_normal((Bt, N, L)), "D": rng.standard_normal(Dm),
           "z": rng.standard_normal((Bt, Dm, L)), "delta_bias": rng.standard_normal(Dm) * 0.3}
    dy = rng.standard_normal((Bt, Dm, L))
    dlast = rng.standard_normal((Bt, Dm, N))

    def f(x):
        y, h = oracle.selective_scan(x["u"], x["delta"], x["A"], x["B"], x["C"], D=x["D"], z=x["z"],
                                     delta_bias=x["delta_bias"], delta_softplus=True, lib=lib)
        return float((y * dy).sum() + (h * dlast).sum())

    tt = {k: torch.tensor(v) for k, v in ins.items()}
    yt, ht = bwd.scan_forward_torch(tt["u"], tt["delta"], tt["A"], tt["B"], tt["C"], D=tt["D"], z=tt["z"],
                                    delta_bias=tt["delta_bias"])
    yo, ho = oracle.selective_scan(ins["u"], ins["delta"], ins["A"], ins["B"], ins["C"], D=ins["D"], z=ins["z"],
                                   delta_bias=ins["delta_bias"], delta_softplus=True, lib=lib)
    _close(yt.detach().numpy(), yo, 1e-12, 1e-13, "autograd forward vs C oracle")
    g = bwd.scan_backward(**ins, delta_softplus=True, dy=dy, dlast=dlast)
    eps = 1e-6
    # every index of every input (118 on this shape): a gradient that is wrong at a single
    # position -- one state, one timestep, the last step's D term -- cannot slip through
    for k, arr in ins.items():
        for idx in np.ndindex(arr.shape):
            xp = {kk: vv.copy() for kk, vv in ins.items()}
            xm = {kk: vv.copy() for kk, vv in ins.items()}
            xp[k][idx] += eps
            xm[k][idx] -= eps
            fd = (f(xp) - f(xm)) / (2 * eps)
            _close(g[k][idx], fd, 1e-6, 1e-7, f"d/d{k}{idx}: autograd vs finite differences")


ALL_PINS = [pin_backward_finite_differences, pin_conv_numpy, pin_conv_torch_module, pin_zoh_step_response, pin_zoh_piecewise_ode, pin_zoh_small_step_limit,
            pin_zoh_decode_equals_scan, pin_lti_convolution, pin_tiny_step, pin_prefix_sum, pin_softplus, pin_gate,
            pin_split_resume, pin_tree_bruteforce, pin_linear_causal, pin_hand_case,
            pin_decode_equals_scan, pin_magnitude]
