"""Independent pins for the fp64 oracle.

Each pin computes what the scan must return from something other than the
oracle's own loop -- a closed form, a textbook special case, a library
routine (numpy / scipy) or a hand-derived fixture -- and raises
AssertionError when the oracle (``lib``: the library under test, which may be
a deliberately broken copy) disagrees.  Chosen so that a dropped term, a
wrong sign, a lagged time index, transposed B/C, a missing softplus/bias or a
gate applied before the skip each fail at least one pin.
"""
from __future__ import annotations

import math
import os

import numpy as np
from scipy.special import expit

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def softplus_ref(u):
    return np.logaddexp(0.0, u)          # numpy's log(e^0 + e^u)


def silu_ref(v):
    return v * expit(v)                  # scipy's logistic sigmoid


def rand_problem(seed, bsz=2, L=12, dim=3, N=4, init=True, lti=False):
    r = np.random.default_rng(seed)
    x = r.standard_normal((bsz, L, dim))
    z = r.standard_normal((bsz, L, dim))
    dl = r.standard_normal((bsz, L, dim))
    bias = np.log(np.expm1(r.uniform(0.05, 0.5, dim)))
    B = r.standard_normal((bsz, L, N))
    C = r.standard_normal((bsz, L, N))
    A = -np.exp(r.uniform(-1.0, 1.5, (dim, N)))
    D = r.standard_normal(dim)
    h0 = r.standard_normal((bsz, dim, N)) if init else None
    if lti:
        dl[:] = dl[:, :1, :]
        B[:] = B[:, :1, :]
        C[:] = C[:, :1, :]
    return dict(x=x, delta=dl, z=z, A=A, B=B, C=C, D=D, delta_bias=bias, initial_state=h0)


def _run(lib, p, **kw):
    args = dict(p)
    args.update(kw)
    return oracle.scan_fwd(lib=lib, **args)


def _rel(a, b):
    return float(np.max(np.abs(a - b) / (1.0 + np.abs(b))))


# P1 -- brute-force closed form y_t = sum_{s<=t} C_t . (prod_{r=s+1..t} dA_r) dBx_s
#       (+ the decayed initial state), skip, gate; O(L^2 N) with explicit products.
def pin_closed_form(lib):
    p = rand_problem(1)
    out, last = _run(lib, p)
    x, z, dl, A, B, C, D = (p[k] for k in ("x", "z", "delta", "A", "B", "C", "D"))
    dt = softplus_ref(dl + p["delta_bias"])
    bsz, L, dim = x.shape
    N = A.shape[1]
    ref = np.zeros_like(out)
    last_ref = np.zeros_like(last)
    for b in range(bsz):
        for d in range(dim):
            for t in range(L):
                hs = np.zeros(N)
                prod0 = np.ones(N)
                for r in range(t + 1):
                    prod0 = prod0 * np.exp(dt[b, r, d] * A[d])
                hs += prod0 * p["initial_state"][b, d]
                for s in range(t + 1):
                    prod = np.ones(N)
                    for r in range(s + 1, t + 1):
                        prod = prod * np.exp(dt[b, r, d] * A[d])
                    hs += prod * dt[b, s, d] * B[b, s] * x[b, s, d]
                ref[b, t, d] = (np.dot(C[b, t], hs) + D[d] * x[b, t, d]) * silu_ref(z[b, t, d])
                if t == L - 1:
                    last_ref[b, d] = hs
    assert _rel(out, ref) < 1e-12, _rel(out, ref)
    assert _rel(last, last_ref) < 1e-12


# P2 -- prefix-sum form: prod_{r=s+1..t} exp(Delta_r A) = exp(A * (S_t - S_s)),
#       S the running sum of Delta (A does not depend on time).
def pin_prefix_sum(lib):
    p = rand_problem(2, bsz=1, L=16, dim=2, N=3, init=False)
    out, _ = _run(lib, p, z=None, D=None)
    dt = softplus_ref(p["delta"] + p["delta_bias"])
    S = np.cumsum(dt, axis=1)
    ref = np.zeros_like(out)
    for d in range(2):
        for t in range(16):
            acc = 0.0
            for s in range(t + 1):
                w = np.exp(p["A"][d] * (S[0, t, d] - S[0, s, d]))
                acc += np.dot(p["C"][0, t], w * p["B"][0, s]) * dt[0, s, d] * p["x"][0, s, d]
            ref[0, t, d] = acc
    assert _rel(out, ref) < 1e-12, _rel(out, ref)


# P3 -- LTI special case = global convolution mode: with Delta, B, C constant in
#       time, y = K * x + D x with K_k = sum_n C_n exp(k Delta A_n) Delta B_n.
def pin_lti_convolution(lib):
    p = rand_problem(3, bsz=1, L=20, dim=2, N=4, init=False, lti=True)
    out, _ = _run(lib, p, z=None)
    dt = softplus_ref(p["delta"][0, 0] + p["delta_bias"])        # (dim,)
    ref = np.zeros_like(out)
    for d in range(2):
        K = np.array([np.sum(p["C"][0, 0] * np.exp(k * dt[d] * p["A"][d]) * dt[d] * p["B"][0, 0])
                      for k in range(20)])
        conv = np.convolve(p["x"][0, :, d], K)[:20]               # numpy's direct convolution
        ref[0, :, d] = conv + p["D"][d] * p["x"][0, :, d]
    assert _rel(out, ref) < 1e-12, _rel(out, ref)


# P4 -- Delta -> 0 ("small Delta keeps the state and ignores the input"):
#       softplus(-1e4) underflows to exactly 0, so dA = 1, dBx = 0 and
#       y_t = (C_t . h_0 + D x_t) silu(z_t), the state unchanged.
def pin_small_delta(lib):
    p = rand_problem(4, bsz=2, L=7, dim=3, N=4, init=True)
    p["delta"] = np.full_like(p["delta"], -1e4)
    out, last = _run(lib, p)
    ref = (np.einsum("bln,bdn->bld", p["C"], p["initial_state"]) + p["D"] * p["x"]) * silu_ref(p["z"])
    assert np.array_equal(last, p["initial_state"])
    assert _rel(out, ref) < 1e-14, _rel(out, ref)


# P5 -- large Delta ("large Delta resets the state, focuses on the current input"):
#       dA ~ e^{-60|A|} ~ 0, so h_t = Delta_t B_t x_t and
#       y_t = (Delta_t x_t (C_t . B_t) + D x_t) silu(z_t).
def pin_large_delta(lib):
    p = rand_problem(5, bsz=1, L=9, dim=3, N=4, init=True)
    p["A"] = -1.0 - np.abs(p["A"])
    p["delta"] = np.full_like(p["delta"], 60.0)
    p["delta_bias"] = np.zeros(3)
    out, last = _run(lib, p)
    dt = softplus_ref(60.0)
    cb = np.sum(p["C"] * p["B"], axis=-1)[:, :, None]
    ref = (dt * p["x"] * cb + p["D"] * p["x"]) * silu_ref(p["z"])
    assert _rel(out, ref) < 1e-12, _rel(out, ref)
    assert _rel(last[0], dt * p["x"][0, -1][:, None] * p["B"][0, -1][None, :]) < 1e-12


# P6 -- split + carry: [0, L1) then [L1, L) from the first part's last state
#       equals the unsplit run (bit for bit: same operations in the same order).
def pin_split_carry(lib):
    p = rand_problem(6, bsz=2, L=15, dim=3, N=4, init=True)
    out, last = _run(lib, p)
    L1 = 6
    cut = lambda a, sl: None if a is None else a[:, sl]
    first = {k: (cut(v, slice(0, L1)) if k in ("x", "delta", "z", "B", "C") else v) for k, v in p.items()}
    o1, l1 = _run(lib, first)
    second = {k: (cut(v, slice(L1, None)) if k in ("x", "delta", "z", "B", "C") else v) for k, v in p.items()}
    second["initial_state"] = l1
    o2, l2 = _run(lib, second)
    assert np.array_equal(np.concatenate([o1, o2], axis=1), out)
    assert np.array_equal(l2, last)


# P7 -- decode = scan: T single-token steps from h_0 equal the scan of T tokens.
def pin_decode_equals_scan(lib):
    p = rand_problem(7, bsz=2, L=10, dim=3, N=4, init=True)
    out, last = _run(lib, p)
    st = p["initial_state"]
    for t in range(10):
        o, st = oracle.state_update(st, p["x"][:, t], p["delta"][:, t], p["A"], p["B"][:, t],
                                    p["C"][:, t], p["D"], p["z"][:, t], p["delta_bias"], lib=lib)
        assert np.array_equal(o, out[:, t])
    assert np.array_equal(st, last)


# P8 -- N = 1 with constant decay r = e^{Delta a}, B = C = 1, x = 1: a first-order
#       IIR filter whose response is the geometric sum y_t = Delta (1 - r^t)/(1 - r).
def pin_first_order_iir(lib):
    L, Dl, a = 30, 0.3, -0.7
    r = math.exp(Dl * a)
    ones = np.ones((1, L, 1))
    out, last = oracle.scan_fwd(ones, np.full((1, L, 1), Dl), np.array([[a]]), ones, ones,
                                delta_softplus=False, lib=lib)
    ref = np.array([Dl * (1 - r ** t) / (1 - r) for t in range(1, L + 1)])
    assert _rel(out[0, :, 0], ref) < 1e-13
    assert abs(last[0, 0, 0] - ref[-1]) < 1e-13


# The hand-derived fixture tests/golden/worked_example.txt.
def _golden():
    env = {"ln2": math.log(2.0), "ln3": math.log(3.0)}
    rows = {}
    with open(os.path.join(GOLDEN, "worked_example.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, rest = line.split(None, 1)
            rows[key] = [[eval(tok, {}, env) for tok in grp.split()] for grp in rest.split("|")]
    return rows


def pin_worked_example(lib):
    g = _golden()
    x = np.array(g["x"][0]).reshape(1, 3, 1)
    out, last = oracle.scan_fwd(x, np.array(g["delta"][0]).reshape(1, 3, 1),
                                np.array(g["A"][0]).reshape(1, 2),
                                np.array(g["B"]).reshape(1, 3, 2), np.array(g["C"]).reshape(1, 3, 2),
                                D=np.array(g["D"][0]), z=np.array(g["z"][0]).reshape(1, 3, 1),
                                delta_bias=np.array(g["bias"][0]), lib=lib)
    assert _rel(out.ravel(), np.array([v[0] for v in g["y"]])) < 1e-15
    assert _rel(last.ravel(), np.array(g["last"][0])) < 1e-15


# Nonlinearities: softplus(0) = ln 2, softplus(u) - softplus(-u) = u, silu(ln 3)
# = (3/4) ln 3, silu(v) - silu(-v) = v; and against numpy/scipy on a grid.
def pin_nonlinearities(lib):
    eps = np.finfo(np.float64).eps
    assert abs(oracle.softplus(0.0, lib=lib) - math.log(2.0)) <= 2 * eps
    assert abs(oracle.silu(math.log(3.0), lib=lib) - 0.75 * math.log(3.0)) <= 4 * eps
    for u in np.linspace(-40, 40, 161):
        sp = oracle.softplus(u, lib=lib)
        assert abs(sp - softplus_ref(u)) <= 1e-15 * max(1.0, abs(sp)) + 1e-300
        assert abs(sp - oracle.softplus(-u, lib=lib) - u) < 1e-13
        sv = oracle.silu(u, lib=lib)
        assert abs(sv - silu_ref(u)) <= 1e-15 * max(1.0, abs(sv))
    assert oracle.softplus(-800.0, lib=lib) == 0.0
    assert oracle.softplus(800.0, lib=lib) == 800.0


# ---- causal depthwise conv1d (+ SiLU) in front of the scan

def _conv_problem(seed, bsz=2, L=11, dim=3, K=4):
    r = np.random.default_rng(seed)
    return (r.standard_normal((bsz, L, dim)), r.standard_normal((dim, K)), r.standard_normal(dim),
            r.standard_normal((bsz, dim, K - 1)))


# C1 -- numpy's direct convolution: out[:, d] = act(np.convolve(x[:, d], w[d][::-1])[:L] + b),
#       with the K-1 earlier inputs (the state) prepended.
def pin_conv_numpy(lib):
    x, w, b, st = _conv_problem(11)
    out, st_out = oracle.conv1d_fwd(x, w, b, st, lib=lib)
    bsz, L, dim = x.shape
    K = w.shape[1]
    for bb in range(bsz):
        for d in range(dim):
            seq = np.concatenate([st[bb, d], x[bb, :, d]])
            full = np.convolve(seq, w[d][::-1])[K - 1:K - 1 + L]
            assert np.max(np.abs(out[bb, :, d] - silu_ref(full + b[d]))) < 1e-13
            assert np.array_equal(st_out[bb, d], seq[-(K - 1):])
    out0, _ = oracle.conv1d_fwd(x, w, b, None, activation=False, lib=lib)
    d = 1
    ref0 = np.convolve(x[0, :, d], w[d][::-1])[:L] + b[d]           # zero history
    assert np.max(np.abs(out0[0, :, d] - ref0)) < 1e-13


# C2 -- special taps: identity (w = e_{K-1}) gives act(x + b); a pure delay
#       (w = e_0) gives act(x[t-K+1] + b) with the history before t = 0.
def pin_conv_taps(lib):
    x, w, b, st = _conv_problem(12, K=3)
    K = 3
    ident = np.zeros_like(w); ident[:, K - 1] = 1.0
    out, _ = oracle.conv1d_fwd(x, ident, b, st, lib=lib)
    assert np.max(np.abs(out - silu_ref(x + b))) < 1e-15
    delay = np.zeros_like(w); delay[:, 0] = 1.0
    out, _ = oracle.conv1d_fwd(x, delay, None, st, activation=False, lib=lib)
    assert np.array_equal(out[:, K - 1:], x[:, :-(K - 1)])
    assert np.array_equal(out[:, :K - 1], np.transpose(st, (0, 2, 1)))


# C3 -- split + state carry: [0, L1) then [L1, L) from the first part's final
#       state equals the unsplit call (bit for bit), also when L1 < K - 1.
def pin_conv_split(lib):
    x, w, b, st = _conv_problem(13, L=10, K=5)
    out, st_out = oracle.conv1d_fwd(x, w, b, st, lib=lib)
    for L1 in (2, 6):
        o1, s1 = oracle.conv1d_fwd(x[:, :L1], w, b, st, lib=lib)
        o2, s2 = oracle.conv1d_fwd(x[:, L1:], w, b, s1, lib=lib)
        assert np.array_equal(np.concatenate([o1, o2], 1), out)
        assert np.array_equal(s2, st_out)


# ------------------------------------------------------- exact ZOH and LTI mode

# Z1 -- the exact zero-order hold through scipy's matrix exponential: for each
#       (step, channel, state) the augmented system [[Delta a, Delta], [0, 0]]
#       exponentiates to [[Abar, Bbar / b], [0, 1]]; the recurrence is then run
#       in numpy with those coefficients
def pin_zoh_expm(lib):
    from scipy.linalg import expm
    p = rand_problem(51, bsz=2, L=7, dim=3, N=4)
    out, last = oracle.scan_fwd(lib=lib, zoh=True, **p)
    bsz, L, dim = p["x"].shape
    N = p["A"].shape[1]
    ref = np.empty_like(out)
    ref_last = np.empty_like(last)
    for b in range(bsz):
        for d in range(dim):
            h = p["initial_state"][b, d].copy()
            for t in range(L):
                dt = softplus_ref(p["delta"][b, t, d] + p["delta_bias"][d])
                y = 0.0
                for n in range(N):
                    E = expm(np.array([[dt * p["A"][d, n], dt], [0.0, 0.0]]))
                    h[n] = E[0, 0] * h[n] + E[0, 1] * p["B"][b, t, n] * p["x"][b, t, d]
                    y += p["C"][b, t, n] * h[n]
                y += p["D"][d] * p["x"][b, t, d]
                ref[b, t, d] = y * silu_ref(p["z"][b, t, d])
            ref_last[b, d] = h
    assert _rel(out, ref) < 1e-11 and _rel(last, ref_last) < 1e-11


# Z2 -- N = 1, constant step and input: a first-order filter with gain
#       g = (r - 1) / a, r = exp(Delta a); h_t = g (1 - r^(t+1)) / (1 - r)
def pin_zoh_first_order(lib):
    L, a, dt = 30, -0.7, 0.4
    one = np.ones((1, L, 1))
    out, last = oracle.scan_fwd(one, np.full((1, L, 1), dt), np.array([[a]]), one, one,
                                delta_softplus=False, lib=lib, zoh=True)
    r = math.exp(dt * a)
    g = (r - 1.0) / a
    t = np.arange(L)
    ref = g * (1.0 - r ** (t + 1)) / (1.0 - r)
    assert np.max(np.abs(out[0, :, 0] - ref)) < 1e-13
    assert abs(last[0, 0, 0] - ref[-1]) < 1e-13


def _lti_params(seed, dim=3, N=4):
    r = np.random.default_rng(seed)
    return (r.uniform(0.05, 0.6, dim), -np.exp(r.uniform(-1.0, 1.5, (dim, N))),
            r.standard_normal((dim, N)), r.standard_normal((dim, N)))


# L1 -- the LTI kernel is the impulse response of the recurrence: for each
#       channel, the scan (first-order or exact ZOH) over a unit impulse with
#       constant step, B, C returns K[d][t]
def pin_lti_kernel_impulse(lib):
    delta, A, B, C = _lti_params(52)
    L = 25
    for zoh in (False, True):
        K = oracle.lti_kernel(delta, A, B, C, L, zoh=zoh, lib=lib)
        for d in range(A.shape[0]):
            x = np.zeros((1, L, 1))
            x[0, 0, 0] = 1.0
            y, _ = oracle.scan_fwd(x, np.full((1, L, 1), delta[d]), A[d:d + 1],
                                   np.broadcast_to(B[d], (1, L, B.shape[1])),
                                   np.broadcast_to(C[d], (1, L, C.shape[1])),
                                   delta_softplus=False, lib=lib, zoh=zoh)
            assert np.max(np.abs(K[d] - y[0, :, 0])) < 1e-13, (zoh, d)


# L2 -- the convolution mode against numpy's convolution, plus skip and gate
def pin_lti_conv_numpy(lib):
    delta, A, B, C = _lti_params(53)
    r = np.random.default_rng(54)
    bsz, L, dim = 2, 19, A.shape[0]
    K = oracle.lti_kernel(delta, A, B, C, L, lib=lib)
    x = r.standard_normal((bsz, L, dim))
    z = r.standard_normal((bsz, L, dim))
    Dv = r.standard_normal(dim)
    y = oracle.lti_conv(K, x, D=Dv, z=z, lib=lib)
    for b in range(bsz):
        for d in range(dim):
            ref = np.convolve(K[d], x[b, :, d])[:L] + Dv[d] * x[b, :, d]
            assert np.max(np.abs(y[b, :, d] - ref * silu_ref(z[b, :, d]))) < 1e-12
    y0 = oracle.lti_conv(K, x, lib=lib)
    assert np.max(np.abs(y0[0, :, 1] - np.convolve(K[1], x[0, :, 1])[:L])) < 1e-12


# ------------------------------------------------------- selection projections
# oracle.selection_proj is numpy (no C library): ``lib`` is unused here, and
# the C-source mutations cannot reach it; its own pins are these two.

# P1 -- brute-force triple loops in plain Python on a tiny problem
def pin_proj_bruteforce(lib):
    r = np.random.default_rng(61)
    bsz, L, dim, R, N = 2, 3, 5, 2, 3
    x = r.standard_normal((bsz, L, dim))
    Wx = r.standard_normal((R + 2 * N, dim))
    Wdt = r.standard_normal((dim, R))
    dt_low, Bm, Cm, delta = oracle.selection_proj(x, Wx, Wdt, R)
    for b in range(bsz):
        for t in range(L):
            xd = [sum(x[b, t, k] * Wx[j, k] for k in range(dim)) for j in range(R + 2 * N)]
            assert np.allclose(dt_low[b, t], xd[:R], atol=1e-13)
            assert np.allclose(Bm[b, t], xd[R:R + N], atol=1e-13)
            assert np.allclose(Cm[b, t], xd[R + N:], atol=1e-13)
            for d in range(dim):
                ref = sum(xd[j] * Wdt[d, j] for j in range(R))
                assert abs(delta[b, t, d] - ref) < 1e-12


# P2 -- selector weights: rows of the identity pick input channels out
def pin_proj_selectors(lib):
    r = np.random.default_rng(62)
    bsz, L, dim, R, N = 1, 4, 8, 2, 3
    x = r.standard_normal((bsz, L, dim))
    Wx = np.zeros((R + 2 * N, dim))
    for j in range(R + 2 * N):
        Wx[j, j] = 1.0                      # xdbl[:, j] = x[:, j]
    Wdt = np.zeros((dim, R))
    Wdt[:, 0] = 1.0                         # delta[:, d] = dt_low[:, 0] = x[:, 0]
    dt_low, Bm, Cm, delta = oracle.selection_proj(x, Wx, Wdt, R)
    assert np.array_equal(dt_low, x[..., :R]) and np.array_equal(Bm, x[..., R:R + N])
    assert np.array_equal(Cm, x[..., R + N:R + 2 * N])
    assert np.array_equal(delta, np.repeat(x[..., :1], dim, axis=-1))


# ------------------------------------------------------------------ backward
# The gradients of the scan (oracle.scan_bwd) are pinned by differentiating
# the forward numerically and by torch's autograd on an fp64 loop of its own.

_BWD_KEYS = (("x", "dx"), ("delta", "ddelta"), ("A", "dA"), ("B", "dB"), ("C", "dC"),
             ("D", "dD"), ("z", "dz"), ("delta_bias", "ddelta_bias"),
             ("initial_state", "dinitial_state"))


def _bwd_problem(seed, bsz=2, L=5, dim=3, N=4, **kw):
    p = rand_problem(seed, bsz=bsz, L=L, dim=dim, N=N)
    r = np.random.default_rng(seed + 1)
    dout = r.standard_normal((bsz, L, dim))
    dlast = r.standard_normal((bsz, dim, N))
    for k, v in kw.items():
        p[k] = v
    return p, dout, dlast


def _loss(lib, p, dout, dlast, softplus=True):
    out, last = oracle.scan_fwd(lib=lib, delta_softplus=softplus, **p)
    return float(np.sum(out * dout) + (np.sum(last * dlast) if dlast is not None else 0.0))


# G1 -- central differences of the forward, coordinate by coordinate
#       (error O(eps^2) + roundoff/eps, about 1e-9 here)
def pin_bwd_finite_differences(lib):
    for case in range(3):
        if case == 0:
            p, dout, dlast = _bwd_problem(31)
            softplus = True
        elif case == 1:     # no optional inputs, no final-state gradient
            p, dout, dlast = _bwd_problem(32, z=None, D=None, delta_bias=None, initial_state=None)
            dlast = None
            softplus = True
        else:               # raw step sizes (positive), no softplus
            p, dout, dlast = _bwd_problem(33)
            p["delta"] = np.abs(p["delta"]) * 0.3 + 0.05
            p["delta_bias"] = None
            softplus = False
        g = oracle.scan_bwd(lib=lib, dout=dout, dlast_state=dlast, delta_softplus=softplus, **p)
        eps = 1e-6
        for name, gk in _BWD_KEYS:
            if p.get(name) is None:
                continue
            arr = p[name]
            fd = np.zeros_like(arr)
            for i in np.ndindex(arr.shape):
                up, dn = arr.copy(), arr.copy()
                up[i] += eps
                dn[i] -= eps
                fd[i] = (_loss(lib, dict(p, **{name: up}), dout, dlast, softplus)
                         - _loss(lib, dict(p, **{name: dn}), dout, dlast, softplus)) / (2 * eps)
            err = np.max(np.abs(g[gk] - fd)) / (1.0 + np.max(np.abs(fd)))
            assert err < 1e-7, (case, name, err)


# G2 -- directional derivative of a longer problem along a random direction
#       over every input at once: sum_i grad_i v_i = d/de L(theta + e v)
def pin_bwd_directional(lib):
    p, dout, dlast = _bwd_problem(34, bsz=2, L=40, dim=5, N=8)
    g = oracle.scan_bwd(lib=lib, dout=dout, dlast_state=dlast, **p)
    r = np.random.default_rng(35)
    v = {name: r.standard_normal(p[name].shape) for name, _ in _BWD_KEYS}
    eps = 1e-6
    up = {k: (p[k] + eps * v[k] if k in v else p[k]) for k in p}
    dn = {k: (p[k] - eps * v[k] if k in v else p[k]) for k in p}
    fd = (_loss(lib, up, dout, dlast) - _loss(lib, dn, dout, dlast)) / (2 * eps)
    an = sum(float(np.sum(g[gk] * v[name])) for name, gk in _BWD_KEYS)
    assert abs(an - fd) < 1e-7 * (1.0 + abs(fd)), (an, fd)


# G3 -- torch autograd through an fp64 loop written here (a second
#       implementation of the forward, differentiated by the library)
def pin_bwd_autograd(lib):
    import torch
    p, dout, dlast = _bwd_problem(36, bsz=2, L=9, dim=4, N=3)
    t = {k: torch.tensor(v, dtype=torch.float64, requires_grad=True) for k, v in p.items()}
    bsz, L, dim = p["x"].shape
    h = t["initial_state"]                                   # (b, d, n)
    outs = []
    for s in range(L):
        dt = torch.nn.functional.softplus(t["delta"][:, s] + t["delta_bias"])   # (b, d)
        decay = torch.exp(dt[..., None] * t["A"][None])
        h = decay * h + (dt * t["x"][:, s])[..., None] * t["B"][:, s][:, None, :]
        y = (h * t["C"][:, s][:, None, :]).sum(-1) + t["D"] * t["x"][:, s]
        outs.append(y * torch.nn.functional.silu(t["z"][:, s]))
    out = torch.stack(outs, 1)
    loss = (out * torch.tensor(dout)).sum() + (h * torch.tensor(dlast)).sum()
    loss.backward()
    g = oracle.scan_bwd(lib=lib, dout=dout, dlast_state=dlast, **p)
    for name, gk in _BWD_KEYS:
        ref = t[name].grad.numpy()
        assert np.max(np.abs(g[gk] - ref)) < 1e-11 * (1.0 + np.max(np.abs(ref))), name


# G4 -- the per-thread partial sums: any thread count gives the same
#       gradients up to fp64 rounding
def pin_bwd_thread_count(lib):
    p, dout, dlast = _bwd_problem(37, bsz=3, L=16, dim=7, N=4)
    g1 = oracle.scan_bwd(lib=lib, dout=dout, dlast_state=dlast, nthreads=1, **p)
    g3 = oracle.scan_bwd(lib=lib, dout=dout, dlast_state=dlast, nthreads=3, **p)
    for _, gk in _BWD_KEYS:
        assert np.max(np.abs(g1[gk] - g3[gk])) < 1e-12 * (1.0 + np.max(np.abs(g1[gk]))), gk


ALL_PINS = [pin_closed_form, pin_prefix_sum, pin_lti_convolution, pin_small_delta,
            pin_large_delta, pin_split_carry, pin_decode_equals_scan, pin_first_order_iir,
            pin_worked_example, pin_nonlinearities, pin_conv_numpy, pin_conv_taps, pin_conv_split,
            pin_bwd_finite_differences, pin_bwd_directional, pin_bwd_autograd, pin_bwd_thread_count,
            pin_zoh_expm, pin_zoh_first_order, pin_lti_kernel_impulse, pin_lti_conv_numpy,
            pin_proj_bruteforce, pin_proj_selectors]
