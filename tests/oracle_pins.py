"""Pins for the fp64 oracle: checks against facts that do not come from the
oracle itself.  Each pin takes ``scan(u, delta, A, B, C, D, z, delta_bias,
softplus) -> (y, h_last)`` and returns the largest error it saw, so the same
pins run against the committed oracle (tests/test_oracle_pins.py) and against
deliberately broken copies of it (tests/test_oracle_mutants.py).

What each pin rests on:
  bruteforce      the unrolled closed form of the linear recurrence,
                  y_t = sum_{s<=t} sum_n C_t[n] exp(A[n] * sum_{r=s+1..t} dt_r)
                        dt_s B_s[n] u_s + D u_t, evaluated in 40-digit mpmath
                  with softplus and SiLU from their textbook definitions
                  ("State Space Models (SSM)" summary page, section 3.2, and
                  the recurrence/readout of section 1.2).
  lti_direct /    time-invariant delta, B, C: y = u * K with
  lti_fft         K_k = sum_n C[n] exp(k dt A[n]) dt B[n] (the convolution
                  kernel K = (C B, C A B, C A^2 B, ...) of the itwiki page's
                  "순환 형태와 합성곱 형태" section, with the diagonal-A
                  Vandermonde form of the youngju.dev S4Layer listing),
                  convolved directly and through a zero-padded FFT.
  associativity   splitting the sequence anywhere and composing the two
                  halves' (decay, state) pairs gives the full result (the
                  associative-scan property of the Obsidian "Mamba" note, 5.1).
  special cases   N = 1, L = 1 scalar recurrence; A = 0 (prefix sum); C = 0
                  (y = D u gate); delta = 0 on a suffix keeps the state
                  (itwiki "Mamba의 선택 메커니즘": small Delta keeps the state);
                  z = 0 gives y = 0; A < 0, delta > 0 keeps h bounded.
  golden          tests/golden/hand_worked.json, worked by hand.
  bruteforce_h0   the closed form with an initial state h0, whose term
                  C_t[n] exp(A[n] * sum_{r=0..t} dt_r) h0[n] is added to y_t
                  (the state h0 decays through every step, step 0 included).
  chaining        a sequence run in two parts, the second starting from the
                  first part's final state, equals the run in one part; and
                  L single recurrent steps equal one L-step scan (the
                  generation-time recurrence of the Obsidian "Mamba" note,
                  4.2, carries only the state).
Pins that pass an initial state call ``scan(..., h0=h0)``.

The exact zero-order-hold discretisation (``scan(..., zoh=True)``) is pinned by:
  zoh_lti         time-invariant inputs: y = u * K with K_k = sum_n C[n]
                  exp(k dt A[n]) (exp(dt A[n]) - 1) / A[n] B[n] (the itwiki
                  page's "이산화" Bbar inside its convolution kernel K), direct
                  and by FFT.
  zoh_ode         with B_t u_t held constant over each step, ZOH is the exact
                  solution of h' = A h + B u: scipy's DOP853 integration of the
                  continuous system, step by step, at rtol 1e-12.
  zoh_limit       A = 0 gives exactly the Euler result; |A| = 1e-7 agrees
                  with it to ~dt^2 |A|.

The causal convolution + SiLU prologue (``conv`` functions with the signature
``conv(x, w, cb) -> u``) is pinned separately:
  conv_numpy      each channel against numpy.convolve (full convolution of x
                  with the kernel, the first L outputs) plus the bias, then
                  SiLU from its definition z / (1 + e^-z).
  conv_k1         K = 1 is the pointwise silu(w x + cb).
  conv_causal     changing x at step s changes no u before s, and changes u
                  at s .. s + K - 1.
  conv_impulse    a unit impulse at step s with zero bias gives
                  u[s + j] = silu(w[K-1-j]) (the taps in reverse order).
"""
from __future__ import annotations

import json
import math
import os

import mpmath
import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "hand_worked.json")


def _rel_err(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if got.shape != ref.shape:
        return float("inf")
    if got.size == 0:
        return 0.0
    return float(np.max(np.abs(got - ref) / (1.0 + np.abs(ref))))


def random_problem(rng, batch, L, dim, N, softplus=True, bias=True, gate=True, skip=True,
                   a_neg=True):
    u = rng.standard_normal((batch, L, dim))
    if softplus:
        delta = rng.standard_normal((batch, L, dim)) - 1.0
    else:
        delta = np.exp(rng.uniform(np.log(1e-2), np.log(5e-1), size=(batch, L, dim)))
    A = -np.exp(rng.uniform(-1.0, 1.5, size=(dim, N))) if a_neg else rng.standard_normal((dim, N))
    B = rng.standard_normal((batch, L, N))
    C = rng.standard_normal((batch, L, N))
    D = rng.standard_normal(dim) if skip else None
    z = rng.standard_normal((batch, L, dim)) if gate else None
    db = 0.5 * rng.standard_normal(dim) if bias else None
    return dict(u=u, delta=delta, A=A, B=B, C=C, D=D, z=z, delta_bias=db, softplus=softplus)


def _call(scan, p, h0=None, zoh=False):
    args = (p["u"], p["delta"], p["A"], p["B"], p["C"], p["D"], p["z"], p["delta_bias"],
            p["softplus"])
    kw = {}
    if h0 is not None:
        kw["h0"] = h0
    if zoh:
        kw["zoh"] = True
    return scan(*args, **kw)


# ---------------------------------------------------------------- brute force
def bruteforce(p, dps=40, h0=None):
    """Unrolled closed form in high precision (see module docstring); h0 is an
    optional initial state (batch, dim, N)."""
    mpmath.mp.dps = dps
    u, delta, A, B, C = p["u"], p["delta"], p["A"], p["B"], p["C"]
    D, z, db, sp = p["D"], p["z"], p["delta_bias"], p["softplus"]
    batch, L, dim = u.shape
    N = A.shape[1]
    y = np.zeros((batch, L, dim))
    h = np.zeros((batch, dim, N))
    mpf = mpmath.mpf
    for b in range(batch):
        for d in range(dim):
            dts = []
            for t in range(L):
                x = mpf(float(delta[b, t, d])) + (mpf(float(db[d])) if db is not None else 0)
                if sp:
                    x = mpmath.log(1 + mpmath.exp(x))       # softplus, textbook form
                dts.append(x)
            for t in range(L):
                acc = mpf(0)
                if h0 is not None:                            # the initial state's share
                    head = sum(dts[:t + 1], mpf(0))           # sum of dt over [0, t]
                    for n in range(N):
                        acc += (mpf(float(C[b, t, n])) * mpmath.exp(mpf(float(A[d, n])) * head)
                                * mpf(float(h0[b, d, n])))
                for s in range(t + 1):
                    tail = sum(dts[s + 1:t + 1], mpf(0))     # sum of dt over (s, t]
                    for n in range(N):
                        a = mpf(float(A[d, n]))
                        acc += (mpf(float(C[b, t, n])) * mpmath.exp(a * tail) * dts[s]
                                * mpf(float(B[b, s, n])) * mpf(float(u[b, s, d])))
                if D is not None:
                    acc += mpf(float(D[d])) * mpf(float(u[b, t, d]))
                if z is not None:
                    zz = mpf(float(z[b, t, d]))
                    acc *= zz / (1 + mpmath.exp(-zz))
                y[b, t, d] = float(acc)
            for n in range(N):
                a = mpf(float(A[d, n]))
                hn = mpf(0)
                if h0 is not None:
                    hn = mpmath.exp(a * sum(dts, mpf(0))) * mpf(float(h0[b, d, n]))
                for s in range(L):
                    tail = sum(dts[s + 1:L], mpf(0))
                    hn += (mpmath.exp(a * tail) * dts[s] * mpf(float(B[b, s, n]))
                           * mpf(float(u[b, s, d])))
                h[b, d, n] = float(hn)
    return y, h


def pin_bruteforce(scan, seed=0):
    rng = np.random.default_rng(seed)
    worst = 0.0
    for kw in (dict(),
               dict(softplus=False, bias=False, gate=False, skip=False),
               dict(softplus=True, bias=False, gate=True, skip=False),
               dict(softplus=False, bias=True, gate=False, skip=True, a_neg=False)):
        p = random_problem(rng, batch=2, L=6, dim=3, N=5, **kw)
        y, h = _call(scan, p)
        yr, hr = bruteforce(p)
        worst = max(worst, _rel_err(y, yr), _rel_err(h, hr))
    return worst


# ---------------------------------------------------------------- time-invariant
def _lti_problem(rng, batch=2, L=384, dim=5, N=16, skip=False):
    dt = np.exp(rng.uniform(np.log(1e-3), np.log(1e-1), size=dim))
    A = -np.broadcast_to(np.arange(1, N + 1, dtype=np.float64), (dim, N)).copy()
    A[1] *= 0.37                      # one channel with a non-integer spectrum
    bvec = rng.standard_normal(N)
    cvec = rng.standard_normal(N)
    u = rng.standard_normal((batch, L, dim))
    p = dict(u=u, delta=np.broadcast_to(dt, (batch, L, dim)).copy(), A=A,
             B=np.broadcast_to(bvec, (batch, L, N)).copy(),
             C=np.broadcast_to(cvec, (batch, L, N)).copy(),
             D=(np.linspace(0.5, 1.5, dim) if skip else None), z=None, delta_bias=None,
             softplus=False)
    return p, dt, bvec, cvec


def lti_kernel(dt, A, bvec, cvec, L):
    """K[d, k] = sum_n C[n] exp(k dt_d A[d,n]) dt_d B[n]  (Vandermonde form)."""
    k = np.arange(L, dtype=np.float64)
    # (dim, N, L) powers exp(k * dt * A)
    pw = np.exp(dt[:, None, None] * A[:, :, None] * k[None, None, :])
    return np.einsum("n,dnl->dl", cvec * bvec, pw) * dt[:, None]


def pin_lti_direct(scan, seed=1, skip=False):
    rng = np.random.default_rng(seed)
    p, dt, bvec, cvec = _lti_problem(rng, skip=skip)
    y, _ = _call(scan, p)
    batch, L, dim = p["u"].shape
    K = lti_kernel(dt, p["A"], bvec, cvec, L)
    yr = np.zeros_like(y)
    for b in range(batch):
        for d in range(dim):
            yr[b, :, d] = np.convolve(p["u"][b, :, d], K[d])[:L]
    if p["D"] is not None:
        yr += p["D"][None, None, :] * p["u"]
    return _rel_err(y, yr)


def pin_lti_fft(scan, seed=2):
    rng = np.random.default_rng(seed)
    p, dt, bvec, cvec = _lti_problem(rng, L=1000)
    y, _ = _call(scan, p)
    batch, L, dim = p["u"].shape
    K = lti_kernel(dt, p["A"], bvec, cvec, L)
    kf = np.fft.rfft(K, n=2 * L, axis=-1)                          # (dim, L+1)
    uf = np.fft.rfft(np.transpose(p["u"], (0, 2, 1)), n=2 * L, axis=-1)
    yr = np.fft.irfft(uf * kf[None], n=2 * L, axis=-1)[..., :L]
    yr = np.transpose(yr, (0, 2, 1))
    return _rel_err(y, yr)


# ---------------------------------------------------------------- associativity
def pin_associativity(scan, seed=3):
    """Run [0, s) and [s, L) separately from zero state; compose with the
    decay exp(A * sum of dt over [s, t]) of the prefix state."""
    rng = np.random.default_rng(seed)
    worst = 0.0
    for split in (1, 7, 16):
        p = random_problem(rng, batch=2, L=23, dim=4, N=6, gate=False, skip=False)
        y, h = _call(scan, p)
        pre = {k: (v[:, :split] if isinstance(v, np.ndarray) and v.ndim == 3 else v)
               for k, v in p.items()}
        suf = {k: (v[:, split:] if isinstance(v, np.ndarray) and v.ndim == 3 else v)
               for k, v in p.items()}
        yp, hp = _call(scan, pre)
        ys, hs = _call(scan, suf)
        dt = p["delta"] + (p["delta_bias"][None, None, :] if p["delta_bias"] is not None else 0)
        dt = np.logaddexp(0.0, dt) if p["softplus"] else dt          # (batch, L, dim)
        cum = np.cumsum(dt[:, split:], axis=1)                        # (batch, Ls, dim)
        decay = np.exp(cum[..., None] * p["A"][None, None])           # (batch, Ls, dim, N)
        carry = np.einsum("btn,btdn,bdn->btd", p["C"][:, split:], decay, hp)
        worst = max(worst, _rel_err(y[:, :split], yp), _rel_err(y[:, split:], ys + carry),
                    _rel_err(h, hs + decay[:, -1] * hp))
    return worst


# ---------------------------------------------------------------- special cases
def pin_special_cases(scan, seed=4):
    rng = np.random.default_rng(seed)
    worst = 0.0
    # N = 1, L = 1: y = C dt B u + D u, h = dt B u
    p = random_problem(rng, 3, 1, 2, 1, softplus=False, bias=False, gate=False)
    y, h = _call(scan, p)
    dt = p["delta"][:, 0, :]
    hr = dt * p["B"][:, 0, :] * p["u"][:, 0, :]
    worst = max(worst, _rel_err(h[:, :, 0], hr),
                _rel_err(y[:, 0, :], p["C"][:, 0, :] * hr + p["D"] * p["u"][:, 0, :]))
    # A = 0: the state is the running sum of dt B u
    p = random_problem(rng, 2, 9, 3, 4, softplus=True, gate=False, skip=False)
    p["A"] = np.zeros_like(p["A"])
    y, h = _call(scan, p)
    dt = np.logaddexp(0.0, p["delta"] + p["delta_bias"])
    hs = np.cumsum(dt[..., None] * p["B"][:, :, None, :] * p["u"][..., None], axis=1)
    worst = max(worst, _rel_err(h, hs[:, -1]),
                _rel_err(y, np.einsum("btn,btdn->btd", p["C"], hs)))
    # C = 0: y = D u silu(z)
    p = random_problem(rng, 2, 5, 3, 4)
    p["C"] = np.zeros_like(p["C"])
    y, _ = _call(scan, p)
    zz = p["z"]
    worst = max(worst, _rel_err(y, p["D"] * p["u"] * zz / (1 + np.exp(-zz))))
    # z = 0: the gate closes
    p = random_problem(rng, 2, 5, 3, 4)
    p["z"] = np.zeros_like(p["z"])
    y, _ = _call(scan, p)
    worst = max(worst, float(np.max(np.abs(y))))
    # delta = 0 on a suffix keeps the state (no softplus), and a softplus input
    # driven to -1e4 (softplus -> 0) does the same
    for sp in (False, True):
        p = random_problem(rng, 2, 12, 3, 4, softplus=sp, bias=False, gate=False)
        _, h_pre = _call(scan, {**p, "u": p["u"][:, :8], "delta": p["delta"][:, :8],
                                "B": p["B"][:, :8], "C": p["C"][:, :8]})
        p["delta"][:, 8:] = -1e4 if sp else 0.0
        _, h = _call(scan, p)
        worst = max(worst, _rel_err(h, h_pre))
    # A < 0, delta > 0: |h[n]| <= max|dt B u| / (1 - max exp(dt A))
    p = random_problem(rng, 2, 200, 3, 4, softplus=False, bias=False, gate=False)
    _, h = _call(scan, p)
    dt = p["delta"]
    dbu = np.abs(dt[..., None] * p["B"][:, :, None, :] * p["u"][..., None])   # (b,t,d,n)
    da = np.exp(dt[..., None] * p["A"][None, None])
    bound = dbu.max(axis=1) / (1.0 - da.max(axis=1))
    excess = np.max(np.abs(h) - bound)
    worst = max(worst, 0.0 if excess <= 0 else float(excess) + 1.0)
    return worst


# ---------------------------------------------------------------- golden
def _ev(x):
    if isinstance(x, str):
        return eval(x, {"__builtins__": {}}, {"ln2": math.log(2.0), "ln3": math.log(3.0)})
    if isinstance(x, list):
        return [_ev(v) for v in x]
    return x


def pin_golden(scan):
    with open(GOLDEN) as f:
        cases = json.load(f)["cases"]
    worst = 0.0
    for c in cases:
        arr = lambda k: None if c[k] is None else np.array(_ev(c[k]), dtype=np.float64)
        y, h = scan(arr("u"), arr("delta"), arr("A"), arr("B"), arr("C"), arr("D"), arr("z"),
                    arr("delta_bias"), c["softplus"])
        worst = max(worst, _rel_err(y, arr("y")), _rel_err(h, arr("h_last")))
    return worst


# ---------------------------------------------------------------- initial state
def pin_bruteforce_h0(scan, seed=6):
    rng = np.random.default_rng(seed)
    worst = 0.0
    for kw in (dict(), dict(softplus=False, bias=False, gate=False, skip=False),
               dict(softplus=True, bias=True, gate=True, skip=True, a_neg=False)):
        p = random_problem(rng, batch=2, L=5, dim=3, N=4, **kw)
        h0 = rng.standard_normal((2, 3, 4))
        y, h = _call(scan, p, h0=h0)
        yr, hr = bruteforce(p, h0=h0)
        worst = max(worst, _rel_err(y, yr), _rel_err(h, hr))
    return worst


def pin_chaining(scan, seed=7):
    """Two parts chained through the state equal one part; and L steps of one
    token each equal one L-step scan."""
    rng = np.random.default_rng(seed)
    worst = 0.0
    for split in (1, 5, 12):
        p = random_problem(rng, batch=2, L=13, dim=4, N=6)
        h0 = rng.standard_normal((2, 4, 6))
        y, h = _call(scan, p, h0=h0)
        pre = {k: (v[:, :split] if isinstance(v, np.ndarray) and v.ndim == 3 else v)
               for k, v in p.items()}
        suf = {k: (v[:, split:] if isinstance(v, np.ndarray) and v.ndim == 3 else v)
               for k, v in p.items()}
        yp, hp = _call(scan, pre, h0=h0)
        ys, hs = _call(scan, suf, h0=hp)
        worst = max(worst, _rel_err(y[:, :split], yp), _rel_err(y[:, split:], ys),
                    _rel_err(h, hs))
    p = random_problem(rng, batch=2, L=7, dim=3, N=5)
    y, h = _call(scan, p)
    hk = np.zeros((2, 3, 5))
    for t in range(7):
        one = {k: (v[:, t:t + 1] if isinstance(v, np.ndarray) and v.ndim == 3 else v)
               for k, v in p.items()}
        yk, hk = _call(scan, one, h0=hk)
        worst = max(worst, _rel_err(y[:, t:t + 1], yk))
    return max(worst, _rel_err(h, hk))


# ---------------------------------------------------------------- zero-order hold
def pin_zoh_lti(scan, seed=12):
    rng = np.random.default_rng(seed)
    p, dt, bvec, cvec = _lti_problem(rng, batch=2, L=300, dim=4, N=8)
    y, _ = _call(scan, p, zoh=True)
    A = p["A"]
    k = np.arange(300)
    worst = 0.0
    for d in range(4):
        bbar = np.expm1(dt[d] * A[d]) / A[d] * bvec                     # (N,)
        K = (np.exp(np.outer(k, dt[d] * A[d])) * cvec * bbar).sum(axis=1)  # (L,)
        for b in range(2):
            x = p["u"][b, :, d]
            direct = np.array([np.dot(K[:t + 1][::-1], x[:t + 1]) for t in range(300)])
            n = 600
            fft = np.fft.irfft(np.fft.rfft(x, n) * np.fft.rfft(K, n), n)[:300]
            worst = max(worst, _rel_err(y[b, :, d], direct), _rel_err(y[b, :, d], fft))
    return worst


def pin_zoh_ode(scan, seed=13):
    from scipy.integrate import solve_ivp
    rng = np.random.default_rng(seed)
    p = random_problem(rng, batch=1, L=6, dim=2, N=3, gate=True, skip=True)
    h0 = rng.standard_normal((1, 2, 3))
    y, h = _call(scan, p, h0=h0, zoh=True)
    dt = p["delta"] + p["delta_bias"][None, None, :]
    dt = np.logaddexp(0.0, dt)
    worst = 0.0
    for d in range(2):
        a = p["A"][d]
        state = h0[0, d].copy()
        for t in range(6):
            drive = p["B"][0, t] * p["u"][0, t, d]          # held over the step
            sol = solve_ivp(lambda _s, x: a * x + drive, (0.0, dt[0, t, d]), state,
                            method="DOP853", rtol=1e-12, atol=1e-14)
            state = sol.y[:, -1]
            yt = np.dot(p["C"][0, t], state) + p["D"][d] * p["u"][0, t, d]
            zz = p["z"][0, t, d]
            yt *= zz / (1.0 + np.exp(-zz))
            worst = max(worst, _rel_err(y[0, t, d], yt))
        worst = max(worst, _rel_err(h[0, d], state))
    return worst


def pin_zoh_limit(scan, seed=14):
    rng = np.random.default_rng(seed)
    p = random_problem(rng, batch=2, L=9, dim=3, N=4)
    p["A"] = np.zeros_like(p["A"])
    y0, h0 = _call(scan, p)
    y1, h1 = _call(scan, p, zoh=True)
    worst = 0.0 if (np.array_equal(y0, y1) and np.array_equal(h0, h1)) else 1.0
    p["A"] = np.full_like(p["A"], -1e-7)
    y0, h0 = _call(scan, p)
    y1, h1 = _call(scan, p, zoh=True)
    return max(worst, 1e-4 * _rel_err(y1, y0), 1e-4 * _rel_err(h1, h0))


ZOH_PINS = {
    "zoh_lti": (pin_zoh_lti, 1e-9),
    "zoh_ode": (pin_zoh_ode, 1e-9),
    "zoh_limit": (pin_zoh_limit, 1e-10),
}


# ---------------------------------------------------------------- conv prologue
def _silu(v):
    return v / (1.0 + np.exp(-v))


def pin_conv_numpy(conv, seed=8):
    rng = np.random.default_rng(seed)
    worst = 0.0
    for K, bias in ((4, True), (3, False), (2, True)):
        x = rng.standard_normal((2, 19, 5))
        w = rng.standard_normal((5, K))
        cb = rng.standard_normal(5) if bias else None
        u = conv(x, w, cb)
        ref = np.empty_like(x)
        for b in range(2):
            for d in range(5):
                # Conv1d is a cross-correlation: convolve with the reversed taps
                full = np.convolve(x[b, :, d], w[d, ::-1])
                ref[b, :, d] = full[:19] + (cb[d] if bias else 0.0)
        worst = max(worst, _rel_err(u, _silu(ref)))
    return worst


def pin_conv_k1(conv, seed=9):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((3, 7, 4))
    w = rng.standard_normal((4, 1))
    cb = rng.standard_normal(4)
    return _rel_err(conv(x, w, cb), _silu(x * w[:, 0] + cb))


def pin_conv_causal(conv, seed=10):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((1, 16, 3))
    w = rng.standard_normal((3, 4))
    cb = rng.standard_normal(3)
    u0 = conv(x, w, cb)
    x2 = x.copy()
    x2[:, 9] += 1.0
    u1 = conv(x2, w, cb)
    changed = np.any(u1 != u0, axis=(0, 2))
    ok = (not np.any(changed[:9])) and bool(np.all(changed[9:13])) and not np.any(changed[13:])
    return 0.0 if ok else 1.0


def pin_conv_impulse(conv):
    K = 4
    w = np.array([[0.5, -1.25, 2.0, 0.75]])
    x = np.zeros((1, 12, 1))
    x[0, 5, 0] = 1.0
    u = conv(x, w, np.zeros(1))
    ref = np.zeros(12)            # silu(0) = 0 away from the impulse
    for j in range(K):
        ref[5 + j] = _silu(w[0, K - 1 - j])
    return _rel_err(u[0, :, 0], ref)


CONV_PINS = {
    "conv_numpy": (pin_conv_numpy, 1e-14),
    "conv_k1": (pin_conv_k1, 1e-15),
    "conv_causal": (pin_conv_causal, 0.0),
    "conv_impulse": (pin_conv_impulse, 1e-15),
}


# ---------------------------------------------------------------- backward
def pin_bwd_loop_forward(seed=15):
    """The autograd loop's forward equals the C oracle's."""
    import oracle
    from oracle.backward import selective_scan_fwd_loop
    rng = np.random.default_rng(seed)
    worst = 0.0
    for kw in (dict(), dict(softplus=False, bias=False, gate=False, skip=False)):
        p = random_problem(rng, batch=2, L=7, dim=3, N=4, **kw)
        y = selective_scan_fwd_loop(p["u"], p["delta"], p["A"], p["B"], p["C"], p["D"], p["z"],
                                    p["delta_bias"], p["softplus"])
        yr, _ = _call(oracle.selective_scan_fwd, p)
        worst = max(worst, _rel_err(y, yr))
    return worst


def pin_bwd_finite_differences(bwd, seed=16, eps=1e-6):
    """Every gradient against central differences of the C oracle's forward
    along a random direction per input: <grad_X, v> = d/de <dout, y(X + e v)>."""
    import oracle
    rng = np.random.default_rng(seed)
    worst = 0.0
    for kw in (dict(), dict(softplus=False, bias=True, gate=False, skip=True, a_neg=False)):
        p = random_problem(rng, batch=2, L=6, dim=3, N=4, **kw)
        dout = rng.standard_normal(p["u"].shape)
        grads = bwd(p["u"], p["delta"], p["A"], p["B"], p["C"], p["D"], p["z"],
                    p["delta_bias"], p["softplus"], dout)
        for name, g in grads.items():
            v = rng.standard_normal(np.shape(p[name]))
            plus = {**p, name: p[name] + eps * v}
            minus = {**p, name: p[name] - eps * v}
            yp, _ = _call(oracle.selective_scan_fwd, plus)
            ym, _ = _call(oracle.selective_scan_fwd, minus)
            fd = float(np.sum(dout * (yp - ym)) / (2 * eps))
            an = float(np.sum(g * v))
            worst = max(worst, abs(fd - an) / (1.0 + abs(fd)))
    return worst


def pin_bwd_state_finite_differences(bwd, seed=17, eps=1e-6):
    """With an initial state h0 and a gradient dh_last on the last state:
    every gradient, h0's included, against central differences of the C
    oracle's forward from h0 along a random direction per input:
    <grad_X, v> = d/de (<dout, y(X + e v)> + <dh_last, h_last(X + e v)>)."""
    import oracle
    rng = np.random.default_rng(seed)
    worst = 0.0
    for kw in (dict(), dict(softplus=False, bias=True, gate=False, skip=True, a_neg=False)):
        p = random_problem(rng, batch=2, L=6, dim=3, N=4, **kw)
        p["h0"] = rng.standard_normal((2, 3, 4))
        dout = rng.standard_normal(p["u"].shape)
        dh = rng.standard_normal((2, 3, 4))
        grads = bwd(p["u"], p["delta"], p["A"], p["B"], p["C"], p["D"], p["z"],
                    p["delta_bias"], p["softplus"], dout, h0=p["h0"], dh_last=dh)
        assert "h0" in grads
        for name, g in grads.items():
            v = rng.standard_normal(np.shape(p[name]))
            plus = {**p, name: p[name] + eps * v}
            minus = {**p, name: p[name] - eps * v}
            yp, hp = _call(oracle.selective_scan_fwd, plus, h0=plus["h0"])
            ym, hm = _call(oracle.selective_scan_fwd, minus, h0=minus["h0"])
            fd = float((np.sum(dout * (yp - ym)) + np.sum(dh * (hp - hm))) / (2 * eps))
            an = float(np.sum(g * v))
            worst = max(worst, abs(fd - an) / (1.0 + abs(fd)))
    return worst


def pin_bwd_chaining(bwd, seed=18, cut=4):
    """The gradients of a sequence equal those of its two pieces chained:
    the second piece starts from the first's last state, and its h0 gradient
    is the first piece's dh_last; per-step gradients concatenate and the
    shared ones (A, D, delta_bias) add."""
    import oracle
    rng = np.random.default_rng(seed)
    p = random_problem(rng, batch=2, L=9, dim=3, N=4)
    dout = rng.standard_normal(p["u"].shape)
    whole = bwd(p["u"], p["delta"], p["A"], p["B"], p["C"], p["D"], p["z"], p["delta_bias"],
                p["softplus"], dout)
    cut_t = lambda a, s: None if a is None else a[:, s]  # noqa: E731
    p1 = {k: (cut_t(v, slice(0, cut)) if k in ("u", "delta", "B", "C", "z") else v)
          for k, v in p.items()}
    p2 = {k: (cut_t(v, slice(cut, None)) if k in ("u", "delta", "B", "C", "z") else v)
          for k, v in p.items()}
    _, hmid = _call(oracle.selective_scan_fwd, p1)
    g2 = bwd(p2["u"], p2["delta"], p2["A"], p2["B"], p2["C"], p2["D"], p2["z"],
             p2["delta_bias"], p2["softplus"], dout[:, cut:], h0=hmid)
    g1 = bwd(p1["u"], p1["delta"], p1["A"], p1["B"], p1["C"], p1["D"], p1["z"],
             p1["delta_bias"], p1["softplus"], dout[:, :cut], dh_last=g2["h0"])
    worst = 0.0
    for k in ("u", "delta", "B", "C", "z"):
        worst = max(worst, _rel_err(np.concatenate([g1[k], g2[k]], axis=1), whole[k]))
    for k in ("A", "D", "delta_bias"):
        worst = max(worst, _rel_err(g1[k] + g2[k], whole[k]))
    return worst


ALL_PINS = {
    "bruteforce": (pin_bruteforce, 1e-12),
    "lti_direct": (pin_lti_direct, 1e-9),
    "lti_fft": (pin_lti_fft, 1e-9),
    "associativity": (pin_associativity, 1e-12),
    "special_cases": (pin_special_cases, 1e-12),
    "golden": (pin_golden, 1e-14),
    "bruteforce_h0": (pin_bruteforce_h0, 1e-12),
    "chaining": (pin_chaining, 1e-12),
}
