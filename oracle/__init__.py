"""Oracle for the selective-scan forward pass: a plain fp64 CPU definition.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s cpu_baseline / reference leg may import this package.  The
product path (the CUDA library and its Python binding) never imports it and
shares no code with it.

The arithmetic lives in ``ssm_oracle.c`` (one loop nest, fp64, checked by eye
against the pages: the "State Space Models (SSM)" summary page, section 3.2
"Selective Scan Algorithm", with the softplus / D-skip / SiLU-gate steps of the
SelectiveSSM and MambaBlock listings on the same page and on the youngju.dev
"Mamba와 State Space Model 논문 심층 분석" page).  This module only compiles it
with gcc and marshals numpy arrays into it.

Every function here is pinned by ``tests/test_oracle_pins.py`` (brute-force
closed form, the time-invariant convolution identity computed directly and by
FFT, associativity of the state, special cases, the stability bound and a
hand-worked golden fixture).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssm_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libssm_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle with gcc (IEEE semantics: no fast-math)."""
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
               "-ffp-contract=off", src, "-o", out, "-lm"]
        subprocess.run(cmd, check=True)
    return out


def load(path: str | None = None):
    """Load (building first if needed) and return the ctypes library."""
    global _lib
    with _lock:
        if path is not None:
            lib = ctypes.CDLL(path)
            _declare(lib)
            return lib
        if _lib is None:
            build()
            _lib = ctypes.CDLL(_LIB_PATH)
            _declare(_lib)
        return _lib


def _declare(lib):
    dp = ctypes.POINTER(ctypes.c_double)
    i64 = ctypes.c_int64
    lib.ssm_oracle_fwd.restype = ctypes.c_int
    lib.ssm_oracle_fwd.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp, ctypes.c_int,
                                   dp, dp, i64, i64, i64, i64]
    lib.ssm_oracle_fwd_ex.restype = ctypes.c_int
    lib.ssm_oracle_fwd_ex.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp, dp, ctypes.c_int,
                                      ctypes.c_int, dp, dp, i64, i64, i64, i64]
    lib.ssm_oracle_fwd_h0.restype = ctypes.c_int
    lib.ssm_oracle_fwd_h0.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp, dp, ctypes.c_int,
                                      dp, dp, i64, i64, i64, i64]
    lib.ssm_oracle_causal_conv_silu.restype = ctypes.c_int
    lib.ssm_oracle_causal_conv_silu.argtypes = [dp, dp, dp, dp, i64, i64, i64, i64]


def _f64(a):
    if a is None:
        return None
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def selective_scan_fwd(u, delta, A, B, C, D=None, z=None, delta_bias=None,
                       softplus=False, lib=None, h0=None, zoh=False):
    """Selective-scan forward in fp64.

    u, delta, z: (batch, L, dim); A: (dim, N); B, C: (batch, L, N);
    D, delta_bias: (dim,); h0: (batch, dim, N) initial state.  D, z,
    delta_bias and h0 may be None (h0 None = zero state).  zoh: exact
    zero-order-hold discretisation of B instead of dt * B.
    Inputs are converted to float64 exactly (fp32 or decoded bf16 values).
    Returns (y (batch, L, dim) float64, h_last (batch, dim, N) float64).
    """
    lib = lib or load()
    u, delta, A, B, C = map(_f64, (u, delta, A, B, C))
    D, z, delta_bias, h0 = map(_f64, (D, z, delta_bias, h0))
    batch, L, dim = u.shape
    N = A.shape[1]
    assert delta.shape == (batch, L, dim)
    assert A.shape == (dim, N)
    assert B.shape == (batch, L, N) and C.shape == (batch, L, N)
    if D is not None:
        assert D.shape == (dim,)
    if delta_bias is not None:
        assert delta_bias.shape == (dim,)
    if z is not None:
        assert z.shape == (batch, L, dim)
    y = np.zeros((batch, L, dim), dtype=np.float64)
    h = np.zeros((batch, dim, N), dtype=np.float64)
    if zoh:
        if h0 is not None:
            assert h0.shape == (batch, dim, N)
        rc = lib.ssm_oracle_fwd_ex(_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C),
                                   _ptr(D), _ptr(z), _ptr(delta_bias), _ptr(h0),
                                   int(bool(softplus)), 1, _ptr(y), _ptr(h), batch, L, dim, N)
    elif h0 is None:
        rc = lib.ssm_oracle_fwd(_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C),
                                _ptr(D), _ptr(z), _ptr(delta_bias), int(bool(softplus)),
                                _ptr(y), _ptr(h), batch, L, dim, N)
    else:
        assert h0.shape == (batch, dim, N)
        rc = lib.ssm_oracle_fwd_h0(_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C),
                                   _ptr(D), _ptr(z), _ptr(delta_bias), _ptr(h0),
                                   int(bool(softplus)), _ptr(y), _ptr(h), batch, L, dim, N)
    if rc != 0:
        raise ValueError(f"oracle rejected its arguments (rc={rc})")
    return y, h


def selective_scan_step(h, u, delta, A, B, C, D=None, z=None, delta_bias=None,
                        softplus=False, lib=None):
    """One recurrent (decode) step: the definition above at L = 1, starting
    from state h.  u, delta, z: (batch, dim); B, C: (batch, N); h: (batch,
    dim, N).  Returns (y (batch, dim), new state (batch, dim, N))."""
    u, delta, B, C, z = map(_f64, (u, delta, B, C, z))
    y, hn = selective_scan_fwd(u[:, None], delta[:, None], A, B[:, None], C[:, None], D,
                               None if z is None else z[:, None], delta_bias, softplus,
                               lib=lib, h0=h)
    return y[:, 0], hn


def causal_conv_silu(x, w, cb=None, lib=None):
    """u = silu(causal depthwise conv1d(x) + cb) in fp64 (see ssm_oracle.c).
    x: (batch, L, dim); w: (dim, K); cb: (dim,) or None."""
    lib = lib or load()
    x, w, cb = _f64(x), _f64(w), _f64(cb)
    batch, L, dim = x.shape
    K = w.shape[1]
    assert w.shape == (dim, K) and (cb is None or cb.shape == (dim,))
    u = np.zeros((batch, L, dim), dtype=np.float64)
    rc = lib.ssm_oracle_causal_conv_silu(_ptr(x), _ptr(w), _ptr(cb), _ptr(u), batch, L, dim, K)
    if rc != 0:
        raise ValueError(f"oracle rejected its arguments (rc={rc})")
    return u


def conv_selective_scan_fwd(x, w, cb, delta, A, B, C, D=None, z=None, delta_bias=None,
                            softplus=False, h0=None):
    """The scan whose input is u = causal_conv_silu(x, w, cb) (the two steps in
    order, each as defined above).  Returns (y, h_last)."""
    u = causal_conv_silu(x, w, cb)
    return selective_scan_fwd(u, delta, A, B, C, D, z, delta_bias, softplus, h0=h0)


def selective_scan_fwd_threads(u, delta, A, B, C, D=None, z=None, delta_bias=None,
                               softplus=False, threads: int = 1):
    """Same result as selective_scan_fwd, with the (batch, dim) channels split
    into contiguous dim-blocks run on ``threads`` host threads (ctypes releases
    the GIL during the C call).  Channels are independent, so the split changes
    nothing in the arithmetic; it only uses more host cores."""
    if threads <= 1:
        return selective_scan_fwd(u, delta, A, B, C, D, z, delta_bias, softplus)
    u, delta, A, B, C = map(_f64, (u, delta, A, B, C))
    D, z, delta_bias = map(_f64, (D, z, delta_bias))
    batch, L, dim = u.shape
    N = A.shape[1]
    y = np.zeros((batch, L, dim), dtype=np.float64)
    h = np.zeros((batch, dim, N), dtype=np.float64)
    bounds = np.linspace(0, dim, threads + 1).astype(int)
    lib = load()

    def run(lo, hi):
        sl = slice(lo, hi)
        yy, hh = selective_scan_fwd(
            u[:, :, sl], delta[:, :, sl], A[sl], B, C,
            None if D is None else D[sl], None if z is None else z[:, :, sl],
            None if delta_bias is None else delta_bias[sl], softplus, lib=lib)
        y[:, :, sl] = yy
        h[:, sl, :] = hh

    ts = [threading.Thread(target=run, args=(int(bounds[i]), int(bounds[i + 1])))
          for i in range(threads) if bounds[i + 1] > bounds[i]]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    return y, h
