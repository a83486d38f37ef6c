"""Gradients of the selective-scan forward (test infrastructure only, like
the rest of ``oracle/``): torch fp64 autograd through a plain loop that
restates the definition of ``ssm_oracle.c`` step by step.  The loop is
checked against the C oracle's forward, and the gradients against central
finite differences of the C oracle (tests/oracle_pins.py, backward pins).

The backward pass of the pages' training story (doyouknow.kr Mamba guide,
section 3-3, "recomputation": the state is recomputed in the backward pass
instead of being stored) computes exactly these gradients; how the GPU
recomputes them is its own business, the values are fixed by the forward.
"""
from __future__ import annotations

import numpy as np


def _forward_torch(u, delta, A, B, C, D, z, delta_bias, softplus, h0=None, return_h=False):
    """The definition (Euler B), one step at a time, on torch fp64 tensors,
    from the state h0 (zero when None): returns y (batch, L, dim), and the
    last state (batch, dim, N) too when return_h."""
    import torch

    batch, L, dim = u.shape
    N = A.shape[1]
    h = torch.zeros((batch, dim, N), dtype=torch.float64) if h0 is None else h0
    ys = []
    for t in range(L):
        dt = delta[:, t, :]
        if delta_bias is not None:
            dt = dt + delta_bias
        if softplus:
            dt = torch.nn.functional.softplus(dt, beta=1.0, threshold=1e9)  # log(1 + e^x)
        x = u[:, t, :]
        dA = torch.exp(dt[..., None] * A[None])                   # (batch, dim, N)
        dBu = dt[..., None] * B[:, t, None, :] * x[..., None]     # (batch, dim, N)
        h = dA * h + dBu
        y = (h * C[:, t, None, :]).sum(-1)
        if D is not None:
            y = y + D * x
        if z is not None:
            zz = z[:, t, :]
            y = y * (zz / (1.0 + torch.exp(-zz)))
        ys.append(y)
    y = torch.stack(ys, dim=1) if L > 0 else torch.zeros((batch, 0, dim), dtype=torch.float64)
    return (y, h) if return_h else y


def selective_scan_fwd_loop(u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=False):
    """The forward of the autograd loop, as numpy fp64 (for its pin)."""
    import torch

    t = lambda a: None if a is None else torch.as_tensor(np.asarray(a, dtype=np.float64))  # noqa
    with torch.no_grad():
        y = _forward_torch(t(u), t(delta), t(A), t(B), t(C), t(D), t(z), t(delta_bias), softplus)
    return y.numpy()


def selective_scan_bwd(u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=False,
                       dout=None, h0=None, dh_last=None):
    """Vector-Jacobian product of (y, h_last) with the upstream gradients dout
    (batch, L, dim) and dh_last (batch, dim, N; zero when None), the scan
    starting from h0 (batch, dim, N; zero when None).  Returns a dict of fp64
    numpy gradients with the shapes of the inputs: u, delta, A, B, C, and D,
    z, delta_bias, h0 where given.  With h0 and dh_last a long sequence's
    gradients follow from its pieces: a piece's h0 gradient is the dh_last of
    the piece before it."""
    import torch

    names = ("u", "delta", "A", "B", "C", "D", "z", "delta_bias", "h0")
    vals = (u, delta, A, B, C, D, z, delta_bias, h0)
    ts = {}
    for n, v in zip(names, vals):
        ts[n] = (None if v is None
                 else torch.tensor(np.asarray(v, dtype=np.float64), requires_grad=True))
    y, h = _forward_torch(ts["u"], ts["delta"], ts["A"], ts["B"], ts["C"], ts["D"], ts["z"],
                          ts["delta_bias"], softplus, h0=ts["h0"], return_h=True)
    outs, gouts = [y], [torch.as_tensor(np.asarray(dout, dtype=np.float64))]
    if dh_last is not None:
        outs.append(h)
        gouts.append(torch.as_tensor(np.asarray(dh_last, dtype=np.float64)))
    leaves = [n for n in names if ts[n] is not None]
    if not any(o.requires_grad for o in outs):  # L = 0 and no h0: nothing depends on the inputs
        return {n: np.zeros(ts[n].shape) for n in leaves}
    grads = torch.autograd.grad(outs, [ts[n] for n in leaves], grad_outputs=gouts,
                                allow_unused=True)
    return {n: (np.zeros(ts[n].shape) if gr is None else gr.numpy())
            for n, gr in zip(leaves, grads)}
