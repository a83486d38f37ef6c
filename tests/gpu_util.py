"""Helpers shared by the GPU tests: move seeded inputs to the device, call the
library through its C ABI binding, and compare with the fp64 oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import ssm_workloads as W
import selective_state_space_150_b300 as ssm

TOL = {"f32": 1e-4, "bf16": 2e-2}


def to_dev(a):
    if a is None:
        return None
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def from_dev(t):
    if t is None:
        return None
    if t.dtype == torch.bfloat16:
        return W.decode(t.view(torch.int16).cpu().numpy().view(np.uint16))
    return t.float().cpu().numpy()


def run_gpu(inp, guard: int = 0, want_h=True, stream=None):
    """Run the library on one input dict; returns (y fp32 numpy, h_last numpy).
    With guard > 0 the outputs sit inside larger buffers whose guard bands are
    filled with a sentinel and checked afterwards."""
    d = {k: to_dev(inp[k]) for k in ("u", "delta", "B", "C", "z", "A", "D", "delta_bias")}
    u = d["u"]
    batch, L, dim = u.shape
    N = d["A"].shape[1]
    ny, nh = batch * L * dim, batch * dim * N
    if guard:
        ybuf = torch.full((ny + 2 * guard,), -7.0, dtype=u.dtype, device="cuda")
        hbuf = torch.full((nh + 2 * guard,), -7.0, dtype=torch.float32, device="cuda")
        y = ybuf[guard:guard + ny].view(batch, L, dim)
        h = hbuf[guard:guard + nh].view(batch, dim, N)
    else:
        y = torch.empty_like(u)
        h = torch.empty((batch, dim, N), dtype=torch.float32, device="cuda")
    ssm.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"],
                           d["delta_bias"], inp["softplus"], y=y, h_last=h if want_h else None,
                           stream=stream)
    st = ssm.ssm_scan_last_device_status(stream or torch.cuda.current_stream().cuda_stream)
    assert st == 0, ssm.ssm_status_string(st)
    if guard:
        for buf in (ybuf, hbuf):
            g = torch.cat([buf[:guard], buf[-guard:]]).float()
            assert torch.all(g == -7.0), "output written outside its buffer"
    return from_dev(y), (from_dev(h) if want_h else None)


def oracle_ref(inp_decoded):
    p = inp_decoded
    return oracle.selective_scan_fwd(p["u"], p["delta"], p["A"], p["B"], p["C"], p["D"], p["z"],
                                     p["delta_bias"], p["softplus"])


def rel_err(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    if got.size == 0:
        return 0.0
    if not np.all(np.isfinite(got)):
        return float("inf")
    return float(np.max(np.abs(got - ref) / (1.0 + np.abs(ref))))


def check_full(inp, tol, **kw):
    """GPU vs oracle on every output element."""
    y, h = run_gpu(inp, **kw)
    yr, hr = oracle_ref(W.decoded(inp))
    ey, eh = rel_err(y, yr), (rel_err(h, hr) if h is not None else 0.0)
    assert ey <= tol and eh <= tol, f"y err {ey:.3e}, h_last err {eh:.3e}, tol {tol:.1e}"
    return ey, eh


def check_sampled(inp, wl, tol, n_dim=24, n_batch=2):
    """GPU on the full problem (the same launch as the benchmark) vs the oracle
    on a sample of (batch row, channel) pairs over the whole sequence."""
    y, h = run_gpu(inp)
    bs, ds = W.channel_sample(wl, n_dim=n_dim, n_batch=n_batch)
    sub = W.gather(inp, bs, ds)
    yr, hr = oracle_ref(sub)
    ys = y[bs][:, :, ds]
    hs = h[bs][:, ds, :]
    ey, eh = rel_err(ys, yr), rel_err(hs, hr)
    assert ey <= tol and eh <= tol, f"y err {ey:.3e}, h_last err {eh:.3e}, tol {tol:.1e}"
    return ey, eh
