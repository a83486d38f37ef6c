"""Achieved accuracy of every workload and of every call beyond the plain
forward, against the fp64 oracle, next to the tolerance it must meet.  Each
test asserts its tolerance and records max |gpu - ref| / (1 + |ref|); with
SSM_MARGINS_OUT set, the last test writes the records there as JSON (the
margin is the tolerance divided by the achieved error)."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import ssm_workloads as W
import selective_state_space_150_b300 as ssm
from oracle.backward import selective_scan_bwd as oracle_bwd
from tests.gpu_util import TOL, from_dev, oracle_ref, rel_err, run_gpu, to_dev

pytestmark = pytest.mark.gpu

RECORDS = []
BWD_TOL = {"f32": 2e-4, "bf16": 4e-3}  # bf16 gradients: one rounding of the fp32 result


def record(name, dtype, tol, **errs):
    worst = max(errs.values())
    RECORDS.append({"case": name, "dtype": dtype, "tolerance": tol,
                    "errors": {k: float(v) for k, v in errs.items()},
                    "margin": (tol / worst) if worst > 0 else None})
    assert worst <= tol, (name, errs, tol)


def sampled(wl, n_dim, n_batch):
    inp = W.make_inputs(wl)
    y, h = run_gpu(inp)
    bs, ds = W.channel_sample(wl, n_dim=n_dim, n_batch=n_batch)
    yr, hr = oracle_ref(W.gather(inp, bs, ds))
    return rel_err(y[bs][:, :, ds], yr), rel_err(h[bs][:, ds, :], hr)


@pytest.mark.parametrize("name", ["small_fp32", "lti_fp32", "lti_fp32_skip"])
def test_small_workloads_every_element(name):
    wl = (W.WORKLOADS["lti_fp32"].with_shape(skip=True) if name == "lti_fp32_skip"
          else W.WORKLOADS[name])
    inp = W.make_inputs(wl)
    y, h = run_gpu(inp)
    yr, hr = oracle_ref(W.decoded(inp))
    record(name, wl.dtype, TOL["f32"], y=rel_err(y, yr), h_last=rel_err(h, hr))


@pytest.mark.parametrize("name", ["mamba130m_bf16", "mamba130m_bf16_nogate", "mamba2p8b_bf16"] +
                         [f"longctx_L{L}" for L in W.LONGCTX_LS])
def test_large_workloads_sampled(name):
    wl = W.WORKLOADS[name]
    n_dim = 12 if wl.L > 32768 else 24
    ey, eh = sampled(wl, n_dim=n_dim, n_batch=min(2, wl.batch))
    record(name + " (sampled channels)", wl.dtype, TOL["bf16"], y=ey, h_last=eh)


def _medium(dtype, **flags):
    base = W.WORKLOADS["mamba130m_bf16"] if dtype == "bf16" else W.WORKLOADS["small_fp32"]
    return base.with_shape(name="m", batch=2, L=300, dim=96, N=16, **flags)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_conv_prologue(dtype):
    wl = _medium(dtype)
    inp = W.make_inputs(wl, seed=1)
    rng = np.random.default_rng(2)
    w = (0.5 * rng.standard_normal((wl.dim, 4))).astype(np.float32)
    cb = (0.1 * rng.standard_normal(wl.dim)).astype(np.float32)
    d = {k: to_dev(inp[k]) for k in ("u", "delta", "B", "C", "z", "A", "D", "delta_bias")}
    y, h = ssm.conv_selective_scan_fwd(d["u"], torch.from_numpy(w).cuda(),
                                       torch.from_numpy(cb).cuda(), d["delta"], d["A"], d["B"],
                                       d["C"], d["D"], d["z"], d["delta_bias"], inp["softplus"])
    torch.cuda.synchronize()
    p = W.decoded(inp)
    yr, hr = oracle.conv_selective_scan_fwd(p["u"], w, cb, p["delta"], p["A"], p["B"], p["C"],
                                            p["D"], p["z"], p["delta_bias"], p["softplus"])
    record("conv1d(k=4)+SiLU prologue, 2x300x96x16", dtype, TOL[dtype],
           y=rel_err(from_dev(y), yr), h_last=rel_err(from_dev(h), hr))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_zero_order_hold(dtype):
    wl = _medium(dtype)
    inp = W.make_inputs(wl, seed=3)
    d = {k: to_dev(inp[k]) for k in ("u", "delta", "B", "C", "z", "A", "D", "delta_bias")}
    y, h = ssm.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"],
                                  d["delta_bias"], inp["softplus"], zoh=True)
    torch.cuda.synchronize()
    p = W.decoded(inp)
    yr, hr = oracle.selective_scan_fwd(p["u"], p["delta"], p["A"], p["B"], p["C"], p["D"], p["z"],
                                       p["delta_bias"], p["softplus"], zoh=True)
    record("exact zero-order hold, 2x300x96x16", dtype, TOL[dtype],
           y=rel_err(from_dev(y), yr), h_last=rel_err(from_dev(h), hr))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_initial_state(dtype):
    wl = _medium(dtype)
    inp = W.make_inputs(wl, seed=4)
    h0 = np.random.default_rng(5).standard_normal((wl.batch, wl.dim, wl.N)).astype(np.float32)
    d = {k: to_dev(inp[k]) for k in ("u", "delta", "B", "C", "z", "A", "D", "delta_bias")}
    y, h = ssm.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"],
                                  d["delta_bias"], inp["softplus"], h0=torch.from_numpy(h0).cuda())
    torch.cuda.synchronize()
    p = W.decoded(inp)
    yr, hr = oracle.selective_scan_fwd(p["u"], p["delta"], p["A"], p["B"], p["C"], p["D"], p["z"],
                                       p["delta_bias"], p["softplus"], h0=h0.astype(np.float64))
    record("scan from h0, 2x300x96x16", dtype, TOL[dtype],
           y=rel_err(from_dev(y), yr), h_last=rel_err(from_dev(h), hr))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_recurrent_steps(dtype):
    """24 one-token steps chained through the state, against the oracle's scan."""
    wl = _medium(dtype).with_shape(L=24)
    inp = W.make_inputs(wl, seed=6)
    d = {k: to_dev(inp[k]) for k in ("u", "delta", "B", "C", "z", "A", "D", "delta_bias")}
    h = torch.zeros((wl.batch, wl.dim, wl.N), dtype=torch.float32, device="cuda")
    ys = []
    for t in range(wl.L):
        tok = {k: (None if d[k] is None else d[k][:, t].contiguous())
               for k in ("u", "delta", "B", "C", "z")}
        ys.append(ssm.selective_scan_step(tok["u"], tok["delta"], d["A"], tok["B"], tok["C"], h,
                                          d["D"], tok["z"], d["delta_bias"], inp["softplus"]))
    torch.cuda.synchronize()
    y = np.stack([from_dev(v) for v in ys], axis=1)
    yr, hr = oracle_ref(W.decoded(inp))
    record("24 chained one-token steps, 2x96x16 states", dtype, TOL[dtype],
           y=rel_err(y, yr), h_last=rel_err(from_dev(h), hr))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_backward(dtype):
    base = W.WORKLOADS["small_fp32"]
    wl = base.with_shape(name="g", batch=2, L=96, dim=48, N=16, dtype=dtype, softplus=True,
                         delta_bias=True, gate=True, skip=True, delta_kind="normal_raw")
    inp = W.make_inputs(wl, seed=7)
    dy32 = np.random.default_rng(8).standard_normal((wl.batch, wl.L, wl.dim)).astype(np.float32)
    dy = W.f32_to_bf16_bits(dy32) if dtype == "bf16" else dy32
    d = {k: to_dev(inp[k]) for k in ("u", "delta", "B", "C", "z", "A", "D", "delta_bias")}
    g = ssm.selective_scan_bwd(d["u"], d["delta"], d["A"], d["B"], d["C"], to_dev(dy), d["D"],
                               d["z"], d["delta_bias"], inp["softplus"])
    torch.cuda.synchronize()
    x = W.decoded(inp)
    r = oracle_bwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"], x["delta_bias"],
                   x["softplus"], W.decode(dy) if dtype == "bf16" else dy)
    names = {"u": "du", "delta": "ddelta", "A": "dA", "B": "dB", "C": "dC", "D": "dD",
             "z": "dz", "delta_bias": "ddelta_bias"}
    errs = {names[k]: rel_err(from_dev(g[names[k]]), v) for k, v in r.items()}
    # bf16 tensors take the bf16 tolerance; dA, dD, ddelta_bias stay fp32
    fp32_grads = {k: v for k, v in errs.items() if k in ("dA", "dD", "ddelta_bias")}
    io_grads = {k: v for k, v in errs.items() if k not in fp32_grads}
    record("backward (io gradients), 2x96x48x16", dtype, BWD_TOL[dtype], **io_grads)
    record("backward (dA, dD, ddelta_bias), 2x96x48x16", dtype, BWD_TOL["f32"], **fp32_grads)


def test_zz_write_records():
    out = os.environ.get("SSM_MARGINS_OUT")
    if out:
        with open(out, "w") as f:
            json.dump(RECORDS, f, indent=1)
    assert RECORDS
