"""GPU parity for the initial-state scan (ssm_scan_fwd*_h0) and the one-token
recurrent step (ssm_scan_step*), through the C ABI, against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import ssm_workloads as W
import selective_state_space_150_b300 as ssm
from selective_state_space_150_b300 import ssmscan
from tests.gpu_util import TOL, from_dev, rel_err, to_dev

pytestmark = pytest.mark.gpu

BASE = {"bf16": W.WORKLOADS["mamba130m_bf16"], "f32": W.WORKLOADS["small_fp32"]}


@pytest.fixture(autouse=True)
def _reset_knobs():
    yield
    for k in (ssmscan.SSM_KNOB_SEGMENTS, ssmscan.SSM_KNOB_KERNEL, ssmscan.SSM_KNOB_CHUNK):
        ssm.ssm_set_knob(k, 0)


def problem(dtype, batch, L, dim, N, seed, **flags):
    wl = BASE[dtype].with_shape(name="s", batch=batch, L=L, dim=dim, N=N, **flags)
    inp = W.make_inputs(wl, seed=seed)
    h0 = np.random.default_rng(seed + 1000).standard_normal((batch, dim, N)).astype(np.float32)
    return inp, h0


def dev_inputs(inp):
    return {k: to_dev(inp[k]) for k in ("u", "delta", "B", "C", "z", "A", "D", "delta_bias")}


def oracle_h0(inp, h0, t0=0, t1=None):
    p = W.decoded(inp)
    sl = slice(t0, t1)
    cut = lambda a: None if a is None else a[:, sl]  # noqa: E731
    return oracle.selective_scan_fwd(cut(p["u"]), cut(p["delta"]), p["A"], cut(p["B"]),
                                     cut(p["C"]), p["D"], cut(p["z"]), p["delta_bias"],
                                     p["softplus"], h0=h0)


def gpu_h0(d, softplus, h0_dev, t0=0, t1=None):
    sl = slice(t0, t1)
    cut = lambda t: None if t is None else t[:, sl].contiguous()  # noqa: E731
    y, h = ssm.selective_scan_fwd(cut(d["u"]), cut(d["delta"]), d["A"], cut(d["B"]),
                                  cut(d["C"]), d["D"], cut(d["z"]), d["delta_bias"], softplus,
                                  h0=h0_dev)
    st = ssm.ssm_scan_last_device_status(torch.cuda.current_stream().cuda_stream)
    assert st == 0, ssm.ssm_status_string(st)
    return y, h


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("kernel", [1, 2])
@pytest.mark.parametrize("segs", [1, 4])
@pytest.mark.parametrize("shape", [(2, 150, 72, 16), (1, 333, 40, 5), (2, 97, 64, 64)])
def test_scan_from_h0_matches_oracle(dtype, kernel, segs, shape):
    ssm.ssm_set_knob(ssmscan.SSM_KNOB_KERNEL, kernel)
    ssm.ssm_set_knob(ssmscan.SSM_KNOB_SEGMENTS, segs)
    inp, h0 = problem(dtype, *shape, seed=sum(shape) + segs)
    d = dev_inputs(inp)
    y, h = gpu_h0(d, inp["softplus"], torch.from_numpy(h0).cuda())
    yr, hr = oracle_h0(inp, h0.astype(np.float64))
    assert rel_err(from_dev(y), yr) <= TOL[dtype] and rel_err(from_dev(h), hr) <= TOL[dtype]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_zero_h0_equals_the_zero_state_entry(dtype):
    inp, _ = problem(dtype, 2, 200, 96, 16, seed=3)
    d = dev_inputs(inp)
    y0, h0 = ssm.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"],
                                    d["delta_bias"], inp["softplus"])
    zero = torch.zeros((2, 96, 16), dtype=torch.float32, device="cuda")
    y1, h1 = gpu_h0(d, inp["softplus"], zero)
    assert torch.equal(y0, y1) and torch.equal(h0, h1)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("split", [1, 100, 299])
def test_two_calls_chained_through_the_state_equal_one_call(dtype, split):
    inp, h0 = problem(dtype, 2, 300, 64, 16, seed=split)
    d = dev_inputs(inp)
    h0d = torch.from_numpy(h0).cuda()
    ya, ha = gpu_h0(d, inp["softplus"], h0d, 0, split)
    yb, hb = gpu_h0(d, inp["softplus"], ha, split, None)
    yr, hr = oracle_h0(inp, h0.astype(np.float64))
    y = np.concatenate([from_dev(ya), from_dev(yb)], axis=1)
    assert rel_err(y, yr) <= TOL[dtype] and rel_err(from_dev(hb), hr) <= TOL[dtype]


def step_inputs(inp, t):
    """Token t of a sequence problem, as (batch, dim) / (batch, N) device tensors."""
    d = dev_inputs(inp)
    tok = {k: (None if d[k] is None else d[k][:, t].contiguous())
           for k in ("u", "delta", "B", "C", "z")}
    tok.update(A=d["A"], D=d["D"], delta_bias=d["delta_bias"])
    return tok


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(3, 1, 200, 16), (1, 1, 33, 5), (2, 1, 64, 128), (4, 1, 1536, 16)])
@pytest.mark.parametrize("flags", [
    dict(softplus=True, delta_bias=True, gate=True, skip=True, delta_kind="normal_raw"),
    dict(softplus=False, delta_bias=False, gate=False, skip=False, delta_kind="loguniform_td"),
])
def test_step_matches_oracle(dtype, shape, flags):
    inp, h0 = problem(dtype, *shape, seed=shape[2] + shape[3], **flags)
    tok = step_inputs(inp, 0)
    h = torch.from_numpy(h0).cuda()
    y = ssm.selective_scan_step(tok["u"], tok["delta"], tok["A"], tok["B"], tok["C"], h,
                                tok["D"], tok["z"], tok["delta_bias"], inp["softplus"])
    torch.cuda.synchronize()
    p = W.decoded(inp)
    yr, hr = oracle.selective_scan_step(h0.astype(np.float64), p["u"][:, 0], p["delta"][:, 0],
                                        p["A"], p["B"][:, 0], p["C"][:, 0], p["D"],
                                        None if p["z"] is None else p["z"][:, 0],
                                        p["delta_bias"], p["softplus"])
    assert rel_err(from_dev(y), yr) <= TOL[dtype] and rel_err(from_dev(h), hr) <= TOL[dtype]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_steps_chain_to_the_scan(dtype):
    """24 one-token steps from h0 equal the 24-step scan from h0 (oracle), and
    the GPU scan from the same state within the same tolerance."""
    inp, h0 = problem(dtype, 2, 24, 96, 16, seed=5)
    h = torch.from_numpy(h0).cuda()
    ys = []
    for t in range(24):
        tok = step_inputs(inp, t)
        ys.append(ssm.selective_scan_step(tok["u"], tok["delta"], tok["A"], tok["B"], tok["C"], h,
                                          tok["D"], tok["z"], tok["delta_bias"], inp["softplus"]))
    torch.cuda.synchronize()
    y = np.stack([from_dev(v) for v in ys], axis=1)
    yr, hr = oracle_h0(inp, h0.astype(np.float64))
    assert rel_err(y, yr) <= TOL[dtype] and rel_err(from_dev(h), hr) <= TOL[dtype]
    yg, hg = gpu_h0(dev_inputs(inp), inp["softplus"], torch.from_numpy(h0).cuda())
    assert rel_err(y, from_dev(yg)) <= TOL[dtype]


def test_step_writes_only_its_outputs():
    inp, h0 = problem("bf16", 2, 1, 96, 16, seed=9)
    tok = step_inputs(inp, 0)
    g = 64
    hbuf = torch.full((2 * 96 * 16 + 2 * g,), -7.0, dtype=torch.float32, device="cuda")
    ybuf = torch.full((2 * 96 + 2 * g,), -7.0, dtype=torch.bfloat16, device="cuda")
    h = hbuf[g:-g].view(2, 96, 16)
    h.copy_(torch.from_numpy(h0))
    y = ybuf[g:-g].view(2, 96)
    ssm.selective_scan_step(tok["u"], tok["delta"], tok["A"], tok["B"], tok["C"], h, tok["D"],
                            tok["z"], tok["delta_bias"], True, y=y)
    torch.cuda.synchronize()
    for buf in (hbuf, ybuf):
        assert torch.all(torch.cat([buf[:g], buf[-g:]]).float() == -7.0)
