"""GPU parity for the backward pass (ssm_scan_bwd), through the C ABI,
against the oracle's fp64 autograd gradients (themselves pinned by finite
differences of the C oracle)."""
import numpy as np
import pytest
import torch

import ssm_workloads as W
import selective_state_space_150_b300 as ssm
from oracle.backward import selective_scan_bwd as oracle_bwd
from tests.gpu_util import rel_err

pytestmark = pytest.mark.gpu

TOL = 2e-4     # fp32 gradients against fp64, |err| <= TOL (1 + |ref|)
BASE = W.WORKLOADS["small_fp32"]


def problem(shape, seed, **flags):
    batch, L, dim, N = shape
    wl = BASE.with_shape(name="g", batch=batch, L=L, dim=dim, N=N, **flags)
    inp = W.make_inputs(wl, seed=seed)
    dy = np.random.default_rng(seed + 99).standard_normal((batch, L, dim)).astype(np.float32)
    return inp, dy


def gpu_grads(inp, dy):
    d = {k: (None if inp[k] is None else torch.from_numpy(np.ascontiguousarray(inp[k])).cuda())
         for k in ("u", "delta", "B", "C", "z", "A", "D", "delta_bias")}
    g = ssm.selective_scan_bwd(d["u"], d["delta"], d["A"], d["B"], d["C"],
                               torch.from_numpy(dy).cuda(), d["D"], d["z"], d["delta_bias"],
                               inp["softplus"])
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in g.items()}


def check(inp, dy):
    g = gpu_grads(inp, dy)
    r = oracle_bwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                   inp["delta_bias"], inp["softplus"], dy)
    names = {"u": "du", "delta": "ddelta", "A": "dA", "B": "dB", "C": "dC", "D": "dD",
             "z": "dz", "delta_bias": "ddelta_bias"}
    errs = {names[k]: rel_err(g[names[k]], v) for k, v in r.items()}
    assert max(errs.values()) <= TOL, errs
    return g


FLAGS = [
    dict(softplus=True, delta_bias=True, gate=True, skip=True, delta_kind="normal_raw"),
    dict(softplus=False, delta_bias=False, gate=False, skip=False, delta_kind="loguniform_td"),
    dict(softplus=True, delta_bias=False, gate=True, skip=False, delta_kind="normal_raw"),
]


@pytest.mark.parametrize("flags", FLAGS)
@pytest.mark.parametrize("shape", [(2, 40, 72, 16), (1, 37, 33, 5), (3, 20, 40, 4),
                                   (1, 17, 64, 1), (2, 50, 32, 8)])
def test_backward_matches_oracle(shape, flags):
    inp, dy = problem(shape, seed=sum(shape), **flags)
    check(inp, dy)


def test_backward_is_deterministic():
    inp, dy = problem((2, 64, 96, 16), seed=3, **FLAGS[0])
    g1, g2 = gpu_grads(inp, dy), gpu_grads(inp, dy)
    assert all(np.array_equal(g1[k], g2[k]) for k in g1)


def test_backward_of_an_empty_sequence_is_zero():
    inp, dy = problem((2, 0, 32, 16), seed=4, **FLAGS[0])
    g = gpu_grads(inp, dy)
    assert all(not np.any(v) for v in g.values())
