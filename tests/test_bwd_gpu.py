"""GPU parity for the backward pass (ssm_scan_bwd), through the C ABI,
against the oracle's fp64 autograd gradients (themselves pinned by finite
differences of the C oracle)."""
import numpy as np
import pytest
import torch

import ssm_workloads as W
import selective_state_space_150_b300 as ssm
from oracle.backward import selective_scan_bwd as oracle_bwd
from tests.gpu_util import from_dev, rel_err, to_dev

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
                                   (1, 17, 64, 1), (2, 50, 32, 8),
                                   # N > 16: slices of 16 states, a ragged last slice, and
                                   # runs of 64 steps in the summing kernel
                                   (1, 70, 40, 17), (2, 33, 64, 40), (1, 150, 33, 64)])
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


# ---------------------------------------------------------------- bf16
BF16_TOL = 4e-3  # bf16 gradients: one round-to-nearest-even on the fp32 result (unit roundoff 2^-8)


def gpu_grads_bf16(inp, dy_bits):
    d = {k: to_dev(inp[k]) for k in ("u", "delta", "B", "C", "z", "A", "D", "delta_bias")}
    g = ssm.selective_scan_bwd(d["u"], d["delta"], d["A"], d["B"], d["C"], to_dev(dy_bits),
                               d["D"], d["z"], d["delta_bias"], inp["softplus"])
    torch.cuda.synchronize()
    return {k: from_dev(v) for k, v in g.items()}, {k: v.dtype for k, v in g.items()}


@pytest.mark.parametrize("flags", FLAGS)
@pytest.mark.parametrize("shape", [(2, 40, 72, 16), (1, 37, 33, 5), (2, 50, 32, 8),
                                   (1, 16, 32, 16), (1, 70, 40, 33)])
def test_bf16_backward_matches_oracle(shape, flags):
    batch, L, dim, N = shape
    wl = BASE.with_shape(name="g", batch=batch, L=L, dim=dim, N=N, dtype="bf16", **flags)
    inp = W.make_inputs(wl, seed=sum(shape) + 7)
    dy32 = np.random.default_rng(sum(shape)).standard_normal((batch, L, dim)).astype(np.float32)
    dy_bits = W.f32_to_bf16_bits(dy32)
    g, dtypes = gpu_grads_bf16(inp, dy_bits)
    x = W.decoded(inp)  # the exact values the GPU reads
    r = oracle_bwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"], x["delta_bias"],
                   x["softplus"], W.decode(dy_bits))
    names = {"u": "du", "delta": "ddelta", "A": "dA", "B": "dB", "C": "dC", "D": "dD",
             "z": "dz", "delta_bias": "ddelta_bias"}
    for k, v in r.items():
        n = names[k]
        bf = k in ("u", "delta", "B", "C", "z")
        assert dtypes[n] == (torch.bfloat16 if bf else torch.float32), (n, dtypes[n])
        err = rel_err(g[n], v)
        assert err <= (BF16_TOL if bf else TOL), (n, err)


def test_bf16_backward_rounds_the_fp32_gradients():
    """The bf16 entry widens its inputs exactly and rounds each gradient once:
    fed the same (bf16-representable) values, it equals the fp32 entry's
    gradients rounded to nearest even, element for element, on the
    per-(step, channel) gradients, and matches bit for bit on the fp32 ones."""
    shape = (2, 48, 64, 16)
    batch, L, dim, N = shape
    wl = BASE.with_shape(name="g", batch=batch, L=L, dim=dim, N=N, dtype="bf16", **FLAGS[0])
    inp = W.make_inputs(wl, seed=11)
    dy_bits = W.f32_to_bf16_bits(
        np.random.default_rng(5).standard_normal((batch, L, dim)).astype(np.float32))
    g16, _ = gpu_grads_bf16(inp, dy_bits)
    x = W.decoded(inp)
    x32 = {k: (None if v is None or k == "softplus" else np.ascontiguousarray(v, dtype=np.float32))
           for k, v in x.items()}
    x32["softplus"] = x["softplus"]
    g32 = gpu_grads(x32, W.decode(dy_bits).astype(np.float32))
    for n in ("du", "ddelta", "dz", "dB", "dC"):
        want = W.decode(W.f32_to_bf16_bits(g32[n]))
        assert np.array_equal(g16[n], want), n
    for n in ("dA", "dD", "ddelta_bias"):
        assert np.array_equal(g16[n], g32[n]), n


def test_sliced_backward_is_deterministic():
    inp, dy = problem((1, 80, 64, 48), seed=8, **FLAGS[0])
    g1, g2 = gpu_grads(inp, dy), gpu_grads(inp, dy)
    assert all(np.array_equal(g1[k], g2[k]) for k in g1)


def test_backward_time_invariant_workload_sampled():
    """The time-invariant workload's N = 64 runs as four slices: its gradients
    on a sample of channels and a shortened sequence against the oracle."""
    wl = W.WORKLOADS["lti_fp32"].with_shape(name="g", L=96, dim=48)
    inp = W.make_inputs(wl, seed=12)
    dy = np.random.default_rng(12).standard_normal((wl.batch, wl.L, wl.dim)).astype(np.float32)
    check(inp, dy)


def test_backward_full_size_mamba130m_bf16_sampled():
    """The full Mamba-130M layer shape (batch 8, L 2048, dim 1536, N 16, bf16),
    checked on a sample of batch rows and channels.  dy is zero outside the
    sampled rows, so those rows alone feed dA, dD and ddelta_bias.  Channels
    are independent given B and C, so the sampled rows and channels form a
    problem of their own, which the oracle solves; du, ddelta, dz there and
    dA, dD, ddelta_bias of the sampled channels must match it.  dB and dC sum
    over every channel and are checked against the whole oracle at the
    smaller sizes above."""
    wl = W.WORKLOADS["mamba130m_bf16"]
    inp = W.make_inputs(wl, seed=0)
    rng = np.random.default_rng(21)
    bs, ds = W.channel_sample(wl, n_dim=16, n_batch=2, seed=3)
    # dy is zero outside the sampled batch rows, so dA, dD and ddelta_bias
    # sum over those rows only, and the channels outside the sample get
    # gradients of their own that are not checked
    dy32 = np.zeros((wl.batch, wl.L, wl.dim), dtype=np.float32)
    dy32[bs] = rng.standard_normal((len(bs), wl.L, wl.dim)).astype(np.float32)
    dy_bits = W.f32_to_bf16_bits(dy32)
    g, _ = gpu_grads_bf16(inp, dy_bits)
    sub = W.gather(inp, bs, ds)
    dys = W.decode(dy_bits)[bs][:, :, ds]
    r = oracle_bwd(sub["u"], sub["delta"], sub["A"], sub["B"], sub["C"], sub["D"], sub["z"],
                   sub["delta_bias"], sub["softplus"], dys)
    for name, k in (("du", "u"), ("ddelta", "delta"), ("dz", "z")):
        err = rel_err(g[name][bs][:, :, ds], r[k])
        assert err <= BF16_TOL, (name, err)
    for name, k in (("dA", "A"), ("dD", "D"), ("ddelta_bias", "delta_bias")):
        err = rel_err(g[name][ds], r[k])
        assert err <= TOL, (name, err)



# ---------------------------------------------------------------- pieces of a sequence
def _state_problem(shape, seed, dtype="f32", **flags):
    batch, L, dim, N = shape
    wl = BASE.with_shape(name="g", batch=batch, L=L, dim=dim, N=N, dtype=dtype, **flags)
    inp = W.make_inputs(wl, seed=seed)
    rng = np.random.default_rng(seed + 1)
    h0 = rng.standard_normal((batch, dim, N)).astype(np.float32)
    dh = rng.standard_normal((batch, dim, N)).astype(np.float32)
    dy = rng.standard_normal((batch, L, dim)).astype(np.float32)
    if dtype == "bf16":
        dy = W.f32_to_bf16_bits(dy)
    return inp, h0, dh, dy


def _gpu_state_grads(inp, dy, h0, dh):
    d = {k: to_dev(inp[k]) for k in ("u", "delta", "B", "C", "z", "A", "D", "delta_bias")}
    g = ssm.selective_scan_bwd(d["u"], d["delta"], d["A"], d["B"], d["C"], to_dev(dy), d["D"],
                               d["z"], d["delta_bias"], inp["softplus"],
                               h0=None if h0 is None else to_dev(h0),
                               dh_last=None if dh is None else to_dev(dh))
    torch.cuda.synchronize()
    return {k: from_dev(v) for k, v in g.items()}


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(2, 40, 72, 16), (1, 37, 33, 5), (1, 30, 40, 40)])
@pytest.mark.parametrize("which", ["both", "h0", "dh_last"])
def test_backward_with_states_matches_oracle(dtype, shape, which):
    inp, h0, dh, dy = _state_problem(shape, sum(shape) + 3, dtype, **FLAGS[0])
    h0 = h0 if which in ("both", "h0") else None
    dh = dh if which in ("both", "dh_last") else None
    g = _gpu_state_grads(inp, dy, h0, dh)
    x = W.decoded(inp)
    r = oracle_bwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"], x["delta_bias"],
                   x["softplus"], W.decode(dy), h0=h0, dh_last=dh)
    names = {"u": "du", "delta": "ddelta", "A": "dA", "B": "dB", "C": "dC", "D": "dD",
             "z": "dz", "delta_bias": "ddelta_bias", "h0": "dh0"}
    if "h0" not in r:  # no h0 given: its gradient still comes back, against a zero start
        r["h0"] = oracle_bwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"],
                             x["delta_bias"], x["softplus"], W.decode(dy),
                             h0=np.zeros_like(g["dh0"]), dh_last=dh)["h0"]
    for k, v in r.items():
        bf = dtype == "bf16" and k in ("u", "delta", "B", "C", "z")
        err = rel_err(g[names[k]], v)
        assert err <= (BF16_TOL if bf else TOL), (names[k], err)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(8, 64, 256, 16), (4, 50, 96, 40), (6, 33, 96, 5)])
def test_checkpoints_by_the_forward_pipeline_equal_the_kernels_own_walk(dtype, shape):
    """Where the tiles can move by TMA the backward takes its checkpoints from
    the forward's warp-specialised kernel (checkpoint instantiation); with
    plain loads forced, the backward kernel walks forward itself.  The two
    compute every state with the same arithmetic in the same order, so all
    gradients, dh0 included, agree bit for bit."""
    from selective_state_space_150_b300 import ssmscan as K
    batch, L, dim, N = shape
    plan = ssm.ssm_scan_plan(batch, L, dim, N, 1 if dtype == "bf16" else 0)
    assert plan["tma"] == 1 and plan["kernel"] == 2  # the pipeline applies to this shape
    inp, h0, dh, dy = _state_problem(shape, sum(shape) + 11, dtype, **FLAGS[0])
    a = _gpu_state_grads(inp, dy, h0, dh)
    assert ssm.ssm_set_knob(K.SSM_KNOB_PLAIN_LOADS, 1) == K.SSM_OK
    try:
        b = _gpu_state_grads(inp, dy, h0, dh)
    finally:
        ssm.ssm_set_knob(K.SSM_KNOB_PLAIN_LOADS, 0)
    assert a.keys() == b.keys()
    for k in a:
        assert np.array_equal(a[k], b[k]), k


def test_backward_pieces_chain_to_the_whole():
    """A sequence's gradients from two pieces: the second from the first's last
    state, the first with the second's dh0 as dh_last."""
    shape = (2, 80, 64, 16)
    inp, _, _, dy = _state_problem(shape, 31, **FLAGS[0])
    whole = _gpu_state_grads(inp, dy, None, None)
    cut = 48
    part = lambda s: {k: (v[:, s] if k in ("u", "delta", "B", "C", "z") and v is not None else v)
                      for k, v in inp.items()}  # noqa: E731
    p1, p2 = part(slice(0, cut)), part(slice(cut, None))
    d = {k: to_dev(p1[k]) for k in ("u", "delta", "B", "C", "z", "A", "D", "delta_bias")}
    y1, hmid = ssm.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"],
                                      d["delta_bias"], p1["softplus"])
    g2 = _gpu_state_grads(p2, dy[:, cut:], hmid.cpu().numpy(), None)
    g1 = _gpu_state_grads(p1, dy[:, :cut], None, g2["dh0"])
    for k in ("du", "ddelta", "dz", "dB", "dC"):
        err = rel_err(np.concatenate([g1[k], g2[k]], axis=1), whole[k])
        assert err <= 2e-5, (k, err)
    for k in ("dA", "dD", "ddelta_bias"):
        err = rel_err(g1[k] + g2[k], whole[k])
        assert err <= 2e-5, (k, err)


def test_backward_of_an_empty_piece_passes_dh_last_through():
    inp, h0, dh, dy = _state_problem((2, 0, 32, 16), 5, **FLAGS[0])
    g = _gpu_state_grads(inp, dy, h0, dh)
    assert np.array_equal(g["dh0"], dh)
    assert all(not np.any(v) for k, v in g.items() if k != "dh0")



# ---------------------------------------------------------------- time segments
@pytest.fixture
def bwd_segments():
    """Force the backward's time-segment count for one test, then restore."""
    from selective_state_space_150_b300 import ssmscan as K

    def force(n):
        assert ssm.ssm_set_knob(K.SSM_KNOB_BWD_SEGMENTS, n) == K.SSM_OK
    yield force
    force(0)


@pytest.mark.parametrize("segs", [2, 3, 7])
@pytest.mark.parametrize("shape", [(2, 200, 72, 16), (1, 203, 33, 5), (1, 150, 40, 40)])
def test_segmented_backward_matches_oracle(bwd_segments, shape, segs):
    bwd_segments(segs)
    inp, dy = problem(shape, seed=sum(shape) + segs, **FLAGS[0])
    check(inp, dy)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_segmented_backward_with_states_matches_oracle(bwd_segments, dtype):
    bwd_segments(4)
    inp, h0, dh, dy = _state_problem((2, 130, 40, 16), 77, dtype, **FLAGS[0])
    g = _gpu_state_grads(inp, dy, h0, dh)
    x = W.decoded(inp)
    r = oracle_bwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"], x["delta_bias"],
                   x["softplus"], W.decode(dy), h0=h0, dh_last=dh)
    names = {"u": "du", "delta": "ddelta", "A": "dA", "B": "dB", "C": "dC", "D": "dD",
             "z": "dz", "delta_bias": "ddelta_bias", "h0": "dh0"}
    for k, v in r.items():
        bf = dtype == "bf16" and k in ("u", "delta", "B", "C", "z")
        err = rel_err(g[names[k]], v)
        assert err <= (BF16_TOL if bf else TOL), (names[k], err)


def test_segmented_backward_is_deterministic_and_close_to_one_segment(bwd_segments):
    inp, dy = problem((1, 320, 64, 16), seed=9, **FLAGS[0])
    bwd_segments(1)
    g1 = gpu_grads(inp, dy)
    bwd_segments(5)
    g5, g5b = gpu_grads(inp, dy), gpu_grads(inp, dy)
    for k in g1:
        assert np.array_equal(g5[k], g5b[k]), k
        assert rel_err(g5[k], g1[k]) <= 5e-5, k
