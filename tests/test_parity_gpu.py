"""GPU parity: libssmscan (through its C ABI) against the fp64 oracle on the
same seeded inputs.  Tolerances: |gpu - ref| <= 1e-4 (1 + |ref|) for fp32
inputs and <= 2e-2 (1 + |ref|) for bf16 inputs, elementwise over y and h_last."""
import numpy as np
import pytest
import torch

import ssm_workloads as W
import selective_state_space_150_b300 as ssm
from selective_state_space_150_b300 import ssmscan
from tests.gpu_util import TOL, check_full, check_sampled, oracle_ref, rel_err, run_gpu

pytestmark = pytest.mark.gpu

BASE_BF16 = W.WORKLOADS["mamba130m_bf16"]
BASE_F32 = W.WORKLOADS["small_fp32"]


def wl_for(dtype, batch, L, dim, N, **flags):
    base = BASE_BF16 if dtype == "bf16" else BASE_F32
    return base.with_shape(name="t", batch=batch, L=L, dim=dim, N=N, **flags)


@pytest.fixture(autouse=True)
def _reset_knobs():
    yield
    for k in (ssmscan.SSM_KNOB_STATE_GROUPS, ssmscan.SSM_KNOB_PLAIN_LOADS, ssmscan.SSM_KNOB_STAGES,
              ssmscan.SSM_KNOB_CHUNK, ssmscan.SSM_KNOB_SEGMENTS, ssmscan.SSM_KNOB_KERNEL,
              ssmscan.SSM_KNOB_FORCE_TIMEOUT):
        ssm.ssm_set_knob(k, 0)
    ssm.ssm_set_knob(ssmscan.SSM_KNOB_WAIT_NS, 2_000_000_000)


# Shapes span several chunks with a ragged tail (L not a multiple of 32/64),
# several channel tiles with a ragged last tile, and every N class.
SHAPES = [(1, 1, 1, 1), (2, 37, 40, 16), (1, 100, 136, 16), (3, 65, 8, 4), (2, 33, 24, 64),
          (1, 70, 16, 128), (1, 64, 64, 3), (2, 130, 72, 8), (1, 97, 130, 16), (2, 40, 9, 32)]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", SHAPES)
def test_small_shapes(dtype, shape):
    wl = wl_for(dtype, *shape)
    inp = W.make_inputs(wl, seed=sum(shape))
    check_full(inp, TOL[dtype], guard=64)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("flags", [
    dict(softplus=False, delta_bias=False, gate=False, skip=False, delta_kind="loguniform_td"),
    dict(softplus=True, delta_bias=False, gate=True, skip=False, delta_kind="normal_raw"),
    dict(softplus=False, delta_bias=True, gate=False, skip=True, delta_kind="loguniform_td"),
    dict(softplus=True, delta_bias=True, gate=True, skip=True, delta_kind="normal_raw"),
])
def test_optional_arguments(dtype, flags):
    wl = wl_for(dtype, 2, 77, 48, 16, **flags)
    inp = W.make_inputs(wl, seed=3)
    if flags["delta_bias"] and not flags["softplus"]:
        # without softplus a bias must keep dt > 0 (dt < 0 with A < 0 makes the
        # recurrence grow without bound, in any precision)
        inp["delta_bias"] = np.abs(inp["delta_bias"]) * 0.01
    check_full(inp, TOL[dtype], guard=64)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_h_last_optional(dtype):
    wl = wl_for(dtype, 2, 50, 32, 16)
    inp = W.make_inputs(wl, seed=4)
    y, _ = run_gpu(inp, want_h=False)
    yr, _ = oracle_ref(W.decoded(inp))
    assert rel_err(y, yr) <= TOL[dtype]


@pytest.mark.parametrize("groups", [1, 2, 4, 8])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", [16, 5, 40])
@pytest.mark.parametrize("chunk", [16, 32])
def test_every_state_split(groups, dtype, N, chunk):
    ssm.ssm_set_knob(ssmscan.SSM_KNOB_STATE_GROUPS, groups)
    ssm.ssm_set_knob(ssmscan.SSM_KNOB_CHUNK, chunk)
    wl = wl_for(dtype, 2, 150, 200, N)
    check_full(W.make_inputs(wl, seed=groups + N), TOL[dtype], guard=64)


@pytest.mark.parametrize("stages", [2, 3, 4])
def test_ring_depths_agree(stages):
    wl = wl_for("bf16", 2, 333, 96, 16)
    inp = W.make_inputs(wl, seed=12)
    y0, h0 = run_gpu(inp)
    ssm.ssm_set_knob(ssmscan.SSM_KNOB_STAGES, stages)
    y1, h1 = run_gpu(inp, guard=64)
    assert np.array_equal(y0, y1) and np.array_equal(h0, h1)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_plain_load_path_matches_tma_path(dtype):
    wl = wl_for(dtype, 2, 90, 64, 16)
    inp = W.make_inputs(wl, seed=11)
    y_tma, h_tma = run_gpu(inp)
    ssm.ssm_set_knob(ssmscan.SSM_KNOB_PLAIN_LOADS, 1)
    y_pl, h_pl = run_gpu(inp, guard=64)
    # same arithmetic in the same order: bitwise equal
    assert np.array_equal(y_tma, y_pl) and np.array_equal(h_tma, h_pl)
    yr, hr = oracle_ref(W.decoded(inp))
    assert rel_err(y_pl, yr) <= TOL[dtype]


# ---------------------------------------------------------------- time segments
# Shapes with ragged chunk tails, segments that do not divide the chunks, the
# segment count capped by the chunk count (64 forced on 66 chunks), and N not a
# multiple of the states per lane.
SEG_CASES = [(2, (2, 130, 72, 16)), (3, (1, 1000, 40, 16)), (5, (2, 333, 96, 5)),
             (7, (1, 517, 33, 40)), (64, (1, 2100, 64, 16)), (4, (1, 300, 24, 128))]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("segs,shape", SEG_CASES)
def test_time_segments_match_the_sequential_definition(dtype, segs, shape):
    ssm.ssm_set_knob(ssmscan.SSM_KNOB_SEGMENTS, segs)
    pl = ssm.ssm_scan_plan(*shape, 1 if dtype == "bf16" else 0)
    assert pl["segments"] > 1
    wl = wl_for(dtype, *shape)
    check_full(W.make_inputs(wl, seed=segs), TOL[dtype], guard=64)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_time_segments_carry_long_memory(dtype):
    """dt around 1e-4: the state hardly decays over the whole sequence, so
    every segment's entry state depends on all earlier segments."""
    ssm.ssm_set_knob(ssmscan.SSM_KNOB_SEGMENTS, 6)
    wl = wl_for(dtype, 2, 600, 64, 16, softplus=False, delta_bias=False,
                delta_kind="loguniform_td")
    inp = W.make_inputs(wl, seed=21)
    if dtype == "bf16":
        small = W.decode(inp["delta"]) * 1e-3
        inp["delta"] = W.f32_to_bf16_bits(small.astype(np.float32))
    else:
        inp["delta"] = (inp["delta"] * 1e-3).astype(np.float32)
    check_full(inp, TOL[dtype], guard=64)


@pytest.mark.parametrize("flags", [
    dict(softplus=True, delta_bias=True, gate=True, skip=True, delta_kind="normal_raw"),
    dict(softplus=False, delta_bias=False, gate=False, skip=False, delta_kind="loguniform_td"),
])
def test_time_segments_with_optional_arguments(flags):
    ssm.ssm_set_knob(ssmscan.SSM_KNOB_SEGMENTS, 4)
    wl = wl_for("bf16", 2, 400, 48, 16, **flags)
    check_full(W.make_inputs(wl, seed=22), TOL["bf16"], guard=64)


def test_time_segments_deterministic_and_plain_loads_agree():
    # one chunk length for both paths, so the segments start at the same steps
    ssm.ssm_set_knob(ssmscan.SSM_KNOB_CHUNK, 16)
    ssm.ssm_set_knob(ssmscan.SSM_KNOB_SEGMENTS, 3)
    wl = wl_for("bf16", 1, 700, 64, 16)
    inp = W.make_inputs(wl, seed=23)
    y1, h1 = run_gpu(inp)
    y2, h2 = run_gpu(inp)
    assert np.array_equal(y1, y2) and np.array_equal(h1, h2)
    ssm.ssm_set_knob(ssmscan.SSM_KNOB_PLAIN_LOADS, 1)
    y3, h3 = run_gpu(inp, guard=64)
    assert np.array_equal(y1, y3) and np.array_equal(h1, h3)


# ------------------------------------------------- the two kernels agree bit for bit
# The phase kernel and the warp-specialised kernel do the same arithmetic in
# the same order; with the same chunk length (hence the same segment
# boundaries) their outputs are identical.
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape,segs", [((2, 130, 72, 16), 1), ((1, 333, 96, 5), 1),
                                        ((2, 97, 256, 64), 1), ((1, 70, 16, 128), 1),
                                        ((1, 900, 64, 16), 5), ((2, 517, 40, 40), 3),
                                        ((3, 61, 200, 16), 1), ((1, 250, 136, 32), 2)])
def test_warp_specialised_kernel_matches_phase_kernel(dtype, shape, segs):
    ssm.ssm_set_knob(ssmscan.SSM_KNOB_CHUNK, 16)
    ssm.ssm_set_knob(ssmscan.SSM_KNOB_SEGMENTS, segs)
    wl = wl_for(dtype, *shape)
    inp = W.make_inputs(wl, seed=40 + segs)
    ssm.ssm_set_knob(ssmscan.SSM_KNOB_KERNEL, 2)
    assert ssm.ssm_scan_plan(*shape, 1 if dtype == "bf16" else 0)["kernel"] == 2
    y2, h2 = run_gpu(inp, guard=64)
    ssm.ssm_set_knob(ssmscan.SSM_KNOB_KERNEL, 1)
    assert ssm.ssm_scan_plan(*shape, 1 if dtype == "bf16" else 0)["kernel"] == 1
    y1, h1 = run_gpu(inp, guard=64)
    assert np.array_equal(y1, y2) and np.array_equal(h1, h2)
    yr, hr = oracle_ref(W.decoded(inp))
    assert rel_err(y2, yr) <= TOL[dtype] and rel_err(h2, hr) <= TOL[dtype]


def test_deterministic():
    wl = wl_for("bf16", 2, 300, 256, 16)
    inp = W.make_inputs(wl, seed=5)
    y1, h1 = run_gpu(inp)
    y2, h2 = run_gpu(inp)
    assert np.array_equal(y1, y2) and np.array_equal(h1, h2)


def test_side_stream():
    wl = wl_for("bf16", 2, 64, 64, 16)
    inp = W.make_inputs(wl, seed=6)
    s = torch.cuda.Stream()
    y, h = run_gpu(inp, stream=s.cuda_stream)
    yr, hr = oracle_ref(W.decoded(inp))
    assert rel_err(y, yr) <= TOL["bf16"] and rel_err(h, hr) <= TOL["bf16"]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_zero_length_sequence_gives_zero_state(dtype):
    wl = wl_for(dtype, 2, 0, 16, 16)
    inp = W.make_inputs(wl, seed=7)
    y, h = run_gpu(inp)
    assert y.shape == (2, 0, 16) and np.all(h == 0.0)


def test_bounded_wait_reports_timeout_and_context_survives():
    """Every block first waits on a barrier nothing completes; the wait gives
    up after 1 ms, the block drains its own copies and returns, and the host
    reads SSM_ERR_TIMEOUT.  A normal call afterwards is correct."""
    wl = wl_for("bf16", 2, 96, 64, 16)
    inp = W.make_inputs(wl, seed=8)
    from tests.gpu_util import to_dev
    d = {k: to_dev(inp[k]) for k in ("u", "delta", "B", "C", "z", "A", "D", "delta_bias")}
    ssm.ssm_set_knob(ssmscan.SSM_KNOB_WAIT_NS, 1_000_000)
    ssm.ssm_set_knob(ssmscan.SSM_KNOB_FORCE_TIMEOUT, 1)
    ssm.selective_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"],
                           d["delta_bias"], True)
    st = ssm.ssm_scan_last_device_status(torch.cuda.current_stream().cuda_stream)
    assert st == ssmscan.SSM_ERR_TIMEOUT
    ssm.ssm_set_knob(ssmscan.SSM_KNOB_FORCE_TIMEOUT, 0)
    ssm.ssm_set_knob(ssmscan.SSM_KNOB_WAIT_NS, 2_000_000_000)
    check_full(inp, TOL["bf16"])


# --------------------------------------------------------------- the workloads
def test_workload_small_fp32():
    wl = W.WORKLOADS["small_fp32"]
    check_full(W.make_inputs(wl), TOL["f32"], guard=64)


@pytest.mark.parametrize("skip", [False, True])
def test_workload_time_invariant_fp32(skip):
    wl = W.WORKLOADS["lti_fp32"].with_shape(skip=skip)
    check_full(W.make_inputs(wl), TOL["f32"], guard=64)


def test_workload_time_invariant_equals_convolution():
    """y = u * K computed from the pages' kernel formula, independent of the oracle."""
    from tests.oracle_pins import lti_kernel
    wl = W.WORKLOADS["lti_fp32"]
    inp = W.make_inputs(wl)
    y, _ = run_gpu(inp)
    dt = inp["delta"][0, 0, :].astype(np.float64)
    K = lti_kernel(dt, inp["A"].astype(np.float64), inp["B"][0, 0].astype(np.float64),
                   inp["C"][0, 0].astype(np.float64), wl.L)
    u = inp["u"].astype(np.float64)
    kf = np.fft.rfft(K, n=2 * wl.L, axis=-1)
    uf = np.fft.rfft(np.transpose(u, (0, 2, 1)), n=2 * wl.L, axis=-1)
    yr = np.transpose(np.fft.irfft(uf * kf[None], n=2 * wl.L, axis=-1)[..., :wl.L], (0, 2, 1))
    assert rel_err(y, yr) <= TOL["f32"]


def test_workload_mamba130m_bf16_sampled():
    wl = W.WORKLOADS["mamba130m_bf16"]
    check_sampled(W.make_inputs(wl), wl, TOL["bf16"], n_dim=48, n_batch=3)


def test_workload_mamba2p8b_bf16_sampled():
    wl = W.WORKLOADS["mamba2p8b_bf16"]
    check_sampled(W.make_inputs(wl), wl, TOL["bf16"], n_dim=24, n_batch=2)


@pytest.mark.parametrize("L", W.LONGCTX_LS)
def test_workload_longctx_bf16_sampled(L):
    wl = W.WORKLOADS[f"longctx_L{L}"]
    n_dim = 24 if L <= 32768 else 12
    check_sampled(W.make_inputs(wl), wl, TOL["bf16"], n_dim=n_dim, n_batch=1)
