"""ssm_scan_fwd_bf16_noalloc: the bf16 scan with its time-segment scratch in
the library's static device buffer instead of cudaMallocAsync.

It runs the same plan and kernels as ssm_scan_fwd_bf16, so the two must agree
bit for bit.  The file sorts last so that its GPU tests also run after every
other test has used the device; they must pass alone as well."""
import numpy as np
import pytest
import torch

import ssm_workloads as W
import selective_state_space_150_b300 as ssm
from selective_state_space_150_b300 import ssmscan
from tests.gpu_util import TOL, from_dev, oracle_ref, rel_err, to_dev

BASE = W.WORKLOADS["mamba130m_bf16"]

# (batch, L, dim, N): split into time segments (scratch used), a ragged split
# with N = 5, and a one-pass problem (no scratch at all).
SHAPES = [(1, 4096, 64, 16), (1, 2500, 40, 5), (2, 300, 96, 16)]


def _inputs(shape, seed):
    batch, L, dim, N = shape
    wl = BASE.with_shape(name="noalloc", batch=batch, L=L, dim=dim, N=N)
    inp = W.make_inputs(wl, seed=seed)
    d = {k: to_dev(inp[k]) for k in ("u", "delta", "B", "C", "z", "A", "D", "delta_bias")}
    return inp, d


def _call(fn, d, softplus, stream):
    """Enqueue one call of `fn` (a bf16 C entry point) with fresh outputs."""
    u = d["u"]
    batch, L, dim = u.shape
    N = d["A"].shape[1]
    y = torch.empty_like(u)
    h = torch.empty((batch, dim, N), dtype=torch.float32, device="cuda")
    ptr = lambda t: 0 if t is None else t.data_ptr()  # noqa: E731
    st = fn(ptr(d["u"]), ptr(d["delta"]), ptr(d["A"]), ptr(d["B"]), ptr(d["C"]), ptr(d["D"]),
            ptr(d["z"]), ptr(d["delta_bias"]), int(softplus), y.data_ptr(), h.data_ptr(),
            batch, L, dim, N, stream)
    assert st == ssmscan.SSM_OK, ssm.ssm_status_string(st)
    return y, h


def _bits(t):
    return t.view(torch.int16).cpu().numpy() if t.dtype == torch.bfloat16 else t.cpu().numpy()


@pytest.mark.gpu
@pytest.mark.parametrize("shape", SHAPES)
def test_noalloc_matches_the_allocating_entry_point_on_two_calls_in_a_row(shape):
    stream = torch.cuda.current_stream().cuda_stream
    (inp1, d1), (inp2, d2) = _inputs(shape, 31), _inputs(shape, 32)
    # two no-alloc calls back to back on one stream (the second reuses the
    # static buffer the first one wrote), then the allocating entry point
    y1, h1 = _call(ssm.ssm_scan_fwd_bf16_noalloc, d1, BASE.softplus, stream)
    y2, h2 = _call(ssm.ssm_scan_fwd_bf16_noalloc, d2, BASE.softplus, stream)
    r1, g1 = _call(ssm.ssm_scan_fwd_bf16, d1, BASE.softplus, stream)
    r2, g2 = _call(ssm.ssm_scan_fwd_bf16, d2, BASE.softplus, stream)
    assert ssm.ssm_scan_last_device_status(stream) == ssmscan.SSM_OK
    for a, b in ((y1, r1), (h1, g1), (y2, r2), (h2, g2)):
        assert np.array_equal(_bits(a), _bits(b))
    # and the pair is right, not only equal
    yr, hr = oracle_ref(W.decoded(inp2))
    assert rel_err(from_dev(y2), yr) <= TOL["bf16"] and rel_err(from_dev(h2), hr) <= TOL["bf16"]


def _pool_used_high(reset: bool):
    """High-water mark of the current device's stream-ordered memory pool (the
    pool cudaMallocAsync draws from), optionally reset to 0 first."""
    from cuda.bindings import driver as drv
    from cuda.bindings import runtime as rt

    def ok(ret):
        err = ret[0] if isinstance(ret, tuple) else ret
        assert err == rt.cudaError_t.cudaSuccess, err
        return ret

    pool = ok(rt.cudaDeviceGetMemPool(torch.cuda.current_device()))[1]
    attr = rt.cudaMemPoolAttr.cudaMemPoolAttrUsedMemHigh
    if reset:
        ok(rt.cudaMemPoolSetAttribute(pool, attr, drv.cuuint64_t(0)))
    return int(ok(rt.cudaMemPoolGetAttribute(pool, attr))[1])


@pytest.mark.gpu
def test_noalloc_takes_nothing_from_the_stream_ordered_pool():
    shape = SHAPES[0]
    assert ssm.ssm_scan_plan(*shape, 1)["segments"] > 1   # scratch is needed
    stream = torch.cuda.current_stream().cuda_stream
    _, d = _inputs(shape, 33)
    torch.cuda.synchronize()
    _pool_used_high(reset=True)
    _call(ssm.ssm_scan_fwd_bf16_noalloc, d, BASE.softplus, stream)
    torch.cuda.synchronize()
    assert _pool_used_high(reset=False) == 0
    # the probe does see the allocating entry point's scratch
    _call(ssm.ssm_scan_fwd_bf16, d, BASE.softplus, stream)
    torch.cuda.synchronize()
    assert _pool_used_high(reset=False) >= ssm.ssm_scan_plan(*shape, 1)["scratch_bytes"]
    assert ssm.ssm_scan_last_device_status(stream) == ssmscan.SSM_OK


def _segmented_pair(d, forced, stream):
    """The no-alloc entry point and, with the same forced segment count, the
    allocating one (which always honours the count)."""
    ssm.ssm_set_knob(ssmscan.SSM_KNOB_SEGMENTS, forced)
    try:
        y, h = _call(ssm.ssm_scan_fwd_bf16_noalloc, d, BASE.softplus, stream)
        r, g = _call(ssm.ssm_scan_fwd_bf16, d, BASE.softplus, stream)
    finally:
        ssm.ssm_set_knob(ssmscan.SSM_KNOB_SEGMENTS, 0)
    return y, h, r, g


# batch 1, dim 4096, N 15: one segment's summaries take 4096 * 16 = 2^16 words,
# so 33 segments fill the 2^21-word buffer exactly.  577 chunks of 16 steps
# split into exactly 33 segments (of 18 chunks) when 33 are asked for, and into
# exactly 34 (of 17) when 34 are.
EDGE = (1, 577 * 16, 4096, 15)


def _oracle_sampled(inp, y, h):
    wl = BASE.with_shape(name="noalloc", batch=EDGE[0], L=EDGE[1], dim=EDGE[2], N=EDGE[3])
    bs, ds = W.channel_sample(wl, n_dim=16, n_batch=1)
    yr, hr = oracle_ref(W.gather(inp, bs, ds))
    ys, hs = from_dev(y)[bs][:, :, ds], from_dev(h)[bs][:, ds, :]
    assert rel_err(ys, yr) <= TOL["bf16"] and rel_err(hs, hr) <= TOL["bf16"]


@pytest.mark.gpu
def test_noalloc_at_the_exact_capacity_of_its_buffer():
    """(segments - 1) * batch * dim * (N + 1) = 2^21 words: the no-alloc entry
    point runs those 33 segments, bit for bit like the allocating one."""
    batch, L, dim, N = EDGE
    assert 32 * batch * dim * (N + 1) == ssmscan.SSM_NOALLOC_SCRATCH_FLOATS
    stream = torch.cuda.current_stream().cuda_stream
    inp, d = _inputs(EDGE, 34)
    ssm.ssm_set_knob(ssmscan.SSM_KNOB_SEGMENTS, 33)
    try:
        assert ssm.ssm_scan_plan(*EDGE, 1)["segments"] == 33
    finally:
        ssm.ssm_set_knob(ssmscan.SSM_KNOB_SEGMENTS, 0)
    y, h, r, g = _segmented_pair(d, 33, stream)
    assert ssm.ssm_scan_last_device_status(stream) == ssmscan.SSM_OK
    assert np.array_equal(_bits(y), _bits(r)) and np.array_equal(_bits(h), _bits(g))
    _oracle_sampled(inp, y, h)


@pytest.mark.gpu
def test_noalloc_one_segment_past_its_buffer_plans_fewer_segments():
    """34 segments would need 2^21 + 2^16 words: the no-alloc entry point runs
    the 33 that fit instead (it never refuses), so it equals the allocating
    entry point forced to 33 segments, not the one forced to 34."""
    stream = torch.cuda.current_stream().cuda_stream
    inp, d = _inputs(EDGE, 35)
    ssm.ssm_set_knob(ssmscan.SSM_KNOB_SEGMENTS, 34)
    try:
        assert ssm.ssm_scan_plan(*EDGE, 1)["segments"] == 34
    finally:
        ssm.ssm_set_knob(ssmscan.SSM_KNOB_SEGMENTS, 0)
    y, h, r34, g34 = _segmented_pair(d, 34, stream)
    _, _, r33, g33 = _segmented_pair(d, 33, stream)
    assert ssm.ssm_scan_last_device_status(stream) == ssmscan.SSM_OK
    assert np.array_equal(_bits(y), _bits(r33)) and np.array_equal(_bits(h), _bits(g33))
    assert not (np.array_equal(_bits(y), _bits(r34)) and np.array_equal(_bits(h), _bits(g34)))
    _oracle_sampled(inp, y, h)
