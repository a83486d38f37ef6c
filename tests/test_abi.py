"""C ABI of libssmscan on the host: the library loads, exports every symbol the
header declares, and rejects bad arguments before touching the GPU.  No call
here reaches a kernel launch, so these run without a GPU."""
import ctypes
import os
import re

import pytest

import selective_state_space_150_b300 as ssm
from selective_state_space_150_b300 import ssmscan

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ssmscan.h")


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^SSM_API\s+(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, re.M)))


def test_header_declares_the_boundary():
    assert declared_symbols() == sorted(ssmscan.EXPORTED)


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(ssmscan.LIB_PATH)
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_status_strings():
    for st in range(0, 11):
        s = ssm.ssm_status_string(st)
        assert s and s != "unknown status"
    assert ssm.ssm_status_string(99) == "unknown status"


# fake device addresses: validation must reject before dereferencing or launching
P = 0x10000000
Q = 0x20000000


def fwd(fn, **kw):
    args = dict(u=P, delta=P + 0x100000, A=P + 0x200000, B=P + 0x300000, C=P + 0x400000,
                D=0, z=0, delta_bias=0, softplus_flag=0, y=Q, h_last=0,
                batch=2, L=8, dim=16, N=4, stream=0)
    args.update(kw)
    return fn(**args)


@pytest.mark.parametrize("fn", [ssm.ssm_scan_fwd, ssm.ssm_scan_fwd_bf16,
                                ssm.ssm_scan_fwd_bf16_noalloc])
def test_null_pointers(fn):
    for k in ("u", "delta", "A", "B", "C", "y"):
        assert fwd(fn, **{k: 0}) == ssmscan.SSM_ERR_NULL, k


@pytest.mark.parametrize("fn", [ssm.ssm_scan_fwd, ssm.ssm_scan_fwd_bf16,
                                ssm.ssm_scan_fwd_bf16_noalloc])
def test_bad_sizes(fn):
    assert fwd(fn, batch=-1) == ssmscan.SSM_ERR_SIZE
    assert fwd(fn, L=-3) == ssmscan.SSM_ERR_SIZE
    assert fwd(fn, dim=-1) == ssmscan.SSM_ERR_SIZE
    assert fwd(fn, N=0) == ssmscan.SSM_ERR_SIZE
    assert fwd(fn, N=ssmscan.SSM_MAX_N + 1) == ssmscan.SSM_ERR_UNSUPPORTED_N
    assert fwd(fn, batch=1 << 40, L=1 << 20, dim=1 << 10) == ssmscan.SSM_ERR_SIZE


def test_misaligned_pointers():
    assert fwd(ssm.ssm_scan_fwd, u=P + 2) == ssmscan.SSM_ERR_ALIGN
    assert fwd(ssm.ssm_scan_fwd_bf16, u=P + 1) == ssmscan.SSM_ERR_ALIGN
    assert fwd(ssm.ssm_scan_fwd_bf16, A=P + 0x200002) == ssmscan.SSM_ERR_ALIGN
    assert fwd(ssm.ssm_scan_fwd_bf16, h_last=Q + 0x100002) == ssmscan.SSM_ERR_ALIGN


@pytest.mark.parametrize("fn", [ssm.ssm_scan_fwd, ssm.ssm_scan_fwd_bf16,
                                ssm.ssm_scan_fwd_bf16_noalloc])
def test_outputs_must_not_alias_inputs(fn):
    assert fwd(fn, y=P + 0x100000) == ssmscan.SSM_ERR_ALIAS            # y == delta
    assert fwd(fn, y=P + 0x10) == ssmscan.SSM_ERR_ALIAS                # y inside u
    assert fwd(fn, h_last=P + 0x300000) == ssmscan.SSM_ERR_ALIAS       # h_last == B
    assert fwd(fn, h_last=Q + 0x8) == ssmscan.SSM_ERR_ALIAS            # h_last inside y


@pytest.mark.parametrize("fn", [ssm.ssm_scan_fwd, ssm.ssm_scan_fwd_bf16,
                                ssm.ssm_scan_fwd_bf16_noalloc])
def test_empty_problems_launch_nothing(fn):
    assert fwd(fn, batch=0) == ssmscan.SSM_OK
    assert fwd(fn, dim=0) == ssmscan.SSM_OK


def test_knobs_validate():
    K = ssmscan
    assert ssm.ssm_set_knob(K.SSM_KNOB_WAIT_NS, 10) == K.SSM_ERR_ARG
    assert ssm.ssm_set_knob(K.SSM_KNOB_STATE_GROUPS, 3) == K.SSM_ERR_ARG
    assert ssm.ssm_set_knob(K.SSM_KNOB_CHUNK, 24) == K.SSM_ERR_ARG
    assert ssm.ssm_set_knob(K.SSM_KNOB_SEGMENTS, -1) == K.SSM_ERR_ARG
    assert ssm.ssm_set_knob(K.SSM_KNOB_SEGMENTS, 65) == K.SSM_ERR_ARG
    assert ssm.ssm_set_knob(K.SSM_KNOB_KERNEL, 3) == K.SSM_ERR_ARG
    assert ssm.ssm_set_knob(K.SSM_KNOB_BWD_SEGMENTS, 65) == K.SSM_ERR_ARG
    assert ssm.ssm_set_knob(K.SSM_KNOB_BWD_SEGMENTS, 0) == K.SSM_OK
    assert ssm.ssm_set_knob(99, 0) == K.SSM_ERR_ARG
    assert ssm.ssm_set_knob(K.SSM_KNOB_STATE_GROUPS, 0) == K.SSM_OK
    assert ssm.ssm_set_knob(K.SSM_KNOB_WAIT_NS, 2_000_000_000) == K.SSM_OK


@pytest.mark.parametrize("shape", [(8, 2048, 1536, 16), (4, 8192, 5120, 16), (1, 131072, 5120, 16),
                                   (1, 256, 64, 16), (2, 4096, 256, 64), (3, 5, 7, 1),
                                   (1, 1, 1, 128), (2, 9, 33, 3)])
@pytest.mark.parametrize("dtype", [0, 1])
def test_plans_cover_the_state(shape, dtype):
    pl = ssm.ssm_scan_plan(*shape, dtype)
    batch, L, dim, N = shape
    ws, npt = pl["state_groups"], pl["states_per_lane"]
    assert ws in (1, 2, 4, 8) and npt in (1, 2, 4, 8, 16)
    assert ws * npt >= N and (ws == 1 or (ws - 1) * npt < N)      # no all-padding group
    wc = 1 if ws >= 4 else 4 // ws
    helpers = 5 if pl["kernel"] == 2 else 0          # warp-specialised: producer, 2 prepare, 2 finish
    assert pl["kernel"] in (1, 2) and (pl["kernel"] == 1 or pl["tma"] == 1)
    assert pl["threads"] == 32 * (wc * ws + helpers) and pl["channels_per_block"] == 32 * wc
    assert pl["blocks"] == batch * -(-dim // pl["channels_per_block"])
    assert 0 < pl["smem_bytes"] <= 227 * 1024
    nchunks = -(-L // pl["chunk"])
    seg = pl["segments"]
    assert 1 <= seg <= max(1, nchunks // 8)           # every automatic segment >= 8 chunks
    assert pl["scratch_bytes"] == (seg - 1) * batch * dim * (N + 1) * 4


def test_time_split_only_where_channels_leave_the_gpu_idle():
    # 8 x 1536 channels fill the GPU: one pass, no scratch
    assert ssm.ssm_scan_plan(8, 2048, 1536, 16, 1)["segments"] == 1
    # one row of 5120 channels over 131072 steps: split in time
    assert ssm.ssm_scan_plan(1, 131072, 5120, 16, 1)["segments"] > 1


def test_time_split_needs_a_sequence_that_repays_the_summary_pass():
    seg = lambda *shape: ssm.ssm_scan_plan(*shape, 1)["segments"]
    # two blocks, most SMs idle: split from 1024 steps on
    assert seg(1, 256, 64, 16) == 1 and seg(1, 512, 64, 16) == 1
    assert seg(1, 1024, 64, 16) > 1
    # 160 blocks, about one per SM: one pass below 4096 steps, then at least 12 segments
    assert seg(1, 2048, 5120, 16) == 1 and seg(1, 4095, 5120, 16) == 1
    assert seg(1, 4096, 5120, 16) >= 12 and seg(1, 131072, 5120, 16) >= 12


@pytest.mark.parametrize("forced,L,expect", [(5, 1000, 5), (64, 100, 4), (3, 32, 1), (1, 5000, 1)])
def test_forced_segments_are_capped_by_chunks(forced, L, expect):
    K = ssmscan
    try:
        assert ssm.ssm_set_knob(K.SSM_KNOB_SEGMENTS, forced) == K.SSM_OK
        pl = ssm.ssm_scan_plan(1, L, 64, 16, 1)
        nchunks = -(-L // pl["chunk"])
        per = -(-nchunks // min(forced, nchunks))
        assert pl["segments"] == (-(-nchunks // per) if min(forced, nchunks) > 1 else 1)
        if pl["chunk"] == 32:
            assert pl["segments"] == expect
    finally:
        ssm.ssm_set_knob(K.SSM_KNOB_SEGMENTS, 0)


def test_plan_rejects_bad_arguments():
    with pytest.raises(ssm.SSMError):
        ssm.ssm_scan_plan(1, 1, 1, 0, 1)
    with pytest.raises(ssm.SSMError):
        ssm.ssm_scan_plan(1, 1, 1, 16, 7)


# ---------------------------------------------------------------- initial state / decode step
def fwd_h0(fn, **kw):
    args = dict(u=P, delta=P + 0x100000, A=P + 0x200000, B=P + 0x300000, C=P + 0x400000,
                D=0, z=0, delta_bias=0, h0=P + 0x500000, softplus_flag=0, y=Q, h_last=Q + 0x100000,
                batch=2, L=8, dim=16, N=4, stream=0)
    args.update(kw)
    return fn(**args)


@pytest.mark.parametrize("fn", [ssm.ssm_scan_fwd_h0, ssm.ssm_scan_fwd_bf16_h0])
def test_h0_checks(fn):
    assert fwd_h0(fn, h0=Q + 0x100000) == ssmscan.SSM_ERR_ALIAS      # h0 is h_last
    assert fwd_h0(fn, h0=Q + 0x40) == ssmscan.SSM_ERR_ALIAS          # h0 inside y
    assert fwd_h0(fn, h0=P + 0x500002) == ssmscan.SSM_ERR_ALIGN
    assert fwd_h0(fn, u=0) == ssmscan.SSM_ERR_NULL
    assert fwd_h0(fn, batch=0) == ssmscan.SSM_OK


def step(fn, **kw):
    args = dict(u=P, delta=P + 0x100000, A=P + 0x200000, B=P + 0x300000, C=P + 0x400000,
                D=0, z=0, delta_bias=0, softplus_flag=1, h=Q, y=Q + 0x100000,
                batch=2, dim=16, N=4, stream=0)
    args.update(kw)
    return fn(**args)


@pytest.mark.parametrize("fn", [ssm.ssm_scan_step, ssm.ssm_scan_step_bf16])
def test_step_checks(fn):
    for k in ("u", "delta", "A", "B", "C", "h", "y"):
        assert step(fn, **{k: 0}) == ssmscan.SSM_ERR_NULL, k
    assert step(fn, batch=-1) == ssmscan.SSM_ERR_SIZE
    assert step(fn, N=0) == ssmscan.SSM_ERR_SIZE
    assert step(fn, N=129) == ssmscan.SSM_ERR_UNSUPPORTED_N
    assert step(fn, h=P + 0x100000) == ssmscan.SSM_ERR_ALIAS          # h is delta
    assert step(fn, y=Q + 0x10) == ssmscan.SSM_ERR_ALIAS              # y inside h
    assert step(fn, y=P) == ssmscan.SSM_ERR_ALIAS                     # y is u
    assert step(fn, h=Q + 2) == ssmscan.SSM_ERR_ALIGN
    assert step(fn, batch=0) == ssmscan.SSM_OK and step(fn, dim=0) == ssmscan.SSM_OK


# ---------------------------------------------------------------- conv prologue
def conv_fwd(fn, **kw):
    args = dict(x=P, conv_w=P + 0x600000, conv_b=0, conv_k=4, delta=P + 0x100000,
                A=P + 0x200000, B=P + 0x300000, C=P + 0x400000, D=0, z=0, delta_bias=0,
                softplus_flag=0, y=Q, h_last=0, batch=2, L=8, dim=16, N=4, stream=0)
    args.update(kw)
    return fn(**args)


@pytest.mark.parametrize("fn", [ssm.ssm_conv_scan_fwd, ssm.ssm_conv_scan_fwd_bf16])
def test_conv_checks(fn):
    assert conv_fwd(fn, conv_k=0) == ssmscan.SSM_ERR_SIZE
    assert conv_fwd(fn, conv_k=5) == ssmscan.SSM_ERR_SIZE
    assert conv_fwd(fn, conv_w=0) == ssmscan.SSM_ERR_NULL
    assert conv_fwd(fn, conv_w=P + 0x600002) == ssmscan.SSM_ERR_ALIGN
    assert conv_fwd(fn, y=P + 0x600000) == ssmscan.SSM_ERR_ALIAS     # y over the taps
    assert conv_fwd(fn, batch=0) == ssmscan.SSM_OK


# ---------------------------------------------------------------- host-buffer calls
def test_host_workspace_sizes():
    f = ssm.ssm_scan_host_workspace_bytes
    small = f(8, 2048, 1536, 16, 1)
    assert small > 0 and f(8, 2048, 1536, 16, 0) > small          # fp32 slots are larger
    # two slots of one part (a row group of 1 row here) plus A, D, bias
    per_row = 4 * 2048 * 1536 * 2 + 2 * 2048 * 16 * 2 + 1536 * 16 * 4
    assert 2 * per_row <= small <= 2 * per_row + 1536 * 16 * 4 + 8 * 1536 + 64 * 256
    assert f(1, 131072, 5120, 16, 1) < f(1, 131072, 5120, 16, 1) * 2   # time pieces: finite
    assert f(-1, 1, 1, 1, 1) == -1 and f(1, 1, 1, 0, 1) == -1 and f(1, 1, 1, 1, 2) == -1


@pytest.mark.parametrize("fn", [ssm.ssm_scan_fwd_host, ssm.ssm_scan_fwd_bf16_host])
def test_host_call_checks(fn):
    args = dict(u=P, delta=P, A=P, B=P, C=P, D=0, z=0, delta_bias=0, softplus_flag=0, y=Q,
                h_last=0, batch=2, L=8, dim=16, N=4, workspace=P, workspace_bytes=16, stream=0)
    assert fn(**{**args, "u": 0}) == ssmscan.SSM_ERR_NULL
    assert fn(**{**args, "workspace": 0}) == ssmscan.SSM_ERR_NULL
    assert fn(**args) == ssmscan.SSM_ERR_SIZE                     # workspace too small
    assert fn(**{**args, "batch": 0}) == ssmscan.SSM_OK
    assert fn(**{**args, "N": 200}) == ssmscan.SSM_ERR_UNSUPPORTED_N


@pytest.mark.parametrize("fn", [ssm.ssm_scan_fwd_zoh, ssm.ssm_scan_fwd_bf16_zoh])
def test_zoh_checks(fn):
    assert fwd_h0(fn, u=0) == ssmscan.SSM_ERR_NULL
    assert fwd_h0(fn, h0=Q + 0x100000) == ssmscan.SSM_ERR_ALIAS
    assert fwd_h0(fn, h0=0, batch=0) == ssmscan.SSM_OK


# ---------------------------------------------------------------- backward
def bwd(fn=ssm.ssm_scan_bwd, **kw):
    args = dict(u=P, delta=P + 0x100000, A=P + 0x200000, B=P + 0x300000, C=P + 0x400000, D=0,
                z=0, delta_bias=0, softplus_flag=0, dy=P + 0x500000, du=Q, ddelta=Q + 0x100000,
                dA=Q + 0x200000, dB=Q + 0x300000, dC=Q + 0x400000, dD=0, dz=0, ddelta_bias=0,
                batch=2, L=8, dim=16, N=4, stream=0)
    args.update(kw)
    return fn(**args)


@pytest.mark.parametrize("fn,es", [(ssm.ssm_scan_bwd, 4), (ssm.ssm_scan_bwd_bf16, 2)])
def test_backward_checks(fn, es):
    for k in ("u", "delta", "dy", "du", "ddelta", "A", "dA", "B", "C", "dB", "dC"):
        assert bwd(fn, **{k: 0}) == ssmscan.SSM_ERR_NULL, k
    assert bwd(fn, D=P + 0x600000) == ssmscan.SSM_ERR_NULL        # D given, dD missing
    assert bwd(fn, z=P + 0x600000) == ssmscan.SSM_ERR_NULL        # z given, dz missing
    assert bwd(fn, N=129) == ssmscan.SSM_ERR_UNSUPPORTED_N
    assert bwd(fn, L=-1) == ssmscan.SSM_ERR_SIZE
    assert bwd(fn, du=P) == ssmscan.SSM_ERR_ALIAS                 # du is u
    assert bwd(fn, dB=Q + 0x40) == ssmscan.SSM_ERR_ALIAS          # dB inside du
    assert bwd(fn, du=Q + es // 2) == ssmscan.SSM_ERR_ALIGN       # du off its element size
    assert bwd(fn, dA=Q + 0x200000 + 2) == ssmscan.SSM_ERR_ALIGN  # fp32 dA off 4 bytes
    assert bwd(fn, batch=0) == ssmscan.SSM_OK


@pytest.mark.parametrize("fn", [ssm.ssm_scan_bwd_h0, ssm.ssm_scan_bwd_bf16_h0])
def test_backward_with_states_checks(fn):
    def call(**kw):
        args = dict(h0=0, dh_last=0, dh0=0)
        args.update(kw)
        return bwd(fn, **args)
    H = Q + 0x800000
    assert call(N=129) == ssmscan.SSM_ERR_UNSUPPORTED_N
    assert call(u=0) == ssmscan.SSM_ERR_NULL
    assert call(dh0=H + 2) == ssmscan.SSM_ERR_ALIGN
    assert call(h0=P + 0x600002) == ssmscan.SSM_ERR_ALIGN
    assert call(dh0=Q + 0x40) == ssmscan.SSM_ERR_ALIAS             # dh0 inside du
    assert call(h0=H, dh0=H) == ssmscan.SSM_ERR_ALIAS              # dh0 is h0
    assert call(dh_last=H + 0x40, dh0=H) == ssmscan.SSM_ERR_ALIAS  # dh0 overlaps dh_last
    assert call(batch=0, h0=H, dh0=H + 0x100000) == ssmscan.SSM_OK
