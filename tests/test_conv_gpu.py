"""GPU parity for the scan with the causal conv1d + SiLU prologue
(ssm_conv_scan_fwd*), through the C ABI, against the fp64 oracle's conv
followed by its scan."""
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
    for k in (ssmscan.SSM_KNOB_SEGMENTS, ssmscan.SSM_KNOB_STAGES):
        ssm.ssm_set_knob(k, 0)


def run(dtype, shape, K, seed, bias=True, **flags):
    batch, L, dim, N = shape
    wl = BASE[dtype].with_shape(name="c", batch=batch, L=L, dim=dim, N=N, **flags)
    inp = W.make_inputs(wl, seed=seed)            # its u serves as the conv input x
    rng = np.random.default_rng(seed + 500)
    w = (0.5 * rng.standard_normal((dim, K))).astype(np.float32)
    cb = (0.1 * rng.standard_normal(dim)).astype(np.float32) if bias else None
    d = {k: to_dev(inp[k]) for k in ("u", "delta", "B", "C", "z", "A", "D", "delta_bias")}
    y, h = ssm.conv_selective_scan_fwd(d["u"], torch.from_numpy(w).cuda(),
                                       None if cb is None else torch.from_numpy(cb).cuda(),
                                       d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"],
                                       d["delta_bias"], inp["softplus"])
    st = ssm.ssm_scan_last_device_status(torch.cuda.current_stream().cuda_stream)
    assert st == 0, ssm.ssm_status_string(st)
    p = W.decoded(inp)
    yr, hr = oracle.conv_selective_scan_fwd(p["u"], w, cb, p["delta"], p["A"], p["B"], p["C"],
                                            p["D"], p["z"], p["delta_bias"], p["softplus"])
    return from_dev(y), from_dev(h), yr, hr


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("K", [4, 3, 1])
@pytest.mark.parametrize("shape", [(2, 150, 72, 16), (1, 333, 40, 5), (2, 97, 256, 64),
                                   (1, 70, 16, 128), (3, 2, 64, 16)])
def test_conv_scan_matches_oracle(dtype, K, shape):
    y, h, yr, hr = run(dtype, shape, K, seed=sum(shape) + K)
    assert rel_err(y, yr) <= TOL[dtype] and rel_err(h, hr) <= TOL[dtype]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("segs", [3, 7])
def test_conv_scan_with_time_segments(dtype, segs):
    """Segments start mid-sequence, so each reads its halo from the previous
    segment's rows."""
    ssm.ssm_set_knob(ssmscan.SSM_KNOB_SEGMENTS, segs)
    y, h, yr, hr = run(dtype, (1, 700, 64, 16), 4, seed=segs)
    assert rel_err(y, yr) <= TOL[dtype] and rel_err(h, hr) <= TOL[dtype]


@pytest.mark.parametrize("stages", [2, 4])
def test_conv_scan_without_bias_and_other_rings(stages):
    ssm.ssm_set_knob(ssmscan.SSM_KNOB_STAGES, stages)
    y, h, yr, hr = run("bf16", (2, 211, 128, 16), 4, seed=stages, bias=False,
                       softplus=False, delta_bias=False, gate=False, skip=False,
                       delta_kind="loguniform_td")
    assert rel_err(y, yr) <= TOL["bf16"] and rel_err(h, hr) <= TOL["bf16"]


def test_conv_needs_tma_rows():
    """dim = 12 in bf16 (24-byte rows) cannot move by TMA: refused, no launch."""
    x = torch.zeros((1, 8, 12), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((12, 4), device="cuda")
    A = -torch.ones((12, 16), device="cuda")
    Bm = torch.zeros((1, 8, 16), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ssm.SSMError) as e:
        ssm.conv_selective_scan_fwd(x, w, None, x.clone(), A, Bm, Bm.clone())
    assert e.value.status == ssmscan.SSM_ERR_ALIGN
