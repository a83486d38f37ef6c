"""GPU parity for the host-buffer calls (ssm_scan_fwd*_host): host arrays in,
host arrays out, against the fp64 oracle; parts by batch rows and by time
pieces chained through the state."""
import numpy as np
import pytest
import torch

import ssm_workloads as W
import selective_state_space_150_b300 as ssm
from tests.gpu_util import TOL, oracle_ref, rel_err

pytestmark = pytest.mark.gpu

BASE = {"bf16": W.WORKLOADS["mamba130m_bf16"], "f32": W.WORKLOADS["small_fp32"]}


def host_tensor(a, pin):
    if a is None:
        return None
    t = (torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
         if a.dtype == np.uint16 else torch.from_numpy(np.ascontiguousarray(a)))
    return t.pin_memory() if pin else t.clone()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(8, 300, 96, 16),    # 8 row groups
                                   (5, 97, 40, 5),       # uneven row groups
                                   (2, 3000, 64, 16),    # time pieces
                                   (1, 70, 32, 64)])     # one piece
@pytest.mark.parametrize("pin", [True, False])
def test_host_call_matches_oracle(dtype, shape, pin):
    batch, L, dim, N = shape
    wl = BASE[dtype].with_shape(name="h", batch=batch, L=L, dim=dim, N=N)
    inp = W.make_inputs(wl, seed=sum(shape))
    h = {k: host_tensor(inp[k], pin) for k in ("u", "delta", "B", "C", "z", "A", "D", "delta_bias")}
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    y = torch.full((batch, L, dim), -7.0, dtype=tdt)
    hl = torch.full((batch, dim, N), -7.0, dtype=torch.float32)
    if pin:
        y, hl = y.pin_memory(), hl.pin_memory()
    nbytes = ssm.ssm_scan_host_workspace_bytes(batch, L, dim, N, 1 if dtype == "bf16" else 0)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    fn = ssm.ssm_scan_fwd_bf16_host if dtype == "bf16" else ssm.ssm_scan_fwd_host
    P = lambda t: 0 if t is None else t.data_ptr()  # noqa: E731
    stream = torch.cuda.current_stream().cuda_stream
    st = fn(P(h["u"]), P(h["delta"]), P(h["A"]), P(h["B"]), P(h["C"]), P(h["D"]), P(h["z"]),
            P(h["delta_bias"]), int(inp["softplus"]), P(y), P(hl), batch, L, dim, N, P(ws), nbytes,
            stream)
    assert st == 0, ssm.ssm_status_string(st)
    torch.cuda.synchronize()
    assert ssm.ssm_scan_last_device_status(stream) == 0
    yf = y.float().numpy()
    yr, hr = oracle_ref(W.decoded(inp))
    assert rel_err(yf, yr) <= TOL[dtype] and rel_err(hl.numpy(), hr) <= TOL[dtype]
