"""The torch wrappers refuse tensors the C ABI cannot take before any CUDA
call: host tensors, mixed dtypes, fp16 (CPU only, no GPU needed)."""
import pytest
import torch

import selective_state_space_150_b300 as ssm


def _tensors(dtype=torch.float32):
    b, L, d, n = 1, 4, 8, 4
    return dict(u=torch.zeros(b, L, d, dtype=dtype), delta=torch.zeros(b, L, d, dtype=dtype),
                A=torch.zeros(d, n), B=torch.zeros(b, L, n, dtype=dtype),
                C=torch.zeros(b, L, n, dtype=dtype))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_forward_refuses_host_tensors(dtype):
    t = _tensors(dtype)
    with pytest.raises(TypeError):
        ssm.selective_scan_fwd(t["u"], t["delta"], t["A"], t["B"], t["C"])


def test_forward_refuses_fp16():
    t = _tensors(torch.float16)
    with pytest.raises(TypeError):
        ssm.selective_scan_fwd(t["u"], t["delta"], t["A"], t["B"], t["C"])


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_backward_refuses_host_tensors(dtype):
    t = _tensors(dtype)
    with pytest.raises(TypeError):
        ssm.selective_scan_bwd(t["u"], t["delta"], t["A"], t["B"], t["C"], t["u"].clone())


def test_backward_refuses_mixed_dtypes():
    t = _tensors(torch.bfloat16)
    with pytest.raises(TypeError):
        ssm.selective_scan_bwd(t["u"], t["delta"].float(), t["A"], t["B"], t["C"],
                               t["u"].clone())
