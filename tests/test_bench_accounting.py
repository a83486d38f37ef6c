"""bench.py's algorithmic accounting on CPU, against the figures worked out by
hand for the Mamba-130M layer shape (batch 8, L 2048, dim 1536, N 16, bf16,
softplus + bias, gate, skip) and the layout the kernels read and write."""
import bench
import ssm_workloads as W

WL = W.WORKLOADS["mamba130m_bf16"]


def test_forward_bytes_per_launch():
    bld = 8 * 2048 * 1536
    # u, delta, z read and y written (2 bytes each), B and C (2 bytes, N = 16),
    # h_last (fp32 state), A (fp32) and D, bias (fp32 per channel)
    want = 4 * 2 * bld + 2 * 2 * 8 * 2048 * 16 + 4 * 8 * 1536 * 16 + 4 * 1536 * 16 + 8 * 1536
    assert bench.algorithmic_bytes(WL) == want == 203_272_192
    # 12 352 bytes per token plus the once-per-call arrays
    assert (want - 4 * 8 * 1536 * 16 - 4 * 1536 * 16 - 8 * 1536) // (8 * 2048) == 8 * 1536 + 4 * 16


def test_forward_mufu_and_fp32_ops():
    mufu, fp32 = bench.algorithmic_ops(WL)
    bld = 8 * 2048 * 1536
    assert mufu == bld * 16 + bld * 4 == 503_316_480      # exp per state; softplus, SiLU: 2 + 2
    assert fp32 == 4 * bld * 16 + 4 * bld                  # 4 per state; bias, dt*u, D*u, gate


def test_backward_accounting():
    bld, bln = 8 * 2048 * 1536, 8 * 2048 * 16
    nbytes, mufu, fp32 = bench.bwd_accounting(WL, es=2)
    # reads u, delta, z, dy and writes du, ddelta, dz (2 bytes), B, C read and
    # dB, dC written, plus A, D, bias and their fp32 gradients
    assert nbytes == 2 * bld * 7 + 2 * bln * 4 + 8 * 1536 * 18
    assert mufu == 3 * bld * 16 + bld * 5
    # per (b, t, d, n): two forward walks of 3, the adjoint step's 11, the
    # dB / dC channel sums' 2; per (b, t, d): 8, and 6 for the gate
    assert fp32 == (3 + 3 + 11 + 2) * bld * 16 + (8 + 6) * bld
    assert bench.bwd_accounting(WL, es=4)[0] == 4 * bld * 7 + 4 * bln * 4 + 8 * 1536 * 18


def test_accounting_follows_the_flags():
    plain = WL.with_shape(softplus=False, delta_bias=False, gate=False, skip=False)
    bld = 8 * 2048 * 1536
    assert bench.algorithmic_bytes(plain) == (3 * 2 * bld + 2 * 2 * 8 * 2048 * 16
                                              + 4 * 8 * 1536 * 16 + 4 * 1536 * 16)
    assert bench.algorithmic_ops(plain) == (bld * 16, 4 * bld * 16 + bld)
