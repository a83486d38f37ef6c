"""Python binding of libssmscan (the selective-scan forward on sm_103a).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of libssmscan.so.  The functions named like the C ABI take raw device
pointers (ints) and sizes; ``selective_scan_fwd`` is a convenience wrapper that
takes torch CUDA tensors, allocates the outputs with torch when they are not
given, and raises on a nonzero status.  There is no CPU fallback: importing this
module fails if the shared library is missing.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libssmscan.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"libssmscan.so not found at {LIB_PATH}; build it with "
        "`python selective_state_space_150_b300/build.py` (nvcc, sm_103a)")

_lib = ctypes.CDLL(LIB_PATH)

SSM_OK = 0
SSM_ERR_NULL = 1
SSM_ERR_SIZE = 2
SSM_ERR_ALIGN = 3
SSM_ERR_UNSUPPORTED_N = 4
SSM_ERR_LAUNCH = 5
SSM_ERR_TIMEOUT = 6
SSM_ERR_ALIAS = 7
SSM_ERR_ARG = 8
SSM_ERR_NOMEM = 9
SSM_ERR_SCRATCH = 10
SSM_NOALLOC_SCRATCH_FLOATS = 2097152
SSM_MAX_N = 128

SSM_KNOB_WAIT_NS = 1
SSM_KNOB_FORCE_TIMEOUT = 2
SSM_KNOB_STATE_GROUPS = 3
SSM_KNOB_CHUNK = 4
SSM_KNOB_PLAIN_LOADS = 5
SSM_KNOB_STAGES = 6
SSM_KNOB_SEGMENTS = 7
SSM_KNOB_KERNEL = 8
SSM_KNOB_BWD_SEGMENTS = 9

EXPORTED = ("ssm_scan_fwd", "ssm_scan_fwd_bf16", "ssm_scan_fwd_bf16_noalloc",
            "ssm_scan_fwd_h0", "ssm_scan_fwd_bf16_h0", "ssm_scan_fwd_zoh", "ssm_scan_fwd_bf16_zoh",
            "ssm_scan_step", "ssm_scan_step_bf16",
            "ssm_conv_scan_fwd", "ssm_conv_scan_fwd_bf16", "ssm_scan_host_workspace_bytes",
            "ssm_scan_fwd_host", "ssm_scan_fwd_bf16_host", "ssm_scan_bwd", "ssm_scan_bwd_bf16",
            "ssm_scan_bwd_h0", "ssm_scan_bwd_bf16_h0",
            "ssm_scan_last_device_status", "ssm_status_string", "ssm_scan_plan", "ssm_set_knob")

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_FWD_ARGS = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_int, _vp, _vp,
             _i64, _i64, _i64, _i64, _vp]
for _name in ("ssm_scan_fwd", "ssm_scan_fwd_bf16", "ssm_scan_fwd_bf16_noalloc"):
    getattr(_lib, _name).argtypes = _FWD_ARGS
    getattr(_lib, _name).restype = ctypes.c_int
for _name in ("ssm_scan_fwd_h0", "ssm_scan_fwd_bf16_h0", "ssm_scan_fwd_zoh", "ssm_scan_fwd_bf16_zoh"):
    getattr(_lib, _name).argtypes = _FWD_ARGS[:8] + [_vp] + _FWD_ARGS[8:]
    getattr(_lib, _name).restype = ctypes.c_int
for _name in ("ssm_conv_scan_fwd", "ssm_conv_scan_fwd_bf16"):
    getattr(_lib, _name).argtypes = [_vp, _vp, _vp, ctypes.c_int] + _FWD_ARGS[1:]
    getattr(_lib, _name).restype = ctypes.c_int
for _name in ("ssm_scan_fwd_host", "ssm_scan_fwd_bf16_host"):
    getattr(_lib, _name).argtypes = _FWD_ARGS[:-1] + [_vp, _i64, _vp]
    getattr(_lib, _name).restype = ctypes.c_int
_lib.ssm_scan_host_workspace_bytes.argtypes = [_i64, _i64, _i64, _i64, ctypes.c_int]
_lib.ssm_scan_host_workspace_bytes.restype = _i64
for _name in ("ssm_scan_bwd", "ssm_scan_bwd_bf16"):
    getattr(_lib, _name).argtypes = [_vp] * 8 + [ctypes.c_int] + [_vp] * 9 + [_i64] * 4 + [_vp]
    getattr(_lib, _name).restype = ctypes.c_int
for _name in ("ssm_scan_bwd_h0", "ssm_scan_bwd_bf16_h0"):
    getattr(_lib, _name).argtypes = [_vp] * 8 + [ctypes.c_int] + [_vp] * 12 + [_i64] * 4 + [_vp]
    getattr(_lib, _name).restype = ctypes.c_int
for _name in ("ssm_scan_step", "ssm_scan_step_bf16"):
    getattr(_lib, _name).argtypes = [_vp] * 8 + [ctypes.c_int, _vp, _vp, _i64, _i64, _i64, _vp]
    getattr(_lib, _name).restype = ctypes.c_int
_lib.ssm_scan_last_device_status.argtypes = [_vp]
_lib.ssm_scan_last_device_status.restype = ctypes.c_int
_lib.ssm_status_string.argtypes = [ctypes.c_int]
_lib.ssm_status_string.restype = ctypes.c_char_p
_lib.ssm_scan_plan.argtypes = [_i64, _i64, _i64, _i64, ctypes.c_int, ctypes.POINTER(_i64)]
_lib.ssm_scan_plan.restype = ctypes.c_int
_lib.ssm_set_knob.argtypes = [ctypes.c_int, _i64]
_lib.ssm_set_knob.restype = ctypes.c_int


class SSMError(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        self.status = status
        super().__init__(f"{where}: status {status} ({ssm_status_string(status)})")


# ------------------------------------------------------------ C ABI, verbatim
def ssm_scan_fwd(u, delta, A, B, C, D, z, delta_bias, softplus_flag, y, h_last,
                 batch, L, dim, N, stream) -> int:
    """fp32 entry point; pointer arguments are ints (0 for NULL)."""
    return _lib.ssm_scan_fwd(u or None, delta or None, A or None, B or None, C or None,
                             D or None, z or None, delta_bias or None, int(softplus_flag),
                             y or None, h_last or None, batch, L, dim, N, stream or None)


def ssm_scan_fwd_bf16(u, delta, A, B, C, D, z, delta_bias, softplus_flag, y, h_last,
                      batch, L, dim, N, stream) -> int:
    """bf16 entry point; pointer arguments are ints (0 for NULL)."""
    return _lib.ssm_scan_fwd_bf16(u or None, delta or None, A or None, B or None, C or None,
                                  D or None, z or None, delta_bias or None, int(softplus_flag),
                                  y or None, h_last or None, batch, L, dim, N, stream or None)


def ssm_scan_fwd_bf16_noalloc(u, delta, A, B, C, D, z, delta_bias, softplus_flag, y, h_last,
                              batch, L, dim, N, stream) -> int:
    """bf16 entry point with segment scratch in the library's static device
    buffer (no allocation); pointer arguments are ints (0 for NULL)."""
    return _lib.ssm_scan_fwd_bf16_noalloc(u or None, delta or None, A or None, B or None,
                                          C or None, D or None, z or None, delta_bias or None,
                                          int(softplus_flag), y or None, h_last or None,
                                          batch, L, dim, N, stream or None)


def ssm_scan_fwd_h0(u, delta, A, B, C, D, z, delta_bias, h0, softplus_flag, y, h_last,
                    batch, L, dim, N, stream) -> int:
    """fp32 entry point from an initial state h0; pointer arguments are ints."""
    return _lib.ssm_scan_fwd_h0(u or None, delta or None, A or None, B or None, C or None,
                                D or None, z or None, delta_bias or None, h0 or None,
                                int(softplus_flag), y or None, h_last or None, batch, L, dim, N,
                                stream or None)


def ssm_scan_fwd_bf16_h0(u, delta, A, B, C, D, z, delta_bias, h0, softplus_flag, y, h_last,
                         batch, L, dim, N, stream) -> int:
    """bf16 entry point from an initial state h0; pointer arguments are ints."""
    return _lib.ssm_scan_fwd_bf16_h0(u or None, delta or None, A or None, B or None, C or None,
                                     D or None, z or None, delta_bias or None, h0 or None,
                                     int(softplus_flag), y or None, h_last or None, batch, L,
                                     dim, N, stream or None)


def ssm_conv_scan_fwd(x, conv_w, conv_b, conv_k, delta, A, B, C, D, z, delta_bias,
                      softplus_flag, y, h_last, batch, L, dim, N, stream) -> int:
    """fp32 scan with the causal conv + SiLU prologue; pointers are ints."""
    return _lib.ssm_conv_scan_fwd(x or None, conv_w or None, conv_b or None, int(conv_k),
                                  delta or None, A or None, B or None, C or None, D or None,
                                  z or None, delta_bias or None, int(softplus_flag), y or None,
                                  h_last or None, batch, L, dim, N, stream or None)


def ssm_conv_scan_fwd_bf16(x, conv_w, conv_b, conv_k, delta, A, B, C, D, z, delta_bias,
                           softplus_flag, y, h_last, batch, L, dim, N, stream) -> int:
    """bf16 scan with the causal conv + SiLU prologue; pointers are ints."""
    return _lib.ssm_conv_scan_fwd_bf16(x or None, conv_w or None, conv_b or None, int(conv_k),
                                       delta or None, A or None, B or None, C or None, D or None,
                                       z or None, delta_bias or None, int(softplus_flag),
                                       y or None, h_last or None, batch, L, dim, N,
                                       stream or None)


def ssm_scan_host_workspace_bytes(batch, L, dim, N, dtype: int) -> int:
    """Device workspace bytes the host-buffer entry points need (-1: bad size)."""
    return int(_lib.ssm_scan_host_workspace_bytes(batch, L, dim, N, int(dtype)))


def ssm_scan_fwd_host(u, delta, A, B, C, D, z, delta_bias, softplus_flag, y, h_last, batch, L,
                      dim, N, workspace, workspace_bytes, stream) -> int:
    """fp32 scan on HOST buffers (pointers are ints); workspace is a device pointer."""
    return _lib.ssm_scan_fwd_host(u or None, delta or None, A or None, B or None, C or None,
                                  D or None, z or None, delta_bias or None, int(softplus_flag),
                                  y or None, h_last or None, batch, L, dim, N, workspace or None,
                                  int(workspace_bytes), stream or None)


def ssm_scan_fwd_bf16_host(u, delta, A, B, C, D, z, delta_bias, softplus_flag, y, h_last, batch,
                           L, dim, N, workspace, workspace_bytes, stream) -> int:
    """bf16 scan on HOST buffers (pointers are ints); workspace is a device pointer."""
    return _lib.ssm_scan_fwd_bf16_host(u or None, delta or None, A or None, B or None, C or None,
                                       D or None, z or None, delta_bias or None,
                                       int(softplus_flag), y or None, h_last or None, batch, L,
                                       dim, N, workspace or None, int(workspace_bytes),
                                       stream or None)


def ssm_scan_fwd_zoh(u, delta, A, B, C, D, z, delta_bias, h0, softplus_flag, y, h_last,
                     batch, L, dim, N, stream) -> int:
    """fp32 entry point with the exact zero-order-hold B; pointers are ints."""
    return _lib.ssm_scan_fwd_zoh(u or None, delta or None, A or None, B or None, C or None,
                                 D or None, z or None, delta_bias or None, h0 or None,
                                 int(softplus_flag), y or None, h_last or None, batch, L, dim, N,
                                 stream or None)


def ssm_scan_fwd_bf16_zoh(u, delta, A, B, C, D, z, delta_bias, h0, softplus_flag, y, h_last,
                          batch, L, dim, N, stream) -> int:
    """bf16 entry point with the exact zero-order-hold B; pointers are ints."""
    return _lib.ssm_scan_fwd_bf16_zoh(u or None, delta or None, A or None, B or None, C or None,
                                      D or None, z or None, delta_bias or None, h0 or None,
                                      int(softplus_flag), y or None, h_last or None, batch, L,
                                      dim, N, stream or None)


def ssm_scan_bwd(u, delta, A, B, C, D, z, delta_bias, softplus_flag, dy, du, ddelta, dA, dB, dC,
                 dD, dz, ddelta_bias, batch, L, dim, N, stream) -> int:
    """fp32 backward pass; pointer arguments are ints (0 for NULL)."""
    p = lambda v: v or None  # noqa: E731
    return _lib.ssm_scan_bwd(p(u), p(delta), p(A), p(B), p(C), p(D), p(z), p(delta_bias),
                             int(softplus_flag), p(dy), p(du), p(ddelta), p(dA), p(dB), p(dC),
                             p(dD), p(dz), p(ddelta_bias), batch, L, dim, N, p(stream))


def ssm_scan_bwd_bf16(u, delta, A, B, C, D, z, delta_bias, softplus_flag, dy, du, ddelta, dA,
                      dB, dC, dD, dz, ddelta_bias, batch, L, dim, N, stream) -> int:
    """bf16 backward pass (bf16 u/delta/B/C/z/dy and du/ddelta/dB/dC/dz, fp32
    A/D/bias and their gradients); pointer arguments are ints (0 for NULL)."""
    p = lambda v: v or None  # noqa: E731
    return _lib.ssm_scan_bwd_bf16(p(u), p(delta), p(A), p(B), p(C), p(D), p(z), p(delta_bias),
                                  int(softplus_flag), p(dy), p(du), p(ddelta), p(dA), p(dB),
                                  p(dC), p(dD), p(dz), p(ddelta_bias), batch, L, dim, N,
                                  p(stream))


def ssm_scan_bwd_h0(u, delta, A, B, C, D, z, delta_bias, softplus_flag, dy, du, ddelta, dA, dB,
                    dC, dD, dz, ddelta_bias, h0, dh_last, dh0, batch, L, dim, N, stream) -> int:
    """fp32 backward from h0 with dh_last, writing dh0; pointers are ints."""
    p = lambda v: v or None  # noqa: E731
    return _lib.ssm_scan_bwd_h0(p(u), p(delta), p(A), p(B), p(C), p(D), p(z), p(delta_bias),
                                int(softplus_flag), p(dy), p(du), p(ddelta), p(dA), p(dB), p(dC),
                                p(dD), p(dz), p(ddelta_bias), p(h0), p(dh_last), p(dh0), batch,
                                L, dim, N, p(stream))


def ssm_scan_bwd_bf16_h0(u, delta, A, B, C, D, z, delta_bias, softplus_flag, dy, du, ddelta, dA,
                         dB, dC, dD, dz, ddelta_bias, h0, dh_last, dh0, batch, L, dim, N,
                         stream) -> int:
    """bf16 backward from h0 with dh_last, writing dh0; pointers are ints."""
    p = lambda v: v or None  # noqa: E731
    return _lib.ssm_scan_bwd_bf16_h0(p(u), p(delta), p(A), p(B), p(C), p(D), p(z),
                                     p(delta_bias), int(softplus_flag), p(dy), p(du), p(ddelta),
                                     p(dA), p(dB), p(dC), p(dD), p(dz), p(ddelta_bias), p(h0),
                                     p(dh_last), p(dh0), batch, L, dim, N, p(stream))


def ssm_scan_step(u, delta, A, B, C, D, z, delta_bias, softplus_flag, h, y, batch, dim, N,
                  stream) -> int:
    """fp32 one-token recurrent step (h updated in place); pointers are ints."""
    return _lib.ssm_scan_step(u or None, delta or None, A or None, B or None, C or None,
                              D or None, z or None, delta_bias or None, int(softplus_flag),
                              h or None, y or None, batch, dim, N, stream or None)


def ssm_scan_step_bf16(u, delta, A, B, C, D, z, delta_bias, softplus_flag, h, y, batch, dim, N,
                       stream) -> int:
    """bf16 one-token recurrent step (h updated in place); pointers are ints."""
    return _lib.ssm_scan_step_bf16(u or None, delta or None, A or None, B or None, C or None,
                                   D or None, z or None, delta_bias or None, int(softplus_flag),
                                   h or None, y or None, batch, dim, N, stream or None)


def ssm_scan_last_device_status(stream=0) -> int:
    return _lib.ssm_scan_last_device_status(stream or None)


def ssm_status_string(status: int) -> str:
    return _lib.ssm_status_string(int(status)).decode()


def ssm_scan_plan(batch, L, dim, N, dtype: int):
    """Launch plan as a dict (see include/ssmscan.h); raises on a bad argument."""
    out = (_i64 * 11)()
    st = _lib.ssm_scan_plan(batch, L, dim, N, int(dtype), out)
    if st != SSM_OK:
        raise SSMError(st, "ssm_scan_plan")
    keys = ("state_groups", "states_per_lane", "chunk", "channels_per_block", "threads",
            "blocks", "smem_bytes", "tma", "segments", "scratch_bytes", "kernel")
    return dict(zip(keys, [int(v) for v in out]))


def ssm_set_knob(key: int, value: int) -> int:
    return _lib.ssm_set_knob(int(key), int(value))


# ------------------------------------------------------------ torch convenience
def _ptr(t):
    return 0 if t is None else t.data_ptr()


def _check_io(u, delta, B, C, z, A, D, delta_bias):
    import torch

    if u.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError(f"u must be float32 or bfloat16, got {u.dtype}")
    for t in (u, delta, B, C) + ((z,) if z is not None else ()):
        if t.dtype != u.dtype or not t.is_cuda or not t.is_contiguous():
            raise TypeError("u, delta, B, C, z must share u's dtype and be contiguous CUDA tensors")
    for t in (A, D, delta_bias):
        if t is not None and (t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous()):
            raise TypeError("A, D, delta_bias must be contiguous float32 CUDA tensors")
    return u.dtype == torch.bfloat16


def selective_scan_fwd(u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=False,
                       y=None, h_last=None, stream=None, want_h_last=True, h0=None, zoh=False):
    """Run the kernel on torch CUDA tensors.

    u, delta, z: (batch, L, dim); B, C: (batch, L, N); A: (dim, N) fp32;
    D, delta_bias: (dim,) fp32; h0: (batch, dim, N) fp32 initial state (None:
    zeros); zoh: the exact zero-order-hold B.  u/delta/B/C/z are all fp32
    (fp32 entry point) or all bf16 (bf16 entry point).  Returns (y, h_last).  Work is enqueued on ``stream``
    (default: torch's current stream) without synchronising.
    """
    import torch

    bf16 = _check_io(u, delta, B, C, z, A, D, delta_bias)
    if h0 is not None and (h0.dtype != torch.float32 or not h0.is_cuda or not h0.is_contiguous()):
        raise TypeError("h0 must be a contiguous float32 CUDA tensor")
    batch, L, dim = u.shape
    N = A.shape[1]
    if y is None:
        y = torch.empty_like(u)
    if h_last is None and want_h_last:
        h_last = torch.empty((batch, dim, N), dtype=torch.float32, device=u.device)
    if stream is None:
        stream = torch.cuda.current_stream(u.device).cuda_stream
    if zoh:
        fn = ssm_scan_fwd_bf16_zoh if bf16 else ssm_scan_fwd_zoh
        st = fn(_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                _ptr(delta_bias), _ptr(h0), int(bool(softplus)), _ptr(y), _ptr(h_last),
                batch, L, dim, N, int(stream))
    elif h0 is None:
        fn = ssm_scan_fwd_bf16 if bf16 else ssm_scan_fwd
        st = fn(_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                _ptr(delta_bias), int(bool(softplus)), _ptr(y), _ptr(h_last),
                batch, L, dim, N, int(stream))
    else:
        fn = ssm_scan_fwd_bf16_h0 if bf16 else ssm_scan_fwd_h0
        st = fn(_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                _ptr(delta_bias), _ptr(h0), int(bool(softplus)), _ptr(y), _ptr(h_last),
                batch, L, dim, N, int(stream))
    if st != SSM_OK:
        raise SSMError(st, fn.__name__)
    return y, h_last


def conv_selective_scan_fwd(x, conv_w, conv_b, delta, A, B, C, D=None, z=None, delta_bias=None,
                            softplus=False, y=None, h_last=None, stream=None):
    """The scan of u = silu(causal depthwise conv1d(x) + conv_b) on torch CUDA
    tensors; conv_w: (dim, K) fp32, K <= 4; conv_b: (dim,) fp32 or None.
    Returns (y, h_last)."""
    import torch

    bf16 = _check_io(x, delta, B, C, z, A, D, delta_bias)
    for t in (conv_w, conv_b):
        if t is not None and (t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous()):
            raise TypeError("conv_w, conv_b must be contiguous float32 CUDA tensors")
    batch, L, dim = x.shape
    N = A.shape[1]
    if y is None:
        y = torch.empty_like(x)
    if h_last is None:
        h_last = torch.empty((batch, dim, N), dtype=torch.float32, device=x.device)
    if stream is None:
        stream = torch.cuda.current_stream(x.device).cuda_stream
    fn = ssm_conv_scan_fwd_bf16 if bf16 else ssm_conv_scan_fwd
    st = fn(_ptr(x), _ptr(conv_w), _ptr(conv_b), conv_w.shape[1], _ptr(delta), _ptr(A), _ptr(B),
            _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias), int(bool(softplus)), _ptr(y),
            _ptr(h_last), batch, L, dim, N, int(stream))
    if st != SSM_OK:
        raise SSMError(st, fn.__name__)
    return y, h_last


def selective_scan_step(u, delta, A, B, C, h, D=None, z=None, delta_bias=None, softplus=False,
                        y=None, stream=None):
    """One recurrent step on torch CUDA tensors; ``h`` (batch, dim, N) fp32 is
    updated in place.  u, delta, z: (batch, dim); B, C: (batch, N).  Returns y
    (batch, dim)."""
    import torch

    bf16 = _check_io(u, delta, B, C, z, A, D, delta_bias)
    if h.dtype != torch.float32 or not h.is_cuda or not h.is_contiguous():
        raise TypeError("h must be a contiguous float32 CUDA tensor")
    batch, dim = u.shape
    N = A.shape[1]
    if y is None:
        y = torch.empty_like(u)
    if stream is None:
        stream = torch.cuda.current_stream(u.device).cuda_stream
    fn = ssm_scan_step_bf16 if bf16 else ssm_scan_step
    st = fn(_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias),
            int(bool(softplus)), _ptr(h), _ptr(y), batch, dim, N, int(stream))
    if st != SSM_OK:
        raise SSMError(st, fn.__name__)
    return y


def selective_scan_bwd(u, delta, A, B, C, dy, D=None, z=None, delta_bias=None, softplus=False,
                       stream=None, h0=None, dh_last=None):
    """Gradients of selective_scan_fwd's y given dy, for contiguous CUDA
    tensors that are all fp32, or bf16 u/delta/B/C/z/dy with fp32 A/D/
    delta_bias.  Returns a dict with du, ddelta, dA, dB, dC and dD, dz,
    ddelta_bias where D, z, delta_bias are given; each gradient has the dtype
    of its input.  With h0 (the state before step 0) or dh_last (the gradient
    on the last state), both fp32 (batch, dim, N), the dict also holds dh0."""
    import torch

    bf = u.dtype == torch.bfloat16
    io = torch.bfloat16 if bf else torch.float32
    for t, want in ((u, io), (delta, io), (B, io), (C, io), (z, io), (dy, io),
                    (A, torch.float32), (D, torch.float32), (delta_bias, torch.float32),
                    (h0, torch.float32), (dh_last, torch.float32)):
        if t is not None and (t.dtype != want or not t.is_cuda or not t.is_contiguous()):
            raise TypeError("the backward pass takes contiguous CUDA tensors: all fp32, or bf16 "
                            "u/delta/B/C/z/dy with fp32 A/D/delta_bias")
    batch, L, dim = u.shape
    N = A.shape[1]
    g = {"du": torch.empty_like(u), "ddelta": torch.empty_like(delta), "dA": torch.empty_like(A),
         "dB": torch.empty_like(B), "dC": torch.empty_like(C)}
    if D is not None:
        g["dD"] = torch.empty_like(D)
    if z is not None:
        g["dz"] = torch.empty_like(z)
    if delta_bias is not None:
        g["ddelta_bias"] = torch.empty_like(delta_bias)
    if stream is None:
        stream = torch.cuda.current_stream(u.device).cuda_stream
    args = (_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
            _ptr(delta_bias), int(bool(softplus)), _ptr(dy), _ptr(g["du"]),
            _ptr(g["ddelta"]), _ptr(g["dA"]), _ptr(g["dB"]), _ptr(g["dC"]),
            _ptr(g.get("dD")), _ptr(g.get("dz")), _ptr(g.get("ddelta_bias")))
    if h0 is not None or dh_last is not None:
        g["dh0"] = torch.empty((batch, dim, N), dtype=torch.float32, device=u.device)
        fn = ssm_scan_bwd_bf16_h0 if bf else ssm_scan_bwd_h0
        st = fn(*args, _ptr(h0), _ptr(dh_last), _ptr(g["dh0"]), batch, L, dim, N, int(stream))
    else:
        fn = ssm_scan_bwd_bf16 if bf else ssm_scan_bwd
        st = fn(*args, batch, L, dim, N, int(stream))
    if st != SSM_OK:
        raise SSMError(st, fn.__name__)
    return g
