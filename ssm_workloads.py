"""Seeded synthetic inputs for the selective-scan forward workloads.

This module is the only code shared by the CUDA path's tests/bench and the
oracle's tests.  It draws random inputs and stores them in the dtypes the
library consumes; it holds none of the scan's arithmetic.

Workloads (shapes and distributions as the pages' Mamba configurations give
them: d_state 16, expand 2 x d_model 768 = 1536 channels for the 130M-class
layer, 5120 channels for the 2.8B-class layer; A initialised to -(n+1), the
S4D-real / A_log = log(1..N) initialisation of the SelectiveSSM and MambaBlock
listings; D initialised to ones):

  small_fp32     fp32, batch 1, L 256,  dim 64,   N 16: u, B, C ~ N(0,1);
                 delta = exp(U(ln 1e-3, ln 1e-1)) per (t, d); A = -(n+1); D = 1;
                 no gate, no softplus, no bias.
  lti_fp32       time-invariant check, fp32, batch 2, L 4096, dim 256, N 64:
                 delta per channel = exp(U(ln 1e-3, ln 1e-1)), the same for all
                 (b, t); B[n], C[n] ~ N(0,1) the same for all (b, t); u ~ N(0,1);
                 A = -(n+1); D absent (y = u * K exactly) or D = 1.
  mamba130m_bf16 batch 8, L 2048, dim 1536, N 16: u, z, B, C, delta_raw ~ N(0,1)
                 rounded to bf16; delta_bias (fp32) = softplus^-1(U(1e-3, 1e-1));
                 softplus on; A = -(n+1) fp32; D = 1 fp32; SiLU(z) gate on.
  mamba2p8b_bf16 batch 4, L 8192, dim 5120, N 16, otherwise as mamba130m_bf16.
  longctx_L{L}   batch 1, dim 5120, N 16, L in {2048, 8192, 32768, 131072},
                 otherwise as mamba130m_bf16.

Random draws use numpy's PCG64 generator seeded with ``seed`` (0 by default),
in the fixed order u, delta, B, C, z, delta_bias.  bf16 values are produced by
round-to-nearest-even from the fp32 draw; ``decode`` returns their exact fp32
values.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional

import numpy as np

_CHUNK = 1 << 24  # elements generated per step, to bound host memory


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    L: int
    dim: int
    N: int
    dtype: str            # "f32" or "bf16" (storage dtype of u, delta, B, C, z, y)
    softplus: bool
    delta_bias: bool
    gate: bool            # z given
    skip: bool            # D given
    delta_kind: str       # "loguniform_td", "loguniform_d" (time-invariant), "normal_raw"
    shared_BC: bool = False  # B, C the same vector for all (b, t)

    @property
    def tokens(self) -> int:
        return self.batch * self.L

    def with_L(self, L: int) -> "Workload":
        return dataclasses.replace(self, L=L, name=f"{self.name.split('_L')[0]}_L{L}")

    def with_shape(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS: Dict[str, Workload] = {
    "small_fp32": Workload("small_fp32", 1, 256, 64, 16, "f32", softplus=False,
                           delta_bias=False, gate=False, skip=True,
                           delta_kind="loguniform_td"),
    "lti_fp32": Workload("lti_fp32", 2, 4096, 256, 64, "f32", softplus=False,
                         delta_bias=False, gate=False, skip=False,
                         delta_kind="loguniform_d", shared_BC=True),
    "mamba130m_bf16": Workload("mamba130m_bf16", 8, 2048, 1536, 16, "bf16",
                               softplus=True, delta_bias=True, gate=True, skip=True,
                               delta_kind="normal_raw"),
    "mamba2p8b_bf16": Workload("mamba2p8b_bf16", 4, 8192, 5120, 16, "bf16",
                               softplus=True, delta_bias=True, gate=True, skip=True,
                               delta_kind="normal_raw"),
    # the Mamba-130M layer shape with the SiLU(z) gate off (no z tensor)
    "mamba130m_bf16_nogate": Workload("mamba130m_bf16_nogate", 8, 2048, 1536, 16, "bf16",
                                      softplus=True, delta_bias=True, gate=False, skip=True,
                                      delta_kind="normal_raw"),
}
LONGCTX_LS = (2048, 8192, 32768, 131072)
for _L in LONGCTX_LS:
    WORKLOADS[f"longctx_L{_L}"] = Workload(f"longctx_L{_L}", 1, _L, 5120, 16, "bf16",
                                           softplus=True, delta_bias=True, gate=True,
                                           skip=True, delta_kind="normal_raw")


# ---------------------------------------------------------------- bf16 storage
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (round to nearest, ties to even); returns the
    16-bit patterns as uint16.  Inputs here are finite."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    b = x.view(np.uint32)
    r = ((b >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((b + r) >> np.uint32(16)).astype(np.uint16)


def decode(a: np.ndarray) -> np.ndarray:
    """Exact fp32 values of a stored array (uint16 bf16 patterns or fp32)."""
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << np.uint32(16)).view(np.float32)
    return np.asarray(a, dtype=np.float32)


def _normal(rng: np.random.Generator, shape, store_bf16: bool) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16 if store_bf16 else np.float32)
    for lo in range(0, n, _CHUNK):
        hi = min(n, lo + _CHUNK)
        v = rng.standard_normal(hi - lo, dtype=np.float32)
        out[lo:hi] = f32_to_bf16_bits(v) if store_bf16 else v
    return out.reshape(shape)


def _loguniform(rng, shape, lo=1e-3, hi=1e-1) -> np.ndarray:
    v = rng.uniform(np.log(lo), np.log(hi), size=shape)
    return np.exp(v).astype(np.float32)


def make_inputs(wl: Workload, seed: int = 0) -> Dict[str, Optional[np.ndarray]]:
    """Draw the inputs of one workload.

    Returns a dict with u, delta, B, C, z (uint16 bf16 patterns for bf16
    workloads, float32 for fp32 ones; z may be None), A (dim, N) float32,
    D (dim,) float32 or None, delta_bias (dim,) float32 or None, plus the flag
    ``softplus``.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    bf = wl.dtype == "bf16"
    B_, L, Dm, N = wl.batch, wl.L, wl.dim, wl.N
    inp: Dict[str, Optional[np.ndarray]] = {}

    inp["u"] = _normal(rng, (B_, L, Dm), bf)

    if wl.delta_kind == "loguniform_td":
        d = _loguniform(rng, (B_, L, Dm))
        inp["delta"] = f32_to_bf16_bits(d) if bf else d
    elif wl.delta_kind == "loguniform_d":
        d = _loguniform(rng, (Dm,))
        full = np.broadcast_to(d, (B_, L, Dm)).copy()
        inp["delta"] = f32_to_bf16_bits(full) if bf else full
    elif wl.delta_kind == "normal_raw":
        inp["delta"] = _normal(rng, (B_, L, Dm), bf)
    else:
        raise ValueError(wl.delta_kind)

    if wl.shared_BC:
        bvec = rng.standard_normal(N, dtype=np.float32)
        cvec = rng.standard_normal(N, dtype=np.float32)
        Bf = np.broadcast_to(bvec, (B_, L, N)).copy()
        Cf = np.broadcast_to(cvec, (B_, L, N)).copy()
        inp["B"] = f32_to_bf16_bits(Bf) if bf else Bf
        inp["C"] = f32_to_bf16_bits(Cf) if bf else Cf
    else:
        inp["B"] = _normal(rng, (B_, L, N), bf)
        inp["C"] = _normal(rng, (B_, L, N), bf)

    inp["z"] = _normal(rng, (B_, L, Dm), bf) if wl.gate else None

    if wl.delta_bias:
        # bias = softplus^-1(v) = log(expm1(v)), v ~ U(1e-3, 1e-1): the bias a
        # freshly initialised dt projection carries so that softplus(bias) = v.
        v = rng.uniform(1e-3, 1e-1, size=Dm)
        inp["delta_bias"] = np.log(np.expm1(v)).astype(np.float32)
    else:
        inp["delta_bias"] = None

    inp["A"] = np.broadcast_to(-np.arange(1, N + 1, dtype=np.float32), (Dm, N)).copy()
    inp["D"] = np.ones(Dm, dtype=np.float32) if wl.skip else None
    inp["softplus"] = wl.softplus
    return inp


def channel_sample(wl: Workload, n_dim: int = 24, n_batch: int = 2, seed: int = 1):
    """Pick a set of batch rows and channels for full-size sampled checks:
    always the first and last channel and batch row, plus seeded random ones."""
    rng = np.random.Generator(np.random.PCG64(seed))
    ds = {0, wl.dim - 1}
    ds |= set(int(x) for x in rng.choice(wl.dim, size=min(n_dim, wl.dim), replace=False))
    bs = {0, wl.batch - 1}
    bs |= set(int(x) for x in rng.choice(wl.batch, size=min(n_batch, wl.batch), replace=False))
    return np.array(sorted(bs)), np.array(sorted(ds))


def gather(inp, bs: np.ndarray, ds: np.ndarray):
    """Sub-problem made of batch rows ``bs`` and channels ``ds`` (channels are
    independent, so this is itself a valid, smaller problem).  Returns decoded
    fp32 arrays."""
    out = {}
    for k in ("u", "delta", "z"):
        a = inp[k]
        out[k] = None if a is None else decode(a[bs][:, :, ds])
    for k in ("B", "C"):
        out[k] = decode(inp[k][bs])
    out["A"] = inp["A"][ds]
    out["D"] = None if inp["D"] is None else inp["D"][ds]
    out["delta_bias"] = None if inp["delta_bias"] is None else inp["delta_bias"][ds]
    out["softplus"] = inp["softplus"]
    return out


def decoded(inp):
    """All inputs decoded to exact fp32 arrays (small workloads only)."""
    out = dict(inp)
    for k in ("u", "delta", "B", "C", "z"):
        if inp[k] is not None:
            out[k] = decode(inp[k])
    return out
