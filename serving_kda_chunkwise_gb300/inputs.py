"""Seeded synthetic inputs for KDA, shared by the tests, the smoke check and the bench.

This module holds no arithmetic of the method itself (no gate, no decay, no
recurrence): it only draws random tensors and rounds them to the storage dtype.
Both the CUDA path and the CPU oracle read exactly the values it returns, so the
oracle sees the bf16-rounded inputs widened to fp64.

Recipe (per tensor, in this draw order, numpy PCG64 seeded with ``seed``):
  lengths (varlen only) ~ U{lo..hi}          A_log ~ U(-1, 1) per head
  q, k ~ N(0, 1), then L2-normalised over d_k for every (token, head)
  v ~ N(0, 1)        beta = logistic(N(0, 1))        z ~ N(0, 1) per channel
  S0 ~ N(0, 0.02^2) (when requested)
then q, k, v, beta, z are rounded to the I/O dtype (bf16: round to nearest even).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

# ----------------------------------------------------------------- rounding --


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); return the raw uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(
        np.float32)


@dataclass
class Stored:
    """One tensor in its storage form plus the exact float32 values it holds."""
    values: np.ndarray          # float32, exactly the stored numbers
    bits: np.ndarray | None     # uint16 raw bf16 bits when dtype == "bf16", else None
    dtype: str                  # "bf16" or "f32"

    def as_torch(self, device="cpu"):
        import torch
        if self.dtype == "bf16":
            t = torch.from_numpy(self.bits.view(np.int16)).view(torch.bfloat16)
        else:
            t = torch.from_numpy(self.values)
        return t.to(device)


def store(x: np.ndarray, dtype: str) -> Stored:
    if dtype == "bf16":
        bits = f32_to_bf16_bits(x)
        return Stored(bf16_bits_to_f32(bits), bits, "bf16")
    if dtype == "f32":
        return Stored(np.ascontiguousarray(x, dtype=np.float32), None, "f32")
    raise ValueError(dtype)


# ------------------------------------------------------------------- draws --


def _normal(rng, shape):
    return rng.standard_normal(size=shape, dtype=np.float32)


def _unit_rows(x: np.ndarray) -> np.ndarray:
    n = np.sqrt(np.sum(np.square(x, dtype=np.float64), axis=-1, keepdims=True))
    return (x / np.maximum(n, 1e-30)).astype(np.float32)


def _logistic(x: np.ndarray) -> np.ndarray:
    return (1.0 / (1.0 + np.exp(-x.astype(np.float64)))).astype(np.float32)


@dataclass
class ForwardInputs:
    q: Stored
    k: Stored
    v: Stored
    beta: Stored
    z: Stored
    A_log: np.ndarray                 # float32 [H]
    S0: np.ndarray | None             # float32 [N, H, dk, dv] or None
    cu_seqlens: np.ndarray            # int64 [N + 1]
    g_min: float
    dtype: str
    meta: dict = field(default_factory=dict)

    @property
    def T(self):
        return self.q.values.shape[0]

    @property
    def H(self):
        return self.q.values.shape[1]

    @property
    def dk(self):
        return self.q.values.shape[2]

    @property
    def dv(self):
        return self.v.values.shape[2]

    @property
    def N(self):
        return self.cu_seqlens.shape[0] - 1


def forward_inputs(*, seed: int, H: int, dk: int, dv: int, dtype: str,
                   lengths=None, B: int = 1, T: int = 0, g_min: float = -5.0,
                   with_state: bool = False, varlen_range=None) -> ForwardInputs:
    """Draw one forward problem.

    Either ``lengths`` (explicit per-sequence lengths), ``varlen_range=(count, lo, hi)``
    (lengths drawn ~ U{lo..hi}) or ``B`` equal sequences of length ``T``.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    if varlen_range is not None:
        count, lo, hi = varlen_range
        lens = rng.integers(lo, hi + 1, size=count).astype(np.int64)
    elif lengths is not None:
        lens = np.asarray(lengths, dtype=np.int64)
    else:
        lens = np.full(B, T, dtype=np.int64)
    cu = np.zeros(lens.shape[0] + 1, dtype=np.int64)
    cu[1:] = np.cumsum(lens)
    Tt = int(cu[-1])
    N = lens.shape[0]
    A_log = rng.uniform(-1.0, 1.0, size=H).astype(np.float32)
    q = _unit_rows(_normal(rng, (Tt, H, dk)))
    k = _unit_rows(_normal(rng, (Tt, H, dk)))
    v = _normal(rng, (Tt, H, dv))
    beta = _logistic(_normal(rng, (Tt, H)))
    z = _normal(rng, (Tt, H, dk))
    S0 = (0.02 * _normal(rng, (N, H, dk, dv))).astype(np.float32) if with_state else None
    return ForwardInputs(store(q, dtype), store(k, dtype), store(v, dtype), store(beta, dtype),
                         store(z, dtype), A_log, S0, cu, float(g_min), dtype,
                         meta=dict(seed=seed))


@dataclass
class DecodeInputs:
    q: Stored
    k: Stored
    v: Stored
    beta: Stored
    z: Stored


def decode_state(*, seed: int, N: int, H: int, dk: int, dv: int):
    """Initial decode state S ~ N(0, 0.02^2) [N,H,dk,dv] float32 and A_log ~ U(-1,1) [H]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    A_log = rng.uniform(-1.0, 1.0, size=H).astype(np.float32)
    S = (0.02 * _normal(rng, (N, H, dk, dv))).astype(np.float32)
    return S, A_log


def decode_step_inputs(*, seed: int, step: int, N: int, H: int, dk: int, dv: int,
                       dtype: str = "bf16") -> DecodeInputs:
    """Inputs for decode step ``step``: one new token for each of N sequences."""
    rng = np.random.Generator(np.random.PCG64([seed, step]))
    q = _unit_rows(_normal(rng, (N, H, dk)))
    k = _unit_rows(_normal(rng, (N, H, dk)))
    v = _normal(rng, (N, H, dv))
    beta = _logistic(_normal(rng, (N, H)))
    z = _normal(rng, (N, H, dk))
    return DecodeInputs(store(q, dtype), store(k, dtype), store(v, dtype), store(beta, dtype),
                        store(z, dtype))


# ------------------------------------------------------ the named workloads --

#: The five workloads, by what they are.  ``seed`` = 1000 + index.
WORKLOADS = {
    "fwd_f32_T256_H2_d64": dict(seed=1000, B=1, T=256, H=2, dk=64, dv=64, dtype="f32",
                                with_state=False),
    "fwd_bf16_B2_T4096_H16_d128": dict(seed=1001, B=2, T=4096, H=16, dk=128, dv=128,
                                       dtype="bf16", with_state=True),
    "fwd_bf16_T65536_H32_d128": dict(seed=1002, B=1, T=65536, H=32, dk=128, dv=128,
                                     dtype="bf16", with_state=False),
    "fwd_bf16_varlen64_H32_d128": dict(seed=1003, varlen_range=(64, 128, 16384), H=32, dk=128,
                                       dv=128, dtype="bf16", with_state=True),
}

#: g_min sweep for the long-context workload (same seed-1002 inputs for each value).
LONG_GMIN_SWEEP = (-3.0, -5.0, -6.0)

DECODE_WORKLOAD = dict(seed=1004, N=256, H=32, dk=128, dv=128, steps=1000, dtype="bf16")


def workload(name: str, g_min: float = -5.0, **overrides) -> ForwardInputs:
    kw = dict(WORKLOADS[name])
    kw.update(overrides)
    return forward_inputs(g_min=g_min, **kw)
