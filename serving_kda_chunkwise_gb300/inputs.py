"""Seeded synthetic inputs for KDA, shared by the tests, the smoke check and the bench.

This module holds no arithmetic of the method itself (no gate, no decay, no
recurrence): it only draws random tensors and rounds them to the storage dtype.
Both the CUDA path and the CPU oracle read exactly the values it produces, so the
oracle sees the bf16-rounded inputs widened to fp64.

Recipe.  Every tensor is cut into blocks of ``BLOCK_TOKENS`` tokens (all heads); block
b of tensor X is drawn from numpy PCG64 seeded with SeedSequence([seed, X's id, b]),
so any block can be regenerated on its own, in any order and in parallel, with the
same bits.  Per token and head:
    q, k ~ N(0, 1), L2-normalised over d_k        v ~ N(0, 1)
    beta = logistic(N(0, 1))                       z ~ N(0, 1) per channel
and per problem:  A_log ~ U(-1, 1) per head,  S0 ~ N(0, 0.02^2),  varlen lengths
~ U{lo..hi}.  q, k, v, beta, z are then rounded to the I/O dtype (bf16: nearest even).
For the gated output step: head outputs o ~ N(0, 1) times a per-(token, head) scale
~ U(0.1, 10) (which the norm removes), gate logits ~ N(0, 1), norm weight ~ U(0.5, 1.5).
For quantile balancing: router scores s_ij ~ N(0, 1) + mu_j with a per-expert popularity
mu_j ~ N(0, 0.5^2) (so that some experts are over-chosen), current biases ~ N(0, 0.1^2);
optionally rounded to a grid of 1/4 to force ties.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
from dataclasses import dataclass

import numpy as np

BLOCK_TOKENS = 2048
_IDS = {"q": 1, "k": 2, "v": 3, "beta": 4, "z": 5, "A_log": 6, "S0": 7, "lengths": 8,
        "o_head": 9, "gate": 10, "norm_w": 11, "router": 12, "popularity": 13,
        "expert_bias": 14}

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


def _round(x: np.ndarray, dtype: str) -> np.ndarray:
    """float32 values exactly representable in `dtype`."""
    return bf16_bits_to_f32(f32_to_bf16_bits(x)) if dtype == "bf16" else x


# ------------------------------------------------------------------- draws --


def _gen(*key):
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(list(key))))


def _unit_rows(x: np.ndarray) -> np.ndarray:
    n = np.sqrt(np.einsum("...i,...i->...", x, x, dtype=np.float32))[..., None]
    return x / np.maximum(n, np.float32(1e-30))


def _logistic(x: np.ndarray) -> np.ndarray:
    return (1.0 / (1.0 + np.exp(-x))).astype(np.float32)


def _draw(kind: str, rng, shape) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if kind in ("q", "k"):
        return _unit_rows(x)
    if kind == "beta":
        return _logistic(x)
    return x


def _threads():
    return max(1, min(32, os.cpu_count() or 1))


@dataclass
class ForwardSpec:
    """Everything that defines one seeded forward problem (cheap; draws nothing big)."""
    seed: int
    H: int
    dk: int
    dv: int
    dtype: str
    cu_seqlens: np.ndarray      # int64 [N + 1]
    A_log: np.ndarray           # float32 [H]
    with_state: bool
    g_min: float

    @property
    def T(self):
        return int(self.cu_seqlens[-1])

    @property
    def N(self):
        return self.cu_seqlens.shape[0] - 1

    def width(self, kind):
        return {"q": self.dk, "k": self.dk, "z": self.dk, "v": self.dv, "beta": None}[kind]

    def block(self, kind: str, b: int) -> np.ndarray:
        """Rounded float32 values of tensor `kind` for tokens [b*BT, min((b+1)*BT, T))."""
        t0 = b * BLOCK_TOKENS
        t1 = min(t0 + BLOCK_TOKENS, self.T)
        w = self.width(kind)
        shape = (t1 - t0, self.H) if w is None else (t1 - t0, self.H, w)
        return _round(_draw(kind, _gen(self.seed, _IDS[kind], b), shape), self.dtype)

    def n_blocks(self):
        return (self.T + BLOCK_TOKENS - 1) // BLOCK_TOKENS

    def tokens(self, kind: str, t0: int, t1: int, heads=None) -> np.ndarray:
        """Rounded float32 values for tokens [t0, t1), optionally a subset of heads."""
        hs = None if heads is None else list(heads)

        def piece(b):
            blk = self.block(kind, b)
            lo = max(t0 - b * BLOCK_TOKENS, 0)
            hi = min(t1 - b * BLOCK_TOKENS, blk.shape[0])
            blk = blk[lo:hi]
            return blk if hs is None else np.ascontiguousarray(blk[:, hs])

        blocks = range(t0 // BLOCK_TOKENS, (t1 + BLOCK_TOKENS - 1) // BLOCK_TOKENS)
        with cf.ThreadPoolExecutor(max_workers=_threads()) as ex:
            parts = list(ex.map(piece, blocks))
        if not parts:
            w = self.width(kind)
            nh = self.H if heads is None else len(list(heads))
            return np.zeros((0, nh) if w is None else (0, nh, w), dtype=np.float32)
        return np.concatenate(parts, axis=0)

    def S0(self) -> np.ndarray | None:
        if not self.with_state:
            return None
        rng = _gen(self.seed, _IDS["S0"])
        return (np.float32(0.02) * rng.standard_normal((self.N, self.H, self.dk, self.dv),
                                                       dtype=np.float32))

    # ---- whole tensors -------------------------------------------------------

    def host(self, kind: str) -> Stored:
        """The whole tensor on the host (use for problems that fit comfortably in RAM)."""
        return store(self.tokens(kind, 0, self.T), self.dtype)

    def to_device(self, device="cuda"):
        """All tensors on `device`, generated block by block in parallel host threads.

        Returns a dict of torch tensors: q, k, v, beta, z (I/O dtype), A_log, S0 (fp32 or
        None) and cu (int32 [N + 1]).
        """
        import torch
        tdt = torch.bfloat16 if self.dtype == "bf16" else torch.float32
        out = {}
        for kind in ("q", "k", "v", "beta", "z"):
            w = self.width(kind)
            shape = (self.T, self.H) if w is None else (self.T, self.H, w)
            out[kind] = torch.empty(shape, dtype=tdt, device=device)
        jobs = [(kind, b) for kind in ("q", "k", "v", "beta", "z") for b in range(self.n_blocks())]

        def make(job):
            kind, b = job
            x = self.block(kind, b)
            if self.dtype == "bf16":
                return job, torch.from_numpy(f32_to_bf16_bits(x).view(np.int16)).view(
                    torch.bfloat16)
            return job, torch.from_numpy(x)

        with cf.ThreadPoolExecutor(max_workers=_threads()) as ex:
            for (kind, b), t in ex.map(make, jobs):
                t0 = b * BLOCK_TOKENS
                out[kind][t0:t0 + t.shape[0]].copy_(t)
        out["A_log"] = torch.from_numpy(self.A_log).to(device)
        S0 = self.S0()
        out["S0"] = None if S0 is None else torch.from_numpy(S0).to(device)
        out["cu"] = torch.from_numpy(self.cu_seqlens.astype(np.int32)).to(device)
        return out


def forward_spec(*, seed: int, H: int, dk: int, dv: int, dtype: str, lengths=None, B: int = 1,
                 T: int = 0, g_min: float = -5.0, with_state: bool = False,
                 varlen_range=None) -> ForwardSpec:
    """Either explicit ``lengths``, ``varlen_range=(count, lo, hi)`` (lengths ~ U{lo..hi})
    or ``B`` equal sequences of length ``T``."""
    if varlen_range is not None:
        count, lo, hi = varlen_range
        lens = _gen(seed, _IDS["lengths"]).integers(lo, hi + 1, size=count).astype(np.int64)
    elif lengths is not None:
        lens = np.asarray(lengths, dtype=np.int64)
    else:
        lens = np.full(B, T, dtype=np.int64)
    cu = np.zeros(lens.shape[0] + 1, dtype=np.int64)
    cu[1:] = np.cumsum(lens)
    A_log = _gen(seed, _IDS["A_log"]).uniform(-1.0, 1.0, size=H).astype(np.float32)
    return ForwardSpec(seed, H, dk, dv, dtype, cu, A_log, with_state, float(g_min))


@dataclass
class ForwardInputs:
    """A problem fully materialised on the host (small and medium sizes)."""
    spec: ForwardSpec
    q: Stored
    k: Stored
    v: Stored
    beta: Stored
    z: Stored
    S0: np.ndarray | None

    def __getattr__(self, name):
        return getattr(self.spec, name)


def forward_inputs(**kw) -> ForwardInputs:
    sp = forward_spec(**kw)
    return ForwardInputs(sp, sp.host("q"), sp.host("k"), sp.host("v"), sp.host("beta"),
                         sp.host("z"), sp.S0())


# ------------------------------------------------------------------ decode --


@dataclass
class DecodeInputs:
    q: Stored
    k: Stored
    v: Stored
    beta: Stored
    z: Stored


def decode_state(*, seed: int, N: int, H: int, dk: int, dv: int):
    """Initial decode state S ~ N(0, 0.02^2) [N,H,dk,dv] float32 and A_log ~ U(-1,1) [H]."""
    A_log = _gen(seed, _IDS["A_log"]).uniform(-1.0, 1.0, size=H).astype(np.float32)
    S = np.float32(0.02) * _gen(seed, _IDS["S0"]).standard_normal((N, H, dk, dv),
                                                                   dtype=np.float32)
    return S, A_log


def decode_step_inputs(*, seed: int, step: int, N: int, H: int, dk: int, dv: int,
                       dtype: str = "bf16") -> DecodeInputs:
    """Inputs for decode step ``step``: one new token for each of N sequences."""
    out = {}
    for kind in ("q", "k", "v", "beta", "z"):
        w = {"q": dk, "k": dk, "z": dk, "v": dv, "beta": None}[kind]
        shape = (N, H) if w is None else (N, H, w)
        out[kind] = store(_draw(kind, _gen(seed, 100 + _IDS[kind], step), shape), dtype)
    return DecodeInputs(**out)


def decode_steps_iter(*, seed: int, steps: int, N: int, H: int, dk: int, dv: int,
                      dtype: str = "bf16", lookahead: int = 32):
    """Yield (step, DecodeInputs) in order, drawing upcoming steps in parallel threads."""
    with cf.ThreadPoolExecutor(max_workers=_threads()) as ex:
        futs = {}
        for step in range(steps):
            for s in range(step, min(step + lookahead, steps)):
                if s not in futs:
                    futs[s] = ex.submit(decode_step_inputs, seed=seed, step=s, N=N, H=H, dk=dk,
                                        dv=dv, dtype=dtype)
            yield step, futs.pop(step).result()


@dataclass
class OutputGateInputs:
    o: Stored                   # [T, H, dv] head outputs
    gate: Stored                # [T, H, dv] gate logits (W_g x, given)
    norm_w: np.ndarray | None   # float32 [dv], or None for unit weights


def output_gate_inputs(*, seed: int, T: int, H: int, dv: int, dtype: str,
                       with_weight: bool = True) -> OutputGateInputs:
    nb = -(-T // BLOCK_TOKENS)

    def block(kind, b):
        t0 = b * BLOCK_TOKENS
        n = min(BLOCK_TOKENS, T - t0)
        rng = _gen(seed, _IDS[kind], b)
        x = rng.standard_normal(size=(n, H, dv), dtype=np.float32)
        if kind == "o_head":
            x *= rng.uniform(0.1, 10.0, size=(n, H, 1)).astype(np.float32)
        return x

    out = {}
    for kind in ("o_head", "gate"):
        if T == 0:
            out[kind] = np.zeros((0, H, dv), dtype=np.float32)
            continue
        with cf.ThreadPoolExecutor(max_workers=_threads()) as ex:
            parts = list(ex.map(lambda b: block(kind, b), range(nb)))
        out[kind] = np.concatenate(parts, axis=0)
    w = (_gen(seed, _IDS["norm_w"]).uniform(0.5, 1.5, size=dv).astype(np.float32)
         if with_weight else None)
    return OutputGateInputs(store(out["o_head"], dtype), store(out["gate"], dtype), w)


def qb_inputs(*, seed: int, m: int, n: int, grid: float = 0.0):
    """(scores [m, n] float32, bias [n] float32) for the quantile-balancing update."""
    mu = _gen(seed, _IDS["popularity"]).normal(0.0, 0.5, size=n).astype(np.float32)
    nb = -(-m // BLOCK_TOKENS)

    def block(b):
        t0 = b * BLOCK_TOKENS
        rows = min(BLOCK_TOKENS, m - t0)
        return _gen(seed, _IDS["router"], b).standard_normal(size=(rows, n), dtype=np.float32)

    with cf.ThreadPoolExecutor(max_workers=_threads()) as ex:
        s = np.concatenate(list(ex.map(block, range(nb))), axis=0) + mu[None, :]
    bias = _gen(seed, _IDS["expert_bias"]).normal(0.0, 0.1, size=n).astype(np.float32)
    if grid:
        s = np.round(s / grid) * grid
        bias = np.round(bias / grid) * grid
    return np.ascontiguousarray(s, dtype=np.float32), bias.astype(np.float32)


# ------------------------------------------------------ the named workloads --

#: The forward workloads, by what they are.  ``seed`` = 1000 + index.
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

#: The gated output step at the long-context forward's output shape.
OUTPUT_GATE_WORKLOAD = dict(seed=1005, T=65536, H=32, dv=128, dtype="bf16")

#: Quantile balancing: one routing batch of 65536 tokens over 256 experts, 8 per token.
QB_WORKLOAD = dict(seed=1006, m=65536, n=256, k=8)

#: 256 sequences x 32 heads, one token per step for 1000 steps.
DECODE_WORKLOAD = dict(seed=1004, N=256, H=32, dk=128, dv=128, steps=1000, dtype="bf16")


def workload_spec(name: str, g_min: float = -5.0, **overrides) -> ForwardSpec:
    kw = dict(WORKLOADS[name])
    kw.update(overrides)
    return forward_spec(g_min=g_min, **kw)


def workload(name: str, g_min: float = -5.0, **overrides) -> ForwardInputs:
    kw = dict(WORKLOADS[name])
    kw.update(overrides)
    return forward_inputs(g_min=g_min, **kw)
