"""Shared helpers for the parity tests: move seeded inputs to the device, run the
oracle on (a sample of) the same inputs, and apply the tolerances.

Tolerances (written here once, used by every parity test):
  fp32 I/O  per (sequence, head):  ||o_gpu - o_ref||_F / ||o_ref||_F <= 1e-4, same for S_out.
  bf16 I/O  per (sequence, head), after dividing both outputs by rms(o_ref) over all
            (token, channel) of that (sequence, head):
              |o_gpu - o_ref| <= 2e-2 + 2^-8 |o_ref|   for every element, and
              rms(o_gpu - o_ref) <= 1e-2.
            2e-2 is the stated absolute figure.  2^-8 |o_ref| bounds half a bf16 ulp of the
            reference value: the output is stored in bf16, and one correct rounding of the
            exact result moves it by up to that much (the outputs are heavy-tailed,
            max|o| / rms ~ 20 per head, so the rounded exact answer alone can exceed 2e-2
            of rms; see test_tolerance_reading.py).  Nothing else is allowed beyond 2e-2.
            The rms bound catches errors that are systematic across a head even when each
            element stays inside the band.
            The fp32 final state of a bf16 problem is not rounded on output, so it gets no
            relative term: max|S_gpu - S_ref| <= 2e-2 rms(S_ref) and
            rms(S_gpu - S_ref) <= 1e-2 rms(S_ref).
"""
from __future__ import annotations

import numpy as np

FP32_REL_TOL = 1e-4
BF16_NORM_TOL = 2e-2
BF16_RTOL = 2.0 ** -8
BF16_RMS_TOL = 1e-2


def bf16_norm_err(o_gpu, o_ref):
    """Largest (|o_gpu - o_ref| - 2^-8 |o_ref|) / rms(o_ref): must be <= 2e-2."""
    if o_ref.size == 0:
        return 0.0
    rms = max(np.sqrt(np.mean(o_ref ** 2)), 1e-30)
    excess = np.abs(o_gpu - o_ref) - BF16_RTOL * np.abs(o_ref)
    return float(max(np.max(excess), 0.0) / rms)


def bf16_rms_err(o_gpu, o_ref):
    """rms(o_gpu - o_ref) / rms(o_ref)."""
    if o_ref.size == 0:
        return 0.0
    return float(np.sqrt(np.mean((o_gpu - o_ref) ** 2)) / max(np.sqrt(np.mean(o_ref ** 2)),
                                                                1e-30))


def plain_norm_err(o_gpu, o_ref):
    """max |o_gpu - o_ref| / rms(o_ref): the reading that bf16 rounding alone can fail."""
    if o_ref.size == 0:
        return 0.0
    return float(np.max(np.abs(o_gpu - o_ref)) / max(np.sqrt(np.mean(o_ref ** 2)), 1e-30))


def state_err(S_gpu, S_ref):
    """max |S_gpu - S_ref| / rms(S_ref) for the fp32 final state: must be <= 2e-2."""
    return plain_norm_err(np.asarray(S_gpu, np.float64), np.asarray(S_ref, np.float64))


def _spec(x):
    return getattr(x, "spec", x)


def device_inputs(inp, device="cuda"):
    """Device tensors for a ForwardInputs (host arrays) or a ForwardSpec (drawn in blocks)."""
    import torch
    if hasattr(inp, "spec"):
        d = dict(q=inp.q.as_torch(device), k=inp.k.as_torch(device), v=inp.v.as_torch(device),
                 beta=inp.beta.as_torch(device), z=inp.z.as_torch(device),
                 A_log=torch.from_numpy(inp.A_log).to(device))
        d["S0"] = None if inp.S0 is None else torch.from_numpy(inp.S0).to(device)
        d["cu"] = torch.from_numpy(inp.cu_seqlens.astype(np.int32)).to(device)
        return d
    return inp.to_device(device)


def gpu_forward(inp, use_cu=True, want_state=True, **kw):
    from serving_kda_chunkwise_gb300 import kda
    d = device_inputs(inp)
    sp = _spec(inp)
    o, S = kda.fwd_chunked(d["q"], d["k"], d["v"], d["beta"], d["z"], d["A_log"], sp.g_min,
                           S0=d["S0"], cu_seqlens=d["cu"] if use_cu else None,
                           N=None if use_cu else sp.N, want_state=want_state, **kw)
    o = o.float().cpu().numpy()
    S = None if S is None else S.cpu().numpy()
    del d
    return o, S


def oracle_forward(inp, seqs=None, heads=None, nthreads=None, gate="sigmoid"):
    """Oracle on the exact stored inputs, optionally restricted to some sequences/heads.

    Returns dict {(n, h): (o [len, dv], S [dk, dv])} in float64.
    """
    import oracle
    sp = _spec(inp)
    host = inp if hasattr(inp, "spec") else None
    cu = sp.cu_seqlens
    seqs = range(sp.N) if seqs is None else seqs
    hs = list(range(sp.H) if heads is None else heads)
    S0_all = host.S0 if host is not None else sp.S0()
    out = {}
    for n in seqs:
        a, b = int(cu[n]), int(cu[n + 1])
        if host is not None:
            t = {kind: getattr(host, kind).values[a:b][:, hs] for kind in ("q", "k", "v", "beta", "z")}
        else:
            t = {kind: sp.tokens(kind, a, b, hs) for kind in ("q", "k", "v", "beta", "z")}
        S0 = None if S0_all is None else S0_all[n:n + 1][:, hs]
        o, S = oracle.recurrent(t["q"], t["k"], t["v"], t["beta"], t["z"], sp.A_log[hs], sp.g_min,
                                S0=S0, nthreads=nthreads, gate=gate)
        for ii, h in enumerate(hs):
            out[(n, h)] = (o[:, ii], S[0, ii])
    return out


def check_head(o_gpu, o_ref, S_gpu, S_ref, dtype, what=""):
    """Apply the tolerance to one (sequence, head); returns the two error figures."""
    o_gpu = np.asarray(o_gpu, dtype=np.float64)
    assert np.all(np.isfinite(o_gpu)), f"{what}: non-finite output"
    if dtype == "f32":
        eo = np.linalg.norm(o_gpu - o_ref) / max(np.linalg.norm(o_ref), 1e-30)
        es = 0.0
        if S_ref is not None:
            es = np.linalg.norm(S_gpu - S_ref) / max(np.linalg.norm(S_ref), 1e-30)
        assert eo <= FP32_REL_TOL, f"{what}: output rel err {eo:.3e} > {FP32_REL_TOL}"
        assert es <= FP32_REL_TOL, f"{what}: state rel err {es:.3e} > {FP32_REL_TOL}"
        return eo, es
    eo = bf16_norm_err(o_gpu, o_ref)
    er = bf16_rms_err(o_gpu, o_ref)
    assert er <= BF16_RMS_TOL, f"{what}: normalised rms err {er:.3e} > {BF16_RMS_TOL}"
    es = 0.0
    if S_ref is not None:
        es = state_err(S_gpu, S_ref)
        ers = bf16_rms_err(np.asarray(S_gpu, np.float64), S_ref)
        assert ers <= BF16_RMS_TOL, f"{what}: normalised state rms err {ers:.3e}"
    assert eo <= BF16_NORM_TOL, f"{what}: normalised output err {eo:.3e} > {BF16_NORM_TOL}"
    assert es <= BF16_NORM_TOL, f"{what}: normalised state err {es:.3e} > {BF16_NORM_TOL}"
    return eo, es


def check_forward(inp, o_gpu, S_gpu, ref, check_state=True):
    worst = (0.0, 0.0)
    inp = _spec(inp)
    cu = inp.cu_seqlens
    for (n, h), (o_ref, S_ref) in ref.items():
        a, b = int(cu[n]), int(cu[n + 1])
        e = check_head(o_gpu[a:b, h], o_ref, None if not check_state else S_gpu[n, h],
                       S_ref if check_state else None, inp.dtype, what=f"seq {n} head {h}")
        worst = (max(worst[0], e[0]), max(worst[1], e[1]))
    return worst
