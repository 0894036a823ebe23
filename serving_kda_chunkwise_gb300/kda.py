"""Python binding of libkda.so: same entry-point names as include/kda.h.

Argument marshalling only -- every step of the computation runs in the library's
CUDA kernels.  Torch is used for device memory and streams.  Importing this module
loads ``_build/libkda.so`` and raises if it is missing: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# KDA_LIBRARY may name another build of the same library (e.g. an instrumented one).
LIB_PATH = os.environ.get("KDA_LIBRARY") or os.path.join(_HERE, "_build", "libkda.so")

KDA_OK, KDA_ERR_INVALID_ARG, KDA_ERR_UNSUPPORTED, KDA_ERR_CUDA, KDA_ERR_TIMEOUT, \
    KDA_ERR_DEVICE = range(6)
KDA_F32, KDA_BF16 = 0, 1

C_CHUNK = 64


class KdaError(RuntimeError):
    def __init__(self, status: int, func: str, msg: str):
        self.status = status
        super().__init__(f"{func}: {_lib.kda_status_string(status).decode()}: {msg}")


class ProfileEntry(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 32), ("launches", ctypes.c_int),
                ("total_ms", ctypes.c_double)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"libkda.so not found at {LIB_PATH}; build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'` (needs nvcc)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i64, i32, f32, sz = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float,
                             ctypes.c_size_t)
    lib.kda_version.restype = ctypes.c_int
    lib.kda_version.argtypes = []
    lib.kda_status_string.restype = ctypes.c_char_p
    lib.kda_status_string.argtypes = [ctypes.c_int]
    lib.kda_last_error.restype = ctypes.c_char_p
    lib.kda_last_error.argtypes = []
    lib.kda_gate.restype = ctypes.c_int
    lib.kda_gate.argtypes = [vp, i32, vp, f32, vp, i64, i32, i32, vp]
    lib.kda_fwd_workspace_size.restype = sz
    lib.kda_fwd_workspace_size.argtypes = [i64, i32, i32, i32, i32, i32]
    lib.kda_fwd_chunked.restype = ctypes.c_int
    lib.kda_fwd_chunked.argtypes = [vp, vp, vp, vp, vp, vp, f32, vp, vp, vp, i32, i64, i32, i32,
                                    i32, i32, vp, vp, sz, vp]
    lib.kda_decode_step.restype = ctypes.c_int
    lib.kda_decode_step.argtypes = [vp, vp, vp, vp, vp, vp, f32, vp, i32, i32, i32, i32, i32, vp,
                                    vp]
    lib.kda_output_norm_gate.restype = ctypes.c_int
    lib.kda_output_norm_gate.argtypes = [vp, vp, vp, f32, vp, i64, i32, i32, i32, vp]
    lib.kda_decode_step_gated.restype = ctypes.c_int
    lib.kda_decode_step_gated.argtypes = [vp, vp, vp, vp, vp, vp, f32, vp, vp, vp, f32, i32, i32,
                                          i32, i32, i32, vp, vp]
    lib.kda_quantile_balance_workspace_size.restype = sz
    lib.kda_quantile_balance_workspace_size.argtypes = [i64, i32]
    lib.kda_quantile_balance.restype = ctypes.c_int
    lib.kda_quantile_balance.argtypes = [vp, vp, i64, i32, i32, vp, vp, vp, vp, sz, vp]
    lib.kda_fwd_chunked_softplus.restype = ctypes.c_int
    lib.kda_fwd_chunked_softplus.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i64, i32,
                                             i32, i32, i32, vp, vp, sz, vp]
    lib.kda_bwd_workspace_size.restype = sz
    lib.kda_bwd_workspace_size.argtypes = [i64, i32, i32, i32, i32]
    lib.kda_bwd.restype = ctypes.c_int
    lib.kda_bwd.argtypes = [vp, vp, vp, vp, vp, vp, f32, vp, vp, i32, i64, i32, i32, i32, i32,
                            vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.kda_selftest_timeout.restype = ctypes.c_int
    lib.kda_selftest_timeout.argtypes = [ctypes.c_uint, vp]
    lib.kda_device_status.restype = ctypes.c_int
    lib.kda_device_status.argtypes = [vp]
    lib.kda_profile_begin.restype = ctypes.c_int
    lib.kda_profile_begin.argtypes = []
    lib.kda_profile_end.restype = ctypes.c_int
    lib.kda_profile_end.argtypes = [ctypes.POINTER(ProfileEntry), ctypes.c_int]
    return lib


_lib = _load()


def library():
    """The loaded ctypes handle (for tests that call the C ABI directly)."""
    return _lib


def _check(status: int, func: str):
    if status != KDA_OK:
        raise KdaError(status, func, _lib.kda_last_error().decode())


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return KDA_BF16
    if t.dtype == torch.float32:
        return KDA_F32
    raise TypeError(f"unsupported I/O dtype {t.dtype} (bf16 or fp32)")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need(t: torch.Tensor, name: str, dtype=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


def version() -> int:
    return _lib.kda_version()


def gate(z: torch.Tensor, A_log: torch.Tensor, g_min: float, g_out=None, stream=None):
    """g = g_min * sigmoid(exp(A_log[h]) * z), z: [T, H, dk] -> fp32 [T, H, dk]."""
    _need(z, "z")
    _need(A_log, "A_log", torch.float32)
    T, H, dk = z.shape
    if g_out is None:
        g_out = torch.empty((T, H, dk), dtype=torch.float32, device=z.device)
    _need(g_out, "g_out", torch.float32)
    _check(_lib.kda_gate(_ptr(z), _dt(z), _ptr(A_log), float(g_min), _ptr(g_out), T, H, dk,
                         _stream(stream)), "kda_gate")
    return g_out


def workspace_size(T_total: int, N: int, H: int, dk: int, dv: int, io_dtype) -> int:
    dt = KDA_BF16 if io_dtype == torch.bfloat16 else KDA_F32
    return int(_lib.kda_fwd_workspace_size(int(T_total), int(N), int(H), int(dk), int(dv), dt))


def fwd_chunked(q, k, v, beta, z, A_log, g_min: float, S0=None, cu_seqlens=None, N=None,
                o=None, S_out=None, want_state: bool = True, workspace=None, stream=None):
    """KDA forward over packed sequences (chunked form, C = 64).

    q, k, z: [T, H, dk]; v: [T, H, dv]; beta: [T, H] (all one I/O dtype);
    A_log: fp32 [H]; S0: fp32 [N, H, dk, dv] or None; cu_seqlens: int32 [N+1] on the
    device, or None with N equal sequences (N defaults to 1).
    Returns (o [T, H, dv], S_out [N, H, dk, dv] or None).
    """
    for t, nm in ((q, "q"), (k, "k"), (v, "v"), (beta, "beta"), (z, "z")):
        _need(t, nm, q.dtype)
    _need(A_log, "A_log", torch.float32)
    T, H, dk = q.shape
    dv = v.shape[2]
    if cu_seqlens is not None:
        _need(cu_seqlens, "cu_seqlens", torch.int32)
        N = cu_seqlens.shape[0] - 1
    elif N is None:
        N = 1
    if S0 is not None:
        _need(S0, "S0", torch.float32)
    if o is None:
        o = torch.empty((T, H, dv), dtype=q.dtype, device=q.device)
    _need(o, "o", q.dtype)
    if S_out is None and want_state:
        S_out = torch.empty((N, H, dk, dv), dtype=torch.float32, device=q.device)
    if S_out is not None:
        _need(S_out, "S_out", torch.float32)
    need = workspace_size(T, N, H, dk, dv, q.dtype)
    if need > 0 and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib.kda_fwd_chunked(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(z), _ptr(A_log),
                                float(g_min), _ptr(S0), _ptr(S_out), _ptr(cu_seqlens), int(N),
                                int(T), int(H), int(dk), int(dv), _dt(q), _ptr(o), _ptr(workspace),
                                ws_bytes, _stream(stream)), "kda_fwd_chunked")
    return o, S_out


_copy_streams = {}


def _streams(device):
    key = torch.device(device).index or 0
    if key not in _copy_streams:
        _copy_streams[key] = tuple(torch.cuda.Stream(device=device) for _ in range(3))
    return _copy_streams[key]


def fwd_chunked_host(q, k, v, beta, z, A_log, g_min: float, S0=None, cu_seqlens=None, N=None,
                     o=None, S_out=None, segments: int = 8, device="cuda"):
    """kda_fwd_chunked from (pinned) host tensors to (pinned) host outputs.

    Same arguments as fwd_chunked, all on the host (cu_seqlens an int32 host tensor or None).
    The work is cut into `segments` pieces and pipelined on three streams: the host-to-device
    copy of piece s + 1, the forward of piece s and the device-to-host copy of piece s - 1
    overlap.  One sequence is cut at multiples of 64 tokens, its fp32 state carried on the
    device from piece to piece (the result equals one call over the whole sequence); several
    sequences are grouped whole.  Returns (o, S_out) on the host.
    """
    T, H, dk = q.shape
    dv = v.shape[2]
    dev = torch.device(device)
    if cu_seqlens is None:
        N = 1 if N is None else int(N)
        cu = [T * n // N for n in range(N + 1)]
    else:
        cu = [int(x) for x in cu_seqlens.tolist()]
        N = len(cu) - 1
    # pieces: (first token, end token, first sequence, end sequence)
    if N == 1:
        step = -(-max(T, 1) // max(segments, 1))
        step = -(-step // C_CHUNK) * C_CHUNK
        pieces = [(a, min(a + step, T), 0, 1) for a in range(0, T, step)] or [(0, 0, 0, 1)]
    else:
        pieces, first, target = [], 0, max(T // max(segments, 1), 1)
        for n in range(1, N + 1):
            if cu[n] - cu[first] >= target or n == N:
                pieces.append((cu[first], cu[n], first, n))
                first = n
    if o is None:
        o = torch.empty((T, H, dv), dtype=q.dtype).pin_memory()
    if S_out is None:
        S_out = torch.empty((N, H, dk, dv), dtype=torch.float32).pin_memory()
    s_in, s_comp, s_out = _streams(dev)
    cur = torch.cuda.current_stream(dev)
    for s in (s_in, s_comp, s_out):
        s.wait_stream(cur)
    with torch.cuda.stream(s_in):
        dq, dk_, dv_, db, dz = (torch.empty_like(t, device=dev) for t in (q, k, v, beta, z))
        dA = A_log.to(dev, non_blocking=True)
        S = (torch.zeros((N, H, dk, dv), dtype=torch.float32, device=dev) if S0 is None
             else S0.to(dev, non_blocking=True))
        do = torch.empty((T, H, dv), dtype=q.dtype, device=dev)
        longest = max(b - a for a, b, _, _ in pieces)
        most = max(n1 - n0 for _, _, n0, n1 in pieces)
        need = workspace_size(longest, most, H, dk, dv, q.dtype)
        ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    done_in = []
    for a, b, n0, n1 in pieces:
        with torch.cuda.stream(s_in):
            for dst, src in ((dq, q), (dk_, k), (dv_, v), (db, beta), (dz, z)):
                dst[a:b].copy_(src[a:b], non_blocking=True)
            cu_d = None
            if N > 1:
                cu_d = torch.tensor([c - cu[n0] for c in cu[n0:n1 + 1]], dtype=torch.int32).to(
                    dev, non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(s_in)
            done_in.append((ev, cu_d))
    for (a, b, n0, n1), (ev, cu_d) in zip(pieces, done_in):
        s_comp.wait_event(ev)
        Sp = S[n0:n1]
        if b > a or N > 1:
            fwd_chunked(dq[a:b], dk_[a:b], dv_[a:b], db[a:b], dz[a:b], dA, g_min, S0=Sp,
                        cu_seqlens=cu_d, N=n1 - n0, o=do[a:b], S_out=Sp, workspace=ws,
                        stream=s_comp)
        ev2 = torch.cuda.Event()
        ev2.record(s_comp)
        s_out.wait_event(ev2)
        with torch.cuda.stream(s_out):
            o[a:b].copy_(do[a:b], non_blocking=True)
    with torch.cuda.stream(s_out):
        S_out.copy_(S, non_blocking=True)
    for t in (dq, dk_, dv_, db, dz, dA, S, do, ws):
        t.record_stream(s_out)
    cur.wait_stream(s_out)
    s_out.synchronize()
    return o, S_out


def fwd_chunked_softplus(q, k, v, beta, z, A_log, S0=None, cu_seqlens=None, N=None, o=None,
                         S_out=None, want_state=True, workspace=None, stream=None):
    """The chunked forward with the unbounded gate -e^A softplus(z): the mixed path (bf16,
    d = 128) or the explicit per-pair path.

    Same arguments as fwd_chunked without g_min.  Returns (o, S_out).
    """
    for t, nm in ((q, "q"), (k, "k"), (v, "v"), (beta, "beta"), (z, "z")):
        _need(t, nm, q.dtype)
    _need(A_log, "A_log", torch.float32)
    T, H, dk = q.shape
    dv = v.shape[2]
    if cu_seqlens is not None:
        _need(cu_seqlens, "cu_seqlens", torch.int32)
        N = cu_seqlens.numel() - 1
    elif N is None:
        N = 1
    if o is None:
        o = torch.empty((T, H, dv), dtype=q.dtype, device=q.device)
    if S_out is None and want_state:
        S_out = torch.empty((N, H, dk, dv), dtype=torch.float32, device=q.device)
    if S0 is not None:
        _need(S0, "S0", torch.float32)
    need = workspace_size(T, N, H, dk, dv, q.dtype)
    if need > 0 and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib.kda_fwd_chunked_softplus(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(z),
                                         _ptr(A_log), _ptr(S0), _ptr(S_out), _ptr(cu_seqlens),
                                         int(N), int(T), int(H), int(dk), int(dv), _dt(q),
                                         _ptr(o), _ptr(workspace), ws_bytes, _stream(stream)),
           "kda_fwd_chunked_softplus")
    return o, S_out


def bwd(q, k, v, beta, z, A_log, g_min: float, dout, S0=None, dS_out=None, cu_seqlens=None,
        N=None, want_dS0=True, workspace=None, stream=None):
    """Gradients of fwd_chunked's (o, S_out) for upstream gradients dout (and dS_out).

    Returns a dict: dq, dk, dv, dbeta, dz (io dtype), dA_log [H] fp32, dS0 [N,H,dk,dv] fp32.
    """
    for t, nm in ((q, "q"), (k, "k"), (v, "v"), (beta, "beta"), (z, "z"), (dout, "dout")):
        _need(t, nm, q.dtype)
    _need(A_log, "A_log", torch.float32)
    T, H, dk = q.shape
    dv = v.shape[2]
    if cu_seqlens is not None:
        _need(cu_seqlens, "cu_seqlens", torch.int32)
        N = cu_seqlens.numel() - 1
    elif N is None:
        N = 1
    for t, nm in ((S0, "S0"), (dS_out, "dS_out")):
        if t is not None:
            _need(t, nm, torch.float32)
    dev = q.device
    out = {"dq": torch.empty_like(q), "dk": torch.empty_like(k), "dv": torch.empty_like(v),
           "dbeta": torch.empty_like(beta), "dz": torch.empty_like(z),
           "dA_log": torch.empty(H, dtype=torch.float32, device=dev),
           "dS0": (torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev)
                   if want_dS0 else None)}
    need = int(_lib.kda_bwd_workspace_size(int(T), int(N), int(H), int(dk), int(dv)))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    _check(_lib.kda_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(z), _ptr(A_log),
                        float(g_min), _ptr(S0), _ptr(cu_seqlens), int(N), int(T), int(H),
                        int(dk), int(dv), _dt(q), _ptr(dout), _ptr(dS_out), _ptr(out["dq"]),
                        _ptr(out["dk"]), _ptr(out["dv"]), _ptr(out["dbeta"]), _ptr(out["dz"]),
                        _ptr(out["dA_log"]), _ptr(out["dS0"]), _ptr(workspace),
                        workspace.numel(), _stream(stream)), "kda_bwd")
    return out


def decode_step(q, k, v, beta, z, A_log, g_min: float, S, o=None, stream=None):
    """One decode token per sequence; S [N, H, dk, dv] fp32 is updated in place.

    q, k, z: [N, H, dk]; v: [N, H, dv]; beta: [N, H].  Returns o [N, H, dv].
    """
    for t, nm in ((q, "q"), (k, "k"), (v, "v"), (beta, "beta"), (z, "z")):
        _need(t, nm, q.dtype)
    _need(A_log, "A_log", torch.float32)
    _need(S, "S", torch.float32)
    N, H, dk = q.shape
    dv = v.shape[2]
    if o is None:
        o = torch.empty((N, H, dv), dtype=q.dtype, device=q.device)
    _need(o, "o", q.dtype)
    _check(_lib.kda_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(z), _ptr(A_log),
                                float(g_min), _ptr(S), int(N), int(H), int(dk), int(dv), _dt(q),
                                _ptr(o), _stream(stream)), "kda_decode_step")
    return o


def output_norm_gate(o, gate, norm_w=None, eps: float = 1e-6, y=None, stream=None):
    """y = sigmoid(gate) * norm_w * o / sqrt(mean(o^2) + eps) per (token, head) row.

    o, gate: [T, H, dv] (bf16 or fp32); norm_w: [dv] fp32 or None; y may be o (in place).
    """
    _need(o, "o")
    _need(gate, "gate", o.dtype)
    if norm_w is not None:
        _need(norm_w, "norm_w", torch.float32)
    T, H, dv = o.shape
    if y is None:
        y = torch.empty_like(o)
    _need(y, "y", o.dtype)
    _check(_lib.kda_output_norm_gate(_ptr(o), _ptr(gate), _ptr(norm_w), float(eps), _ptr(y),
                                     int(T), int(H), int(dv), _dt(o), _stream(stream)),
           "kda_output_norm_gate")
    return y


def decode_step_gated(q, k, v, beta, z, A_log, g_min: float, S, gate, norm_w=None,
                      eps: float = 1e-6, y=None, stream=None):
    """decode_step with the gated output step fused: returns y [N, H, dv] in place of o."""
    for t, nm in ((q, "q"), (k, "k"), (v, "v"), (beta, "beta"), (z, "z"), (gate, "gate")):
        _need(t, nm, q.dtype)
    _need(A_log, "A_log", torch.float32)
    _need(S, "S", torch.float32)
    if norm_w is not None:
        _need(norm_w, "norm_w", torch.float32)
    N, H, dk = q.shape
    dv = v.shape[2]
    if y is None:
        y = torch.empty((N, H, dv), dtype=q.dtype, device=q.device)
    _need(y, "y", q.dtype)
    _check(_lib.kda_decode_step_gated(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(z),
                                      _ptr(A_log), float(g_min), _ptr(S), _ptr(gate),
                                      _ptr(norm_w), float(eps), int(N), int(H), int(dk), int(dv),
                                      _dt(q), _ptr(y), _stream(stream)), "kda_decode_step_gated")
    return y


def quantile_balance(scores, bias, k: int, want_bhat=False, want_alpha=False, workspace=None,
                     stream=None):
    """Quantile-balancing bias update: returns bias_new [n] (and bhat [n], alpha [m] when
    asked).  scores: [m, n] fp32 (token-major), bias: [n] fp32."""
    _need(scores, "scores", torch.float32)
    _need(bias, "bias", torch.float32)
    m, n = scores.shape
    dev = scores.device
    b_new = torch.empty(n, dtype=torch.float32, device=dev)
    bhat = torch.empty(n, dtype=torch.float32, device=dev) if want_bhat else None
    alpha = torch.empty(m, dtype=torch.float32, device=dev) if want_alpha else None
    need = int(_lib.kda_quantile_balance_workspace_size(int(m), int(n)))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    _check(_lib.kda_quantile_balance(_ptr(scores), _ptr(bias), int(m), int(n), int(k),
                                     _ptr(b_new), _ptr(bhat), _ptr(alpha), _ptr(workspace),
                                     workspace.numel(), _stream(stream)), "kda_quantile_balance")
    out = [b_new]
    if want_bhat:
        out.append(bhat)
    if want_alpha:
        out.append(alpha)
    return out[0] if len(out) == 1 else tuple(out)


def selftest_timeout(limit_us: int = 50000, stream=None):
    """Enqueue a bounded wait that runs out (see kda_selftest_timeout in kda.h)."""
    _check(_lib.kda_selftest_timeout(int(limit_us), _stream(stream)), "kda_selftest_timeout")


def device_status(stream=None):
    """Wait for the stream and raise if a kernel flagged malformed input or a timeout."""
    _check(_lib.kda_device_status(_stream(stream)), "kda_device_status")


def profile_begin():
    """Start bracketing every library kernel launch with CUDA events (see kda.h)."""
    _check(_lib.kda_profile_begin(), "kda_profile_begin")


def profile_end(max_entries: int = 64):
    """Stop recording; return {kernel name: (launches, total device ms)}."""
    arr = (ProfileEntry * max_entries)()
    n = _lib.kda_profile_end(arr, max_entries)
    if n < 0:
        raise KdaError(KDA_ERR_CUDA, "kda_profile_end", "a CUDA event call failed")
    return {arr[i].name.decode(): (arr[i].launches, arr[i].total_ms) for i in range(n)}
