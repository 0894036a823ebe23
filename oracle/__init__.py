"""fp64 CPU oracle for Kimi Delta Attention (KDA) -- test infrastructure only.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product (the CUDA library under
``serving_kda_chunkwise_gb300``) never does, and this package never imports the
product.  The arithmetic lives in ``kda_oracle.c`` (plain C, fp64); this module
only compiles it with gcc and marshals numpy arrays into it.

What it computes, and the page each step follows, is written at the top of
``kda_oracle.c``:  the token-by-token KDA recurrence and, independently, the
chunkwise-parallel form with an explicit forward-substitution inverse, plus the
lower-bounded sigmoid gate and the gated, RMS-normalised output step.  The
quantile-balancing bias update of the mixture-of-experts router is plain numpy, in
``oracle/quantile_balance.py``; the gradients of the forward are fp64 torch reverse-mode
differentiation of the token recurrence, in ``oracle/kda_backward.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libkda_oracle.so")
_lib = None
_lock = threading.Lock()

_dp = ctypes.POINTER(ctypes.c_double)
_i64p = ctypes.POINTER(ctypes.c_int64)


def build(force: bool = False) -> str:
    """Compile kda_oracle.c into a shared library (plain gcc, -O2, no fast-math)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fno-fast-math",
               "-ffp-contract=off", "-o", tmp, _SRC, "-lm", "-lpthread"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.kda_oracle_gate_value.restype = ctypes.c_double
            lib.kda_oracle_gate_value.argtypes = [ctypes.c_double] * 3
            lib.kda_oracle_gate.restype = None
            lib.kda_oracle_gate.argtypes = [_dp, _dp, ctypes.c_double, _dp,
                                            ctypes.c_int64, ctypes.c_int, ctypes.c_int]
            lib.kda_oracle_gate_softplus_value.restype = ctypes.c_double
            lib.kda_oracle_gate_softplus_value.argtypes = [ctypes.c_double] * 2
            common = [_dp, _dp, _dp, _dp, _dp, _dp, ctypes.c_double, ctypes.c_int, _dp, _dp,
                      _i64p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int]
            lib.kda_oracle_recurrent.restype = ctypes.c_int
            lib.kda_oracle_recurrent.argtypes = common + [_dp, ctypes.c_int]
            lib.kda_oracle_chunked.restype = ctypes.c_int
            lib.kda_oracle_chunked.argtypes = common + [ctypes.c_int, _dp, ctypes.c_int]
            lib.kda_oracle_output_norm_gate.restype = None
            lib.kda_oracle_output_norm_gate.argtypes = [_dp, _dp, _dp, ctypes.c_double, _dp,
                                                        ctypes.c_int64, ctypes.c_int]
            _lib = lib
    return _lib


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_dp)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def gate(z, A_log, g_min: float) -> np.ndarray:
    """g = g_min * sigmoid(exp(A_log[h]) * z) for z of shape [T, H, dk]."""
    z = _f64(z)
    A_log = _f64(A_log)
    T, H, dk = z.shape
    g = np.empty_like(z)
    _load().kda_oracle_gate(_ptr(z), _ptr(A_log), float(g_min), _ptr(g), T, H, dk)
    return g


def gate_value(z: float, A_log: float, g_min: float) -> float:
    return float(_load().kda_oracle_gate_value(float(z), float(A_log), float(g_min)))


def output_norm_gate(o, gate, w=None, eps: float = 1e-6) -> np.ndarray:
    """sigmoid(gate) * w * o / sqrt(mean(o^2) + eps), the mean over the last axis (dv).

    o, gate: [..., dv] (one row per (token, head)); w: [dv] or None (ones).
    """
    o = _f64(o)
    gate = _f64(gate)
    assert gate.shape == o.shape
    dv = o.shape[-1]
    n_rows = o.size // dv if dv else 0
    wc = None if w is None else _f64(w)
    if wc is not None:
        assert wc.shape == (dv,)
    y = np.empty_like(o)
    if n_rows:
        _load().kda_oracle_output_norm_gate(_ptr(o), _ptr(gate), _ptr(wc), float(eps), _ptr(y),
                                            n_rows, dv)
    return y


GATES = {"sigmoid": 0, "softplus": 1}


def gate_softplus_value(z: float, A_log: float) -> float:
    """g = -e^{A_log} softplus(z): the gate the lower bound replaces."""
    return float(_load().kda_oracle_gate_softplus_value(float(z), float(A_log)))


def _run(mode, q, k, v, beta, z, A_log, g_min, S0=None, cu_seqlens=None, C=64,
         nthreads=None, want_state=True, gate="sigmoid"):
    q, k, v, beta, z, A_log = (_f64(x) for x in (q, k, v, beta, z, A_log))
    T, H, dk = q.shape
    dv = v.shape[2]
    assert k.shape == (T, H, dk) and z.shape == (T, H, dk)
    assert v.shape == (T, H, dv) and beta.shape == (T, H) and A_log.shape == (H,)
    if cu_seqlens is None:
        cu = np.array([0, T], dtype=np.int64)
    else:
        cu = np.ascontiguousarray(cu_seqlens, dtype=np.int64)
    N = cu.shape[0] - 1
    assert cu[-1] == T
    S0c = None if S0 is None else _f64(S0)
    if S0c is not None:
        assert S0c.shape == (N, H, dk, dv)
    o = np.zeros((T, H, dv), dtype=np.float64)
    S_out = np.zeros((N, H, dk, dv), dtype=np.float64) if want_state else None
    nt = default_threads() if nthreads is None else int(nthreads)
    lib = _load()
    args = [_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(z), _ptr(A_log), float(g_min),
            GATES[gate], _ptr(S0c), _ptr(S_out), cu.ctypes.data_as(_i64p), N, H, dk, dv]
    if mode == "recurrent":
        rc = lib.kda_oracle_recurrent(*args, _ptr(o), nt)
    else:
        rc = lib.kda_oracle_chunked(*args, int(C), _ptr(o), nt)
    if rc != 0:
        raise ValueError(f"oracle rejected its arguments (code {rc})")
    return o, S_out


def recurrent(q, k, v, beta, z, A_log, g_min, S0=None, cu_seqlens=None, nthreads=None,
              want_state=True, gate="sigmoid"):
    """Token-by-token KDA.  Returns (o [T,H,dv], S_out [N,H,dk,dv]) in float64.

    gate: "sigmoid" (g_min * sigmoid(e^A z)) or "softplus" (-e^A softplus(z); g_min unused).
    """
    return _run("recurrent", q, k, v, beta, z, A_log, g_min, S0, cu_seqlens,
                nthreads=nthreads, want_state=want_state, gate=gate)


def chunked(q, k, v, beta, z, A_log, g_min, S0=None, cu_seqlens=None, C=64, nthreads=None,
            want_state=True, gate="sigmoid"):
    """The same result through the chunkwise-parallel form (chunk length C)."""
    return _run("chunked", q, k, v, beta, z, A_log, g_min, S0, cu_seqlens, C=C,
                nthreads=nthreads, want_state=want_state, gate=gate)


def decode_steps(S, q, k, v, beta, z, A_log, g_min, nthreads=None):
    """One decode step for N independent sequences (a length-1 recurrence each).

    S: [N,H,dk,dv]; q,k,z: [N,H,dk]; v: [N,H,dv]; beta: [N,H].
    Returns (o [N,H,dv], S_new [N,H,dk,dv]).
    """
    N = q.shape[0]
    cu = np.arange(N + 1, dtype=np.int64)
    return recurrent(q, k, v, beta, z, A_log, g_min, S0=S, cu_seqlens=cu, nthreads=nthreads)
