"""kda_fwd_chunked_noalloc: the forward for callers that cannot allocate device memory.

Such callers (a runtime that owns all GPU memory, a plugin barred from the CUDA allocator)
get their scratch from a fixed buffer inside libkda.so instead of a workspace argument.
This file is collected last so that a stop-at-first-failure run has run every other test
before it.  It calls the entry point through the C ABI twice in a row, on different inputs,
and holds each result to the parity rule of the other bf16 tests against kda_fwd_chunked
on the same inputs.
"""
import ctypes

import numpy as np
import pytest

from serving_kda_chunkwise_gb300 import inputs
from kda_testutil import (BF16_NORM_TOL, BF16_RMS_TOL, bf16_norm_err, bf16_rms_err,
                          device_inputs)

pytestmark = pytest.mark.gpu


def _noalloc(lib, d, inp, o, S_out, stream):
    f = lib.kda_fwd_chunked_noalloc
    f.restype = ctypes.c_int
    vp = ctypes.c_void_p
    f.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.c_float, vp, vp, vp, ctypes.c_int,
                  ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp]
    p = lambda t: None if t is None else vp(t.data_ptr())
    return f(p(d["q"]), p(d["k"]), p(d["v"]), p(d["beta"]), p(d["z"]), p(d["A_log"]),
             inp.g_min, p(d["S0"]), p(S_out), p(d["cu"]), inp.N, inp.T, inp.H, 128, 128, 1,
             p(o), vp(stream.cuda_stream))


def test_noalloc_matches_workspace_entry_point_twice():
    import torch
    from serving_kda_chunkwise_gb300 import kda
    lib = kda.library()
    stream = torch.cuda.current_stream()
    for seed, lens in ((101, [300, 77, 130]), (202, [64, 1, 190, 255])):
        inp = inputs.forward_inputs(seed=seed, lengths=lens, H=4, dk=128, dv=128, dtype="bf16",
                                    with_state=True)
        d = device_inputs(inp)
        o_ref, S_ref = kda.fwd_chunked(d["q"], d["k"], d["v"], d["beta"], d["z"], d["A_log"],
                                       inp.g_min, S0=d["S0"], cu_seqlens=d["cu"])
        o = torch.empty_like(o_ref)
        S = torch.empty_like(S_ref)
        rc = _noalloc(lib, d, inp, o, S, stream)
        assert rc == 0, lib.kda_last_error()
        kda.device_status()
        o_n, o_r = o.float().cpu().numpy(), o_ref.float().cpu().numpy().astype(np.float64)
        S_n, S_r = S.cpu().numpy(), S_ref.cpu().numpy().astype(np.float64)
        for n in range(inp.N):
            a, b = inp.cu_seqlens[n], inp.cu_seqlens[n + 1]
            for h in range(inp.H):
                assert bf16_norm_err(o_n[a:b, h], o_r[a:b, h]) <= BF16_NORM_TOL
                assert bf16_rms_err(o_n[a:b, h], o_r[a:b, h]) <= BF16_RMS_TOL
                assert bf16_norm_err(S_n[n, h], S_r[n, h]) <= BF16_NORM_TOL


def test_noalloc_rejects_problems_beyond_its_buffer():
    from serving_kda_chunkwise_gb300 import kda
    lib = kda.library()
    vp = ctypes.c_void_p
    f = lib.kda_fwd_chunked_noalloc
    f.restype = ctypes.c_int
    a = vp(0x10000)
    # T = 65536 tokens x 32 heads needs far more than 64 MiB of scratch
    rc = f(a, a, a, a, a, a, ctypes.c_float(-5.0), None, None, None, 1, ctypes.c_int64(65536),
           32, 128, 128, 1, a, None)
    assert rc == kda.KDA_ERR_INVALID_ARG
    lib.kda_last_error.restype = ctypes.c_char_p
    assert b"built into the library" in lib.kda_last_error()
