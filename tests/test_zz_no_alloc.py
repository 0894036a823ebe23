"""kda_fwd_chunked_noalloc: the forward for callers that cannot allocate device memory.

Such callers (a runtime that owns all GPU memory, a plugin barred from the CUDA allocator)
get their scratch from a fixed buffer inside libkda.so instead of a workspace argument.
This file is collected last so that a stop-at-first-failure run has run every other test
before it.  It calls the entry point through the C ABI twice in a row, on different inputs,
and requires each result to be bitwise equal to kda_fwd_chunked's on the same inputs (the
same kernels run, so the results must be identical; the bf16 parity rule is checked as
well).  A problem that needs no scratch (fp32 I/O, d = 64) takes the same entry point too.
The rejection of problems larger than the buffer needs no GPU and is tested in
test_abi.py.
"""
import ctypes

import numpy as np
import pytest

from serving_kda_chunkwise_gb300 import inputs
from kda_testutil import (BF16_NORM_TOL, BF16_RMS_TOL, bf16_norm_err, bf16_rms_err,
                          device_inputs, state_err)

pytestmark = pytest.mark.gpu


def _noalloc(lib, d, inp, o, S_out, stream, d_head=128, io_dt=1):
    f = lib.kda_fwd_chunked_noalloc
    f.restype = ctypes.c_int
    vp = ctypes.c_void_p
    f.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.c_float, vp, vp, vp, ctypes.c_int,
                  ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp]
    p = lambda t: None if t is None else vp(t.data_ptr())
    return f(p(d["q"]), p(d["k"]), p(d["v"]), p(d["beta"]), p(d["z"]), p(d["A_log"]),
             inp.g_min, p(d["S0"]), p(S_out), p(d["cu"]), inp.N, inp.T, inp.H, d_head, d_head,
             io_dt, p(o), vp(stream.cuda_stream))


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
        assert torch.equal(o, o_ref) and torch.equal(S, S_ref), "noalloc differs from the workspace entry point"
        o_n, o_r = o.float().cpu().numpy(), o_ref.float().cpu().numpy().astype(np.float64)
        S_n, S_r = S.cpu().numpy(), S_ref.cpu().numpy().astype(np.float64)
        for n in range(inp.N):
            a, b = inp.cu_seqlens[n], inp.cu_seqlens[n + 1]
            for h in range(inp.H):
                assert bf16_norm_err(o_n[a:b, h], o_r[a:b, h]) <= BF16_NORM_TOL
                assert bf16_rms_err(o_n[a:b, h], o_r[a:b, h]) <= BF16_RMS_TOL
                assert state_err(S_n[n, h], S_r[n, h]) <= BF16_NORM_TOL


def test_noalloc_without_scratch_fp32():
    """fp32 I/O at d = 64 selects kernels that need no scratch: the call forwards directly."""
    import torch
    from serving_kda_chunkwise_gb300 import kda
    lib = kda.library()
    stream = torch.cuda.current_stream()
    inp = inputs.forward_inputs(seed=303, lengths=[100, 37], H=3, dk=64, dv=64, dtype="f32",
                                with_state=True)
    d = device_inputs(inp)
    o_ref, S_ref = kda.fwd_chunked(d["q"], d["k"], d["v"], d["beta"], d["z"], d["A_log"],
                                   inp.g_min, S0=d["S0"], cu_seqlens=d["cu"])
    o = torch.empty_like(o_ref)
    S = torch.empty_like(S_ref)
    rc = _noalloc(lib, d, inp, o, S, stream, d_head=64, io_dt=0)
    assert rc == 0, lib.kda_last_error()
    kda.device_status()
    assert torch.equal(o, o_ref) and torch.equal(S, S_ref)
