"""The C ABI without a GPU: libkda.so loads, exports every function include/kda.h declares,
and rejects malformed arguments on the host before any CUDA work is enqueued."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")


@pytest.fixture(scope="module")
def lib():
    from serving_kda_chunkwise_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert "kda_fwd_chunked" in names and "kda_decode_step" in names and "kda_gate" in names
    for n in names:
        assert hasattr(lib, n), f"libkda.so does not export {n}"


def test_status_strings_and_version(lib):
    lib.kda_status_string.restype = ctypes.c_char_p
    assert lib.kda_status_string(0) == b"KDA_OK"
    assert lib.kda_status_string(2) == b"KDA_ERR_UNSUPPORTED"
    assert lib.kda_version() >= 100


def _fwd(lib, **over):
    vp = ctypes.c_void_p
    aligned = vp(0x10000)
    args = dict(q=aligned, k=aligned, v=aligned, beta=aligned, z=aligned, A_log=aligned,
                g_min=ctypes.c_float(-5.0), S0=None, S_out=None, cu=None, N=1,
                T=ctypes.c_int64(128), H=2, dk=128, dv=128, dt=1, o=aligned, ws=None,
                ws_bytes=ctypes.c_size_t(0), stream=None)
    args.update(over)
    lib.kda_fwd_chunked.restype = ctypes.c_int
    lib.kda_last_error.restype = ctypes.c_char_p
    rc = lib.kda_fwd_chunked(args["q"], args["k"], args["v"], args["beta"], args["z"],
                             args["A_log"], args["g_min"], args["S0"], args["S_out"], args["cu"],
                             args["N"], args["T"], args["H"], args["dk"], args["dv"], args["dt"],
                             args["o"], args["ws"], args["ws_bytes"], args["stream"])
    return rc, lib.kda_last_error().decode()


def test_fwd_argument_validation(lib):
    vp = ctypes.c_void_p
    cases = [
        (dict(q=None), 1, "q is NULL"),
        (dict(k=vp(0x10004)), 1, "16-byte"),
        (dict(g_min=ctypes.c_float(0.0)), 1, "g_min"),
        (dict(g_min=ctypes.c_float(float("nan"))), 1, "g_min"),
        (dict(dk=96), 2, "only 64 and 128"),
        (dict(dv=32), 2, "only 64 and 128"),
        (dict(dk=0), 1, "positive"),
        (dict(H=0), 1, "H=0"),
        (dict(N=-1), 1, "N=-1"),
        (dict(N=3), 1, "multiple of N"),
        (dict(T=ctypes.c_int64(-1)), 1, "T_total"),
        (dict(dt=7), 1, "kda_dtype_t"),
        (dict(S0=vp(0x10008)), 1, "S0 is not 16-byte aligned"),
    ]
    for over, code, frag in cases:
        rc, msg = _fwd(lib, **over)
        assert rc == code, (over, rc, msg)
        assert frag in msg, (over, msg)
    # nothing to do is not an error and touches no device
    rc, msg = _fwd(lib, N=0, T=ctypes.c_int64(0))
    assert rc == 0, msg


def test_decode_and_gate_validation(lib):
    vp = ctypes.c_void_p
    a = vp(0x10000)
    lib.kda_decode_step.restype = ctypes.c_int
    lib.kda_last_error.restype = ctypes.c_char_p
    rc = lib.kda_decode_step(a, a, a, a, a, a, ctypes.c_float(-5.0), None, 4, 2, 128, 128, 1, a,
                             None)
    assert rc == 1 and b"S is NULL" in lib.kda_last_error()
    rc = lib.kda_decode_step(a, a, a, a, a, a, ctypes.c_float(1.0), a, 4, 2, 128, 128, 1, a, None)
    assert rc == 1
    rc = lib.kda_decode_step(a, a, a, a, a, a, ctypes.c_float(-5.0), a, 4, 2, 64, 96, 1, a, None)
    assert rc == 2
    lib.kda_gate.restype = ctypes.c_int
    rc = lib.kda_gate(a, 1, a, ctypes.c_float(-5.0), a, ctypes.c_int64(10), 2, 6, None)
    assert rc == 1 and b"multiple of 4" in lib.kda_last_error()
    rc = lib.kda_gate(a, 1, a, ctypes.c_float(-5.0), None, ctypes.c_int64(10), 2, 8, None)
    assert rc == 1 and b"g_out is NULL" in lib.kda_last_error()
    rc = lib.kda_gate(None, 1, None, ctypes.c_float(-5.0), None, ctypes.c_int64(0), 2, 8, None)
    assert rc == 0


def test_workspace_size_needs_no_device(lib):
    lib.kda_fwd_workspace_size.restype = ctypes.c_size_t
    lib.kda_fwd_workspace_size.argtypes = [ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_int, ctypes.c_int]
    for dt in (0, 1):
        n = lib.kda_fwd_workspace_size(65536, 1, 32, 128, 128, dt)
        assert n >= 0


def test_output_gate_validation(lib):
    vp, f = ctypes.c_void_p, ctypes.c_float
    a = vp(0x10000)
    lib.kda_output_norm_gate.restype = ctypes.c_int
    lib.kda_decode_step_gated.restype = ctypes.c_int
    lib.kda_last_error.restype = ctypes.c_char_p
    i64 = ctypes.c_int64
    # o, gate, norm_w, eps, y, n_tokens, H, dv, io_dt, stream
    assert lib.kda_output_norm_gate(a, a, None, f(1e-6), a, i64(4), 2, 96, 1, None) == 2
    assert lib.kda_output_norm_gate(a, a, None, f(-1.0), a, i64(4), 2, 128, 1, None) == 1
    assert b"eps" in lib.kda_last_error()
    assert lib.kda_output_norm_gate(a, None, None, f(1e-6), a, i64(4), 2, 128, 1, None) == 1
    assert b"gate is NULL" in lib.kda_last_error()
    assert lib.kda_output_norm_gate(a, a, vp(0x10004), f(1e-6), a, i64(4), 2, 128, 1, None) == 1
    assert b"norm_w is not 16-byte aligned" in lib.kda_last_error()
    assert lib.kda_output_norm_gate(None, None, None, f(0.0), None, i64(0), 2, 64, 0, None) == 0
    # q, k, v, beta, z, A_log, g_min, S, gate, norm_w, eps, N, H, dk, dv, io_dt, y, stream
    rc = lib.kda_decode_step_gated(a, a, a, a, a, a, f(-5.0), a, None, None, f(1e-6), 4, 2, 128,
                                   128, 1, a, None)
    assert rc == 1 and b"gate is NULL" in lib.kda_last_error()
    rc = lib.kda_decode_step_gated(a, a, a, a, a, a, f(-5.0), a, a, None, f(float("nan")), 4, 2,
                                   128, 128, 1, a, None)
    assert rc == 1 and b"eps" in lib.kda_last_error()
    rc = lib.kda_decode_step_gated(a, a, a, a, a, a, f(-5.0), a, a, None, f(1e-6), 4, 2, 128, 96,
                                   1, a, None)
    assert rc == 2


def test_quantile_balance_validation(lib):
    vp = ctypes.c_void_p
    a = vp(0x10000)
    i64 = ctypes.c_int64
    lib.kda_quantile_balance.restype = ctypes.c_int
    lib.kda_quantile_balance_workspace_size.restype = ctypes.c_size_t
    lib.kda_last_error.restype = ctypes.c_char_p
    need = lib.kda_quantile_balance_workspace_size(i64(1000), 64)
    assert need >= 1000 * 4 + 64 * 256 * 4
    # scores, bias, m, n, k, bias_new, bhat, alpha, workspace, ws_bytes, stream
    rc = lib.kda_quantile_balance(a, a, i64(1000), 2000, 8, a, None, None, a,
                                  ctypes.c_size_t(need), None)
    assert rc == 1 and b"n=2000" in lib.kda_last_error()
    rc = lib.kda_quantile_balance(a, a, i64(1000), 64, 64, a, None, None, a,
                                  ctypes.c_size_t(need), None)
    assert rc == 1 and b"k=64" in lib.kda_last_error()
    rc = lib.kda_quantile_balance(a, a, i64(1000), 64, 8, a, None, None, a,
                                  ctypes.c_size_t(need - 1), None)
    assert rc == 1 and b"workspace" in lib.kda_last_error()
    rc = lib.kda_quantile_balance(a, a, i64(0), 64, 8, a, None, None, a,
                                  ctypes.c_size_t(need), None)
    assert rc == 1


def test_softplus_forward_validation(lib):
    vp = ctypes.c_void_p
    a = vp(0x10000)
    i64 = ctypes.c_int64
    lib.kda_fwd_chunked_softplus.restype = ctypes.c_int
    lib.kda_last_error.restype = ctypes.c_char_p
    sz = ctypes.c_size_t
    # q, k, v, beta, z, A_log, S0, S_out, cu, N, T, H, dk, dv, io_dt, o, workspace, ws, stream
    rc = lib.kda_fwd_chunked_softplus(a, a, a, a, a, a, None, None, None, 1, i64(64), 2, 96,
                                      128, 1, a, None, sz(0), None)
    assert rc == 2
    rc = lib.kda_fwd_chunked_softplus(a, a, a, a, None, a, None, None, None, 1, i64(64), 2, 128,
                                      128, 1, a, None, sz(0), None)
    assert rc == 1 and b"z is NULL" in lib.kda_last_error()
    rc = lib.kda_fwd_chunked_softplus(a, a, a, a, a, a, None, None, None, 3, i64(64), 2, 128,
                                      128, 1, a, None, sz(0), None)
    assert rc == 1 and b"multiple of N" in lib.kda_last_error()
    # bf16, d = 128 (the mixed path) needs the forward's workspace
    lib.kda_fwd_workspace_size.restype = ctypes.c_size_t
    need = lib.kda_fwd_workspace_size(i64(64), 1, 2, 128, 128, 1)
    assert need > 0
    rc = lib.kda_fwd_chunked_softplus(a, a, a, a, a, a, None, None, None, 1, i64(64), 2, 128,
                                      128, 1, a, None, sz(0), None)
    assert rc == 1 and b"workspace is NULL" in lib.kda_last_error()
    rc = lib.kda_fwd_chunked_softplus(a, a, a, a, a, a, None, None, None, 1, i64(64), 2, 128,
                                      128, 1, a, a, sz(need - 1), None)
    assert rc == 1 and b"smaller than" in lib.kda_last_error()


def test_bwd_validation(lib):
    vp = ctypes.c_void_p
    a = vp(0x10000)
    i64, f = ctypes.c_int64, ctypes.c_float
    lib.kda_bwd.restype = ctypes.c_int
    lib.kda_bwd_workspace_size.restype = ctypes.c_size_t
    lib.kda_last_error.restype = ctypes.c_char_p
    need = lib.kda_bwd_workspace_size(i64(640), 2, 4, 128, 128)
    # per (chunk, head): the checkpoint, Psi and the end gradient [dk][dv] and Phi [dk][dk],
    # fp32, for the T/64 + N chunks the layout provisions
    assert need >= (640 // 64 + 2) * 4 * (3 * 128 * 128 + 128 * 128) * 4
    assert (lib.kda_bwd_workspace_size(i64(640), 2, 4, 64, 128)
            >= (640 // 64 + 2) * 4 * (3 * 64 * 128 + 64 * 64) * 4)
    assert lib.kda_bwd_workspace_size(i64(640), 2, 4, 96, 128) == 0

    def call(**kw):
        args = dict(q=a, k=a, v=a, beta=a, z=a, A=a, gmin=f(-5.0), S0=None, cu=None, N=2,
                    T=i64(640), H=4, dk=128, dv=128, dt=1, do=a, dS=None, dq=a, dkk=a, dvv=a,
                    db=a, dz=a, dA=a, dS0=None, ws=a, wsb=ctypes.c_size_t(need))
        args.update(kw)
        return lib.kda_bwd(*args.values(), None)

    assert call(dk=96) == 2
    assert call(gmin=f(0.5)) == 1
    assert call(do=None) == 1 and b"dout is NULL" in lib.kda_last_error()
    assert call(wsb=ctypes.c_size_t(need - 1)) == 1 and b"workspace" in lib.kda_last_error()
    assert call(T=i64(641)) == 1 and b"multiple of N" in lib.kda_last_error()


def _noalloc(lib, **over):
    vp = ctypes.c_void_p
    a = vp(0x10000)
    args = dict(q=a, k=a, v=a, beta=a, z=a, A_log=a, g_min=ctypes.c_float(-5.0), S0=None,
                S_out=None, cu=None, N=1, T=ctypes.c_int64(128), H=2, dk=128, dv=128, dt=1, o=a)
    args.update(over)
    f = lib.kda_fwd_chunked_noalloc
    f.restype = ctypes.c_int
    lib.kda_last_error.restype = ctypes.c_char_p
    rc = f(args["q"], args["k"], args["v"], args["beta"], args["z"], args["A_log"], args["g_min"],
           args["S0"], args["S_out"], args["cu"], args["N"], args["T"], args["H"], args["dk"],
           args["dv"], args["dt"], args["o"], None)
    return rc, lib.kda_last_error().decode()


def test_noalloc_rejects_problems_beyond_its_buffer(lib):
    """A problem whose scratch exceeds the built-in 64 MiB is refused before any launch."""
    lib.kda_fwd_workspace_size.restype = ctypes.c_size_t
    lib.kda_fwd_workspace_size.argtypes = [ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_int, ctypes.c_int]
    T = 65536
    assert lib.kda_fwd_workspace_size(T, 1, 32, 128, 128, 1) > (64 << 20)
    rc, msg = _noalloc(lib, T=ctypes.c_int64(T), H=32)
    assert rc == 1 and "built into the library" in msg


def test_noalloc_reports_malformed_arguments_first(lib):
    """A malformed call names the bad argument, even when the problem is also too large."""
    rc, msg = _noalloc(lib, q=None, T=ctypes.c_int64(65536), H=32)
    assert rc == 1 and "q is NULL" in msg
    rc, msg = _noalloc(lib, N=3, T=ctypes.c_int64(65536 + 1), H=32)
    assert rc == 1 and "multiple of N" in msg
