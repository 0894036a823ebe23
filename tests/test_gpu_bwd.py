"""GPU parity of the backward (kda_bwd) against the fp64 reverse-mode oracle
(oracle/kda_backward.py), on the same stored inputs and upstream gradients.

Tolerance, per (sequence, head) and gradient tensor: fp32 I/O ||d - d_ref||_F / ||d_ref||_F
<= 1e-4; bf16 I/O the forward's rule (after dividing by rms(d_ref): |d - d_ref| <= 2e-2 +
2^-8 |d_ref|, the last term half a bf16 ulp of the stored gradient, and rms(d - d_ref) <= 1e-2).  dA_log (summed over sequences) and dS0 are fp32
outputs: relative 1e-4 for fp32 problems, 1e-2 for bf16 problems.
"""
import numpy as np
import pytest

from oracle import kda_backward as kb
from serving_kda_chunkwise_gb300 import inputs
from kda_testutil import BF16_NORM_TOL, BF16_RMS_TOL, bf16_norm_err, bf16_rms_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kda():
    import torch  # noqa: F401
    from serving_kda_chunkwise_gb300 import kda as _k
    return _k


def _close(d, ref, dtype, what):
    d = np.asarray(d, dtype=np.float64)
    assert np.all(np.isfinite(d)), what
    if dtype == "f32":
        rel = np.linalg.norm(d - ref) / max(np.linalg.norm(ref), 1e-30)
        assert rel <= 1e-4, f"{what}: {rel:.3e}"
    else:
        assert bf16_norm_err(d, ref) <= BF16_NORM_TOL, what
        assert bf16_rms_err(d, ref) <= BF16_RMS_TOL, what


def _run(kda, lengths, H, d, dtype, seed, with_dS=True, dv=None, g_min=None):
    import torch
    dv = d if dv is None else dv
    kw = {} if g_min is None else {"g_min": g_min}
    inp = inputs.forward_inputs(seed=seed, lengths=lengths, H=H, dk=d, dv=dv, dtype=dtype,
                                with_state=True, **kw)
    rng = np.random.default_rng(seed + 1)
    T, N = int(inp.cu_seqlens[-1]), len(lengths)
    do = inputs.store(rng.standard_normal((T, H, dv)).astype(np.float32), dtype)
    dS = rng.standard_normal((N, H, d, dv)).astype(np.float32) if with_dS else None
    dev = {nm: getattr(inp, nm).as_torch("cuda") for nm in ("q", "k", "v", "beta", "z")}
    g = kda.bwd(dev["q"], dev["k"], dev["v"], dev["beta"], dev["z"],
                torch.from_numpy(inp.A_log).cuda(), inp.g_min, do.as_torch("cuda"),
                S0=torch.from_numpy(inp.S0).cuda(),
                dS_out=None if dS is None else torch.from_numpy(dS).cuda(),
                cu_seqlens=torch.from_numpy(inp.cu_seqlens.astype(np.int32)).cuda())
    kda.device_status()
    ref = kb.backward(inp.q.values, inp.k.values, inp.v.values, inp.beta.values, inp.z.values,
                      inp.A_log, inp.g_min, do.values, S0=inp.S0, dS_out=dS,
                      cu_seqlens=inp.cu_seqlens)
    cu = inp.cu_seqlens
    for nm in ("dq", "dk", "dv", "dbeta", "dz"):
        got = g[nm].float().cpu().numpy()
        for n in range(N):
            a, b = int(cu[n]), int(cu[n + 1])
            if b == a:
                continue
            for h in range(H):
                _close(got[a:b, h], ref[nm][a:b, h], dtype, f"{nm} seq {n} head {h}")
    tol = 1e-4 if dtype == "f32" else 1e-2
    dA, dS0 = g["dA_log"].cpu().numpy(), g["dS0"].cpu().numpy()
    np.testing.assert_allclose(dA, ref["dA_log"], rtol=tol,
                               atol=tol * np.max(np.abs(ref["dA_log"])))
    for n in range(N):
        for h in range(H):
            rel = np.linalg.norm(dS0[n, h] - ref["dS0"][n, h]) / np.linalg.norm(ref["dS0"][n, h])
            assert rel <= tol, f"dS0 seq {n} head {h}: {rel:.3e}"
    return g


@pytest.mark.parametrize("dtype,d", [("f32", 64), ("f32", 128), ("bf16", 128)])
def test_matches_oracle(kda, dtype, d):
    _run(kda, [70, 0, 129, 1], H=2, d=d, dtype=dtype, seed=71)


@pytest.mark.parametrize("dtype,dk,dv", [("f32", 64, 128), ("f32", 128, 64), ("bf16", 64, 64),
                                         ("bf16", 128, 64), ("bf16", 64, 128)])
def test_other_head_sizes(kda, dtype, dk, dv):
    """d_k != d_v (the state's rows and columns split differently over the threads; on the
    tensor-core path the padded key or value channels of the operand images are zeros) and
    bf16 at d = 64."""
    _run(kda, [90, 17], H=2, d=dk, dv=dv, dtype=dtype, seed=75)


@pytest.mark.parametrize("g_min", [-3.0, -6.0])
def test_gate_bound_range(kda, g_min):
    """bf16 at the ends of the gate bounds used by the benchmark's sweep: at g_min = -6 a
    16-token block spans decay factors up to e^{48} on either side of its reference, the range
    the decayed products' references are built for."""
    _run(kda, [130, 64], H=2, d=128, dtype="bf16", seed=77, g_min=g_min)


def test_without_final_state_gradient(kda):
    _run(kda, [200], H=3, d=64, dtype="f32", seed=72, with_dS=False)


def test_deterministic(kda):
    import torch
    g1 = _run(kda, [150, 33], H=2, d=128, dtype="bf16", seed=73)
    g2 = _run(kda, [150, 33], H=2, d=128, dtype="bf16", seed=73)
    for nm in g1:
        assert torch.equal(g1[nm], g2[nm]), nm


def test_more_chains_than_sms(kda):
    """64 packed sequences of 1..130 tokens at H = 3: 192 (sequence, head) chains, more than the
    GPU has SMs, so each chain CTA of both chains runs several chains in turn (their operand
    images through the same shared-memory stages and bulk copies)."""
    rng = np.random.default_rng(82)
    lengths = [int(x) for x in rng.integers(1, 131, size=64)]
    _run(kda, lengths, H=3, d=64, dtype="bf16", seed=83)


def test_long_sequences(kda):
    """Sequences of 2100 and 1000 tokens (33 and 16 chunks, ragged tails): the checkpoints and
    the per-chunk recompute over many chunks."""
    _run(kda, [2100, 1000], H=2, d=128, dtype="bf16", seed=74)


def test_full_size_window(kda):
    """The benchmark's backward shape and launch configuration (one sequence of T = 65536
    tokens, H = 32, d = 128, bf16, dS_out = 0), with the upstream gradient do nonzero only on
    tokens [t_a, t_b).  The state's gradient is then exactly zero from t_b on, so every
    gradient of a token at or after t_b is exactly zero; and the gradients of the tokens in
    [w0, t_b) are those of the window alone started from the state at w0, which the oracle
    gives exactly: the C token recurrence over [0, w0), then the reverse-mode oracle over
    [w0, t_b).  This crosses the two chains over all 1024 chunks (the state at every chunk
    start, the gradient at every chunk end).  Sampled heads 3 and 29; the window starts and
    ends inside chunks."""
    import torch
    import oracle
    sp = inputs.workload_spec("fwd_bf16_T65536_H32_d128")
    d = sp.to_device("cuda")
    T, H, dk, dv = sp.T, sp.H, sp.dk, sp.dv
    t_a, t_b = 40013, 40163
    w0 = t_a - 100
    rng = np.random.default_rng(76)
    do_win = inputs.store(rng.standard_normal((t_b - t_a, H, dv)).astype(np.float32), "bf16")
    do = torch.zeros((T, H, dv), dtype=torch.bfloat16, device="cuda")
    do[t_a:t_b] = do_win.as_torch("cuda")
    g = kda.bwd(d["q"], d["k"], d["v"], d["beta"], d["z"], d["A_log"], sp.g_min, do,
                dS_out=torch.zeros((1, H, dk, dv), dtype=torch.float32, device="cuda"), N=1)
    kda.device_status()
    for nm in ("dq", "dk", "dv", "dbeta", "dz"):
        assert torch.count_nonzero(g[nm][t_b:]).item() == 0, f"{nm} after the window"
    heads = [3, 29]
    kinds = ("q", "k", "v", "beta", "z")
    pre = {kind: sp.tokens(kind, 0, w0, heads) for kind in kinds}
    _, S_w0 = oracle.recurrent(pre["q"], pre["k"], pre["v"], pre["beta"], pre["z"],
                               sp.A_log[heads], sp.g_min)
    win = {kind: sp.tokens(kind, w0, t_b, heads) for kind in kinds}
    do_ref = np.zeros((t_b - w0, len(heads), dv))
    do_ref[t_a - w0:] = do_win.values[:, heads]
    ref = kb.backward(win["q"], win["k"], win["v"], win["beta"], win["z"], sp.A_log[heads],
                      sp.g_min, do_ref, S0=S_w0)
    for nm in ("dq", "dk", "dv", "dbeta", "dz"):
        got = g[nm][w0:t_b].float().cpu().numpy()
        for ii, h in enumerate(heads):
            _close(got[:, h], ref[nm][:, ii], "bf16", f"{nm} head {h}")
