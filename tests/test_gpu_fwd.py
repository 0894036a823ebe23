"""GPU parity of the chunked forward against the fp64 oracle, on the seeded workloads
(full comparison where the oracle finishes in seconds, sampled (sequence, head) pairs at
full size), plus edge cases, resume/varlen properties and determinism."""
import numpy as np
import pytest

from serving_kda_chunkwise_gb300 import inputs
from kda_testutil import (BF16_NORM_TOL, BF16_RMS_TOL, bf16_norm_err, bf16_rms_err,
                          check_forward, gpu_forward, oracle_forward, state_err)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kda():
    import torch  # noqa: F401
    from serving_kda_chunkwise_gb300 import kda as _k
    return _k


def test_fwd_f32_T256_H2_d64_full():
    inp = inputs.workload("fwd_f32_T256_H2_d64")
    o, S = gpu_forward(inp)
    check_forward(inp, o, S, oracle_forward(inp))


def test_fwd_bf16_B2_T4096_H16_d128_full():
    inp = inputs.workload("fwd_bf16_B2_T4096_H16_d128")
    o, S = gpu_forward(inp, use_cu=False)
    check_forward(inp, o, S, oracle_forward(inp))


@pytest.mark.parametrize("g_min", inputs.LONG_GMIN_SWEEP)
def test_fwd_bf16_T65536_H32_d128_sampled(g_min):
    inp = inputs.workload_spec("fwd_bf16_T65536_H32_d128", g_min=g_min)
    o, S = gpu_forward(inp, use_cu=False)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(S))
    check_forward(inp, o, S, oracle_forward(inp, heads=[0, 13, 31]))


def test_fwd_bf16_varlen64_H32_d128_sampled():
    inp = inputs.workload_spec("fwd_bf16_varlen64_H32_d128")
    o, S = gpu_forward(inp)
    lens = np.diff(inp.cu_seqlens)
    seqs = [int(np.argmin(lens)), int(np.argmax(lens)), 7, 40]
    check_forward(inp, o, S, oracle_forward(inp, seqs=seqs, heads=[0, 21]))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("d", [64, 128])
def test_fwd_ragged_and_empty(dtype, d):
    lens = [1, 0, 63, 64, 65, 130, 0, 200, 17]
    inp = inputs.forward_inputs(seed=5, lengths=lens, H=3, dk=d, dv=d, dtype=dtype,
                                with_state=True, g_min=-6.0)
    o, S = gpu_forward(inp)
    check_forward(inp, o, S, oracle_forward(inp))
    # an empty sequence passes its initial state through unchanged
    np.testing.assert_array_equal(S[1], inp.S0[1])


@pytest.mark.parametrize("dk,dv", [(128, 64), (64, 128)])
def test_fwd_rectangular_heads(dk, dv):
    inp = inputs.forward_inputs(seed=9, lengths=[150, 77], H=2, dk=dk, dv=dv, dtype="bf16",
                                with_state=True)
    o, S = gpu_forward(inp)
    check_forward(inp, o, S, oracle_forward(inp))


def test_fwd_resume_equals_single_call(kda):
    """Splitting sequences at chunk and non-chunk boundaries and chaining S_out -> S0
    reproduces one call."""
    import torch
    inp = inputs.forward_inputs(seed=21, B=2, T=1000, H=4, dk=128, dv=128, dtype="bf16",
                                with_state=True)
    from kda_testutil import device_inputs
    d = device_inputs(inp)
    o_full, S_full = kda.fwd_chunked(d["q"], d["k"], d["v"], d["beta"], d["z"], d["A_log"],
                                     inp.g_min, S0=d["S0"], cu_seqlens=d["cu"])
    for split in (64, 333):
        parts_o = []
        S = d["S0"]
        for lo, hi in ((0, split), (split, 1000)):
            idx = torch.cat([torch.arange(lo, hi), torch.arange(1000 + lo, 1000 + hi)]).cuda()
            cu = torch.tensor([0, hi - lo, 2 * (hi - lo)], dtype=torch.int32, device="cuda")
            o, S = kda.fwd_chunked(d["q"][idx].contiguous(), d["k"][idx].contiguous(),
                                   d["v"][idx].contiguous(), d["beta"][idx].contiguous(),
                                   d["z"][idx].contiguous(), d["A_log"], inp.g_min, S0=S,
                                   cu_seqlens=cu)
            parts_o.append((idx, o))
        o_chain = torch.empty_like(o_full)
        for idx, o in parts_o:
            o_chain[idx] = o
        # chained vs single call differ only by rounding: same per-head rule as the parity tests
        oc, of = o_chain.float().cpu().numpy(), o_full.float().cpu().numpy().astype(np.float64)
        for n in range(2):
            for h in range(4):
                sl = slice(1000 * n, 1000 * (n + 1))
                assert bf16_norm_err(oc[sl, h], of[sl, h]) <= BF16_NORM_TOL
                assert bf16_rms_err(oc[sl, h], of[sl, h]) <= BF16_RMS_TOL
                sc = S[n, h].cpu().numpy()
                sf = S_full[n, h].cpu().numpy().astype(np.float64)
                assert state_err(sc, sf) <= BF16_NORM_TOL


def test_fwd_state_aliasing_and_determinism(kda):
    import torch
    inp = inputs.forward_inputs(seed=31, lengths=[300, 129], H=2, dk=128, dv=128, dtype="bf16",
                                with_state=True)
    from kda_testutil import device_inputs
    d = device_inputs(inp)
    runs = []
    for _ in range(3):
        o, S = kda.fwd_chunked(d["q"], d["k"], d["v"], d["beta"], d["z"], d["A_log"], inp.g_min,
                               S0=d["S0"], cu_seqlens=d["cu"])
        runs.append((o.clone(), S.clone()))
    for o, S in runs[1:]:
        assert torch.equal(o, runs[0][0]) and torch.equal(S, runs[0][1])
    S_inplace = d["S0"].clone()
    o2, _ = kda.fwd_chunked(d["q"], d["k"], d["v"], d["beta"], d["z"], d["A_log"], inp.g_min,
                            S0=S_inplace, S_out=S_inplace, cu_seqlens=d["cu"])
    assert torch.equal(o2, runs[0][0]) and torch.equal(S_inplace, runs[0][1])


def test_fwd_output_canaries(kda):
    """Nothing is written outside o / S_out (guard regions around both stay intact)."""
    import torch
    inp = inputs.forward_inputs(seed=41, lengths=[77, 190], H=2, dk=128, dv=128, dtype="bf16",
                                with_state=True)
    from kda_testutil import device_inputs
    d = device_inputs(inp)
    T, H, dv = 267, 2, 128
    pad = 4096
    o_buf = torch.full((pad + T * H * dv + pad,), 7.0, dtype=torch.bfloat16, device="cuda")
    S_buf = torch.full((pad + 2 * H * 128 * dv + pad,), 9.0, dtype=torch.float32, device="cuda")
    o = o_buf[pad:pad + T * H * dv].view(T, H, dv)
    S = S_buf[pad:pad + 2 * H * 128 * dv].view(2, H, 128, dv)
    kda.fwd_chunked(d["q"], d["k"], d["v"], d["beta"], d["z"], d["A_log"], inp.g_min, S0=d["S0"],
                    cu_seqlens=d["cu"], o=o, S_out=S)
    torch.cuda.synchronize()
    assert torch.all(o_buf[:pad] == 7.0) and torch.all(o_buf[-pad:] == 7.0)
    assert torch.all(S_buf[:pad] == 9.0) and torch.all(S_buf[-pad:] == 9.0)


def test_fwd_decode_consistency(kda):
    """1000 decode steps equal one chunked forward over the same 1000 tokens."""
    import torch
    inp = inputs.forward_inputs(seed=51, B=1, T=1000, H=2, dk=128, dv=128, dtype="bf16",
                                with_state=True)
    from kda_testutil import device_inputs
    d = device_inputs(inp)
    o_fwd, S_fwd = kda.fwd_chunked(d["q"], d["k"], d["v"], d["beta"], d["z"], d["A_log"],
                                   inp.g_min, S0=d["S0"], cu_seqlens=d["cu"])
    S = d["S0"].clone()
    outs = []
    for t in range(1000):
        outs.append(kda.decode_step(d["q"][t:t + 1], d["k"][t:t + 1], d["v"][t:t + 1],
                                    d["beta"][t:t + 1], d["z"][t:t + 1], d["A_log"], inp.g_min,
                                    S))
    o_dec = torch.cat(outs).float().cpu().numpy()
    o_f = o_fwd.float().cpu().numpy().astype(np.float64)
    for h in range(2):
        assert bf16_norm_err(o_dec[:, h], o_f[:, h]) <= BF16_NORM_TOL
        assert bf16_rms_err(o_dec[:, h], o_f[:, h]) <= BF16_RMS_TOL
        assert state_err(S[0, h].cpu().numpy(), S_fwd[0, h].cpu().numpy().astype(np.float64)) \
            <= BF16_NORM_TOL


def test_fwd_invariant_state_held(kda):
    """beta = 0 and alpha = 1 (z = -inf): the state is carried unchanged and o = S0^T q."""
    import torch
    inp = inputs.forward_inputs(seed=61, lengths=[100, 30], H=2, dk=128, dv=128, dtype="f32",
                                with_state=True)
    from kda_testutil import device_inputs
    d = device_inputs(inp)
    d["beta"].zero_()
    d["z"].fill_(-float("inf"))
    o, S = kda.fwd_chunked(d["q"], d["k"], d["v"], d["beta"], d["z"], d["A_log"], inp.g_min,
                           S0=d["S0"], cu_seqlens=d["cu"])
    assert torch.equal(S, d["S0"])
    ref = torch.einsum("thi,hij->thj", d["q"][:100].double(), d["S0"][0].double())
    assert torch.allclose(o[:100].double(), ref, rtol=1e-5, atol=1e-7)


def test_fwd_bad_seqlens_reported(kda):
    import torch
    inp = inputs.forward_inputs(seed=71, lengths=[64, 64], H=1, dk=64, dv=64, dtype="f32")
    from kda_testutil import device_inputs
    d = device_inputs(inp)
    bad = torch.tensor([0, 100, 90], dtype=torch.int32, device="cuda")   # decreasing
    kda.fwd_chunked(d["q"], d["k"], d["v"], d["beta"], d["z"], d["A_log"], -5.0, cu_seqlens=bad)
    with pytest.raises(kda.KdaError) as ei:
        kda.device_status()
    assert ei.value.status == kda.KDA_ERR_DEVICE
    kda.device_status()   # cleared


def test_fwd_tensor_core_path_matches_cuda_core_path(kda, monkeypatch):
    """The tcgen05 path (bf16, d=128) against the fp32 CUDA-core path on the same inputs."""
    inp = inputs.forward_inputs(seed=81, lengths=[333, 64, 1, 190], H=3, dk=128, dv=128,
                                dtype="bf16", with_state=True, g_min=-6.0)
    o_tc, S_tc = gpu_forward(inp)
    monkeypatch.setenv("KDA_FWD_PATH", "generic")
    assert kda.workspace_size(inp.T, inp.N, inp.H, 128, 128, __import__("torch").bfloat16) == 0
    o_cc, S_cc = gpu_forward(inp)
    for n in range(inp.N):
        a, b = inp.cu_seqlens[n], inp.cu_seqlens[n + 1]
        for h in range(inp.H):
            assert bf16_norm_err(o_tc[a:b, h], o_cc[a:b, h].astype(np.float64)) < 2e-2
            assert state_err(S_tc[n, h], S_cc[n, h].astype(np.float64)) <= BF16_NORM_TOL
            assert bf16_rms_err(S_tc[n, h], S_cc[n, h].astype(np.float64)) <= BF16_RMS_TOL


def test_fwd_fused_matches_two_launch(kda, monkeypatch):
    """Equal-length sequences without cu_seqlens take the fused form (one cooperative launch,
    packages handed from the intra stage to the chain stage through a ring in L2).  It runs
    the same arithmetic as the two-launch form, so the results are bitwise equal, and both
    meet the parity rule against the oracle."""
    inp = inputs.forward_inputs(seed=91, B=3, T=2000, H=5, dk=128, dv=128, dtype="bf16",
                                with_state=True, g_min=-6.0)
    kda.profile_begin()
    o_f, S_f = gpu_forward(inp, use_cu=False)
    names = kda.profile_end()
    assert "fwd_fused_kernel" in names and "chain_kernel" not in names
    monkeypatch.setenv("KDA_FWD_FUSED", "0")
    kda.profile_begin()
    o_2, S_2 = gpu_forward(inp, use_cu=False)
    names = kda.profile_end()
    assert "chain_kernel" in names and "fwd_fused_kernel" not in names
    assert np.array_equal(o_f, o_2) and np.array_equal(S_f, S_2)
    check_forward(inp, o_f, S_f, oracle_forward(inp))


@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 128), (128, 64)])
def test_fwd_bf16_small_heads_on_tensor_cores(kda, monkeypatch, dk, dv):
    """bf16 heads of 64 channels take the tensor-core path, zero-padded to 128 inside (the
    tensor maps read zeros past the head, and zero channels add nothing to q.k, the state or
    o).  The fused form and the two-launch form agree bitwise and meet the parity rule,
    initial and final state included."""
    inp = inputs.forward_inputs(seed=92, B=2, T=1280, H=3, dk=dk, dv=dv, dtype="bf16",
                                with_state=True)
    kda.profile_begin()
    o_f, S_f = gpu_forward(inp, use_cu=False)
    names = kda.profile_end()
    assert "fwd_fused_kernel" in names and "fwd_generic_kernel" not in names
    monkeypatch.setenv("KDA_FWD_FUSED", "0")
    kda.profile_begin()
    o_2, S_2 = gpu_forward(inp, use_cu=False)
    names = kda.profile_end()
    assert "intra_kernel" in names and "chain_kernel" in names
    assert np.array_equal(o_f, o_2) and np.array_equal(S_f, S_2)
    check_forward(inp, o_f, S_f, oracle_forward(inp))


def test_fwd_bf16_d64_output_canaries(kda):
    """The zero-padded tensor-core path writes only o and S_out of a 64-channel head
    (guard regions around both stay intact), fused and two-launch forms."""
    import torch
    for B, lens in ((2, None), (None, [77, 190])):
        if B:
            inp = inputs.forward_inputs(seed=43, B=B, T=1024, H=2, dk=64, dv=64, dtype="bf16",
                                        with_state=True)
        else:
            inp = inputs.forward_inputs(seed=42, lengths=lens, H=2, dk=64, dv=64, dtype="bf16",
                                        with_state=True)
        from kda_testutil import device_inputs
        d = device_inputs(inp)
        N = len(inp.cu_seqlens) - 1
        T, H, dv = int(inp.cu_seqlens[-1]), 2, 64
        pad = 4096
        o_buf = torch.full((pad + T * H * dv + pad,), 7.0, dtype=torch.bfloat16, device="cuda")
        S_buf = torch.full((pad + N * H * 64 * dv + pad,), 9.0, dtype=torch.float32, device="cuda")
        o = o_buf[pad:pad + T * H * dv].view(T, H, dv)
        S = S_buf[pad:pad + N * H * 64 * dv].view(N, H, 64, dv)
        kw = dict(N=N) if B else dict(cu_seqlens=d["cu"])
        kda.fwd_chunked(d["q"], d["k"], d["v"], d["beta"], d["z"], d["A_log"], inp.g_min,
                        S0=d["S0"], o=o, S_out=S, **kw)
        torch.cuda.synchronize()
        assert torch.all(o_buf[:pad] == 7.0) and torch.all(o_buf[-pad:] == 7.0)
        assert torch.all(S_buf[:pad] == 9.0) and torch.all(S_buf[-pad:] == 9.0)
        check_forward(inp, o.float().cpu().numpy(), S.cpu().numpy(), oracle_forward(inp))
