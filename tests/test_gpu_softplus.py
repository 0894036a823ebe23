"""GPU parity of the comparison variant: the chunked forward with the gate the bound replaces,
g = -e^{A_h} Softplus(z) ("Kimi k3 技术报告详解（1）", section "Chunkwise parallel form"),
against the fp64 token recurrence.  bf16 with d = 128 runs the mixed path (off-diagonal
sub-tiles on the tensor cores, diagonal sub-tiles per pair), everything else the explicit
per-pair path.  Same tolerances as the bounded forward (kda_testutil)."""
import numpy as np
import pytest

from serving_kda_chunkwise_gb300 import inputs
from kda_testutil import check_forward, oracle_forward

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kda():
    import torch  # noqa: F401
    from serving_kda_chunkwise_gb300 import kda as _k
    return _k


def _gpu(kda, inp, use_cu=True):
    import torch
    dev = {k: getattr(inp, k).as_torch("cuda") for k in ("q", "k", "v", "beta", "z")}
    if use_cu:
        kw = dict(cu_seqlens=torch.from_numpy(inp.cu_seqlens.astype(np.int32)).cuda())
    else:  # equal lengths without cu_seqlens
        kw = dict(N=len(inp.cu_seqlens) - 1)
    o, S = kda.fwd_chunked_softplus(
        dev["q"], dev["k"], dev["v"], dev["beta"], dev["z"], torch.from_numpy(inp.A_log).cuda(),
        S0=None if inp.S0 is None else torch.from_numpy(inp.S0).cuda(), **kw)
    kda.device_status()
    return o.float().cpu().numpy(), S.cpu().numpy()


def _shift_z(inp, dz):
    """Move every z by dz (re-rounded to the I/O type): dz > 0 means stronger decay."""
    inp.z = inputs.store(inp.z.values + np.float32(dz), inp.dtype)
    return inp


@pytest.mark.parametrize("dtype,d", [("f32", 64), ("bf16", 128), ("f32", 128), ("bf16", 64)])
def test_matches_recurrence(kda, dtype, d):
    inp = inputs.forward_inputs(seed=61, lengths=[100, 64, 1, 300, 0, 129], H=2, dk=d, dv=d,
                                dtype=dtype, with_state=True)
    o, S = _gpu(kda, inp)
    check_forward(inp, o, S, oracle_forward(inp, gate="softplus"))


def test_strong_decay_stays_finite(kda):
    """z around +3: g ~ -3 e^A per token, a chunk's decay far below any fp32 number; the
    explicit path forms every factor as e^(<= 0) and stays finite."""
    inp = _shift_z(inputs.forward_inputs(seed=62, lengths=[256, 70], H=2, dk=128, dv=128,
                                         dtype="bf16", with_state=True), 3.0)
    o, S = _gpu(kda, inp)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(S))
    check_forward(inp, o, S, oracle_forward(inp, gate="softplus"))


def test_no_decay_and_no_writes_holds_state(kda):
    inp = inputs.forward_inputs(seed=63, lengths=[90], H=2, dk=64, dv=64, dtype="f32",
                                with_state=True)
    inp.z.values[:] = -np.inf
    inp.beta.values[:] = 0.0
    o, S = _gpu(kda, inp)
    assert np.array_equal(S, inp.S0)
    ref = np.einsum("thc,hcj->thj", inp.q.values.astype(np.float64), inp.S0[0].astype(np.float64))
    np.testing.assert_allclose(o, ref, rtol=1e-5, atol=1e-7)


def test_full_size_sampled(kda):
    """The benchmark's comparison shape (T = 65536, H = 32, d = 128, bf16): heads 0 and 17
    against the token recurrence."""
    sp = inputs.workload_spec("fwd_bf16_T65536_H32_d128")
    d = sp.to_device("cuda")
    o, S = kda.fwd_chunked_softplus(d["q"], d["k"], d["v"], d["beta"], d["z"], d["A_log"], N=1)
    kda.device_status()
    o = o.float().cpu().numpy()
    S = S.cpu().numpy()
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(S))
    check_forward(sp, o, S, oracle_forward(sp, heads=[0, 17], gate="softplus"))


def test_mixed_path_kernels_and_fused_form(kda, monkeypatch):
    """bf16, d = 128 takes the mixed path; equal lengths without cu_seqlens take its fused
    form (bitwise equal to the two-launch form), and both meet the parity rule."""
    inp = inputs.forward_inputs(seed=64, B=2, T=1280, H=4, dk=128, dv=128, dtype="bf16",
                                with_state=True)
    kda.profile_begin()
    o_f, S_f = _gpu(kda, inp, use_cu=False)
    names = kda.profile_end()
    assert "fwd_fused_mixed_kernel" in names and "fwd_generic_kernel" not in names
    monkeypatch.setenv("KDA_FWD_FUSED", "0")
    kda.profile_begin()
    o_2, S_2 = _gpu(kda, inp, use_cu=False)
    names = kda.profile_end()
    assert "intra_mixed_kernel" in names and "chain_kernel" in names
    assert np.array_equal(o_f, o_2) and np.array_equal(S_f, S_2)
    check_forward(inp, o_f, S_f, oracle_forward(inp, gate="softplus"))


@pytest.mark.parametrize("dz", [-2.0, 1.5, 6.0])
def test_mixed_path_decay_range(kda, dz):
    """From weak (z - 2) to very strong (z + 6: g ~ -6 e^A per token, a 16-token sub-tile's
    decay past the fp32 range) decay, with ragged tails: every factor of the mixed path is
    <= 1, so the result stays finite and meets the parity rule."""
    inp = _shift_z(inputs.forward_inputs(seed=65, lengths=[64 * 5 + 17, 64 * 3 - 5, 7], H=3,
                                         dk=128, dv=128, dtype="bf16", with_state=True), dz)
    o, S = _gpu(kda, inp)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(S))
    check_forward(inp, o, S, oracle_forward(inp, gate="softplus"))


def test_mixed_path_matches_explicit_path(kda, monkeypatch):
    """The mixed path and the explicit per-pair path on the same bf16 inputs both meet the
    parity rule against the oracle."""
    inp = inputs.forward_inputs(seed=66, lengths=[200, 333], H=2, dk=128, dv=128,
                                dtype="bf16", with_state=True)
    ref = oracle_forward(inp, gate="softplus")
    o_m, S_m = _gpu(kda, inp)
    monkeypatch.setenv("KDA_FWD_PATH", "generic")
    o_e, S_e = _gpu(kda, inp)
    check_forward(inp, o_m, S_m, ref)
    check_forward(inp, o_e, S_e, ref)
