"""GPU parity of the comparison variant: the chunked forward with the gate the bound replaces,
g = -e^{A_h} Softplus(z) ("Kimi k3 技术报告详解（1）", section "Chunkwise parallel form"), on the
explicit per-pair path, against the fp64 token recurrence.  Same tolerances as the bounded
forward (kda_testutil)."""
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


def _gpu(kda, inp):
    import torch
    dev = {k: getattr(inp, k).as_torch("cuda") for k in ("q", "k", "v", "beta", "z")}
    o, S = kda.fwd_chunked_softplus(
        dev["q"], dev["k"], dev["v"], dev["beta"], dev["z"], torch.from_numpy(inp.A_log).cuda(),
        S0=None if inp.S0 is None else torch.from_numpy(inp.S0).cuda(),
        cu_seqlens=torch.from_numpy(inp.cu_seqlens.astype(np.int32)).cuda())
    kda.device_status()
    return o.float().cpu().numpy(), S.cpu().numpy()


def _shift_z(inp, dz):
    """Move every z by dz (re-rounded to the I/O type): dz > 0 means stronger decay."""
    inp.z = inputs.store(inp.z.values + np.float32(dz), inp.dtype)
    return inp


@pytest.mark.parametrize("dtype,d", [("f32", 64), ("bf16", 128), ("f32", 128)])
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
