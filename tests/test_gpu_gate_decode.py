"""GPU parity: the gate kernel and the decode kernel against the fp64 oracle."""
import numpy as np
import pytest

import oracle
from serving_kda_chunkwise_gb300 import inputs
from kda_testutil import BF16_NORM_TOL, FP32_REL_TOL, bf16_norm_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kda():
    import torch  # noqa: F401
    from serving_kda_chunkwise_gb300 import kda as _k
    return _k


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("g_min", [-3.0, -5.0, -6.0])
def test_gate_matches_oracle(kda, dtype, g_min):
    import torch
    rng = np.random.Generator(np.random.PCG64(5))
    z = inputs.store(rng.standard_normal((333, 3, 128)).astype(np.float32) * 3, dtype)
    z.values[0, 0, :4] = [0.0, np.inf, -np.inf, 40.0]
    if dtype == "bf16":
        z = inputs.store(z.values, "bf16")
    A = rng.uniform(-1, 1, 3).astype(np.float32)
    g = kda.gate(z.as_torch("cuda"), torch.from_numpy(A).cuda(), g_min).cpu().numpy()
    ref = oracle.gate(z.values, A, g_min)
    np.testing.assert_allclose(g, ref, rtol=2e-6, atol=1e-7)
    assert g[0, 0, 1] == np.float32(g_min) and g[0, 0, 2] == 0.0


def test_gate_empty_and_odd_shapes(kda):
    import torch
    z = torch.zeros((0, 2, 8), dtype=torch.bfloat16, device="cuda")
    A = torch.zeros(2, dtype=torch.float32, device="cuda")
    assert kda.gate(z, A, -5.0).shape == (0, 2, 8)
    z = torch.randn((7, 5, 12), device="cuda")
    g = kda.gate(z, torch.zeros(5, device="cuda"), -5.0).cpu().numpy()
    np.testing.assert_allclose(g, oracle.gate(z.cpu().numpy(), np.zeros(5), -5.0), rtol=2e-6,
                               atol=1e-7)


def _decode_run(kda, N, H, dk, dv, steps, dtype, sample, seed=77, g_min=-5.0):
    import torch
    S_np, A = inputs.decode_state(seed=seed, N=N, H=H, dk=dk, dv=dv)
    S = torch.from_numpy(S_np).cuda()
    At = torch.from_numpy(A).cuda()
    S_ref = {nh: S_np[nh].astype(np.float64) for nh in sample}
    worst = 0.0
    for step, x in inputs.decode_steps_iter(seed=seed, steps=steps, N=N, H=H, dk=dk, dv=dv,
                                            dtype=dtype):
        o = kda.decode_step(x.q.as_torch("cuda"), x.k.as_torch("cuda"), x.v.as_torch("cuda"),
                            x.beta.as_torch("cuda"), x.z.as_torch("cuda"), At, g_min, S)
        o = o.float().cpu().numpy()
        for (n, h) in sample:
            o_r, S_new = oracle.decode_steps(S_ref[(n, h)][None, None], x.q.values[n:n + 1, h:h + 1],
                                             x.k.values[n:n + 1, h:h + 1],
                                             x.v.values[n:n + 1, h:h + 1],
                                             x.beta.values[n:n + 1, h:h + 1],
                                             x.z.values[n:n + 1, h:h + 1], A[h:h + 1], g_min,
                                             nthreads=1)
            S_ref[(n, h)] = S_new[0, 0]
            if dtype == "bf16":
                err = bf16_norm_err(o[n, h], o_r[0, 0])
            else:  # fp32: relative 2-norm of this (sequence, head)'s output vector
                err = np.linalg.norm(o[n, h] - o_r[0, 0]) / max(np.linalg.norm(o_r[0, 0]), 1e-30)
            worst = max(worst, err)
            tol = BF16_NORM_TOL if dtype == "bf16" else FP32_REL_TOL
            assert err <= tol, f"step {step} seq {n} head {h}: {err:.3e}"
    S_fin = S.cpu().numpy()
    for (n, h), Sr in S_ref.items():
        rel = np.linalg.norm(S_fin[n, h] - Sr) / np.linalg.norm(Sr)
        assert rel <= (1e-5 if dtype == "f32" else 1e-4), f"state seq {n} head {h}: {rel:.3e}"
    return worst


@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 64), (128, 64), (64, 128)])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_decode_small(kda, dk, dv, dtype):
    _decode_run(kda, N=3, H=4, dk=dk, dv=dv, steps=20, dtype=dtype,
                sample=[(0, 0), (1, 3), (2, 1)])


def test_decode_full_size_1000_steps(kda):
    """N=256 sequences x 32 heads, d=128, 1000 seeded steps; sampled states vs the oracle."""
    w = inputs.DECODE_WORKLOAD
    sample = [(0, 0), (17, 5), (128, 31), (255, 12)]
    _decode_run(kda, N=w["N"], H=w["H"], dk=w["dk"], dv=w["dv"], steps=w["steps"],
                dtype=w["dtype"], sample=[(n, h) for n, h in sample], seed=w["seed"])
