"""GPU parity: the gated output step (section "Gated MLA" of "Kimi k3 技术报告详解（1）"),
standalone and fused into the decode step, against the fp64 oracle.

Tolerance.  The step is elementwise after one row reduction, so the only sizeable error is
the final rounding of y to the I/O type: |y - y_ref| <= 2^-8 |y_ref| + 1e-6 for bf16 output
(one rounding is at most 2^-9 relative) and 1e-5 |y_ref| + 1e-6 for fp32.  The fused decode
output inherits the decode step's own error and is held to the decode tolerance.
"""
import numpy as np
import pytest

import oracle
from serving_kda_chunkwise_gb300 import inputs
from kda_testutil import BF16_NORM_TOL, bf16_norm_err

pytestmark = pytest.mark.gpu

RTOL = {"bf16": 2.0 ** -8, "f32": 1e-5}
ATOL = 1e-6


@pytest.fixture(scope="module")
def kda():
    import torch  # noqa: F401
    from serving_kda_chunkwise_gb300 import kda as _k
    return _k


def _run(kda, x, eps, in_place=False):
    import torch
    o = x.o.as_torch("cuda")
    g = x.gate.as_torch("cuda")
    w = None if x.norm_w is None else torch.from_numpy(x.norm_w).cuda()
    y = kda.output_norm_gate(o, g, w, eps, y=o if in_place else None)
    return y.float().cpu().numpy()


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("dv", [64, 128])
@pytest.mark.parametrize("T,with_weight", [(1, True), (37, False), (1000, True)])
def test_matches_oracle(kda, dtype, dv, T, with_weight):
    x = inputs.output_gate_inputs(seed=41 + T, T=T, H=3, dv=dv, dtype=dtype,
                                  with_weight=with_weight)
    eps = 1e-6
    y = _run(kda, x, eps)
    ref = oracle.output_norm_gate(x.o.values, x.gate.values, x.norm_w, eps)
    np.testing.assert_allclose(y, ref, rtol=RTOL[dtype], atol=ATOL)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_in_place_equals_out_of_place(kda, dtype):
    x = inputs.output_gate_inputs(seed=7, T=513, H=5, dv=128, dtype=dtype)
    assert np.array_equal(_run(kda, x, 1e-5), _run(kda, x, 1e-5, in_place=True))


def test_edge_rows(kda):
    """Zero rows give 0; saturated gates give 0 and the bare normalised row; empty is a no-op."""
    import torch
    x = inputs.output_gate_inputs(seed=9, T=6, H=2, dv=128, dtype="f32", with_weight=False)
    x.o.values[0] = 0.0
    x.gate.values[1] = -200.0
    x.gate.values[2] = 200.0
    y = _run(kda, x, 1e-6)
    assert np.all(y[0] == 0.0) and np.all(np.abs(y[1]) < 1e-30)
    ref = oracle.output_norm_gate(x.o.values, x.gate.values, None, 1e-6)
    np.testing.assert_allclose(y[2], ref[2], rtol=1e-5, atol=ATOL)
    np.testing.assert_allclose(np.mean(y[2].astype(np.float64) ** 2, axis=-1), 1.0, rtol=1e-4)
    e = torch.empty((0, 4, 64), dtype=torch.bfloat16, device="cuda")
    assert kda.output_norm_gate(e, e.clone(), None, 1e-6).shape == (0, 4, 64)


def test_full_size_sampled(kda):
    """The shape the benchmark times (T=65536, H=32, dv=128, bf16), 4096 sampled rows."""
    import torch
    w = inputs.OUTPUT_GATE_WORKLOAD
    x = inputs.output_gate_inputs(**w)
    eps = 1e-6
    y = kda.output_norm_gate(x.o.as_torch("cuda"), x.gate.as_torch("cuda"),
                             torch.from_numpy(x.norm_w).cuda(), eps)
    rows = np.random.Generator(np.random.PCG64(3)).choice(w["T"] * w["H"], 4096, replace=False)
    t, h = rows // w["H"], rows % w["H"]
    ys = y[torch.from_numpy(t).cuda(), torch.from_numpy(h).cuda()].float().cpu().numpy()
    ref = oracle.output_norm_gate(x.o.values[t, h], x.gate.values[t, h], x.norm_w, eps)
    np.testing.assert_allclose(ys, ref, rtol=RTOL["bf16"], atol=ATOL)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 64)])
def test_decode_gated(kda, dtype, dk, dv):
    """The fused decode step: the state evolves exactly as in the plain step, and y is the
    gated, normalised output of the oracle's decode step."""
    import torch
    N, H, eps = 3, 4, 1e-6
    S_host, A = inputs.decode_state(seed=51, N=N, H=H, dk=dk, dv=dv)
    S_plain = torch.from_numpy(S_host).cuda()
    S_gated = S_plain.clone()
    S_ref = S_host.astype(np.float64)
    Ad = torch.from_numpy(A).cuda()
    wv = np.random.Generator(np.random.PCG64(53)).uniform(0.5, 1.5, dv).astype(np.float32)
    for step in range(5):
        x = inputs.decode_step_inputs(seed=51, step=step, N=N, H=H, dk=dk, dv=dv, dtype=dtype)
        gate = inputs.store(np.random.Generator(np.random.PCG64(60 + step)).standard_normal(
            (N, H, dv)).astype(np.float32), dtype)
        dev = {k_: getattr(x, k_).as_torch("cuda") for k_ in ("q", "k", "v", "beta", "z")}
        o = kda.decode_step(dev["q"], dev["k"], dev["v"], dev["beta"], dev["z"], Ad, -5.0,
                            S_plain)
        y = kda.decode_step_gated(dev["q"], dev["k"], dev["v"], dev["beta"], dev["z"], Ad, -5.0,
                                  S_gated, gate.as_torch("cuda"), torch.from_numpy(wv).cuda(),
                                  eps)
        assert torch.equal(S_plain, S_gated), f"step {step}: the state differs"
        o_ref, S_ref = oracle.decode_steps(S_ref, x.q.values, x.k.values, x.v.values,
                                           x.beta.values, x.z.values, A, -5.0)
        y_ref = oracle.output_norm_gate(o_ref, gate.values, wv, eps)
        yg = y.float().cpu().numpy()
        if dtype == "bf16":
            for n in range(N):
                for h in range(H):
                    assert bf16_norm_err(yg[n, h], y_ref[n, h]) <= BF16_NORM_TOL
        else:
            np.testing.assert_allclose(yg, y_ref, rtol=1e-4, atol=1e-5)
        # and against the standalone step applied to the plain decode output
        y2 = kda.output_norm_gate(o, gate.as_torch("cuda"), torch.from_numpy(wv).cuda(), eps)
        np.testing.assert_allclose(yg, y2.float().cpu().numpy(),
                                   rtol=(2.0 ** -7 if dtype == "bf16" else 1e-5), atol=1e-5)
