"""Pins for the oracle's negative-softplus gate: the gate the lower bound replaces.

Source: "Kimi k3 技术报告详解（1）——架构再升华", section "Chunkwise parallel form": before the
bound, g = -e^{A_h} Softplus(z) in (-inf, 0) and alpha = exp(g); the bound replaces it with
g_min Sigmoid(e^{A_h} z).  The recurrence itself is unchanged, so the pins are the gate's
closed forms plus the recurrence pins that involve the gate.

What pins what:
  closed forms      z = 0 gives -e^A ln 2; Softplus(z) - Softplus(-z) = z, so
                    g(z) - g(-z) = -e^A z; for large z, g ~ -e^A z (no lower bound: the
                    gate passes any g_min)
  no decay at -inf  z -> -inf gives g = -0, alpha = 1: with beta = 0 the state is held
  pure decay        with k = 0, o_t = (Diag(prod of alpha) S0)^T q_t, alpha from the gate
  two orderings     the chunked form agrees with the recurrence (moderate z, where the fp64
                    decay products stay in range)
"""
import math

import numpy as np
import pytest

import oracle


@pytest.mark.parametrize("A", [-1.0, 0.0, 0.7])
def test_closed_forms(A):
    e = math.exp(A)
    assert oracle.gate_softplus_value(0.0, A) == pytest.approx(-e * math.log(2.0), rel=1e-15)
    for z in (0.3, 2.0, 17.0):
        d = oracle.gate_softplus_value(z, A) - oracle.gate_softplus_value(-z, A)
        assert d == pytest.approx(-e * z, rel=1e-13)
    assert oracle.gate_softplus_value(40.0, A) == pytest.approx(-e * 40.0, rel=1e-15)
    assert oracle.gate_softplus_value(10.0, A) < -6.0 * e  # below any g_min in [-6, -3]
    assert -1e-17 < oracle.gate_softplus_value(-40.0, A) < 0.0


def _rand(seed, T, H, dk, dv):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, dv))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, H))))
    z = rng.standard_normal((T, H, dk))
    A = rng.uniform(-1.0, 1.0, H)
    S0 = 0.02 * rng.standard_normal((1, H, dk, dv))
    return q, k, v, beta, z, A, S0


def test_state_held_without_decay_or_writes():
    q, k, v, beta, z, A, S0 = _rand(1, 20, 2, 8, 5)
    beta[:] = 0.0
    z[:] = -np.inf
    o, S = oracle.recurrent(q, k, v, beta, z, A, -5.0, S0=S0, gate="softplus")
    assert np.array_equal(S, S0)
    np.testing.assert_allclose(o, np.einsum("thc,hcj->thj", q, S0[0]), rtol=1e-14, atol=1e-16)


def test_pure_decay_closed_form():
    q, k, v, beta, z, A, S0 = _rand(2, 15, 2, 6, 4)
    k[:] = 0.0
    o, _ = oracle.recurrent(q, k, v, beta, z, A, -5.0, S0=S0, gate="softplus")
    sp = np.logaddexp(0.0, z)                                  # softplus, independent form
    logalpha = -np.exp(A)[None, :, None] * sp                  # [T, H, dk]
    cum = np.cumsum(logalpha, axis=0)
    ref = np.einsum("thc,thc,hcj->thj", q, np.exp(cum), S0[0])
    np.testing.assert_allclose(o, ref, rtol=1e-12, atol=1e-15)


@pytest.mark.parametrize("C", [1, 16, 64])
def test_chunked_matches_recurrence(C):
    q, k, v, beta, z, A, S0 = _rand(3, 150, 2, 16, 8)
    o_r, S_r = oracle.recurrent(q, k, v, beta, z, A, -5.0, S0=S0, gate="softplus")
    o_c, S_c = oracle.chunked(q, k, v, beta, z, A, -5.0, S0=S0, C=C, gate="softplus")
    scale = np.sqrt(np.mean(o_r ** 2))
    assert np.max(np.abs(o_c - o_r)) / scale < 1e-10
    assert np.max(np.abs(S_c - S_r)) / np.sqrt(np.mean(S_r ** 2)) < 1e-10


def test_softplus_differs_from_bounded_gate():
    """The two gates give different results (the switch reaches the recurrence)."""
    q, k, v, beta, z, A, S0 = _rand(4, 30, 1, 8, 4)
    o1, _ = oracle.recurrent(q, k, v, beta, z, A, -5.0, S0=S0, gate="softplus")
    o2, _ = oracle.recurrent(q, k, v, beta, z, A, -5.0, S0=S0, gate="sigmoid")
    assert np.max(np.abs(o1 - o2)) > 1e-3
