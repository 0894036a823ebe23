"""Pins for the fp64 oracle, each against something other than the oracle itself.

Sources: the KDA recurrence and chunkwise-parallel form from "Kimi k3 技术报告详解（1）——架构再升华"
(sections "Kimi Delta Attention" and "Chunkwise parallel form"); the bounded gate from the same page
and from "A Look at Kimi K3: Three Core Innovations and Engineering Tuning Guide" section 2.2.

What pins what:
  gate        closed-form special values (z = 0, z = ln 3, z = +-inf), the reflection
              g(z) + g(-z) = g_min, the A_h scaling law, the range (g_min, 0), the printed
              value e^-5 ~ 0.0067, and the page's torch pseudocode.
  recurrence  state held (beta = 0, alpha = 1); delta-rule exact overwrite with one-hot and
              orthonormal keys; brute-force unrolling into explicit matrix products on tiny
              inputs; the transposed delta-rule formula of the page at alpha = 1; linearity
              in (V, S0); pure-decay closed form at k = 0; varlen = separate calls; resume.
  chunked     agreement with the recurrence to 1e-10 for C in {1, 4, 16, 64}, ragged tails,
              g_min in {-3, -5, -6}.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def _problem(seed, T, H, dk, dv, N_state=1, unit=True):
    r = _rng(seed)
    q = r.standard_normal((T, H, dk))
    k = r.standard_normal((T, H, dk))
    if unit:
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = r.standard_normal((T, H, dv))
    beta = 1.0 / (1.0 + np.exp(-r.standard_normal((T, H))))
    z = r.standard_normal((T, H, dk))
    A_log = r.uniform(-1, 1, H)
    S0 = 0.02 * r.standard_normal((N_state, H, dk, dv))
    return q, k, v, beta, z, A_log, S0


# ------------------------------------------------------------------ gate --


@pytest.mark.parametrize("g_min", [-3.0, -5.0, -6.0])
def test_gate_special_values(g_min):
    for A in (-1.0, 0.0, 0.7):
        assert oracle.gate_value(0.0, A, g_min) == g_min / 2        # sigmoid(0) = 1/2
        assert oracle.gate_value(-math.inf, A, g_min) == 0.0        # alpha = 1: no decay
        assert oracle.gate_value(math.inf, A, g_min) == g_min       # the lower bound
    # sigmoid(ln 3) = 3/4 exactly in real arithmetic
    assert oracle.gate_value(math.log(3.0), 0.0, g_min) == pytest.approx(0.75 * g_min, rel=1e-15)


def test_gate_reflection_scaling_and_range():
    r = _rng(7)
    z = r.standard_normal((50, 3, 16)) * 4
    A = r.uniform(-1, 1, 3)
    for g_min in (-3.0, -5.0, -6.0):
        g = oracle.gate(z, A, g_min)
        g_neg = oracle.gate(-z, A, g_min)
        np.testing.assert_allclose(g + g_neg, g_min, rtol=0, atol=1e-14)   # s(x)+s(-x)=1
        g0 = oracle.gate(z * np.exp(A)[None, :, None], np.zeros(3), g_min)  # e^{A} scales z
        np.testing.assert_allclose(g, g0, rtol=1e-14, atol=0)
        assert np.all(g < 0) and np.all(g > g_min)
        alpha = np.exp(g)
        assert np.all(alpha < 1) and np.all(alpha > math.exp(g_min))
        # monotone non-increasing in z for g_min < 0
        zs = np.sort(z.reshape(-1))
        gs = oracle.gate(zs.reshape(-1, 1, 1), np.zeros(1), g_min).reshape(-1)
        assert np.all(np.diff(gs) <= 0)


def test_gate_printed_lower_bound():
    fx = json.load(open(os.path.join(GOLDEN, "gate_bound.json")))
    for case in fx["cases"]:
        g_min = case["g_min"]
        lowest = math.exp(oracle.gate_value(math.inf, 0.0, g_min))
        assert round(lowest, case["digits"]) == case["alpha_lower_bound"]


def test_gate_matches_page_pseudocode():
    torch = pytest.importorskip("torch")
    r = _rng(3)
    z = r.standard_normal((40, 4, 8))
    A = r.uniform(-1, 1, 4)
    ref = (-5.0 * torch.sigmoid(torch.exp(torch.from_numpy(A))[None, :, None]
                                * torch.from_numpy(z))).numpy()
    np.testing.assert_allclose(oracle.gate(z, A, -5.0), ref, rtol=1e-14, atol=1e-15)


# ------------------------------------------------------------ recurrence --


def test_state_held_when_beta_zero_and_no_decay():
    q, k, v, beta, z, A, S0 = _problem(11, 37, 2, 16, 12)
    beta[:] = 0.0
    z[:] = -np.inf                      # alpha = 1
    o, S = oracle.recurrent(q, k, v, beta, z, A, -5.0, S0=S0)
    np.testing.assert_array_equal(S, S0)
    np.testing.assert_allclose(o, np.einsum("thi,hij->thj", q, S0[0]), rtol=1e-13, atol=1e-16)


def test_delta_rule_one_hot_overwrite():
    T, H, dk, dv = 20, 1, 8, 5
    q, k, v, beta, z, A, S0 = _problem(12, T, H, dk, dv)
    z[:] = -np.inf
    beta[:] = 1.0
    idx = _rng(5).integers(0, dk, size=T)
    k[:] = 0.0
    k[np.arange(T), 0, idx] = 1.0
    S = S0[0, 0].copy()
    for t in range(T):
        _, S_new = oracle.recurrent(q[t:t + 1], k[t:t + 1], v[t:t + 1], beta[t:t + 1],
                                    z[t:t + 1], A, -5.0, S0=S[None, None])
        others = np.arange(dk) != idx[t]
        # every other row is untouched bit for bit; row idx[t] becomes v^T (S_i + (v - S_i))
        np.testing.assert_array_equal(S_new[0, 0][others], S[others])
        np.testing.assert_allclose(S_new[0, 0][idx[t]], v[t, 0], rtol=0, atol=1e-15)
        S = S_new[0, 0]


def test_delta_rule_orthonormal_keys_store_values():
    dk, dv, T = 16, 6, 10
    q, _, v, beta, z, A, S0 = _problem(13, T, 1, dk, dv)
    Qm, _ = np.linalg.qr(_rng(9).standard_normal((dk, dk)))
    k = Qm[:, :T].T.reshape(T, 1, dk).copy()
    z[:] = -np.inf
    beta[:] = 1.0
    _, S = oracle.recurrent(q, k, v, beta, z, A, -5.0, S0=S0)
    for t in range(T):
        np.testing.assert_allclose(S[0, 0].T @ k[t, 0], v[t, 0], rtol=0, atol=1e-12)


def _brute_force(q, k, v, beta, alpha, S0):
    """S_T = (A_T...A_1) S0 + sum_t (A_T...A_{t+1}) B_t with dense A_t, B_t."""
    T, dk = q.shape
    A_mats = [(np.eye(dk) - beta[t] * np.outer(k[t], k[t])) @ np.diag(alpha[t]) for t in range(T)]
    B_mats = [beta[t] * np.outer(k[t], v[t]) for t in range(T)]
    outs = []
    for tt in range(1, T + 1):
        P = np.eye(dk)
        for t in range(tt):
            P = A_mats[t] @ P
        S = P @ S0
        for t in range(tt):
            Pt = np.eye(dk)
            for s in range(t + 1, tt):
                Pt = A_mats[s] @ Pt
            S = S + Pt @ B_mats[t]
        outs.append((S.T @ q[tt - 1], S))
    return outs


@pytest.mark.parametrize("dk,dv,T", [(2, 2, 5), (3, 4, 8), (4, 3, 7)])
def test_brute_force_unrolling(dk, dv, T):
    q, k, v, beta, z, A, S0 = _problem(20 + dk, T, 1, dk, dv, unit=False)
    g_min = -5.0
    alpha = np.exp(oracle.gate(z, A, g_min))[:, 0]
    o, S = oracle.recurrent(q, k, v, beta, z, A, g_min, S0=S0)
    ref = _brute_force(q[:, 0], k[:, 0], v[:, 0], beta[:, 0], alpha, S0[0, 0])
    for t in range(T):
        np.testing.assert_allclose(o[t, 0], ref[t][0], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(S[0, 0], ref[-1][1], rtol=1e-12, atol=1e-14)


def test_page_delta_rule_orientation_at_unit_decay():
    """At alpha = 1 the page's delta rule S_t = S_{t-1}(I - b k k^T) + b v k^T, o_t = S_t q_t
    (value-by-key orientation) must give the same outputs as the key-by-value recurrence."""
    T, dk, dv = 25, 8, 6
    q, k, v, beta, z, A, S0 = _problem(31, T, 1, dk, dv)
    z[:] = -np.inf
    o, S = oracle.recurrent(q, k, v, beta, z, A, -5.0, S0=S0)
    Sv = S0[0, 0].T.copy()                               # d_v x d_k
    for t in range(T):
        kt, vt, bt = k[t, 0], v[t, 0], beta[t, 0]
        Sv = Sv @ (np.eye(dk) - bt * np.outer(kt, kt)) + bt * np.outer(vt, kt)
        np.testing.assert_allclose(o[t, 0], Sv @ q[t, 0], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(S[0, 0], Sv.T, rtol=1e-12, atol=1e-14)


def test_linearity_in_values_and_state():
    q, k, v1, beta, z, A, S01 = _problem(41, 30, 2, 8, 8)
    _, _, v2, _, _, _, S02 = _problem(42, 30, 2, 8, 8)
    o1, s1 = oracle.recurrent(q, k, v1, beta, z, A, -5.0, S0=S01)
    o2, s2 = oracle.recurrent(q, k, v2, beta, z, A, -5.0, S0=S02)
    o3, s3 = oracle.recurrent(q, k, v1 + v2, beta, z, A, -5.0, S0=S01 + S02)
    np.testing.assert_allclose(o3, o1 + o2, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(s3, s1 + s2, rtol=1e-12, atol=1e-13)


def test_pure_decay_when_keys_vanish():
    q, k, v, beta, z, A, S0 = _problem(51, 40, 2, 8, 5)
    k[:] = 0.0
    g_min = -3.0
    g = oracle.gate(z, A, g_min)
    o, S = oracle.recurrent(q, k, v, beta, z, A, g_min, S0=S0)
    logdecay = np.cumsum(g, axis=0)                      # sum of g over tokens 1..t
    for t in range(40):
        St = np.exp(logdecay[t])[:, :, None] * S0[0]     # Diag(gamma^{1->t}) S0 per head
        np.testing.assert_allclose(o[t], np.einsum("hi,hij->hj", q[t], St), rtol=1e-12,
                                   atol=1e-16)


def test_varlen_equals_separate_and_resume():
    lens = [5, 0, 67, 1, 130]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T = int(cu[-1])
    q, k, v, beta, z, A, S0 = _problem(61, T, 2, 8, 6, N_state=len(lens))
    o, S = oracle.recurrent(q, k, v, beta, z, A, -5.0, S0=S0, cu_seqlens=cu)
    for n in range(len(lens)):
        a, b = cu[n], cu[n + 1]
        on, Sn = oracle.recurrent(q[a:b], k[a:b], v[a:b], beta[a:b], z[a:b], A, -5.0,
                                  S0=S0[n:n + 1])
        np.testing.assert_array_equal(o[a:b], on)
        np.testing.assert_array_equal(S[n], Sn[0])
    # resume: split the longest sequence at an arbitrary point and chain the state
    a, b = cu[4], cu[5]
    m = a + 77
    o1, S1 = oracle.recurrent(q[a:m], k[a:m], v[a:m], beta[a:m], z[a:m], A, -5.0, S0=S0[4:5])
    o2, S2 = oracle.recurrent(q[m:b], k[m:b], v[m:b], beta[m:b], z[m:b], A, -5.0, S0=S1)
    np.testing.assert_allclose(np.concatenate([o1, o2]), o[a:b], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(S2[0], S[4], rtol=1e-13, atol=1e-15)


# ---------------------------------------------------------------- chunked --


def _rel(a, b):
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


@pytest.mark.parametrize("C", [1, 4, 16, 64])
@pytest.mark.parametrize("g_min", [-3.0, -5.0, -6.0])
def test_chunked_matches_recurrence(C, g_min):
    lens = [150, 64, 3]
    cu = np.concatenate([[0], np.cumsum(lens)])
    q, k, v, beta, z, A, S0 = _problem(71, int(cu[-1]), 2, 16, 12, N_state=3)
    o_r, S_r = oracle.recurrent(q, k, v, beta, z, A, g_min, S0=S0, cu_seqlens=cu)
    o_c, S_c = oracle.chunked(q, k, v, beta, z, A, g_min, S0=S0, cu_seqlens=cu, C=C)
    assert _rel(o_c, o_r) < 1e-10
    assert _rel(S_c, S_r) < 1e-10


def test_chunked_matches_recurrence_full_width():
    """d = 64 and d = 128 with C = 64 at the most negative bound, two full chunks + a tail."""
    for d, T in ((64, 150), (128, 140)):
        q, k, v, beta, z, A, S0 = _problem(81 + d, T, 1, d, d)
        z *= 3.0                                  # push many gates to the bound
        o_r, S_r = oracle.recurrent(q, k, v, beta, z, A, -6.0, S0=S0)
        o_c, S_c = oracle.chunked(q, k, v, beta, z, A, -6.0, S0=S0, C=64)
        assert _rel(o_c, o_r) < 1e-10
        assert _rel(S_c, S_r) < 1e-10
