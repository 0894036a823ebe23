"""Pins for the backward oracle (fp64 torch reverse-mode differentiation of the token
recurrence of "Kimi k3 技术报告详解（1）", section "Kimi Delta Attention").

What pins what:
  forward          the torch program's outputs equal the C oracle's token recurrence
                   (itself pinned in test_oracle_pins.py) to 1e-12
  finite diffs     central differences of the loss in every input (q, k, v, beta, z, A_log,
                   S0) agree with the returned gradients on tiny problems (a dropped term or
                   a transposed operand in the forward changes one of them)
  two orderings    the hand-derived reverse of the chunk form (backward_chunked), chunk by
                   chunk, agrees with the reverse mode through the token recurrence
  closed forms     with beta = 0 and alpha = 1 (z = -inf) the state is S0 throughout, so
                   dq_t = S0 do_t, dS0 = sum_t q_t do_t^T + dS_out, and dv = dk = 0
"""
import numpy as np
import pytest

import oracle
from oracle import kda_backward as kb


def _prob(seed, T, H, dk, dv, lengths=None):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, dv))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, H))))
    z = rng.standard_normal((T, H, dk))
    A = rng.uniform(-1.0, 1.0, H)
    cu = None if lengths is None else np.concatenate([[0], np.cumsum(lengths)])
    N = 1 if lengths is None else len(lengths)
    S0 = 0.3 * rng.standard_normal((N, H, dk, dv))
    do = rng.standard_normal((T, H, dv))
    dS = rng.standard_normal((N, H, dk, dv))
    return q, k, v, beta, z, A, S0, do, dS, cu


def test_forward_matches_c_oracle():
    q, k, v, beta, z, A, S0, do, dS, cu = _prob(1, 40, 2, 8, 6, lengths=[15, 0, 25])
    o, S = kb.forward(q, k, v, beta, z, A, -5.0, S0=S0, cu_seqlens=cu)
    o_c, S_c = oracle.recurrent(q, k, v, beta, z, A, -5.0, S0=S0, cu_seqlens=cu)
    np.testing.assert_allclose(o, o_c, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(S, S_c, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("lengths", [None, [3, 0, 4]])
def test_gradients_match_central_differences(lengths):
    T = 6 if lengths is None else sum(lengths)
    q, k, v, beta, z, A, S0, do, dS, cu = _prob(2, T, 2, 3, 2, lengths=lengths)
    g = kb.backward(q, k, v, beta, z, A, -4.0, do, S0=S0, dS_out=dS, cu_seqlens=cu)
    args = dict(q=q, k=k, v=v, beta=beta, z=z, A_log=A, S0=S0)

    def loss(**kw):
        a = dict(args)
        a.update(kw)
        o, S = kb.forward(a["q"], a["k"], a["v"], a["beta"], a["z"], a["A_log"], -4.0,
                          S0=a["S0"], cu_seqlens=cu)
        return float(np.sum(o * do) + np.sum(S * dS))

    h = 1e-6
    for name, x in args.items():
        grad = g["d" + name] if name != "A_log" else g["dA_log"]
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            num[idx] = (loss(**{name: xp}) - loss(**{name: xm})) / (2 * h)
        np.testing.assert_allclose(grad, num, rtol=1e-6, atol=1e-8, err_msg=name)


def test_closed_form_without_decay_or_writes():
    q, k, v, beta, z, A, S0, do, dS, cu = _prob(3, 9, 2, 5, 4)
    beta[:] = 0.0
    z[:] = -np.inf
    g = kb.backward(q, k, v, beta, z, A, -5.0, do, S0=S0, dS_out=dS)
    np.testing.assert_allclose(g["dq"], np.einsum("hij,thj->thi", S0[0], do), rtol=1e-13)
    np.testing.assert_allclose(g["dS0"][0], np.einsum("thi,thj->hij", q, do) + dS[0],
                               rtol=1e-13)
    assert np.all(g["dv"] == 0.0) and np.all(g["dk"] == 0.0)


@pytest.mark.parametrize("C", [1, 4, 16, 64])
def test_chunked_ordering_matches_reverse_mode(C):
    """Two independent orderings of the same gradients: torch's reverse mode through the
    token recurrence, and the hand-derived reverse of the chunk form, chunk by chunk.  C = 1
    reduces the chunk form to the token step; ragged last chunks, an empty sequence and
    d_k != d_v included."""
    lengths = [70, 0, 37, 5]
    q, k, v, beta, z, A, S0, do, dS, cu = _prob(4, sum(lengths), 2, 6, 3, lengths=lengths)
    ref = kb.backward(q, k, v, beta, z, A, -5.0, do, S0=S0, dS_out=dS, cu_seqlens=cu)
    got = kb.backward_chunked(q, k, v, beta, z, A, -5.0, do, S0=S0, dS_out=dS, cu_seqlens=cu,
                              C=C)
    for nm in ("dq", "dk", "dv", "dbeta", "dz", "dA_log", "dS0"):
        scale = np.max(np.abs(ref[nm])) if ref[nm].size else 1.0
        assert np.max(np.abs(got[nm] - ref[nm])) <= 1e-10 * max(scale, 1e-30), nm
