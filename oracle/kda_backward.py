"""Gradients of the KDA forward, plain fp64 PyTorch on the CPU -- test infrastructure only
(the product never imports it, and it imports nothing from the product).

Source: "Kimi k3 技术报告详解（1）——架构再升华", section "Kimi Delta Attention": per sequence
and head, with S d_k x d_v,
    g_t = g_min Sigmoid(e^{A_h} z_t)        (section "Chunkwise parallel form")
    S'_t = Diag(exp(g_t)) S_{t-1}
    u_t  = beta_t (v_t - S'_t^T k_t)
    S_t  = S'_t + k_t u_t^T                  (= (I - beta k k^T) Diag(alpha) S + beta k v^T)
    o_t  = S_t^T q_t
The forward is written out token by token with torch operations (heads batched), and the
gradients of  L = sum_t <do_t, o_t> + <dS_out, S_T>  with respect to q, k, v, beta, z,
A_log and S0 come from torch's reverse-mode differentiation of that program.  The pages
print no backward; this is the exact derivative of the forward they define.

`backward_chunked` is a second, independent ordering of the same gradients: the chunk form
of the forward (section "Chunkwise parallel form") with explicit fp64 decay products, and its
reverse derived by hand, carried back chunk by chunk (numpy only, no autodiff).
"""
from __future__ import annotations

import numpy as np
import torch


def _forward(q, k, v, beta, z, A_log, g_min, S0, cu):
    """Token recurrence; returns (o [T, H, dv], S_out [N, H, dk, dv]) as torch fp64."""
    T, H, dk = q.shape
    dv = v.shape[2]
    N = len(cu) - 1
    scale = torch.exp(A_log)                                       # [H]
    outs, finals = [], []
    for n in range(N):
        S = S0[n] if S0 is not None else torch.zeros((H, dk, dv), dtype=q.dtype)
        for t in range(int(cu[n]), int(cu[n + 1])):
            g = g_min * torch.sigmoid(scale[:, None] * z[t])       # [H, dk]
            Sp = torch.exp(g)[:, :, None] * S                      # Diag(alpha) S
            w = v[t] - torch.einsum("hij,hi->hj", Sp, k[t])        # v - S'^T k
            u = beta[t][:, None] * w
            S = Sp + k[t][:, :, None] * u[:, None, :]
            outs.append(torch.einsum("hij,hi->hj", S, q[t]))
        finals.append(S)
    o = torch.stack(outs) if outs else torch.zeros((0, H, dv), dtype=q.dtype)
    return o, torch.stack(finals)


def forward(q, k, v, beta, z, A_log, g_min: float, S0=None, cu_seqlens=None):
    """The forward (numpy in, numpy fp64 out) -- pinned against the C oracle."""
    t = [torch.as_tensor(np.asarray(x, dtype=np.float64)) for x in (q, k, v, beta, z, A_log)]
    T = t[0].shape[0]
    cu = [0, T] if cu_seqlens is None else [int(x) for x in cu_seqlens]
    S0t = None if S0 is None else torch.as_tensor(np.asarray(S0, dtype=np.float64))
    with torch.no_grad():
        o, S = _forward(*t, float(g_min), S0t, cu)
    return o.numpy(), S.numpy()


def backward(q, k, v, beta, z, A_log, g_min: float, do, S0=None, dS_out=None,
             cu_seqlens=None):
    """Gradients of sum(do * o) + sum(dS_out * S_out).

    Returns a dict of fp64 numpy arrays: dq, dk, dv [T, H, d], dbeta [T, H], dz [T, H, dk],
    dA_log [H], dS0 [N, H, dk, dv] (zeros' gradient when S0 is None).
    """
    names = ("q", "k", "v", "beta", "z", "A_log")
    leaves = {nm: torch.tensor(np.asarray(x, dtype=np.float64), requires_grad=True)
              for nm, x in zip(names, (q, k, v, beta, z, A_log))}
    T, H, dk = leaves["q"].shape
    dv = leaves["v"].shape[2]
    cu = [0, T] if cu_seqlens is None else [int(x) for x in cu_seqlens]
    N = len(cu) - 1
    S0t = torch.tensor(np.zeros((N, H, dk, dv)) if S0 is None else np.asarray(S0, np.float64),
                       requires_grad=True)
    o, S = _forward(*(leaves[nm] for nm in names), float(g_min), S0t, cu)
    loss = (o * torch.as_tensor(np.asarray(do, dtype=np.float64))).sum()
    if dS_out is not None:
        loss = loss + (S * torch.as_tensor(np.asarray(dS_out, dtype=np.float64))).sum()
    loss.backward()
    out = {"d" + nm: leaves[nm].grad.numpy() for nm in names}
    out["dS0"] = S0t.grad.numpy()
    return out


def _chunk_backward(Q, K, V, B, Z, a_log, g_min, S, dO, dS):
    """One chunk of one (sequence, head): the chunk form of the forward written out with
    explicit fp64 decay products, and its reverse-mode derivatives by hand.

    Forward ("Chunkwise parallel form"): G = cumsum(g), Γ = e^G, γ^C = e^{G_last};
    K⁺ = Γ⊙K, K⁻ = K/Γ, Q⁺ = Γ⊙Q, K^c = K⊙(γ^C/Γ); L = StrictTril(Diag(β) K⁺ K⁻ᵀ);
    N = (I+L)⁻¹, M = N Diag(β); W = M K⁺, U = M V, Ṽ = U − W S; A = Tril(Q⁺ K⁻ᵀ);
    O = Q⁺ S + A Ṽ; S_end = Diag(γ^C) S + K^cᵀ Ṽ.
    Returns (dQ, dK, dV, dβ, dz, dA_log contribution, dS at the chunk start).
    """
    x = np.exp(a_log) * Z
    sg = 1.0 / (1.0 + np.exp(-x))
    G = np.cumsum(g_min * sg, axis=0)
    Gm = np.exp(G)
    gC = Gm[-1]
    Kp, Km, Qp, Kc = Gm * K, K / Gm, Gm * Q, K * (gC / Gm)
    C = K.shape[0]
    KK = Kp @ Km.T
    L = np.tril(B[:, None] * KK, -1)
    N = np.linalg.solve(np.eye(C) + L, np.eye(C))
    M = N * B[None, :]
    W, U = M @ Kp, M @ V
    Vt = U - W @ S
    A = np.tril(Qp @ Km.T)
    # reverse
    dVt = A.T @ dO + Kc @ dS
    dS0 = Qp.T @ dO + gC[:, None] * dS - W.T @ dVt
    dA = np.tril(dO @ Vt.T)
    dQp = dO @ S.T + dA @ Km
    dKm = dA.T @ Qp
    dKc = Vt @ dS.T
    dW = -dVt @ S.T
    dM = dW @ Kp.T + dVt @ V.T
    dKp = M.T @ dW
    dV = M.T @ dVt
    dB = np.sum(N * dM, axis=0)
    dL = -np.tril(N.T @ (dM * B[None, :]) @ N.T, -1)
    dB += np.sum(dL * KK, axis=1)
    dKp += (B[:, None] * dL) @ Km
    dKm += (B[:, None] * dL).T @ Kp
    dK = Gm * dKp + dKm / Gm + (gC / Gm) * dKc
    dQ = Gm * dQp
    dG = dKp * Kp - dKm * Km + dQp * Qp - dKc * Kc
    dG[-1] += np.sum(dKc * Kc, axis=0) + gC * np.sum(dS * S, axis=1)
    dg = np.cumsum(dG[::-1], axis=0)[::-1]
    dx = dg * g_min * sg * (1.0 - sg)
    return dQ, dK, dV, dB, dx * np.exp(a_log), float(np.sum(dx * x)), dS0


def backward_chunked(q, k, v, beta, z, A_log, g_min: float, do, S0=None, dS_out=None,
                     cu_seqlens=None, C: int = 64):
    """The same gradients as `backward`, in a second, independent ordering: chunk by chunk
    (C rows; the last chunk of a sequence may be shorter), states at the chunk starts from the
    chunk-form forward, and the gradient carried back chunk by chunk by the hand-derived
    reverse of that form.  fp64 numpy; returns the same dict as `backward`."""
    q, k, v, beta, z, do = (np.asarray(a, dtype=np.float64) for a in (q, k, v, beta, z, do))
    A_log = np.asarray(A_log, dtype=np.float64)
    T, H, dk = q.shape
    dv = v.shape[2]
    cu = [0, T] if cu_seqlens is None else [int(x) for x in cu_seqlens]
    Nseq = len(cu) - 1
    out = {"dq": np.zeros_like(q), "dk": np.zeros_like(k), "dv": np.zeros_like(v),
           "dbeta": np.zeros_like(beta), "dz": np.zeros_like(z), "dA_log": np.zeros(H),
           "dS0": np.zeros((Nseq, H, dk, dv))}
    for n in range(Nseq):
        a, b = cu[n], cu[n + 1]
        starts = list(range(a, b, C))
        for h in range(H):
            S = (np.zeros((dk, dv)) if S0 is None else np.asarray(S0, np.float64)[n, h].copy())
            states = []
            for t0 in starts:  # forward: the state at every chunk start
                t1 = min(t0 + C, b)
                states.append(S)
                x = np.exp(A_log[h]) * z[t0:t1, h]
                G = np.cumsum(g_min / (1.0 + np.exp(-x)), axis=0)
                Gm = np.exp(G)
                Kp, Km, Kc = Gm * k[t0:t1, h], k[t0:t1, h] / Gm, k[t0:t1, h] * (Gm[-1] / Gm)
                Bv = beta[t0:t1, h]
                L = np.tril(Bv[:, None] * (Kp @ Km.T), -1)
                M = np.linalg.solve(np.eye(t1 - t0) + L, np.diag(Bv))
                Vt = M @ v[t0:t1, h] - (M @ Kp) @ S
                S = Gm[-1][:, None] * S + Kc.T @ Vt
            dS = (np.zeros((dk, dv)) if dS_out is None
                  else np.asarray(dS_out, np.float64)[n, h].copy())
            for ci in range(len(starts) - 1, -1, -1):  # backward, last chunk first
                t0 = starts[ci]
                t1 = min(t0 + C, b)
                r = _chunk_backward(q[t0:t1, h], k[t0:t1, h], v[t0:t1, h], beta[t0:t1, h],
                                    z[t0:t1, h], A_log[h], g_min, states[ci], do[t0:t1, h], dS)
                out["dq"][t0:t1, h], out["dk"][t0:t1, h], out["dv"][t0:t1, h] = r[0], r[1], r[2]
                out["dbeta"][t0:t1, h], out["dz"][t0:t1, h] = r[3], r[4]
                out["dA_log"][h] += r[5]
                dS = r[6]
            out["dS0"][n, h] = dS
    return out
