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
