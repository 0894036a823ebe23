"""Quantile-balancing bias update, plain numpy -- test infrastructure only (see the package
docstring: the product never imports it, and it imports nothing from the product).

Source: "Kimi k3 技术报告详解（1）——架构再升华", section on load balancing, "Quantile
Balancing (QB)"; also "A Look at Kimi K3 ..." section 4.2 (thresholds from per-expert
quantiles of the routing scores).  With router scores s [m tokens, n experts], k experts
chosen per token and the current expert biases b [n]:

  1. alpha_i = the (k+1)-th largest of s_i + b over the experts: the token's threshold
     (expert j is chosen for token i when s_ij + b_j > alpha_i).
  2. margin_ij = s_ij - alpha_i.
  3. Expert j would receive sum_i 1[margin_ij > -bhat_j] tokens under a candidate bias
     bhat_j; to make that exactly q = floor(m k / n), bhat_j = -(the (q+1)-th largest
     margin of column j), i.e. minus the (1 - k/n) quantile of the column.
  4. The new bias is bhat minus its mean (the common offset is a free degree of freedom).

Readings where the pages are silent: alpha uses the current biases (the (t) superscript on
alpha); q is rounded down when m k / n is not an integer; "(q+1)-th largest" counts equal
values separately (a sort, descending).  The scores and biases are fp32 and so are
s + b and the margins (they decide which element is selected, so the oracle forms them in
the precision the GPU uses); the mean is taken in fp64.
"""
from __future__ import annotations

import numpy as np


def target_count(m: int, n: int, k: int) -> int:
    """q: the number of tokens each expert should receive."""
    return (m * k) // n


def token_thresholds(s, b, k: int) -> np.ndarray:
    """alpha [m]: the (k+1)-th largest of s_i + b for each token (fp32)."""
    s = np.asarray(s, dtype=np.float32)
    b = np.asarray(b, dtype=np.float32)
    m, n = s.shape
    if not 0 <= k < n:
        raise ValueError(f"need 0 <= k < n (k={k}, n={n})")
    biased = s + b[None, :]                       # fp32
    return -np.sort(-biased, axis=1)[:, k]        # descending order, position k


def quantile_balance(s, b, k: int):
    """Returns (b_new [n] float64, bhat [n] float32, alpha [m] float32)."""
    s = np.asarray(s, dtype=np.float32)
    m, n = s.shape
    q = target_count(m, n, k)
    if q >= m:
        raise ValueError(f"q = {q} must be < m = {m}")
    alpha = token_thresholds(s, b, k)
    margin = s - alpha[:, None]                   # fp32
    bhat = -(-np.sort(-margin, axis=0))[q, :]     # minus the (q+1)-th largest per column
    bhat = bhat.astype(np.float32)
    b_new = bhat.astype(np.float64) - np.mean(bhat.astype(np.float64))
    return b_new, bhat, alpha
