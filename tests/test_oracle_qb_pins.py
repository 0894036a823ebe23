"""Pins for the quantile-balancing oracle against what the pages fix.

Source: "Kimi k3 技术报告详解（1）——架构再升华", "Quantile Balancing (QB)": alpha_i is the
(k+1)-th largest score of token i; with margin_ij = s_ij - alpha_i, expert j receives
sum_i 1[margin_ij > -bhat_j] tokens, and bhat_j is chosen so that this count is exactly q;
the mean of the biases is then removed.

What pins what:
  k chosen per token  with alpha from the current biases, exactly k experts of every token
                      have s_ij + b_j > alpha_i (a wrong order statistic or a dropped bias)
  exact count q       under bhat, every expert receives exactly q = floor(m k / n) tokens
                      where its threshold margin is not tied, and in general at most q
                      strictly above it and at least q + 1 reaching it (a wrong rank, sign
                      or axis breaks it)
  mean removal        the new biases sum to zero and differ from bhat by one constant
  shift invariance    adding a constant to every score leaves the update unchanged
  rank by counting    on tiny inputs, selection by explicit counting (x is the r-th largest
                      when fewer than r values exceed it and at least r reach it) agrees
"""
import numpy as np
import pytest

from oracle import quantile_balance as qb


def _scores(seed, m, n):
    rng = np.random.default_rng(seed)
    popularity = rng.normal(0.0, 0.5, size=n).astype(np.float32)
    s = rng.standard_normal((m, n)).astype(np.float32) + popularity[None, :]
    b = rng.normal(0.0, 0.1, size=n).astype(np.float32)
    return s, b


@pytest.mark.parametrize("m,n,k", [(1000, 16, 2), (4096, 64, 8), (333, 7, 3)])
def test_thresholds_select_exactly_k(m, n, k):
    s, b = _scores(1, m, n)
    alpha = qb.token_thresholds(s, b, k)
    chosen = (s + b[None, :]) > alpha[:, None]
    assert np.all(chosen.sum(axis=1) == k)


@pytest.mark.parametrize("m,n,k", [(1000, 16, 2), (4096, 64, 8), (333, 7, 3), (50, 50, 1)])
def test_every_expert_receives_exactly_q(m, n, k):
    s, b = _scores(2, m, n)
    b_new, bhat, alpha = qb.quantile_balance(s, b, k)
    q = qb.target_count(m, n, k)
    margin = s - alpha[:, None]
    above = (margin > -bhat[None, :]).sum(axis=0)
    reach = (margin >= -bhat[None, :]).sum(axis=0)
    # -bhat_j is the (q+1)-th largest margin: at most q above it, at least q+1 reach it ...
    assert np.all(above <= q) and np.all(reach >= q + 1), (above, reach)
    # ... so the count is exactly q wherever that margin is not tied.  Ties are structural:
    # the token whose (k+1)-th choice is expert j has margin exactly -b_j there.
    untied = reach == above + 1
    assert untied.sum() >= n // 2
    assert np.all(above[untied] == q)


def test_mean_removed():
    s, b = _scores(3, 2048, 32)
    b_new, bhat, _ = qb.quantile_balance(s, b, 4)
    assert abs(b_new.sum()) < 1e-12
    d = b_new - bhat.astype(np.float64)
    np.testing.assert_allclose(d, d[0], rtol=0, atol=1e-12)


def test_shift_invariance():
    rng = np.random.default_rng(4)
    # scores on a dyadic grid, so that adding 0.5 is exact in fp32
    s = (rng.integers(-4096, 4096, size=(700, 12)) / 1024.0).astype(np.float32)
    b = (rng.integers(-64, 64, size=12) / 1024.0).astype(np.float32)
    r1 = qb.quantile_balance(s, b, 3)
    r2 = qb.quantile_balance(s + np.float32(0.5), b, 3)
    assert np.array_equal(r1[1], r2[1]) and np.array_equal(r1[0], r2[0])


def _rth_largest_by_counting(values, r):
    """The r-th largest (1-based) of a list, by counting (ties counted separately)."""
    for x in values:
        above = sum(1 for y in values if y > x)
        reach = sum(1 for y in values if y >= x)
        if above < r <= reach:
            return x
    raise AssertionError("no r-th largest")


@pytest.mark.parametrize("seed", range(5))
def test_tiny_inputs_by_counting(seed):
    m, n, k = 12, 5, 2
    s, b = _scores(10 + seed, m, n)
    s[3, :] = s[3, 0]  # a row of ties
    b_new, bhat, alpha = qb.quantile_balance(s, b, k)
    q = qb.target_count(m, n, k)
    for i in range(m):
        row = [np.float32(s[i, j] + b[j]) for j in range(n)]
        assert alpha[i] == _rth_largest_by_counting(row, k + 1)
    for j in range(n):
        col = [np.float32(s[i, j] - alpha[i]) for i in range(m)]
        assert bhat[j] == -_rth_largest_by_counting(col, q + 1)
