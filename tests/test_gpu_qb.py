"""GPU parity: the quantile-balancing bias update against the numpy oracle.

Source: "Kimi k3 技术报告详解（1）——架构再升华", "Quantile Balancing (QB)".  The token
thresholds alpha and the per-expert bhat are selections among fp32 values that both sides
form in fp32 (s + b, s - alpha), so they must agree bit for bit; the new biases
bhat - mean(bhat) differ only by the rounding of the mean.
"""
import numpy as np
import pytest

from oracle import quantile_balance as qb
from serving_kda_chunkwise_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kda():
    import torch  # noqa: F401
    from serving_kda_chunkwise_gb300 import kda as _k
    return _k


def _check(kda, s, b, k):
    import torch
    b_new, bhat, alpha = kda.quantile_balance(torch.from_numpy(s).cuda(),
                                              torch.from_numpy(b).cuda(), k, want_bhat=True,
                                              want_alpha=True)
    r_new, r_bhat, r_alpha = qb.quantile_balance(s, b, k)
    assert np.array_equal(alpha.cpu().numpy(), r_alpha)
    assert np.array_equal(bhat.cpu().numpy(), r_bhat)
    np.testing.assert_allclose(b_new.cpu().numpy(), r_new, rtol=0,
                               atol=1e-6 * max(1.0, float(np.max(np.abs(r_bhat)))))


@pytest.mark.parametrize("m,n,k", [(1000, 16, 2), (4096, 64, 8), (333, 7, 3), (5000, 1024, 31),
                                   (2048, 100, 0), (3, 5, 4), (1, 4, 1), (10000, 33, 32)])
def test_matches_oracle(kda, m, n, k):
    s, b = inputs.qb_inputs(seed=m + n + k, m=m, n=n)
    _check(kda, s, b, k)


@pytest.mark.parametrize("m,n,k", [(4000, 48, 6), (777, 9, 2)])
def test_ties(kda, m, n, k):
    """Scores and biases on a grid of 1/4: many equal values, counted separately."""
    s, b = inputs.qb_inputs(seed=5 + m, m=m, n=n, grid=0.25)
    assert len(np.unique(s)) < s.size // 10
    _check(kda, s, b, k)


@pytest.mark.parametrize("m,n,k", [(8192, 256, 8), (12000, 64, 5), (200000, 16, 3),
                                   (262144, 4, 1), (300000, 8, 2), (8192, 1024, 31),
                                   (16384, 32, 0)])
def test_sampled_bracket_sizes(kda, m, n, k):
    """Sizes at and around the sampled-bracket path's limits (8192 <= m <= 2^18, n a
    multiple of 4): the smallest m, a non-power-of-two sample count, sparser samples, the
    largest m and one past it (the radix path), the most experts, and k = 0 (q = 0: the
    largest margin, no upper bound to the bracket)."""
    s, b = inputs.qb_inputs(seed=m + 3 * n + k, m=m, n=n)
    _check(kda, s, b, k)


@pytest.mark.parametrize("m,n,k,grid", [(16384, 64, 6, 0.25), (65536, 64, 4, 1.0)])
def test_sampled_bracket_ties(kda, m, n, k, grid):
    """Coarse grids: the wanted margin is tied with thousands of others (on the grid of 1,
    more candidates than an expert's list holds, so the selection falls back to the whole
    column)."""
    s, b = inputs.qb_inputs(seed=11 + m + n, m=m, n=n, grid=grid)
    _check(kda, s, b, k)


def test_sampled_bracket_misses(kda):
    """A sample that misrepresents some experts: with m = 16384 every second token is
    sampled; expert 0 scores far higher on the sampled tokens, expert 1 far lower, and
    expert 2 far higher on the others, so their brackets miss the wanted margin and the
    selection recomputes them from the whole column."""
    m, n, k = 16384, 32, 2
    s, b = inputs.qb_inputs(seed=41, m=m, n=n)
    s[0::2, 0] += 20.0
    s[0::2, 1] -= 20.0
    s[1::2, 2] += 20.0
    _check(kda, s, b, k)


def test_sampled_bracket_wide(kda):
    """Half the experts per token (p = 1/2): the bracket holds about 36 k margins of each
    expert, more than the selection stages in shared memory (it reads them from the list) and
    more than a thread's candidate slots (the counting pass appends straight to the list)."""
    m, n, k = 262144, 4, 2
    s, b = inputs.qb_inputs(seed=91, m=m, n=n)
    _check(kda, s, b, k)


@pytest.mark.parametrize("stride", [32, 16])
def test_thresholds_concentrated(kda, stride):
    """Scores raised by 5 on every 32nd (16th) expert: the row's largest values sit in one
    (two) of the 32 lanes of the threshold kernel's warp, so one lane gives up value after
    value in its rounds."""
    m, n, k = 3000, 256, 8
    s, b = inputs.qb_inputs(seed=70 + stride, m=m, n=n)
    s[:, ::stride] += 5.0
    _check(kda, s, b, k)


def test_full_size(kda):
    """The benchmark's batch: 65536 tokens, 256 experts, 8 per token."""
    w = inputs.QB_WORKLOAD
    s, b = inputs.qb_inputs(seed=w["seed"], m=w["m"], n=w["n"])
    _check(kda, s, b, w["k"])


def test_repeatable_with_shared_workspace(kda):
    import torch
    s, b = inputs.qb_inputs(seed=77, m=3000, n=128)
    sd, bd = torch.from_numpy(s).cuda(), torch.from_numpy(b).cuda()
    ws = torch.empty(kda.library().kda_quantile_balance_workspace_size(3000, 128),
                     dtype=torch.uint8, device="cuda")
    first = kda.quantile_balance(sd, bd, 4, workspace=ws)
    for _ in range(3):
        assert torch.equal(kda.quantile_balance(sd, bd, 4, workspace=ws), first)
