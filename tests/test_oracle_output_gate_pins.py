"""Pins for the oracle's gated output step, each against a property fixed by the definition.

Source: "Kimi k3 技术报告详解（1）——架构再升华", section "Gated MLA": the layer output is
W_o [Sigmoid(W_g x_t) (.) RMSNorm(o~_t)].  The oracle computes the part between the two
projections, per (token, head) row of d_v channels:
    y = Sigmoid(gate) * w * o / sqrt(mean(o^2) + eps).

What pins what (a plausible slip fails at least one):
  unit RMS          gate -> +inf, w = 1, eps = 0: every row of y has mean square exactly 1
                    (normalising over the wrong axis, a sum for the mean, a missing root)
  scale invariance  eps = 0: y(c o) = y(o) for c > 0 (a missing or partial normalisation)
  sigmoid values    gate = 0, +-ln 3 give factors 1/2, 3/4, 1/4 of the ungated row
                    (another squashing function, a sign slip in the exponent)
  weight            y(w) = w * y(1) channel by channel (weight on the wrong axis)
  eps closed form   a constant row c gives c / sqrt(c^2 + eps) (eps outside the root)
  zero row          o = 0, eps > 0 gives 0, not NaN
"""
import math

import numpy as np
import pytest

import oracle

BIG = 745.0  # Sigmoid(745) == 1.0 in fp64 (e^-745 is below half an ulp of 1)


def _rows(seed, n=6, dv=128):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((n, 3, dv)) * rng.uniform(0.1, 10.0, size=(n, 3, 1))


def test_unit_rms_per_head_row():
    o = _rows(1)
    y = oracle.output_norm_gate(o, np.full_like(o, BIG), None, 0.0)
    ms = np.mean(y * y, axis=-1)
    np.testing.assert_allclose(ms, 1.0, rtol=0, atol=1e-13)
    # a different row scale per head must not leak across heads
    assert o.std(axis=-1).std() > 0.1


@pytest.mark.parametrize("c", [1e-3, 7.0, 1e3])
def test_scale_invariance(c):
    o = _rows(2, dv=64)
    g = np.random.default_rng(3).standard_normal(o.shape)
    np.testing.assert_allclose(oracle.output_norm_gate(c * o, g, None, 0.0),
                               oracle.output_norm_gate(o, g, None, 0.0), rtol=1e-13, atol=1e-15)


@pytest.mark.parametrize("gate,factor", [(0.0, 0.5), (math.log(3.0), 0.75), (-math.log(3.0), 0.25)])
def test_sigmoid_values(gate, factor):
    o = _rows(4)
    ungated = oracle.output_norm_gate(o, np.full_like(o, BIG), None, 1e-6)
    y = oracle.output_norm_gate(o, np.full_like(o, gate), None, 1e-6)
    np.testing.assert_allclose(y, factor * ungated, rtol=1e-14, atol=1e-15)


def test_weight_scales_each_channel():
    o = _rows(5)
    g = np.random.default_rng(6).standard_normal(o.shape)
    w = np.random.default_rng(7).uniform(-2.0, 2.0, size=o.shape[-1])
    np.testing.assert_allclose(oracle.output_norm_gate(o, g, w, 1e-5),
                               w * oracle.output_norm_gate(o, g, None, 1e-5), rtol=1e-14,
                               atol=1e-15)


@pytest.mark.parametrize("c,eps", [(0.01, 1e-4), (3.0, 0.5), (-2.0, 0.0)])
def test_eps_closed_form_on_constant_rows(c, eps):
    o = np.full((2, 1, 128), c)
    y = oracle.output_norm_gate(o, np.full_like(o, BIG), None, eps)
    np.testing.assert_allclose(y, c / math.sqrt(c * c + eps), rtol=1e-14)


def test_zero_row_is_zero():
    o = np.zeros((1, 2, 64))
    y = oracle.output_norm_gate(o, np.ones_like(o), None, 1e-6)
    assert np.all(y == 0.0)
