"""Pins of the AdamW oracle (CPU only).

Closed forms that do not go through the oracle's code: after the first step,
and after any number of steps with a constant gradient, the bias-corrected
moments are exactly g and g^2, so each step moves W to
W (1 - lr wd) - lr g / (|g| + eps).
"""

import numpy as np
import pytest

from oracle import adamw_oracle as A

HP = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)


def rel(x, y):
    return float(np.max(np.abs(np.asarray(x, np.float64) - y) / np.maximum(np.abs(y), 1e-30)))


def test_first_step_closed_form():
    rng = np.random.default_rng(40)
    W = rng.standard_normal(1000) * 0.02
    g = rng.standard_normal(1000) * np.exp(rng.uniform(-8, 2, 1000))
    Wn, m, v = A.adamw_step(W, g, np.zeros(1000), np.zeros(1000), step=1, **HP)
    want = W * (1 - HP["lr"] * HP["weight_decay"]) - HP["lr"] * g / (np.abs(g) + HP["eps"])
    assert rel(Wn, want) < 1e-12
    assert rel(m, 0.1 * g) < 1e-15 and rel(v, 0.05 * g * g) < 1e-14


def test_constant_gradient_every_step_closed_form():
    rng = np.random.default_rng(41)
    g = rng.standard_normal(500)
    W = rng.standard_normal(500) * 0.02
    m = np.zeros(500)
    v = np.zeros(500)
    for t in range(1, 40):
        W_prev = W
        W, m, v = A.adamw_step(W, g, m, v, step=t, **HP)
        want = W_prev * (1 - HP["lr"] * HP["weight_decay"]) - HP["lr"] * g / (np.abs(g) + HP["eps"])
        assert rel(W, want) < 1e-9


def test_zero_gradient_is_pure_decay():
    W = np.linspace(-1, 1, 101)
    Wn, m, v = A.adamw_step(W, np.zeros(101), np.zeros(101), np.zeros(101), step=3, **HP)
    assert np.array_equal(Wn, W * (1 - HP["lr"] * HP["weight_decay"]))
    assert not m.any() and not v.any()


def test_fp32_statement_within_a_few_ulps_of_fp64():
    rng = np.random.default_rng(42)
    n = 20000
    W = (rng.standard_normal(n) * 0.02).astype(np.float32)
    m = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    v = (rng.uniform(0, 1e-5, n)).astype(np.float32)
    g = (rng.standard_normal(n) * 1e-2).astype(np.float32)
    W32, m32, v32 = A.adamw_step_fp32(W, g, m, v, step=7, **HP)
    W64, m64, v64 = A.adamw_step(W, g, m, v, step=7, **HP)
    # each sum may cancel: bound the error by a few ulps of its terms' magnitudes
    u = 2.0 ** -24
    m_scale = 0.9 * np.abs(m.astype(np.float64)) + 0.1 * np.abs(g.astype(np.float64))
    assert np.all(np.abs(m32 - m64) <= 3 * u * m_scale)
    v_scale = 0.95 * v.astype(np.float64) + 0.05 * g.astype(np.float64) ** 2
    assert np.all(np.abs(v32 - v64) <= 4 * u * v_scale)
    assert np.max(np.abs(W32 - W64)) < 4e-8


def test_fp32_statement_exact_on_dyadic_values():
    # beta1 = beta2 = 1/2, t = 1: every intermediate is a short dyadic number
    W = np.array([0.5, -0.25, 1.0], np.float32)
    g = np.array([1.0, -2.0, 4.0], np.float32)
    Wn, m, v = A.adamw_step_fp32(W, g, np.zeros(3, np.float32), np.zeros(3, np.float32), lr=0.5, beta1=0.5,
                                 beta2=0.5, eps=0.0, weight_decay=0.0, step=1)
    assert np.array_equal(m, g / 2) and np.array_equal(v, g * g / 2)
    assert np.array_equal(Wn, W - 0.5 * np.sign(g))


@pytest.mark.parametrize("t", [1, 2, 10, 1000])
def test_constants(t):
    k = A.adamw_constants(1e-3, 0.9, 0.95, 1e-8, 0.1, t)
    assert k["step_size"] == np.float32(1e-3 / (1 - 0.9 ** t))
    assert k["bc2"] == np.float32(1 - 0.95 ** t)
