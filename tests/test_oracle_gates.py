"""Pins of the oracle's gate function (the GatedDeltaNet shell's beta and g) against closed forms."""
import math

import numpy as np

from oracle import gates


def test_gate_special_values():
    # softplus(0) = ln 2, sigmoid(0) = 1/2; with A_log = 0 and a = -dt_bias, g = -ln 2 exactly
    g, beta = gates.gates_from_raw(np.array([-0.3]), np.array([0.0]), np.array([0.0]), np.array([0.3]))
    assert g[0] == -math.log(2.0)
    assert beta[0] == 0.5
    # exp(A_log) scales g; beta is the logistic of b
    g2, _ = gates.gates_from_raw(np.array([0.0]), np.array([0.0]), np.array([math.log(3.0)]), np.array([0.0]))
    assert abs(g2[0] + 3.0 * math.log(2.0)) < 1e-15
    assert abs(gates.sigmoid(2.0) - 1.0 / (1.0 + math.exp(-2.0))) < 1e-16


def test_softplus_identity_and_asymptotes():
    x = np.linspace(-40, 40, 8001)
    np.testing.assert_allclose(gates.softplus(x) - gates.softplus(-x), x, atol=1e-12)
    big = np.array([50.0, 200.0, 800.0])
    np.testing.assert_allclose(gates.softplus(big), big, rtol=1e-15)
    small = np.array([-50.0, -200.0])
    np.testing.assert_allclose(gates.softplus(small), np.exp(small), rtol=1e-12)
    assert np.all(np.isfinite(gates.sigmoid(np.array([-1000.0, 1000.0]))))


def test_gates_ranges():
    rng = np.random.default_rng(0)
    a, b = rng.normal(size=(1000, 8)), rng.normal(size=(1000, 8))
    A_log, dt_bias = rng.normal(-0.5, 0.5, size=8), rng.normal(0, 0.5, size=8)
    g, beta = gates.gates_from_raw(a, b, A_log, dt_bias)
    assert np.all(g < 0) and np.all((beta > 0) & (beta < 1))   # decay exp(g) in (0, 1)
    assert np.all(np.diff(gates.gates_from_raw(np.sort(a[:, 0]), b[:, 0], A_log[0], dt_bias[0])[0]) <= 0)
