"""Pins of the oracle's gate function (the GatedDeltaNet shell's beta and g) against closed forms."""
import math

import numpy as np
import pytest

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


def test_gated_rmsnorm_closed_forms():
    dv = 16
    alt = np.tile([1.0, -1.0], dv // 2)
    w = np.linspace(0.5, 1.5, dv)
    z = np.linspace(-3, 3, dv)
    for c in (0.01, 2.5, 300.0):   # the RMS of c * alt is |c|: the result does not depend on c (eps = 0)
        np.testing.assert_allclose(gates.gated_rmsnorm(c * alt, z, w, 0.0), alt * w * gates.silu(z), rtol=1e-14)
    # silu(0) = 0 closes the gate; silu(z) -> z for large z, -> 0 for very negative z
    assert np.all(gates.gated_rmsnorm(alt, np.zeros(dv), w, 1e-6) == 0)
    np.testing.assert_allclose(gates.silu(np.array([40.0])), [40.0], rtol=1e-15)
    assert abs(gates.silu(-40.0)) < 1e-15
    # eps shrinks the normalised vector: RMS(o / sqrt(ms + eps)) = sqrt(ms / (ms + eps))
    o = 0.01 * alt
    y = gates.gated_rmsnorm(o, np.full(dv, 50.0), np.ones(dv), 1e-4)
    np.testing.assert_allclose(np.sqrt(np.mean((y / gates.silu(50.0)) ** 2)), np.sqrt(1e-4 / (1e-4 + 1e-4)), rtol=1e-12)


def _fd(f, x, eps=1e-6):
    x = np.array(x, dtype=np.float64)
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        hi, lo = x.copy(), x.copy()
        hi[i] += eps
        lo[i] -= eps
        g[i] = (f(hi) - f(lo)) / (2 * eps)
    return g


def test_silu_grad_matches_differences_and_closed_values():
    z = np.linspace(-8, 8, 33)
    # central differences of a sum of 33 terms (~30): cancellation error ~ 30 * 2^-52 / 1e-6 ~ 1e-8
    np.testing.assert_allclose(gates.silu_grad(z), _fd(lambda t: np.sum(gates.silu(t)), z), rtol=1e-7, atol=3e-8)
    assert gates.silu_grad(0.0) == 0.5   # sigmoid(0) (1 + 0)


def test_gated_rmsnorm_backward_matches_finite_differences():
    """All three gradients of a weighted sum of the gate's outputs, rows of 8 values, eps both tiny and
    comparable to the mean square."""
    rng = np.random.default_rng(3)
    o, z, w = rng.normal(size=(5, 8)), rng.normal(size=(5, 8)), rng.normal(1.0, 0.2, size=8)
    dy = rng.normal(size=(5, 8))
    for eps in (1e-6, 0.3):
        do, dz, dw = gates.gated_rmsnorm_backward(o, z, w, eps, dy)
        loss = lambda oo=o, zz=z, ww=w: float(np.sum(gates.gated_rmsnorm(oo, zz, ww, eps) * dy))
        np.testing.assert_allclose(do, _fd(lambda t: loss(oo=t), o), rtol=1e-6, atol=1e-8)
        np.testing.assert_allclose(dz, _fd(lambda t: loss(zz=t), z), rtol=1e-6, atol=1e-8)
        np.testing.assert_allclose(dw, _fd(lambda t: loss(ww=t), w), rtol=1e-6, atol=1e-8)


def test_gated_rmsnorm_backward_is_scale_free_in_o():
    """With eps = 0 the gate depends on the direction of each row only: do is orthogonal to o and
    halves when o doubles; a planted slip (the projection term dropped) breaks both."""
    rng = np.random.default_rng(4)
    o, z, w, dy = rng.normal(size=(3, 16)), rng.normal(size=(3, 16)), rng.normal(size=16), rng.normal(size=(3, 16))
    do = gates.gated_rmsnorm_backward(o, z, w, 0.0, dy)[0]
    np.testing.assert_allclose(np.sum(do * o, axis=-1), 0.0, atol=1e-12)
    np.testing.assert_allclose(gates.gated_rmsnorm_backward(2 * o, z, w, 0.0, dy)[0], do / 2, rtol=1e-12)
    inv = 1.0 / np.sqrt(np.mean(o * o, axis=-1, keepdims=True))
    slip = inv * dy * w * gates.silu(z)
    assert np.max(np.abs(np.sum(slip * o, axis=-1))) > 1e-3


@pytest.mark.parametrize("slip", ["sigmoid_for_silu_grad", "no_inv_on_do", "dz_without_weight", "dw_without_gate"])
def test_gated_rmsnorm_backward_pin_catches_planted_slips(slip):
    """Each plausible slip in the gate's chain rule, written into a copy of its formulas, is caught by
    the finite-difference pin above (some gradient off by far more than its tolerance)."""
    rng = np.random.default_rng(5)
    o, z, w, dy = rng.normal(size=(4, 8)), rng.normal(size=(4, 8)), rng.normal(1.0, 0.2, size=8), rng.normal(size=(4, 8))
    eps = 1e-6
    inv = 1.0 / np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + eps)
    oh, s = o * inv, gates.silu(z)
    gy = dy * w * s
    do = (1.0 if slip == "no_inv_on_do" else inv) * (gy - oh * np.mean(gy * oh, axis=-1, keepdims=True))
    dz = dy * oh * (1.0 if slip == "dz_without_weight" else w) * (
        gates.sigmoid(z) if slip == "sigmoid_for_silu_grad" else gates.silu_grad(z))
    dw = np.sum(dy * oh * (1.0 if slip == "dw_without_gate" else s), axis=0)
    loss = lambda oo=o, zz=z, ww=w: float(np.sum(gates.gated_rmsnorm(oo, zz, ww, eps) * dy))
    worst = max(np.max(np.abs(do - _fd(lambda t: loss(oo=t), o))), np.max(np.abs(dz - _fd(lambda t: loss(zz=t), z))),
                np.max(np.abs(dw - _fd(lambda t: loss(ww=t), w))))
    assert worst > 1e-3, f"{slip} went unnoticed ({worst:.2e})"
