"""Pins of the oracle's causal short convolution: numpy.convolve, impulse response, causality,
splitting a sequence at the cache, packed sequences."""
import numpy as np
import pytest

from oracle import conv, gates



@pytest.mark.parametrize("K", [1, 2, 4])
def test_matches_numpy_convolve(K):
    rng = np.random.default_rng(K)
    T, C = 37, 5
    x, w = rng.normal(size=(1, T, C)), rng.normal(size=(C, K))
    y, _ = conv.causal_conv1d(x, w)
    for c in range(C):
        pre = np.convolve(x[0, :, c], w[c, ::-1])[:T]    # causal: output t uses x[t-K+1 .. t]
        np.testing.assert_allclose(y[0, :, c], gates.silu(pre), rtol=1e-13, atol=1e-15)


def test_impulse_response_and_causality():
    K, T, C = 4, 12, 3
    w = np.arange(1, K * C + 1, dtype=np.float64).reshape(C, K) / 10
    x = np.zeros((1, T, C))
    x[0, 5] = 1.0
    y, _ = conv.causal_conv1d(x, w)
    for c in range(C):
        expect = np.zeros(T)
        expect[5:5 + K] = w[c, ::-1]        # token 5 + j sees the impulse through w[c, K-1-j]
        np.testing.assert_allclose(y[0, :, c], gates.silu(expect), rtol=1e-14)
    x2 = x.copy()
    x2[0, 9] = 7.0                          # a later input cannot change earlier outputs
    y2, _ = conv.causal_conv1d(x2, w)
    np.testing.assert_array_equal(y2[0, :9], y[0, :9])


def test_cache_splits_a_sequence_exactly():
    rng = np.random.default_rng(3)
    K, T, C = 4, 20, 6
    x, w = rng.normal(size=(2, T, C)), rng.normal(size=(C, K))
    cache0 = rng.normal(size=(2, K - 1, C))
    y, c_end = conv.causal_conv1d(x, w, cache0)
    for cut in (1, 2, 3, 11):
        ya, ca = conv.causal_conv1d(x[:, :cut], w, cache0)
        yb, cb = conv.causal_conv1d(x[:, cut:], w, ca)
        np.testing.assert_allclose(np.concatenate([ya, yb], 1), y, rtol=1e-14)
        np.testing.assert_allclose(cb, c_end, rtol=1e-14)
    # one token at a time (the decode step) gives the same outputs
    c = cache0
    for t in range(T):
        yt, c = conv.causal_conv1d(x[:, t:t + 1], w, c)
        np.testing.assert_allclose(yt[:, 0], y[:, t], rtol=1e-14)


def test_packed_equals_separate():
    rng = np.random.default_rng(4)
    lens = [3, 0, 9, 1]
    K, C = 4, 5
    x, w = rng.normal(size=(1, sum(lens), C)), rng.normal(size=(C, K))
    cache = rng.normal(size=(len(lens), K - 1, C))
    cu = np.concatenate([[0], np.cumsum(lens)])
    y, co = conv.causal_conv1d(x, w, cache, cu_seqlens=cu)
    for i in range(len(lens)):
        yi, ci = conv.causal_conv1d(x[:, cu[i]:cu[i + 1]], w, cache[i:i + 1])
        np.testing.assert_array_equal(y[:, cu[i]:cu[i + 1]], yi)
        np.testing.assert_array_equal(co[i], ci[0])


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


@pytest.mark.parametrize("case", [
    dict(B=2, T=6, C=3, K=4, cache=True, dco=True),
    dict(B=1, T=9, C=2, K=3, cache=False, dco=False),
    dict(lens=(4, 0, 1, 5), C=3, K=4, cache=True, dco=True),   # packed; an empty and a short sequence
    dict(B=1, T=5, C=2, K=1, cache=False, dco=False),           # no history: a pointwise map
])
def test_conv_backward_matches_finite_differences(case):
    rng = np.random.default_rng(9)
    lens = case.get("lens")
    B, T = (1, sum(lens)) if lens else (case["B"], case["T"])
    C, K = case["C"], case["K"]
    nseq = len(lens) if lens else B
    cu = np.concatenate([[0], np.cumsum(lens)]) if lens else None
    x = rng.normal(size=(B, T, C))
    w = rng.normal(size=(C, K))
    cache = rng.normal(size=(nseq, K - 1, C)) if case["cache"] else None
    dy = rng.normal(size=(B, T, C))
    dco = rng.normal(size=(nseq, K - 1, C)) if case["dco"] else None

    def loss(xx=x, ww=w, cc=cache):
        y, co = conv.causal_conv1d(xx, ww, cc, cu_seqlens=cu)
        return float(np.sum(y * dy) + (np.sum(co * dco) if dco is not None else 0.0))

    dx, dw, dc = conv.causal_conv1d_backward(x, w, dy, cache, cu_seqlens=cu, dcache_out=dco)
    np.testing.assert_allclose(dx, _fd(lambda t: loss(xx=t), x), rtol=1e-6, atol=1e-8)
    np.testing.assert_allclose(dw, _fd(lambda t: loss(ww=t), w), rtol=1e-6, atol=1e-8)
    if cache is not None:
        np.testing.assert_allclose(dc, _fd(lambda t: loss(cc=t), cache), rtol=1e-6, atol=1e-8)


def test_conv_backward_closed_form_single_tap():
    """K = 1: y = silu(w x) per element, so dx = w silu'(w x) dy and dw_c = sum_t x silu'(w x) dy."""
    from oracle.gates import silu_grad
    rng = np.random.default_rng(10)
    x, w, dy = rng.normal(size=(2, 7, 4)), rng.normal(size=(4, 1)), rng.normal(size=(2, 7, 4))
    dx, dw, _ = conv.causal_conv1d_backward(x, w, dy)
    u = x * w[:, 0]
    np.testing.assert_allclose(dx, w[:, 0] * silu_grad(u) * dy, rtol=1e-13)
    np.testing.assert_allclose(dw[:, 0], np.sum(x * silu_grad(u) * dy, axis=(0, 1)), rtol=1e-12)


def test_conv_backward_pins_catch_a_reversed_window():
    """Applying the taps in the wrong order (w[:, K-1-j]) is caught by the difference pin."""
    rng = np.random.default_rng(11)
    x, w, dy = rng.normal(size=(1, 6, 2)), rng.normal(size=(2, 4)), rng.normal(size=(1, 6, 2))
    dx = conv.causal_conv1d_backward(x, w[:, ::-1], dy)[0]
    fd = _fd(lambda t: float(np.sum(conv.causal_conv1d(t, w)[0] * dy)), x)
    assert np.max(np.abs(dx - fd)) > 1e-2
