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
