"""Depthwise causal short convolution + SiLU in fp64.  TEST INFRASTRUCTURE.

Only the tests use this module.  "Transformer by Hand, ch. 7", listing "qwen/deltanet.py": conv1d with
groups = channels, kernel K, padding K - 1, outputs cut to the first T, then SiLU (each channel sees its
own previous K - 1 tokens); the learn-llm "linear attention" page: at inference the last K - 1 inputs
are cached.  Written out as the sum, per sequence, over a window padded on the left with the cache;
causal_conv1d_backward is the chain rule through that sum and the SiLU.
"""
import numpy as np

from .gates import silu


def causal_conv1d(x, w, cache_in=None, cu_seqlens=None):
    """x [B, T, C]; w [C, K]; cache_in [nseq, K-1, C] or None.  Returns (y [B, T, C], cache_out [nseq, K-1, C])."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    B, T, C = x.shape
    K = w.shape[1]
    if cu_seqlens is None:
        spans = [(b, 0, T) for b in range(B)]
    else:
        cu = np.asarray(cu_seqlens, dtype=np.int64)
        spans = [(0, int(cu[i]), int(cu[i + 1])) for i in range(len(cu) - 1)]
    y = np.zeros_like(x)
    cache_out = np.zeros((len(spans), K - 1, C))
    for i, (b, t0, t1) in enumerate(spans):
        past = np.zeros((K - 1, C)) if cache_in is None else np.asarray(cache_in[i], dtype=np.float64)
        xp = np.concatenate([past, x[b, t0:t1]], axis=0)          # [K-1 + n, C]
        for t in range(t1 - t0):
            window = xp[t:t + K]                                  # oldest first; last row = token t
            y[b, t0 + t] = silu(np.sum(w.T * window, axis=0))
        cache_out[i] = xp[xp.shape[0] - (K - 1):] if K > 1 else np.zeros((0, C))
    return y, cache_out


def causal_conv1d_backward(x, w, dy, cache_in=None, cu_seqlens=None, dcache_out=None):
    """Gradients through causal_conv1d given dy = dL/dy [B, T, C] (and dcache_out = dL/dcache_out
    [nseq, K-1, C] or None): with xp the cache-padded inputs of a sequence and u_t = sum_j w[:, j] xp[t + j]
    the pre-activation of token t, du_t = dy_t silu'(u_t), dxp[t + j] += w[:, j] du_t and
    dw[:, j] += du_t xp[t + j]; the cache_out rows are copies of the last K - 1 rows of xp.
    Returns (dx [B, T, C], dw [C, K], dcache_in [nseq, K-1, C]) in fp64."""
    from .gates import silu_grad
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    dy = np.asarray(dy, dtype=np.float64)
    B, T, C = x.shape
    K = w.shape[1]
    if cu_seqlens is None:
        spans = [(b, 0, T) for b in range(B)]
    else:
        cu = np.asarray(cu_seqlens, dtype=np.int64)
        spans = [(0, int(cu[i]), int(cu[i + 1])) for i in range(len(cu) - 1)]
    dx = np.zeros_like(x)
    dw = np.zeros((C, K))
    dcache = np.zeros((len(spans), K - 1, C))
    for i, (b, t0, t1) in enumerate(spans):
        past = np.zeros((K - 1, C)) if cache_in is None else np.asarray(cache_in[i], dtype=np.float64)
        xp = np.concatenate([past, x[b, t0:t1]], axis=0)
        dxp = np.zeros_like(xp)
        for t in range(t1 - t0):
            window = xp[t:t + K]
            du = dy[b, t0 + t] * silu_grad(np.sum(w.T * window, axis=0))
            dxp[t:t + K] += w.T * du
            dw += (window * du).T
        if dcache_out is not None and K > 1:
            dxp[xp.shape[0] - (K - 1):] += np.asarray(dcache_out[i], dtype=np.float64)
        dx[b, t0:t1] = dxp[K - 1:]
        dcache[i] = dxp[:K - 1]
    return dx, dw, dcache
