"""Gates of the GatedDeltaNet shell in fp64.  TEST INFRASTRUCTURE.

Only the tests use this module.  "Transformer by Hand, ch. 7", listing "qwen/deltanet.py",
GatedDeltaNet.forward, and the parts table below it:
    beta = sigmoid(in_proj_b(x))                                   write strength in (0, 1)
    g    = -exp(A_log) * softplus(in_proj_a(x) + dt_bias)          log decay, always <= 0
Their backward (silu_grad, gated_rmsnorm_backward) is the chain rule written out.
Here a = in_proj_a(x) and b = in_proj_b(x) are given directly (the projections need trained
weights and are out of scope).  softplus and sigmoid are numpy's logaddexp and an overflow-safe
logistic.
"""
import numpy as np


def softplus(x):
    """log(1 + e^x)."""
    return np.logaddexp(0.0, np.asarray(x, dtype=np.float64))


def sigmoid(x):
    x = np.asarray(x, dtype=np.float64)
    e = np.exp(-np.abs(x))
    return np.where(x >= 0, 1.0 / (1.0 + e), e / (1.0 + e))


def gates_from_raw(a, b, A_log, dt_bias):
    """a, b [..., Hv]; A_log, dt_bias [Hv].  Returns (g, beta) in fp64."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    A_log = np.asarray(A_log, dtype=np.float64)
    dt_bias = np.asarray(dt_bias, dtype=np.float64)
    g = -np.exp(A_log) * softplus(a + dt_bias)
    return g, sigmoid(b)


def silu(z):
    z = np.asarray(z, dtype=np.float64)
    return z * sigmoid(z)


def gated_rmsnorm(o, z, weight, eps):
    """Output gate of the shell (GatedRMSNorm(out, z), "the output is normalised per head and then
    multiplied by the gate silu(z)"): o / sqrt(mean(o^2) + eps) * weight * silu(z) over the last axis
    (the dv values of one token and value head).  The GatedRMSNorm body is not printed on the pages;
    this is the reading taken (RMS over the head's values, weight after the normalisation)."""
    o = np.asarray(o, dtype=np.float64)
    ms = np.mean(o * o, axis=-1, keepdims=True)
    return o / np.sqrt(ms + eps) * np.asarray(weight, dtype=np.float64) * silu(z)


def silu_grad(z):
    """d silu / dz = sigmoid(z) (1 + z (1 - sigmoid(z)))."""
    z = np.asarray(z, dtype=np.float64)
    s = sigmoid(z)
    return s * (1.0 + z * (1.0 - s))


def gated_rmsnorm_backward(o, z, weight, eps, dy):
    """Gradients of a loss through y = gated_rmsnorm(o, z, weight, eps) given dy = dL/dy: with
    inv = (mean(o^2) + eps)^-1/2, o_hat = o inv and gy = dy weight silu(z),
        do = inv (gy - o_hat mean(gy o_hat)),   dz = dy o_hat weight silu'(z),
        dweight = sum over all rows of dy o_hat silu(z).
    Returns (do, dz, dweight) in fp64."""
    o, z, dy = (np.asarray(x, dtype=np.float64) for x in (o, z, dy))
    weight = np.asarray(weight, dtype=np.float64)
    inv = 1.0 / np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + eps)
    oh = o * inv
    s = silu(z)
    gy = dy * weight * s
    do = inv * (gy - oh * np.mean(gy * oh, axis=-1, keepdims=True))
    dz = dy * oh * weight * silu_grad(z)
    dw = np.sum((dy * oh * s).reshape(-1, o.shape[-1]), axis=0)
    return do, dz, dw
