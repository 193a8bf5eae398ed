"""Backward pass of the gated delta-rule recurrence in fp64.  TEST INFRASTRUCTURE.

Only the tests and the benchmark's CPU legs use this module.  The forward is the token loop of
"Transformer by Hand, ch. 7", section "The formula" and `delta_rule` in listing "qwen/deltanet.py"
(per sequence and value head, a_t = exp(g_t)):

    p_t = S_{t-1}^T k_t,   u_t = beta_t (v_t - a_t p_t),   S_t = a_t S_{t-1} + k_t u_t^T,
    o_t = scale * S_t^T q_t.

The learn-llm "linear attention" page trains this loop through autograd; here its gradient is
written out by hand as the adjoint of that loop, walked backwards in time.  With L the scalar loss
and lam = dL/dS_t (starting from dL/dS_final):

    lam   += scale q_t do_t^T                              (o_t reads S_t)
    dq_t   = scale (a_t S_{t-1} do_t + k_t (u_t . do_t))   (= scale S_t do_t)
    du     = lam^T k_t,   dk_t = lam u_t                   (S_t gets k_t u_t^T)
    dv_t   = beta_t du,   dbeta_t = du . (v_t - a_t p_t)   (u_t)
    dp     = -a_t beta_t du
    da     = <lam, S_{t-1}> - beta_t du . p_t              (a_t S_{t-1} and a_t p_t)
    dk_t  += S_{t-1} dp                                    (p_t reads S_{t-1} with k_t)
    dg_t   = a_t da
    lam    = a_t lam + k_t dp^T                            (dL/dS_{t-1})

and dS0 = lam at the start of the sequence.  The states S_{t-1} of the forward are kept (fp64);
with GQA, dq and dk of a query/key head sum over the value heads that read it.

backward_frontend() adds the chain rule through the fused front end of the GatedDeltaNet shell (the
l2 norm of q and k, the gates from the raw projections a, b with A_log and dt_bias).
"""
from __future__ import annotations

from typing import Optional

import numpy as np


def _spans(B, T, cu_seqlens):
    if cu_seqlens is None:
        return [(b, 0, T) for b in range(B)]
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    return [(0, int(cu[i]), int(cu[i + 1])) for i in range(len(cu) - 1)]


def backward(q, k, v, g, beta, dout, S0=None, dS_final=None, cu_seqlens=None, scale: float = 1.0):
    """q, k [B, T, Hqk, dk]; v, dout [B, T, Hv, dv]; g, beta [B, T, Hv]; S0, dS_final [nseq, Hv, dk, dv] or
    None.  Returns dq, dk, dv, dg, dbeta, dS0 (fp64, shaped like q, k, v, g, beta, S0)."""
    q, k, v, g, beta, dout = (np.asarray(x, dtype=np.float64) for x in (q, k, v, g, beta, dout))
    B, T, Hqk, DK = q.shape
    Hv, DV = v.shape[2], v.shape[3]
    G = Hv // Hqk
    spans = _spans(B, T, cu_seqlens)
    dq, dk = np.zeros_like(q), np.zeros_like(k)
    dv, dg, dbeta = np.zeros_like(v), np.zeros_like(g), np.zeros_like(beta)
    dS0 = np.zeros((len(spans), Hv, DK, DV))
    for i, (b, t0, t1) in enumerate(spans):
        for h in range(Hv):
            hk = h // G
            # forward, keeping S_{t-1} for every token
            S = np.zeros((DK, DV)) if S0 is None else np.array(S0[i, h], dtype=np.float64)
            prev = []
            for t in range(t0, t1):
                a = np.exp(g[b, t, h])
                prev.append(S)
                p = S.T @ k[b, t, hk]
                u = beta[b, t, h] * (v[b, t, h] - a * p)
                S = a * S + np.outer(k[b, t, hk], u)
            # backward
            lam = np.zeros((DK, DV)) if dS_final is None else np.array(dS_final[i, h], dtype=np.float64)
            for t in range(t1 - 1, t0 - 1, -1):
                Sp = prev[t - t0]
                a, bt = np.exp(g[b, t, h]), beta[b, t, h]
                kt, qt, vt, do = k[b, t, hk], q[b, t, hk], v[b, t, h], dout[b, t, h]
                p = Sp.T @ kt
                u = bt * (vt - a * p)
                lam = lam + scale * np.outer(qt, do)
                dq[b, t, hk] += scale * (a * (Sp @ do) + kt * (u @ do))
                du = lam.T @ kt
                dp = -a * bt * du
                dk[b, t, hk] += lam @ u + Sp @ dp
                dv[b, t, h] = bt * du
                dbeta[b, t, h] = du @ (vt - a * p)
                da = np.sum(lam * Sp) - bt * (du @ p)
                dg[b, t, h] = a * da
                lam = a * lam + np.outer(kt, dp)
            dS0[i, h] = lam
    return dq, dk, dv, dg, dbeta, dS0


# ---------------------------------------------------------------- the fused front end
# The GatedDeltaNet shell of "Transformer by Hand, ch. 7" (listing "qwen/deltanet.py") feeds the
# recurrence l2-normalised q and k and the gates beta = sigmoid(b), g = -exp(A_log) softplus(a + dt_bias)
# of the raw projections a, b.  The chain rule through those maps, per (token, head) row:
#   x_n = r x, r = (x . x + eps)^(-1/2):          dx = r dx_n - r^3 (x . dx_n) x
#   g = -exp(A_log) softplus(a + dt_bias):       da = dg (-exp(A_log)) sigmoid(a + dt_bias),
#                                                dA_log = sum over tokens of dg g, d dt_bias = sum of da
#   beta = sigmoid(b):                           db = dbeta beta (1 - beta)
# (eps = 1e-6, the reading of the unprinted l2norm epsilon the forward uses).
L2_EPS = 1e-6


def l2_normalize(x, eps: float = L2_EPS):
    """x / sqrt(x . x + eps) over the last axis (fp64)."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


def l2_normalize_backward(x, dxn, eps: float = L2_EPS):
    """Gradient with respect to x of a loss whose gradient with respect to x_n = l2_normalize(x) is dxn."""
    x = np.asarray(x, dtype=np.float64)
    dxn = np.asarray(dxn, dtype=np.float64)
    r = 1.0 / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)
    return r * dxn - r ** 3 * np.sum(x * dxn, axis=-1, keepdims=True) * x


def gates_backward(a, b, A_log, dt_bias, dg, dbeta):
    """Gradients with respect to a, b [..., Hv], A_log and dt_bias [Hv] given dg, dbeta [..., Hv]."""
    from .gates import gates_from_raw, sigmoid
    a, b, dg, dbeta = (np.asarray(x, dtype=np.float64) for x in (a, b, dg, dbeta))
    A_log = np.asarray(A_log, dtype=np.float64)
    dt_bias = np.asarray(dt_bias, dtype=np.float64)
    g, beta = gates_from_raw(a, b, A_log, dt_bias)
    da = dg * (-np.exp(A_log)) * sigmoid(a + dt_bias)
    db = dbeta * beta * (1.0 - beta)
    lead = tuple(range(dg.ndim - 1))
    return da, db, np.sum(dg * g, axis=lead), np.sum(da, axis=lead)


def backward_frontend(q, k, v, a, b, dout, A_log=None, dt_bias=None, normalize_qk: bool = False, S0=None,
                      dS_final=None, cu_seqlens=None, scale: float = 1.0):
    """The backward pass through the fused front end and the recurrence: q, k are the raw rows (normalised
    inside when normalize_qk), a, b the raw gate projections when A_log / dt_bias are given (else they are
    g and beta themselves).  Returns dq, dk, dv, da, db, dS0, dA_log, ddt_bias (the last two None without
    raw gates); all fp64."""
    qn = l2_normalize(q) if normalize_qk else np.asarray(q, dtype=np.float64)
    kn = l2_normalize(k) if normalize_qk else np.asarray(k, dtype=np.float64)
    if A_log is not None:
        from .gates import gates_from_raw
        g, beta = gates_from_raw(a, b, A_log, dt_bias)
    else:
        g, beta = a, b
    dq, dk, dv, dg, dbeta, dS0 = backward(qn, kn, v, g, beta, dout, S0=S0, dS_final=dS_final,
                                          cu_seqlens=cu_seqlens, scale=scale)
    if normalize_qk:
        dq, dk = l2_normalize_backward(q, dq), l2_normalize_backward(k, dk)
    if A_log is None:
        return dq, dk, dv, dg, dbeta, dS0, None, None
    da, db, dA_log, ddt = gates_backward(a, b, A_log, dt_bias, dg, dbeta)
    return dq, dk, dv, da, db, dS0, dA_log, ddt
