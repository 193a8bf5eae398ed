"""fp64 chunk-parallel (WY/UT) form of the recurrence.  TEST INFRASTRUCTURE.

Only the tests use this module: it pins that the chunk algebra the GPU prefill
is built on equals the token loop (the learn-llm "linear attention" page says the
chunked implementations are mathematically equivalent to the token loop; the
handbook's history table names the chunk-parallel algorithm of Yang et al. 2024).
The algebra is derived here from the update in "Transformer by Hand, ch. 7",
section "The formula"; it is written with plain numpy matrix products and a
library linear solve, with no blocking beyond the chunks themselves.

Inside one chunk of n tokens, with G_r = g_1 + ... + g_r and gamma_r = exp(G_r):

  unrolling S_r = a_r S_{r-1} + k_r u_r^T, u_r = beta_r (v_r - a_r S_{r-1}^T k_r), gives
      S_r = gamma_r S0 + sum_{s<=r} exp(G_r - G_s) k_s u_s^T;
  substituting into u_r:
      (I + diag(beta) A) U = diag(beta) V - diag(beta*gamma) K S0,
      A_rs = exp(G_r - G_s) (k_r . k_s) for s < r, else 0;
  so with T = (I + diag(beta) A)^-1,  W = T diag(beta*gamma) K,  U~ = T diag(beta) V:
      U = U~ - W S0
      O = scale * (diag(gamma) Q S0 + (M * Q K^T) U),   M_rs = exp(G_r - G_s) [s <= r]
      S_n = gamma_n S0 + (diag(exp(G_n - G)) K)^T U.

Decay ratios are always formed as exp(G_r - G_s) with s <= r (never 1/gamma_s).
"""
from __future__ import annotations

import numpy as np


def chunk_step(Q, K, V, g, beta, S0, scale=1.0):
    """One chunk (n tokens) of one (sequence, value head).  Returns (O [n, dv], S_n)."""
    n = Q.shape[0]
    G = np.cumsum(g)
    gamma = np.exp(G)
    D = G[:, None] - G[None, :]                  # G_r - G_s
    lower = np.tril(np.ones((n, n), dtype=bool), -1)
    causal = np.tril(np.ones((n, n), dtype=bool), 0)
    A = np.where(lower, np.exp(np.where(lower, D, 0.0)) * (K @ K.T), 0.0)
    Tmat = np.linalg.solve(np.eye(n) + beta[:, None] * A, np.eye(n))
    W = Tmat @ ((beta * gamma)[:, None] * K)
    Ut = Tmat @ (beta[:, None] * V)
    U = Ut - W @ S0
    M = np.where(causal, np.exp(np.where(causal, D, 0.0)), 0.0)
    O = scale * (gamma[:, None] * (Q @ S0) + (M * (Q @ K.T)) @ U)
    decay_to_end = np.exp(G[-1] - G)
    S_n = gamma[-1] * S0 + (decay_to_end[:, None] * K).T @ U
    return O, S_n


def chunk_step_folded(Q, K, V, g, beta, S0, scale=1.0):
    """The same chunk with U eliminated, so that the state moves by one affine map per chunk.

    With b = exp(G_n - G) and K~ = diag(b) K, substituting U = U~ - W S0 into the update and the
    outputs gives
        S_n = gamma_n S0 + (-K~^T W) S0 + K~^T U~
        O   = (scale diag(gamma) Q - P W) S0 + P U~,   P = scale (M * Q K^T)
    (the first line is the form in which a chunk step needs a single product with the state)."""
    n = Q.shape[0]
    G = np.cumsum(g)
    gamma = np.exp(G)
    D = G[:, None] - G[None, :]
    lower = np.tril(np.ones((n, n), dtype=bool), -1)
    causal = np.tril(np.ones((n, n), dtype=bool), 0)
    A = np.where(lower, np.exp(np.where(lower, D, 0.0)) * (K @ K.T), 0.0)
    Tmat = np.linalg.solve(np.eye(n) + beta[:, None] * A, np.eye(n))
    W = Tmat @ ((beta * gamma)[:, None] * K)
    Ut = Tmat @ (beta[:, None] * V)
    Kt = np.exp(G[-1] - G)[:, None] * K
    P = scale * np.where(causal, np.exp(np.where(causal, D, 0.0)), 0.0) * (Q @ K.T)
    S_n = gamma[-1] * S0 + (-Kt.T @ W) @ S0 + Kt.T @ Ut
    O = (scale * gamma[:, None] * Q - P @ W) @ S0 + P @ Ut
    return O, S_n


def forward(q, k, v, g, beta, S0=None, cu_seqlens=None, chunk=64, scale=1.0, folded=False):
    """Same interface and layouts as :func:`oracle.recurrence.forward` (fp64 results).  With
    folded=True every chunk goes through :func:`chunk_step_folded`."""
    step = chunk_step_folded if folded else chunk_step
    q, k, v, g, beta = (np.asarray(t, dtype=np.float64) for t in (q, k, v, g, beta))
    B, T, Hqk, dk = q.shape
    Hv, dv = v.shape[2], v.shape[3]
    group = Hv // Hqk
    if cu_seqlens is None:
        spans = [(b, 0, T) for b in range(B)]
    else:
        cu = np.asarray(cu_seqlens, dtype=np.int64)
        spans = [(0, int(cu[i]), int(cu[i + 1])) for i in range(len(cu) - 1)]
    out = np.zeros((B, T, Hv, dv))
    S_final = np.zeros((len(spans), Hv, dk, dv))
    for i, (b, t0, t1) in enumerate(spans):
        for h in range(Hv):
            hk = h // group
            S = np.zeros((dk, dv)) if S0 is None else np.array(S0[i, h], dtype=np.float64)
            for c0 in range(t0, t1, chunk):
                c1 = min(c0 + chunk, t1)
                O, S = step(q[b, c0:c1, hk], k[b, c0:c1, hk], v[b, c0:c1, h], g[b, c0:c1, h],
                            beta[b, c0:c1, h], S, scale)
                out[b, c0:c1, h] = O
            S_final[i, h] = S
    return out, S_final
