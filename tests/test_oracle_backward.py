"""Pins of the oracle's backward pass: central finite differences of the fp64 forward oracle on tiny
problems, a closed form (no writes: pure decay), and planted mistakes that the pins must catch."""
import numpy as np
import pytest

from oracle import backward as ob
from oracle import recurrence as orc


def _problem(seed, B=1, T=7, Hqk=1, Hv=2, dk=4, dv=3, lens=None, s0=True):
    rng = np.random.default_rng(seed)
    if lens is not None:
        B, T = 1, sum(lens)
    q = rng.normal(size=(B, T, Hqk, dk))
    k = rng.normal(size=(B, T, Hqk, dk)) / np.sqrt(dk)
    v = rng.normal(size=(B, T, Hv, dv))
    g = -np.abs(rng.normal(0.3, 0.2, size=(B, T, Hv)))
    beta = 1.0 / (1.0 + np.exp(-rng.normal(size=(B, T, Hv))))
    nseq = B if lens is None else len(lens)
    S0 = 0.5 * rng.normal(size=(nseq, Hv, dk, dv)) if s0 else None
    cu = None if lens is None else np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    dout = rng.normal(size=(B, T, Hv, dv))
    dSf = rng.normal(size=(nseq, Hv, dk, dv))
    return dict(q=q, k=k, v=v, g=g, beta=beta, S0=S0, cu=cu, dout=dout, dSf=dSf)


def _loss(x, scale, **over):
    y = dict(x, **over)
    o, S = orc.forward(y["q"], y["k"], y["v"], y["g"], y["beta"], S0=y["S0"], cu_seqlens=y["cu"], scale=scale)
    return float(np.sum(o * x["dout"]) + np.sum(S * x["dSf"]))


def _fd(x, name, scale, eps=1e-6):
    base = np.array(x[name], dtype=np.float64)
    grad = np.zeros_like(base)
    it = np.nditer(base, flags=["multi_index"])
    for _ in it:
        idx = it.multi_index
        hi, lo = base.copy(), base.copy()
        hi[idx] += eps
        lo[idx] -= eps
        grad[idx] = (_loss(x, scale, **{name: hi}) - _loss(x, scale, **{name: lo})) / (2 * eps)
    return grad


def _analytic(x, scale, fn=ob.backward):
    return dict(zip(("q", "k", "v", "g", "beta", "S0"),
                    fn(x["q"], x["k"], x["v"], x["g"], x["beta"], x["dout"], S0=x["S0"], dS_final=x["dSf"],
                       cu_seqlens=x["cu"], scale=scale)))


@pytest.mark.parametrize("case", [
    dict(seed=1),                                         # GQA: two value heads read one q/k head
    dict(seed=2, B=2, Hqk=2, Hv=2, T=5),                  # batched, one value head per q/k head
    dict(seed=3, lens=(3, 0, 5, 1)),                      # packed sequences, an empty one, state reset
    dict(seed=4, s0=False, T=9, dk=3, dv=5),              # zero initial state, dk != dv
])
@pytest.mark.parametrize("scale", [1.0, 0.5])
def test_gradients_match_finite_differences(case, scale):
    x = _problem(**case)
    an = _analytic(x, scale)
    for name in ("q", "k", "v", "g", "beta") + (("S0",) if x["S0"] is not None else ()):
        fd = _fd(x, name, scale)
        np.testing.assert_allclose(an[name], fd, rtol=1e-6, atol=1e-7, err_msg=name)


def test_pure_decay_closed_form():
    """beta = 0: nothing is written, S_t = e^{G_t} S0 and o_t = scale e^{G_t} S0^T q_t, so
    dS0 = sum_t scale e^{G_t} q_t do_t^T + e^{G_T} dS_final, dv = 0, dk = 0,
    dq_t = scale e^{G_t} S0 do_t and dg_t = sum_{s >= t} (scale e^{G_s} q_s^T S0 do_s) + e^{G_T} <dS_final, S0>."""
    x = _problem(5, T=6, Hv=1)
    x["beta"] = np.zeros_like(x["beta"])
    scale = 0.7
    an = _analytic(x, scale)
    g = x["g"][0, :, 0]
    Gc = np.cumsum(g)
    S0, q, do, dSf = x["S0"][0, 0], x["q"][0, :, 0], x["dout"][0, :, 0], x["dSf"][0, 0]
    dS0 = sum(scale * np.exp(Gc[t]) * np.outer(q[t], do[t]) for t in range(6)) + np.exp(Gc[-1]) * dSf
    np.testing.assert_allclose(an["S0"][0, 0], dS0, rtol=1e-12)
    np.testing.assert_allclose(an["q"][0, :, 0], [scale * np.exp(Gc[t]) * S0 @ do[t] for t in range(6)], rtol=1e-12)
    assert np.all(an["v"] == 0) and np.allclose(an["k"], 0, atol=1e-15)
    term = np.array([scale * np.exp(Gc[s]) * q[s] @ S0 @ do[s] for s in range(6)])
    dg = np.array([term[t:].sum() for t in range(6)]) + np.exp(Gc[-1]) * np.sum(dSf * S0)
    np.testing.assert_allclose(an["g"][0, :, 0], dg, rtol=1e-12)


MUTATIONS = {
    # one plausible mistake each, planted in a copy of the oracle's source; (gradient that must move)
    "dk_without_lookup_term": ("dk[b, t, hk] += lam @ u + Sp @ dp", "dk[b, t, hk] += lam @ u", "k"),
    "adjoint_not_decayed": ("lam = a * lam + np.outer(kt, dp)", "lam = lam + np.outer(kt, dp)", "S0"),
    "dg_without_chain_rule": ("dg[b, t, h] = a * da", "dg[b, t, h] = da", "g"),
    "dbeta_sign": ("dbeta[b, t, h] = du @ (vt - a * p)", "dbeta[b, t, h] = du @ (vt + a * p)", "beta"),
    "da_without_lookup_term": ("da = np.sum(lam * Sp) - bt * (du @ p)", "da = np.sum(lam * Sp)", "g"),
    "dq_from_old_state": ("dq[b, t, hk] += scale * (a * (Sp @ do) + kt * (u @ do))",
                          "dq[b, t, hk] += scale * (Sp @ do)", "q"),
}


def _mutant(kind):
    src = open(ob.__file__).read()
    old, new, _ = MUTATIONS[kind]
    assert src.count(old) == 1, kind
    ns = {}
    exec(compile(src.replace(old, new), "mutant_backward", "exec"), ns)
    return ns["backward"]


@pytest.mark.parametrize("kind", sorted(MUTATIONS))
def test_planted_mistakes_fail_the_finite_difference_pin(kind):
    x = _problem(6, T=5, Hv=1)
    an = _analytic(x, 1.0, fn=_mutant(kind))
    name = MUTATIONS[kind][2]
    fd = _fd(x, name, 1.0)
    assert not np.allclose(an[name], fd, rtol=1e-6, atol=1e-7)
