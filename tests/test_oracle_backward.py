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


# ---------------------------------------------------------------- the fused front end
from oracle import gates as og  # noqa: E402


def _fe_problem(seed, lens=None, B=1, T=6, Hqk=1, Hv=2, dk=4, dv=3):
    x = _problem(seed, B=B, T=T, Hqk=Hqk, Hv=Hv, dk=dk, dv=dv, lens=lens)
    rng = np.random.default_rng(100 + seed)
    shp = x["g"].shape
    x["q"] = x["q"] * rng.uniform(0.5, 2.0, size=x["q"].shape[:-1] + (1,))    # off the unit sphere
    x["k"] = x["k"] * rng.uniform(0.5, 2.0, size=x["k"].shape[:-1] + (1,)) * np.sqrt(x["k"].shape[-1])
    x["a"] = rng.normal(0.5, 1.0, size=shp)
    x["b"] = rng.normal(size=shp)
    x["A_log"] = rng.normal(-0.5, 0.3, size=shp[-1])
    x["dt_bias"] = rng.normal(0.0, 0.5, size=shp[-1])
    return x


def _fe_loss(x, scale, **over):
    y = dict(x, **over)
    g, beta = og.gates_from_raw(y["a"], y["b"], y["A_log"], y["dt_bias"])
    o, S = orc.forward(y["q"], y["k"], y["v"], g, beta, S0=y["S0"], cu_seqlens=y["cu"], scale=scale, normalize_qk=True)
    return float(np.sum(o * x["dout"]) + np.sum(S * x["dSf"]))


def _fe_fd(x, name, scale, eps=1e-6):
    base = np.array(x[name], dtype=np.float64)
    grad = np.zeros_like(base)
    it = np.nditer(base, flags=["multi_index"])
    for _ in it:
        idx = it.multi_index
        hi, lo = base.copy(), base.copy()
        hi[idx] += eps
        lo[idx] -= eps
        grad[idx] = (_fe_loss(x, scale, **{name: hi}) - _fe_loss(x, scale, **{name: lo})) / (2 * eps)
    return grad


def _fe_analytic(x, scale):
    r = ob.backward_frontend(x["q"], x["k"], x["v"], x["a"], x["b"], x["dout"], A_log=x["A_log"],
                             dt_bias=x["dt_bias"], normalize_qk=True, S0=x["S0"], dS_final=x["dSf"],
                             cu_seqlens=x["cu"], scale=scale)
    return dict(zip(("q", "k", "v", "a", "b", "S0", "A_log", "dt_bias"), r))


@pytest.mark.parametrize("case", [dict(seed=11), dict(seed=12, lens=(2, 0, 4)), dict(seed=13, B=2, Hqk=2, Hv=2, T=4)])
def test_front_end_gradients_match_finite_differences(case):
    """The raw-row l2 norm (done by the C forward) and the gates from raw a, b (oracle.gates): every
    gradient of backward_frontend against central differences of the composed forward."""
    x = _fe_problem(**case)
    an = _fe_analytic(x, 0.8)
    for name in ("q", "k", "v", "a", "b", "S0", "A_log", "dt_bias"):
        fd = _fe_fd(x, name, 0.8)
        np.testing.assert_allclose(an[name], fd, rtol=1e-6, atol=1e-7, err_msg=name)


def test_l2_backward_is_orthogonal_to_the_row_and_scale_equivariant():
    """x_n depends only on the direction of x (up to eps), so dx is orthogonal to x and halves when x
    doubles."""
    rng = np.random.default_rng(7)
    x, dxn = rng.normal(size=(5, 8)), rng.normal(size=(5, 8))
    dx = ob.l2_normalize_backward(x, dxn, eps=0.0)
    np.testing.assert_allclose(np.sum(dx * x, axis=-1), 0.0, atol=1e-13)
    np.testing.assert_allclose(ob.l2_normalize_backward(2 * x, dxn, eps=0.0), dx / 2, rtol=1e-12)
    # along x itself the gradient vanishes; across it, it is dxn / |x|
    u = x[0] / np.linalg.norm(x[0])
    np.testing.assert_allclose(ob.l2_normalize_backward(x[:1], u[None], eps=0.0), 0.0, atol=1e-14)


def test_gate_gradients_closed_values():
    """At a + dt_bias = 0: sigmoid = 1/2, so da = -exp(A_log) dg / 2; at b = 0: db = dbeta / 4;
    dA_log = sum dg g with g = -exp(A_log) ln 2."""
    A_log, dt = np.array([0.3]), np.array([0.7])
    a, b = np.full((3, 1), -0.7), np.zeros((3, 1))
    dg, dbeta = np.array([[1.0], [2.0], [-0.5]]), np.array([[4.0], [1.0], [2.0]])
    da, db, dA, ddt = ob.gates_backward(a, b, A_log, dt, dg, dbeta)
    np.testing.assert_allclose(da, -np.exp(0.3) * dg / 2, rtol=1e-14)
    np.testing.assert_allclose(db, dbeta / 4, rtol=1e-14)
    np.testing.assert_allclose(dA, [np.sum(dg) * -np.exp(0.3) * np.log(2.0)], rtol=1e-14)
    np.testing.assert_allclose(ddt, [np.sum(da)], rtol=1e-14)


@pytest.mark.parametrize("mistake", ["no_projection", "r_squared", "no_sigmoid", "beta_not_squashed"])
def test_front_end_pins_catch_planted_mistakes(mistake, monkeypatch):
    """A plausible slip in the chain rule of the front end fails the finite-difference pin."""
    good_l2, good_gates = ob.l2_normalize_backward, ob.gates_backward

    def bad_l2(x, dxn, eps=ob.L2_EPS):
        x, dxn = np.asarray(x, dtype=np.float64), np.asarray(dxn, dtype=np.float64)
        r = 1.0 / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)
        if mistake == "no_projection":
            return r * dxn
        return r * dxn - r ** 2 * np.sum(x * dxn, axis=-1, keepdims=True) * x

    def bad_gates(a, b, A_log, dt_bias, dg, dbeta):
        da, db, dA, ddt = good_gates(a, b, A_log, dt_bias, dg, dbeta)
        if mistake == "no_sigmoid":
            da = np.asarray(dg) * -np.exp(np.asarray(A_log))
            ddt = np.sum(da, axis=tuple(range(np.ndim(dg) - 1)))
        else:
            db = np.asarray(dbeta, dtype=np.float64)
        return da, db, dA, ddt

    if mistake in ("no_projection", "r_squared"):
        monkeypatch.setattr(ob, "l2_normalize_backward", bad_l2)
    else:
        monkeypatch.setattr(ob, "gates_backward", bad_gates)
    x = _fe_problem(11)
    an = _fe_analytic(x, 1.0)
    names = ("q", "k") if mistake in ("no_projection", "r_squared") else ("a", "b", "dt_bias")
    worst = max(np.max(np.abs(an[n] - _fe_fd(x, n, 1.0))) for n in names)
    assert worst > 1e-3, f"{mistake} went unnoticed ({worst:.2e})"
