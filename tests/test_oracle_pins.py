"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Every test here checks the oracle (oracle.recurrence) against something other
than itself: values the pages print for worked examples (tests/golden/), closed
forms, invariants, brute force, an independent statement of the update from the
other page, or the independent chunk-form derivation.  No GPU is needed.
"""
import math

import numpy as np
import pytest

from conftest import read_golden
from gdn_inputs import normals, unit_rows
from oracle import chunked
from oracle import recurrence as orc


def run1(q, k, v, g, beta, S0=None, mode=orc.MODE_DELTA, scale=1.0, normalize_qk=False):
    """One sequence, one head: q, k [T, dk]; v [T, dv]; g, beta [T]."""
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    T = q.shape[0]
    out, sf = orc.forward(q.reshape(1, T, 1, -1), k.reshape(1, T, 1, -1), v.reshape(1, T, 1, -1),
                          np.asarray(g, dtype=np.float64).reshape(1, T, 1),
                          np.asarray(beta, dtype=np.float64).reshape(1, T, 1),
                          S0=None if S0 is None else np.asarray(S0, dtype=np.float64)[None, None],
                          mode=mode, scale=scale, normalize_qk=normalize_qk, threads=1)
    return out[0, :, 0], sf[0, 0]


def gv(vals):
    return np.array([float(x) for x in vals])


# ---------------------------------------------------------------- worked 2-D example
def test_toy_table_and_reads():
    """Handbook ch. 7, ch07_toy.py output part 1: two writes, then three reads."""
    gold = read_golden("toy_2d.txt")
    k1, k2, z = [1.0, 0.0], [0.0, 1.0], [0.0, 0.0]
    q = [k1, k2, [1.0, 0.0], [0.0, 1.0], [0.6, 0.8]]
    k = [k1, k2, z, z, z]
    v = [[3.0, 1.0], [-1.0, 2.0], z, z, z]
    beta = [1, 1, 0, 0, 0]
    out, S = run1(q, k, v, np.zeros(5), beta)
    np.testing.assert_allclose(S.ravel(), gv(gold["table"]), atol=1e-12)
    np.testing.assert_allclose(out[2], gv(gold["read_q_1_0"]), atol=1e-12)
    np.testing.assert_allclose(out[3], gv(gold["read_q_0_1"]), atol=1e-12)
    np.testing.assert_allclose(out[4], gv(gold["read_q_06_08"]), atol=1e-12)


@pytest.mark.parametrize("name,mode,alpha", [("linear", orc.MODE_PLAIN_ADD, 1.0),
                                             ("delta", orc.MODE_DELTA, 1.0),
                                             ("gated05", orc.MODE_DELTA, 0.5)])
def test_toy_overwrite(name, mode, alpha):
    """ch07_toy.py output part 2: rewrite k1 -> (5, 0) from the table, read k1 and k2."""
    gold = read_golden("toy_2d.txt")
    table = gv(gold["table"]).reshape(2, 2)
    for qv, key in (([1.0, 0.0], f"{name}_k1"), ([0.0, 1.0], f"{name}_k2")):
        out, _ = run1([qv], [[1.0, 0.0]], [[5.0, 0.0]], [math.log(alpha)], [1.0], S0=table, mode=mode)
        np.testing.assert_allclose(out[0], gv(gold[key]), atol=1e-12)


@pytest.mark.parametrize("alpha", ["1.0", "0.9", "0.5"])
def test_decay_powers(alpha):
    """ch07_toy.py output part 3: beta = 0 leaves exp(sum g) * S0 after 10 and 50 steps."""
    gold = read_golden("toy_2d.txt")[f"decay_{alpha}"]
    a = float(alpha)
    for n, fmt, want in ((10, "{:.3f}", gold[0]), (50, "{:.3g}", gold[1])):
        _, S = run1(np.ones((n, 1)), np.ones((n, 1)), np.ones((n, 1)), np.full(n, math.log(a)),
                    np.zeros(n), S0=np.ones((1, 1)))
        assert fmt.format(S[0, 0]) == want
        assert S[0, 0] == pytest.approx(a ** n, rel=1e-13)


def test_embedded_2d_example_in_32_dims():
    """The 2-D example zero-padded to dk = dv = 32 gives the same numbers and zeros elsewhere."""
    d = 32
    E = lambda x: np.concatenate([np.asarray(x, dtype=np.float64), np.zeros(d - 2)])
    q = [E([1, 0]), E([0, 1]), E([0.6, 0.8])]
    k = [E([1, 0]), E([0, 1]), E([0, 0])]
    v = [E([3, 1]), E([-1, 2]), E([0, 0])]
    out, S = run1(q, k, v, np.zeros(3), [1, 1, 0])
    np.testing.assert_allclose(out[2], E([1.0, 2.2]), atol=1e-12)
    want = np.zeros((d, d))
    want[:2, :2] = [[3, 1], [-1, 2]]
    np.testing.assert_allclose(S, want, atol=1e-12)


# ---------------------------------------------------------------- closed forms
def test_repeated_write_distances():
    """ch07_deltanet.py part 3: same (k, v) six times, q = k, g = 0, beta = 0.5.

    Delta rule: |o_t - v| = |v| 2^-t.  Plain add: |o_t - v| = |v| |1 - t/2|.  The
    printed {:6.3f} values follow with |v| = 9.3454 (the page's torch draw is not
    reproducible here, so |v| is set to a value consistent with every printed digit).
    """
    gold = read_golden("repeated_write.txt")
    dk = 128
    k = unit_rows(normals(11, 0, dk))
    v = normals(11, 1, dk)
    v *= 9.3454 / np.linalg.norm(v)
    Q = np.tile(k, (6, 1))
    V = np.tile(v, (6, 1))
    for mode, key in ((orc.MODE_DELTA, "delta"), (orc.MODE_PLAIN_ADD, "plain")):
        out, _ = run1(Q, Q, V, np.zeros(6), np.full(6, 0.5), mode=mode, scale=dk ** -0.5)
        dist = np.linalg.norm(out * dk ** 0.5 - v, axis=1)
        assert [f"{x:6.3f}".strip() for x in dist] == gold[key]
        t = np.arange(1, 7)
        closed = np.linalg.norm(v) * (0.5 ** t if key == "delta" else np.abs(1 - t / 2))
        np.testing.assert_allclose(dist, closed, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("alpha", [1.0, 0.7, 0.05])
def test_write_invariant(alpha):
    """beta = 1, |k| = 1: right after the write, S'^T k = v; beta = 0.5 lands half way
    between the decayed old value and v (learn-llm page, S'k = Sk + beta (v - Sk)|k|^2;
    handbook question 2)."""
    rng = np.random.default_rng(1)
    dk, dv = 16, 12
    S0 = rng.normal(size=(dk, dv))
    k = unit_rows(rng.normal(size=dk))
    v = rng.normal(size=dv)
    _, S1 = run1([k], [k], [v], [math.log(alpha)], [1.0], S0=S0)
    np.testing.assert_allclose(S1.T @ k, v, atol=1e-12)
    _, Sh = run1([k], [k], [v], [math.log(alpha)], [0.5], S0=S0)
    np.testing.assert_allclose(Sh.T @ k, 0.5 * (alpha * S0.T @ k + v), atol=1e-12)


def test_divergence_with_long_key():
    """|k|^2 = 4, beta = 1: the read-back error is multiplied by |1 - beta |k|^2| = 3 per write."""
    dk, dv = 8, 5
    rng = np.random.default_rng(2)
    k = 2.0 * unit_rows(rng.normal(size=dk))
    v = rng.normal(size=dv)
    n = 6
    out, _ = run1(np.tile(k, (n, 1)), np.tile(k, (n, 1)), np.tile(v, (n, 1)), np.zeros(n), np.ones(n))
    err = np.linalg.norm(v - out, axis=1)
    np.testing.assert_allclose(err, np.linalg.norm(v) * 3.0 ** np.arange(1, n + 1), rtol=1e-10)


@pytest.mark.parametrize("mode", [orc.MODE_DELTA, orc.MODE_PLAIN_ADD])
def test_orthogonal_recall_exact(mode):
    """128 mutually orthogonal unit keys in a 128 x 128 table read back exactly
    (ch07_toy.py output part 4: 0% error for both linear attention and the delta rule)."""
    dk = dv = 128
    Kmat, _ = np.linalg.qr(normals(5, 0, dk * dk).reshape(dk, dk))
    K = Kmat.T                                    # rows are orthonormal keys
    V = normals(5, 1, dk * dv).reshape(dk, dv)
    Q = np.concatenate([np.zeros((dk, dk)), K])   # write phase, then read phase with q = k_j
    Kin = np.concatenate([K, np.zeros((dk, dk))])
    Vin = np.concatenate([V, np.zeros((dk, dv))])
    beta = np.concatenate([np.ones(dk), np.zeros(dk)])
    out, _ = run1(Q, Kin, Vin, np.zeros(2 * dk), beta, mode=mode)
    np.testing.assert_allclose(out[dk:], V, atol=1e-12)


@pytest.mark.parametrize("decay", [False, True])
def test_linear_attention_bruteforce(decay):
    """Plain add is linear attention: o_t = sum_{j<=t} exp(sum_{i=j+1..t} g_i) beta_j (q_t.k_j) v_j
    (handbook section "The memory table": the sum over keys equals (sum_j k_j v_j^T)^T q)."""
    rng = np.random.default_rng(3)
    T, dk, dv = 40, 6, 5
    q, k, v = rng.normal(size=(T, dk)), rng.normal(size=(T, dk)), rng.normal(size=(T, dv))
    g = -rng.uniform(0.0, 0.3, size=T) if decay else np.zeros(T)
    beta = rng.uniform(0.1, 1.0, size=T) if decay else np.ones(T)
    out, _ = run1(q, k, v, g, beta, mode=orc.MODE_PLAIN_ADD, scale=0.75)
    want = np.zeros((T, dv))
    for t in range(T):
        for j in range(t + 1):
            w = math.exp(sum(g[j + 1:t + 1])) * beta[j] * float(q[t] @ k[j])
            want[t] += w * v[j]
    np.testing.assert_allclose(out, 0.75 * want, rtol=1e-12, atol=1e-12)


def test_transposed_update_table():
    """The learn-llm page's update table writes the state as dv x dk:
    S_t = S_{t-1} (alpha_t (I - beta_t k k^T)) + beta_t v k^T.  Its transpose is the oracle's S."""
    rng = np.random.default_rng(4)
    T, dk, dv = 20, 5, 3
    q, k, v = rng.normal(size=(T, dk)), unit_rows(rng.normal(size=(T, dk))), rng.normal(size=(T, dv))
    g = -rng.uniform(0, 0.5, size=T)
    beta = rng.uniform(0, 1, size=T)
    S0 = rng.normal(size=(dk, dv))
    out, S = run1(q, k, v, g, beta, S0=S0)
    St = S0.T.copy()
    for t in range(T):
        a = math.exp(g[t])
        St = St @ (a * (np.eye(dk) - beta[t] * np.outer(k[t], k[t]))) + beta[t] * np.outer(v[t], k[t])
        np.testing.assert_allclose(out[t], St @ q[t], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(S, St.T, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- structure
def test_grouped_heads_follow_repeat_interleave():
    """Value head h reads query/key head h // (Hv/Hqk), as repeat_interleave in the GatedDeltaNet shell."""
    rng = np.random.default_rng(5)
    B, T, Hqk, Hv, d = 2, 9, 2, 6, 4
    q, k = rng.normal(size=(B, T, Hqk, d)), rng.normal(size=(B, T, Hqk, d))
    v = rng.normal(size=(B, T, Hv, d))
    g, beta = -rng.uniform(0, 1, size=(B, T, Hv)), rng.uniform(0, 1, size=(B, T, Hv))
    out, sf = orc.forward(q, k, v, g, beta)
    rep = Hv // Hqk
    out2, sf2 = orc.forward(np.repeat(q, rep, axis=2), np.repeat(k, rep, axis=2), v, g, beta)
    np.testing.assert_array_equal(out, out2)
    np.testing.assert_array_equal(sf, sf2)


def test_normalize_flag_matches_prenormalised():
    rng = np.random.default_rng(6)
    B, T, H, d = 1, 12, 2, 8
    q, k = rng.normal(size=(B, T, H, d)) * 3, rng.normal(size=(B, T, H, d)) * 0.5
    v = rng.normal(size=(B, T, H, d))
    g, beta = -rng.uniform(0, 1, size=(B, T, H)), rng.uniform(0, 1, size=(B, T, H))
    o1, s1 = orc.forward(q, k, v, g, beta, normalize_qk=True)
    o2, s2 = orc.forward(unit_rows(q), unit_rows(k), v, g, beta)
    np.testing.assert_allclose(o1, o2, rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(s1, s2, rtol=1e-5, atol=1e-6)


def test_packed_sequences_equal_separate_runs():
    rng = np.random.default_rng(7)
    lens = [5, 17, 1, 9]
    T = sum(lens)
    Hqk, Hv, d = 1, 2, 4
    q, k = rng.normal(size=(1, T, Hqk, d)), rng.normal(size=(1, T, Hqk, d))
    v = rng.normal(size=(1, T, Hv, d))
    g, beta = -rng.uniform(0, 1, size=(1, T, Hv)), rng.uniform(0, 1, size=(1, T, Hv))
    S0 = rng.normal(size=(len(lens), Hv, d, d))
    cu = np.concatenate([[0], np.cumsum(lens)])
    out, sf = orc.forward(q, k, v, g, beta, S0=S0, cu_seqlens=cu)
    for i in range(len(lens)):
        sl = slice(cu[i], cu[i + 1])
        o_i, s_i = orc.forward(q[:, sl], k[:, sl], v[:, sl], g[:, sl], beta[:, sl], S0=S0[i:i + 1])
        np.testing.assert_array_equal(out[:, sl], o_i)
        np.testing.assert_array_equal(sf[i], s_i[0])


def test_split_and_resume_equals_one_run():
    """Feeding the returned state back in (delta_rule returns the final S) resumes exactly."""
    rng = np.random.default_rng(8)
    T, H, d = 23, 2, 6
    q, k = rng.normal(size=(1, T, H, d)), rng.normal(size=(1, T, H, d))
    v = rng.normal(size=(1, T, H, d))
    g, beta = -rng.uniform(0, 1, size=(1, T, H)), rng.uniform(0, 1, size=(1, T, H))
    out, sf = orc.forward(q, k, v, g, beta)
    for cut in (1, 11, 22):
        oa, sa = orc.forward(q[:, :cut], k[:, :cut], v[:, :cut], g[:, :cut], beta[:, :cut])
        ob, sb = orc.forward(q[:, cut:], k[:, cut:], v[:, cut:], g[:, cut:], beta[:, cut:], S0=sa)
        np.testing.assert_allclose(np.concatenate([oa, ob], axis=1), out, rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(sb, sf, rtol=1e-13, atol=1e-13)


def test_decode_step_is_one_token_of_the_loop():
    rng = np.random.default_rng(9)
    N, Hqk, Hv, d = 3, 1, 2, 5
    q, k = rng.normal(size=(N, Hqk, d)), rng.normal(size=(N, Hqk, d))
    v = rng.normal(size=(N, Hv, d))
    g, beta = -rng.uniform(0, 1, size=(N, Hv)), rng.uniform(0, 1, size=(N, Hv))
    S = rng.normal(size=(N, Hv, d, d))
    o, S1 = orc.decode_step(q, k, v, g, beta, S, scale=0.5)
    for n in range(N):
        for h in range(Hv):
            St = math.exp(g[n, h]) * S[n, h]
            p = St.T @ k[n, 0]
            St = St + np.outer(k[n, 0], beta[n, h] * (v[n, h] - p))
            np.testing.assert_allclose(S1[n, h], St, rtol=1e-13, atol=1e-13)
            np.testing.assert_allclose(o[n, h], 0.5 * St.T @ q[n, 0], rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------- chunk algebra
@pytest.mark.parametrize("chunk", [1, 16, 64])
def test_chunk_form_equals_token_loop(chunk):
    """The chunk-parallel (WY/UT) algebra equals the token loop to fp64 rounding, for ragged
    tails, grouped heads, packed sequences and a random initial state."""
    rng = np.random.default_rng(10 + chunk)
    lens = [100, 37, 64]
    T = sum(lens)
    Hqk, Hv, dk, dv = 2, 4, 16, 8
    q = unit_rows(rng.normal(size=(1, T, Hqk, dk)))
    k = unit_rows(rng.normal(size=(1, T, Hqk, dk)))
    v = rng.normal(size=(1, T, Hv, dv))
    g = np.log(1 / (1 + np.exp(-rng.normal(3, 1, size=(1, T, Hv)))))
    beta = 1 / (1 + np.exp(-rng.normal(size=(1, T, Hv))))
    S0 = 0.1 * rng.normal(size=(len(lens), Hv, dk, dv))
    cu = np.concatenate([[0], np.cumsum(lens)])
    o_ref, s_ref = orc.forward(q, k, v, g, beta, S0=S0, cu_seqlens=cu, scale=0.3)
    o_chk, s_chk = chunked.forward(q, k, v, g, beta, S0=S0, cu_seqlens=cu, chunk=chunk, scale=0.3)
    np.testing.assert_allclose(o_chk, o_ref, rtol=0, atol=1e-12 * np.abs(o_ref).max())
    np.testing.assert_allclose(s_chk, s_ref, rtol=0, atol=1e-12 * np.abs(s_ref).max())


@pytest.mark.parametrize("chunk", [16, 64])
def test_folded_chunk_form_equals_token_loop(chunk):
    """The chunk step with U eliminated (one affine map of the state per chunk:
    S_n = (gamma_n I - K~^T W) S0 + K~^T U~) equals the token loop, ragged and packed, with GQA."""
    rng = np.random.default_rng(20 + chunk)
    lens = [150, 9, 64]
    T = sum(lens)
    Hqk, Hv, dk, dv = 2, 4, 16, 8
    q = unit_rows(rng.normal(size=(1, T, Hqk, dk)))
    k = unit_rows(rng.normal(size=(1, T, Hqk, dk)))
    v = rng.normal(size=(1, T, Hv, dv))
    g = np.log(1 / (1 + np.exp(-rng.normal(3, 1, size=(1, T, Hv)))))
    beta = 1 / (1 + np.exp(-rng.normal(size=(1, T, Hv))))
    S0 = 0.1 * rng.normal(size=(len(lens), Hv, dk, dv))
    cu = np.concatenate([[0], np.cumsum(lens)])
    o_ref, s_ref = orc.forward(q, k, v, g, beta, S0=S0, cu_seqlens=cu, scale=0.5)
    o_f, s_f = chunked.forward(q, k, v, g, beta, S0=S0, cu_seqlens=cu, chunk=chunk, scale=0.5, folded=True)
    np.testing.assert_allclose(o_f, o_ref, rtol=0, atol=1e-12 * np.abs(o_ref).max())
    np.testing.assert_allclose(s_f, s_ref, rtol=0, atol=1e-12 * np.abs(s_ref).max())


def test_chunk_form_survives_strong_decay():
    """Cumulated decay far below fp64's range (sum g < -745 inside one chunk) stays finite,
    because decay ratios are exp(G_r - G_s) with s <= r."""
    rng = np.random.default_rng(12)
    T, H, d = 64, 1, 8
    q, k = unit_rows(rng.normal(size=(1, T, H, d))), unit_rows(rng.normal(size=(1, T, H, d)))
    v = rng.normal(size=(1, T, H, d))
    g = np.full((1, T, H), -20.0)
    beta = np.full((1, T, H), 0.9)
    o_ref, s_ref = orc.forward(q, k, v, g, beta)
    o_chk, s_chk = chunked.forward(q, k, v, g, beta, chunk=64)
    assert np.all(np.isfinite(o_chk))
    np.testing.assert_allclose(o_chk, o_ref, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(s_chk, s_ref, rtol=1e-10, atol=1e-12)
