"""The recurrent core of one GatedDeltaNet layer end to end on the GPU, against the composed oracle:
causal conv + SiLU of the packed q/k/v projection (three channel slices), gates from the raw a/b
projections, l2 norm of q and k, the recurrence (scale dk^-1/2), and the gated RMS norm with silu(z)
("Transformer by Hand, ch. 7", GatedDeltaNet.forward).  The oracle composes its fp64 pieces and
applies the same dtype casts the interfaces apply (the conv's outputs are bf16 tensors).

Also the serving invariant: a prefill of T0 tokens hands its conv caches and states to decode, and
the decode steps reproduce a prefill of T0 + n tokens."""
import numpy as np
import pytest

import gdn_inputs as gi
from oracle import conv as oconv
from oracle import gates as ogates
from oracle import recurrence as orc

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from gpu_util import rel_err, up  # noqa: E402
import gated_deltanet_recurrence_03_gb300 as gdn  # noqa: E402

TOL = 2e-2
B, T, Hqk, Hv, D, K = 2, 100, 2, 4, 128, 4
CQ, CV = Hqk * D, Hv * D
C = 2 * CQ + CV
SLICES = ((0, CQ), (CQ, 2 * CQ), (2 * CQ, C))


def _inputs(seed=41):
    w = gi.Workload("layer", "prefill", "bf16", B=B, T=T, Hqk=Hqk, Hv=Hv, dk=D, dv=D, s0_std=0.1, seed=seed)
    proj = gi.round_to_dtype(gi.normals(seed, 20, B * T * C).reshape(B, T, C), "bf16")
    cw = gi.round_to_dtype(0.5 * gi.normals(seed, 21, C * K).reshape(C, K), "f32")
    raw = gi.make_raw_gates(w)
    og = gi.make_output_gate(w, (B, T, Hv, D))
    S0 = gi.make_prefill_inputs(w)["S0"]
    return w, proj, cw, raw, og, S0


def _gpu_prefill(proj, cw, raw, og, S0, t0, t1, caches=None):
    """Layer prefill over tokens [t0, t1) of every sequence; returns out, S_final and conv caches."""
    bf = torch.bfloat16
    x = up(np.ascontiguousarray(proj[:, t0:t1]), bf)
    n = t1 - t0
    parts, new_caches = [], []
    for i, (c0, c1) in enumerate(SLICES):
        cache_in = None if caches is None else caches[i]
        y, cache_out = gdn.gdn_causal_conv1d_fwd(x[:, :, c0:c1], up(cw[c0:c1], torch.float32), cache_in)
        parts.append(y)
        new_caches.append(cache_out)
    q = parts[0].view(B, n, Hqk, D)
    k = parts[1].view(B, n, Hqk, D)
    v = parts[2].view(B, n, Hv, D)
    a, b = (up(np.ascontiguousarray(raw[n_][:, t0:t1]), bf) for n_ in ("a", "b"))
    z = up(np.ascontiguousarray(og["z"][:, t0:t1]), bf)
    out, Sf = gdn.gdn_chunk_fwd(q, k, v, a, b, S0, scale=D ** -0.5, normalize_qk=True,
                                raw_gates=(up(raw["A_log"], torch.float32), up(raw["dt_bias"], torch.float32)),
                                output_gate=(z, up(og["norm_weight"], torch.float32), 1e-6))
    return out, Sf, new_caches


def _oracle_layer(proj, cw, raw, og, S0, steps=None):
    ys = []
    for c0, c1 in SLICES:
        y, _ = oconv.causal_conv1d(proj[:, :, c0:c1], cw[c0:c1])
        ys.append(gi.round_to_dtype(y, "bf16"))          # the conv hands bf16 tensors on
    q = ys[0].reshape(B, -1, Hqk, D)
    k = ys[1].reshape(B, -1, Hqk, D)
    v = ys[2].reshape(B, -1, Hv, D)
    g, beta = ogates.gates_from_raw(raw["a"], raw["b"], raw["A_log"], raw["dt_bias"])
    o, S = orc.forward(q, k, v, g, beta, S0=S0, scale=D ** -0.5, normalize_qk=True)
    y = ogates.gated_rmsnorm(o, og["z"], og["norm_weight"], 1e-6)
    return y, S


def test_layer_prefill_matches_composed_oracle():
    w, proj, cw, raw, og, S0 = _inputs()
    out, Sf, _ = _gpu_prefill(proj, cw, raw, og, up(S0, torch.float32), 0, T)
    torch.cuda.synchronize()
    gdn.check_device_status()
    ref_y, ref_S = _oracle_layer(proj, cw, raw, og, S0)
    assert rel_err(ref_y, out.float().cpu().numpy()) <= TOL
    assert rel_err(ref_S, Sf.cpu().numpy()) <= TOL


def test_prefill_hands_over_to_decode():
    """prefill(T0) -> conv caches + states -> decode steps == prefill(T0 + n), and == the oracle."""
    w, proj, cw, raw, og, S0 = _inputs(seed=42)
    T0 = 90
    bf = torch.bfloat16
    full, Sf_full, caches_full = _gpu_prefill(proj, cw, raw, og, up(S0, torch.float32), 0, T)
    _, S, caches = _gpu_prefill(proj, cw, raw, og, up(S0, torch.float32), 0, T0)
    rg = (up(raw["A_log"], torch.float32), up(raw["dt_bias"], torch.float32))
    nw = up(og["norm_weight"], torch.float32)
    outs = []
    for t in range(T0, T):
        xt = up(np.ascontiguousarray(proj[:, t]), bf)
        y = [gdn.gdn_causal_conv1d_step(xt[:, c0:c1], up(cw[c0:c1], torch.float32), caches[i])
             for i, (c0, c1) in enumerate(SLICES)]
        o = gdn.gdn_recurrent_step(y[0].view(B, Hqk, D), y[1].view(B, Hqk, D), y[2].view(B, Hv, D),
                                   up(np.ascontiguousarray(raw["a"][:, t]), bf),
                                   up(np.ascontiguousarray(raw["b"][:, t]), bf), S, scale=D ** -0.5,
                                   normalize_qk=True, raw_gates=rg,
                                   output_gate=(up(np.ascontiguousarray(og["z"][:, t]), bf), nw, 1e-6))
        outs.append(o)
    torch.cuda.synchronize()
    gdn.check_device_status()
    dec = torch.stack(outs, 1).float().cpu().numpy()
    assert rel_err(full[:, T0:].float().cpu().numpy(), dec) <= TOL
    assert rel_err(Sf_full.cpu().numpy(), S.cpu().numpy()) <= TOL
    for i in range(3):   # the conv caches hold inputs: identical after either route
        np.testing.assert_array_equal(caches_full[i].float().cpu().numpy(), caches[i].float().cpu().numpy())
    ref_y, ref_S = _oracle_layer(proj, cw, raw, og, S0)
    assert rel_err(ref_y[:, T0:], dec) <= TOL
    assert rel_err(ref_S, S.cpu().numpy()) <= TOL
