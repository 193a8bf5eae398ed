"""GPU front end against the oracle: gates formed in-kernel from the raw projections
(GDN_RAW_GATES) and in-kernel l2 normalisation of q and k (GDN_NORMALIZE_QK), on the tensor-core
prefill, the chunked prefill of other shapes (the binding always passes the workspace) and decode;
the token-serial prefill's front end is covered through the C ABI in test_gpu_prefill_paths."""
import numpy as np
import pytest

import gdn_inputs as gi
from oracle import gates as ogates
from oracle import recurrence as orc

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from gpu_util import TOL, rel_err, up  # noqa: E402
import gated_deltanet_recurrence_03_gb300 as gdn  # noqa: E402

CASES = {
    "tc_bf16_d128": gi.Workload("fe", "prefill", "bf16", B=2, T=150, Hqk=2, Hv=4, dk=128, dv=128, s0_std=0.1, seed=31),
    "chunked_f32_d64": gi.Workload("fe", "prefill", "f32", B=2, T=70, Hqk=1, Hv=2, dk=64, dv=64, chunk=32,
                                  s0_std=0.1, seed=32),
    "chunked_bf16_d32": gi.Workload("fe", "prefill", "bf16", B=1, T=90, Hqk=2, Hv=2, dk=32, dv=32, s0_std=0.1, seed=33),
}


def _prefill(w, x, q, k, raw, normalize):
    dt = w.dtype
    if raw is not None:
        g_in, b_in = raw["a"], raw["b"]
        rg = (up(raw["A_log"], torch.float32), up(raw["dt_bias"], torch.float32))
    else:
        g_in, b_in, rg = x["g"], x["beta"], None
    out, sf = gdn.gdn_chunk_fwd(up(q, dt), up(k, dt), up(x["v"], dt), up(g_in, dt), up(b_in, dt),
                                up(x["S0"], torch.float32), chunk=w.chunk, normalize_qk=normalize, raw_gates=rg)
    torch.cuda.synchronize()
    gdn.check_device_status()
    return out.float().cpu().numpy(), sf.cpu().numpy()


@pytest.mark.parametrize("name", sorted(CASES))
def test_prefill_raw_gates(name):
    w = CASES[name]
    x = gi.make_prefill_inputs(w)
    raw = gi.make_raw_gates(w)
    got_o, got_s = _prefill(w, x, x["q"], x["k"], raw, False)
    g, beta = ogates.gates_from_raw(raw["a"], raw["b"], raw["A_log"], raw["dt_bias"])
    ref_o, ref_s = orc.forward(x["q"], x["k"], x["v"], g, beta, S0=x["S0"])
    eo, es = rel_err(ref_o, got_o), rel_err(ref_s, got_s)
    assert eo <= TOL[w.dtype] and es <= TOL[w.dtype], (eo, es)


@pytest.mark.parametrize("name", sorted(CASES))
def test_prefill_normalize_qk(name):
    w = CASES[name]
    x = gi.make_prefill_inputs(w)
    q = gi.round_to_dtype(x["q"] * 3.0, w.dtype)      # not unit length any more
    k = gi.round_to_dtype(x["k"] * 0.4, w.dtype)
    got_o, got_s = _prefill(w, x, q, k, None, True)
    ref_o, ref_s = orc.forward(q, k, x["v"], x["g"], x["beta"], S0=x["S0"], normalize_qk=True)
    eo, es = rel_err(ref_o, got_o), rel_err(ref_s, got_s)
    assert eo <= TOL[w.dtype] and es <= TOL[w.dtype], (eo, es)


def test_tc_raw_gates_and_normalize_together():
    w = CASES["tc_bf16_d128"]
    x = gi.make_prefill_inputs(w)
    raw = gi.make_raw_gates(w)
    q = gi.round_to_dtype(x["q"] * 2.0, w.dtype)
    k = gi.round_to_dtype(x["k"] * 0.7, w.dtype)
    got_o, got_s = _prefill(w, x, q, k, raw, True)
    g, beta = ogates.gates_from_raw(raw["a"], raw["b"], raw["A_log"], raw["dt_bias"])
    ref_o, ref_s = orc.forward(q, k, x["v"], g, beta, S0=x["S0"], normalize_qk=True)
    eo, es = rel_err(ref_o, got_o), rel_err(ref_s, got_s)
    assert eo <= 2e-2 and es <= 2e-2, (eo, es)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_raw_gates(dtype):
    w = gi.Workload("fe", "decode", dtype, B=4, T=6, Hqk=2, Hv=4, dk=128, dv=128, s0_std=0.1, seed=34)
    d = gi.make_decode_inputs(w)
    raw = gi.make_raw_gates(w, lead_shape=(w.T, w.B))
    S = up(d["S0"], torch.float32)
    rg = (up(raw["A_log"], torch.float32), up(raw["dt_bias"], torch.float32))
    outs = []
    for t in range(w.T):
        outs.append(gdn.gdn_recurrent_step(up(d["q"][t], dtype), up(d["k"][t], dtype), up(d["v"][t], dtype),
                                           up(raw["a"][t], dtype), up(raw["b"][t], dtype), S, raw_gates=rg))
    torch.cuda.synchronize()
    got_o = torch.stack(outs).float().cpu().numpy()
    g, beta = ogates.gates_from_raw(raw["a"], raw["b"], raw["A_log"], raw["dt_bias"])
    tr = lambda a: np.swapaxes(a, 0, 1)
    ref_o, ref_s = orc.forward(tr(d["q"]), tr(d["k"]), tr(d["v"]), tr(g), tr(beta), S0=d["S0"])
    eo, es = rel_err(ref_o, tr(got_o)), rel_err(ref_s, S.cpu().numpy())
    assert eo <= TOL[dtype] and es <= TOL[dtype], (eo, es)


@pytest.mark.parametrize("name", sorted(CASES))
def test_prefill_output_gate(name):
    w = CASES[name]
    x = gi.make_prefill_inputs(w)
    og = gi.make_output_gate(w, x["v"].shape)
    dt = w.dtype
    out, sf = gdn.gdn_chunk_fwd(up(x["q"], dt), up(x["k"], dt), up(x["v"], dt), up(x["g"], dt), up(x["beta"], dt),
                                up(x["S0"], torch.float32), chunk=w.chunk,
                                output_gate=(up(og["z"], dt), up(og["norm_weight"], torch.float32), 1e-6))
    torch.cuda.synchronize()
    ref_o, ref_s = orc.forward(x["q"], x["k"], x["v"], x["g"], x["beta"], S0=x["S0"])
    ref_y = ogates.gated_rmsnorm(ref_o, og["z"], og["norm_weight"], 1e-6)
    ey, es = rel_err(ref_y, out.float().cpu().numpy()), rel_err(ref_s, sf.cpu().numpy())
    assert ey <= TOL[dt] and es <= TOL[dt], (ey, es)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_output_gate(dtype):
    w = gi.Workload("fe", "decode", dtype, B=4, T=3, Hqk=2, Hv=4, dk=128, dv=128, s0_std=0.1, seed=35)
    d = gi.make_decode_inputs(w)
    og = gi.make_output_gate(w, d["v"].shape)
    S = up(d["S0"], torch.float32)
    wn = up(og["norm_weight"], torch.float32)
    outs = []
    for t in range(w.T):
        outs.append(gdn.gdn_recurrent_step(up(d["q"][t], dtype), up(d["k"][t], dtype), up(d["v"][t], dtype),
                                           up(d["g"][t], dtype), up(d["beta"][t], dtype), S,
                                           output_gate=(up(og["z"][t], dtype), wn, 1e-6)))
    torch.cuda.synchronize()
    tr = lambda a: np.swapaxes(a, 0, 1)
    ref_o, ref_s = orc.forward(tr(d["q"]), tr(d["k"]), tr(d["v"]), tr(d["g"]), tr(d["beta"]), S0=d["S0"])
    ref_y = ogates.gated_rmsnorm(ref_o, tr(og["z"]), og["norm_weight"], 1e-6)
    ey = rel_err(ref_y, tr(torch.stack(outs).float().cpu().numpy()))
    es = rel_err(ref_s, S.cpu().numpy())
    assert ey <= TOL[dtype] and es <= TOL[dtype], (ey, es)
