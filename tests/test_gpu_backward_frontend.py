"""GPU backward through the fused front end (gdn_recurrent_bwd with GDN_NORMALIZE_QK and / or
GDN_RAW_GATES) against the fp64 oracle (oracle.backward.backward_frontend): the gradients with respect
to the raw q, k (before the l2 norm), v, the raw gate projections a, b, S0, and the per-head A_log and
dt_bias.  Both sides read the same rounded inputs and the GPU path computes in fp32, so the bound is
max|d - ref| / max|ref| <= 1e-4 per gradient for both input dtypes."""
import numpy as np
import pytest

import gdn_inputs as gi
from oracle import backward as ob

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from gpu_util import rel_err, up  # noqa: E402
import gated_deltanet_recurrence_03_gb300 as gdn  # noqa: E402

TOL = 1e-4


def run(w, normalize, raw_gates, scale=1.0, seqlens=None):
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    x, y = gi.make_prefill_inputs(w), gi.make_backward_inputs(w)
    q, k = x["q"], x["k"]
    if normalize:   # off the unit sphere, row lengths varying, so that the norm's gradient matters
        lead = q.shape[:-1] + (1,)
        q = gi.round_to_dtype(q * np.linspace(0.5, 3.0, q.shape[1])[None, :, None, None] * np.ones(lead), w.dtype)
        k = gi.round_to_dtype(k * np.linspace(2.0, 0.3, k.shape[1])[None, :, None, None] * np.ones(lead), w.dtype)
    raw = gi.make_raw_gates(w) if raw_gates else None
    ga, gb = (raw["a"], raw["b"]) if raw_gates else (x["g"], x["beta"])
    cu = None if seqlens is None else np.concatenate([[0], np.cumsum(seqlens)]).astype(np.int64)
    rg = (up(raw["A_log"], torch.float32), up(raw["dt_bias"], torch.float32)) if raw_gates else None
    got = gdn.gdn_recurrent_bwd(up(q, dt), up(k, dt), up(x["v"], dt), up(ga, dt), up(gb, dt), up(x["S0"], torch.float32),
                                up(y["dout"], dt), up(y["dSf"], torch.float32), scale=scale,
                                cu_seqlens=None if cu is None else torch.from_numpy(cu.astype(np.int32)).cuda(),
                                normalize_qk=normalize, raw_gates=rg)
    torch.cuda.synchronize()
    gdn.check_device_status()
    ref = ob.backward_frontend(q, k, x["v"], ga, gb, y["dout"], A_log=raw["A_log"] if raw_gates else None,
                               dt_bias=raw["dt_bias"] if raw_gates else None, normalize_qk=normalize, S0=x["S0"],
                               dS_final=y["dSf"], cu_seqlens=cu, scale=scale)
    names = ("q", "k", "v", "a" if raw_gates else "g", "b" if raw_gates else "beta", "S0", "A_log", "dt_bias")
    errs = {n: rel_err(r, g.cpu().numpy()) for n, r, g in zip(names, ref, got) if r is not None}
    bad = {n: e for n, e in errs.items() if not e <= TOL}
    assert not bad, errs
    return errs


@pytest.mark.parametrize("normalize,raw_gates", [(True, False), (False, True), (True, True)],
                         ids=["normalize", "raw_gates", "both"])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_front_end_backward_tensor_core_shape(dtype, normalize, raw_gates):
    """dk = dv = 128, two value heads per query/key head, a ragged last chunk."""
    w = gi.Workload("fe_bwd", "prefill", dtype, B=2, T=150, Hqk=2, Hv=4, dk=128, dv=128, s0_std=0.1, seed=41)
    run(w, normalize, raw_gates, scale=0.5)


def test_front_end_backward_packed_small_heads():
    """Packed sequences (an empty one and a one-token one) with head dims 64 / 32, both front-end parts."""
    lens = (70, 0, 1, 33)
    w = gi.Workload("fe_bwd_packed", "prefill", "bf16", B=1, T=sum(lens), Hqk=1, Hv=3, dk=64, dv=32, s0_std=0.1,
                    seqlens=lens, seed=42)
    run(w, True, True, seqlens=lens)


def test_front_end_backward_packed_tensor_core_shape():
    """Packed sequences (an empty one, a one-token one, one across three chunks) at dk = dv = 128 in bf16:
    every kernel on the raw rows, the chunk-local kernel reading the per-slot l2 scalars back."""
    lens = (70, 0, 1, 130)
    w = gi.Workload("fe_bwd_packed128", "prefill", "bf16", B=1, T=sum(lens), Hqk=2, Hv=4, dk=128, dv=128,
                    s0_std=0.1, seqlens=lens, seed=45)
    run(w, True, True, seqlens=lens)


def test_front_end_backward_many_value_heads():
    """More than 256 value heads: the per-head parameter sums take the one-block-per-head path."""
    w = gi.Workload("fe_bwd_wide", "prefill", "f32", B=1, T=24, Hqk=1, Hv=264, dk=32, dv=32, s0_std=0.1, seed=46)
    run(w, False, True)


def test_front_end_backward_of_unit_rows_matches_the_plain_backward():
    """Rows already of unit length: the l2 norm changes them by eps only, so the front-end path's q / k
    gradients (projected onto the tangent space) and the plain path's differ by the radial component,
    while v, g, beta and S0 gradients agree to rounding."""
    w = gi.Workload("fe_bwd_unit", "prefill", "f32", B=1, T=96, Hqk=1, Hv=2, dk=64, dv=64, s0_std=0.1, seed=43)
    x, y = gi.make_prefill_inputs(w), gi.make_backward_inputs(w)
    f32 = torch.float32
    args = [up(x[n], f32) for n in ("q", "k", "v", "g", "beta")] + [up(x["S0"], f32), up(y["dout"], f32),
                                                                   up(y["dSf"], f32)]
    plain = gdn.gdn_recurrent_bwd(*args)
    fe = gdn.gdn_recurrent_bwd(*args, normalize_qk=True)
    torch.cuda.synchronize()
    for i in (2, 3, 4, 5):
        assert rel_err(plain[i].cpu().numpy(), fe[i].cpu().numpy()) <= 1e-5
    q = up(x["q"], f32)
    radial = (plain[0] * q).sum(-1, keepdim=True) * q
    assert rel_err((plain[0] - radial).cpu().numpy(), fe[0].cpu().numpy()) <= 1e-4


def test_front_end_backward_is_deterministic():
    w = gi.Workload("fe_bwd_det", "prefill", "bf16", B=1, T=200, Hqk=2, Hv=4, dk=128, dv=128, s0_std=0.1, seed=44)
    x, y, raw = gi.make_prefill_inputs(w), gi.make_backward_inputs(w), gi.make_raw_gates(w)
    bf = torch.bfloat16
    args = [up(x["q"], bf), up(x["k"], bf), up(x["v"], bf), up(raw["a"], bf), up(raw["b"], bf),
            up(x["S0"], torch.float32), up(y["dout"], bf), up(y["dSf"], torch.float32)]
    rg = (up(raw["A_log"], torch.float32), up(raw["dt_bias"], torch.float32))
    r1 = gdn.gdn_recurrent_bwd(*args, normalize_qk=True, raw_gates=rg)
    r2 = gdn.gdn_recurrent_bwd(*args, normalize_qk=True, raw_gates=rg)
    torch.cuda.synchronize()
    for a, b in zip(r1, r2):
        assert torch.equal(a, b)
