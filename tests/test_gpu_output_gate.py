"""The output gate on its own (gdn_output_gate_fwd) and its backward (gdn_output_gate_bwd) against the
fp64 oracle (oracle.gates.gated_rmsnorm and gated_rmsnorm_backward).  Forward outputs are compared at
the dtype's tolerance; the gradients are fp32 from the same rounded inputs: 1e-4 of max|ref| each."""
import numpy as np
import pytest

import gdn_inputs as gi
from oracle import gates as og

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from gpu_util import TOL, rel_err, up  # noqa: E402
import gated_deltanet_recurrence_03_gb300 as gdn  # noqa: E402


def _inputs(dtype, rows, dv, seed):
    o = gi.round_to_dtype(gi.normals(seed, 0, rows * dv).reshape(rows, dv), dtype)
    z = gi.round_to_dtype(1.5 * gi.normals(seed, 1, rows * dv).reshape(rows, dv), dtype)
    w = gi.round_to_dtype(1.0 + 0.2 * gi.normals(seed, 2, dv), "f32")
    dy = gi.round_to_dtype(gi.normals(seed, 3, rows * dv).reshape(rows, dv), dtype)
    return o, z, w, dy


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("dv", [32, 64, 128])
@pytest.mark.parametrize("rows", [1, 37, 4099])
def test_output_gate_forward_and_backward(dtype, dv, rows):
    o, z, w, dy = _inputs(dtype, rows, dv, seed=50 + dv + rows)
    eps = 1e-6 if rows != 37 else 0.05   # an eps comparable to small rows' mean square in one case
    if rows == 37:
        o[:5] *= 0.01
    y = gdn.gdn_output_gate_fwd(up(o, dtype), up(z, dtype), up(w, torch.float32), eps)
    go, gz, gw = gdn.gdn_output_gate_bwd(up(o, dtype), up(z, dtype), up(w, torch.float32), up(dy, dtype), eps)
    torch.cuda.synchronize()
    ey = rel_err(og.gated_rmsnorm(o, z, w, eps), y.float().cpu().numpy())
    assert ey <= TOL[dtype], ey
    ref = og.gated_rmsnorm_backward(o, z, w, eps, dy)
    errs = [rel_err(r, g.cpu().numpy()) for r, g in zip(ref, (go, gz, gw))]
    assert max(errs) <= 1e-4, errs


def test_output_gate_in_place_and_same_as_the_prefill_epilogue():
    """In place (y = o) gives the same bytes as out of place, and the standalone gate applied to the
    prefill's raw output gives the same bytes as gdn_chunk_fwd with the gate fused."""
    w = gi.Workload("gate_pf", "prefill", "bf16", B=1, T=130, Hqk=1, Hv=2, dk=128, dv=128, s0_std=0.1, seed=55)
    x = gi.make_prefill_inputs(w)
    bf = torch.bfloat16
    args = [up(x[n], bf) for n in ("q", "k", "v", "g", "beta")] + [up(x["S0"], torch.float32)]
    og_in = gi.make_output_gate(w, (w.B, w.T, w.Hv, w.dv))
    zt, wt = up(og_in["z"], bf), up(og_in["norm_weight"], torch.float32)
    o_raw, _ = gdn.gdn_chunk_fwd(*args)
    o_fused, _ = gdn.gdn_chunk_fwd(*args, output_gate=(zt, wt, 1e-6))
    y = gdn.gdn_output_gate_fwd(o_raw, zt, wt, 1e-6)
    o_copy = o_raw.clone()
    gdn.gdn_output_gate_fwd(o_copy, zt, wt, 1e-6, out=o_copy)
    torch.cuda.synchronize()
    assert torch.equal(y, o_fused)
    assert torch.equal(o_copy, y)


def test_output_gate_backward_deterministic_and_empty():
    o, z, w, dy = _inputs("bf16", 20000, 128, seed=56)
    bf = torch.bfloat16
    a = [up(o, bf), up(z, bf), up(w, torch.float32), up(dy, bf)]
    r1 = gdn.gdn_output_gate_bwd(*a)
    r2 = gdn.gdn_output_gate_bwd(*a)
    e = gdn.gdn_output_gate_bwd(*(t[:0] if t.dim() == 2 else t for t in a))
    torch.cuda.synchronize()
    for p, q in zip(r1, r2):
        assert torch.equal(p, q)
    assert e[0].numel() == 0 and torch.equal(e[2], torch.zeros_like(e[2]))
