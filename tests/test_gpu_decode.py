"""GPU decode (gdn_recurrent_step through the C ABI) against the fp64 oracle on the same inputs.

The state is carried on the device across steps, as the decode workload does; the oracle runs the
same tokens as one sequence per decode slot.
"""
import numpy as np
import pytest

import gdn_inputs as gi
from oracle import recurrence as orc

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from gpu_util import TOL, rel_err, up  # noqa: E402
import gated_deltanet_recurrence_03_gb300 as gdn  # noqa: E402


def run_steps(w, d, steps, dtype, scale=1.0, normalize_qk=False, seq_subset=None):
    S = up(d["S0"], torch.float32)
    qs, ks, vs, gs, bs = (up(d[n][:steps], dtype) for n in ("q", "k", "v", "g", "beta"))
    outs = torch.empty_like(vs)
    for t in range(steps):
        gdn.gdn_recurrent_step(qs[t], ks[t], vs[t], gs[t], bs[t], S, out=outs[t], scale=scale,
                               normalize_qk=normalize_qk)
    torch.cuda.synchronize()
    gdn.check_device_status()
    got_o = outs.float().cpu().numpy()              # [steps, N, Hv, dv]
    got_s = S.cpu().numpy()
    sel = slice(None) if seq_subset is None else seq_subset
    # oracle: each decode slot is one sequence of `steps` tokens
    tr = lambda a: np.swapaxes(a[:steps], 0, 1)[sel]
    ref_o, ref_s = orc.forward(tr(d["q"]), tr(d["k"]), tr(d["v"]), tr(d["g"]), tr(d["beta"]), S0=d["S0"][sel],
                               scale=scale, normalize_qk=normalize_qk)
    return rel_err(ref_o, np.swapaxes(got_o, 0, 1)[sel]), rel_err(ref_s, got_s[sel])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(128, 128), (32, 32), (64, 128), (128, 32)])
def test_decode_small(dtype, dk, dv):
    w = gi.Workload("dec", "decode", dtype, B=5, T=9, Hqk=2, Hv=4, dk=dk, dv=dv, s0_std=0.1, seed=7)
    d = gi.make_decode_inputs(w)
    eo, es = run_steps(w, d, 9, dtype)
    assert eo <= TOL[dtype] and es <= TOL[dtype], (eo, es)


def test_decode_normalize_and_scale():
    w = gi.Workload("dec", "decode", "f32", B=3, T=4, Hqk=1, Hv=2, dk=64, dv=64, s0_std=0.1, seed=8)
    d = gi.make_decode_inputs(w)
    d["q"] = d["q"] * 2.5
    d["k"] = d["k"] * 0.3
    eo, es = run_steps(w, d, 4, "f32", scale=0.125, normalize_qk=True)
    assert eo <= 1e-4 and es <= 1e-4, (eo, es)


def test_decode_continues_prefill():
    """prefill(T) then decode(n) equals prefill(T + n)."""
    w = gi.scaled(gi.WORKLOADS["prefill_gqa_8k"], B=2, T=80, Hqk=2, Hv=4)
    x = gi.make_prefill_inputs(w)
    dt = torch.bfloat16
    q, k, v, g, b = (up(x[n], dt) for n in ("q", "k", "v", "g", "beta"))
    S0 = up(x["S0"], torch.float32)
    o_full, s_full = gdn.gdn_chunk_fwd(q, k, v, g, b, S0)
    T0 = 70
    _, S = gdn.gdn_chunk_fwd(q[:, :T0].contiguous(), k[:, :T0].contiguous(), v[:, :T0].contiguous(),
                             g[:, :T0].contiguous(), b[:, :T0].contiguous(), S0)
    outs = []
    for t in range(T0, 80):
        outs.append(gdn.gdn_recurrent_step(q[:, t].contiguous(), k[:, t].contiguous(), v[:, t].contiguous(),
                                           g[:, t].contiguous(), b[:, t].contiguous(), S))
    torch.cuda.synchronize()
    assert rel_err(o_full[:, T0:].float().cpu().numpy(), torch.stack(outs, 1).float().cpu().numpy()) <= 2e-2
    assert rel_err(s_full.cpu().numpy(), S.cpu().numpy()) <= 2e-2


@pytest.mark.slow
def test_decode_256x512_full_sampled():
    """The full decode workload (256 x 32 heads, 512 steps, 512 MiB of state); every output and the
    final state of a sample of sequences are compared."""
    w = gi.WORKLOADS["decode_256x512"]
    d = gi.make_decode_inputs(w)
    eo, es = run_steps(w, d, w.T, "bf16", seq_subset=[0, 77, 255])
    assert eo <= 2e-2 and es <= 2e-2, (eo, es)
