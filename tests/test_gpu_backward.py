"""GPU backward pass (gdn_recurrent_bwd through the C ABI) against the fp64 oracle backward.

The gradients are computed in fp32 from the same (rounded) inputs on both sides, so the bound is
the fp32 one for both input dtypes: max|d - ref| / max|ref| <= 1e-4 per gradient."""
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
NAMES = ("q", "k", "v", "g", "beta", "S0")


def run(w, x, y, scale=1.0, with_s0=True, with_dsf=True):
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    cu = x.get("cu_seqlens")
    S0 = x.get("S0") if with_s0 else None
    dSf = y["dSf"] if with_dsf else None
    got = gdn.gdn_recurrent_bwd(*(up(x[n], dt) for n in ("q", "k", "v", "g", "beta")),
                                None if S0 is None else up(S0, torch.float32), up(y["dout"], dt),
                                None if dSf is None else up(dSf, torch.float32), scale=scale,
                                cu_seqlens=None if cu is None else torch.from_numpy(np.asarray(cu, np.int32)).cuda())
    torch.cuda.synchronize()
    gdn.check_device_status()
    ref = ob.backward(x["q"], x["k"], x["v"], x["g"], x["beta"], y["dout"], S0=S0, dS_final=dSf, cu_seqlens=cu,
                      scale=scale)
    errs = {n: rel_err(r, gg.cpu().numpy()) for n, r, gg in zip(NAMES, ref, got)}
    bad = {n: e for n, e in errs.items() if not e <= TOL}
    assert not bad, f"{w.name}: {errs}"
    return errs


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(32, 32), (64, 128), (128, 64), (128, 128)])
def test_backward_small(dtype, dk, dv):
    w = gi.Workload("bwd", "prefill", dtype, B=2, T=37, Hqk=1, Hv=2, dk=dk, dv=dv, s0_std=0.1, seed=11)
    run(w, gi.make_prefill_inputs(w), gi.make_backward_inputs(w), scale=0.5)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_backward_packed_with_empty_and_short(dtype):
    lens = (0, 1, 16, 17, 0, 40)
    w = gi.Workload("bwd_packed", "prefill", dtype, B=1, T=sum(lens), Hqk=2, Hv=4, dk=64, dv=64, s0_std=0.1,
                    seqlens=lens, seed=12)
    x, y = gi.make_prefill_inputs(w), gi.make_backward_inputs(w)
    run(w, x, y)
    run(w, x, y, with_s0=False, with_dsf=False)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_backward_packed_multichunk_odd_grouping_strong_decay(dtype):
    """Packed sequences spanning several 64-token chunks (full, partial and a 1-token tail), three value
    heads per query/key head, and one head with strong decay (~e^-3.5 per token, whose decay ratios
    underflow within a chunk)."""
    lens = (130, 0, 64, 1, 200)
    w = gi.Workload("bwd_packed_mc", "prefill", dtype, B=1, T=sum(lens), Hqk=1, Hv=3, dk=64, dv=32, s0_std=0.1,
                    seqlens=lens, seed=14)
    x, y = gi.make_prefill_inputs(w), gi.make_backward_inputs(w)
    g = np.array(x["g"], dtype=np.float64)
    g[:, :, 1] = g[:, :, 1] * 60.0 - 0.5
    x["g"] = gi.round_to_dtype(g, dtype)
    run(w, x, y, scale=0.7)


def test_backward_longer_gqa_d128():
    w = gi.scaled(gi.WORKLOADS["prefill_gqa_8k"], B=1, T=300, Hqk=2, Hv=4)
    run(w, gi.make_prefill_inputs(w), gi.make_backward_inputs(w))


def test_backward_matches_torch_autograd_of_the_loop_on_gpu():
    """A second, independent reference on the device: torch autograd of the token loop in fp64."""
    w = gi.Workload("bwd_ag", "prefill", "f32", B=1, T=20, Hqk=1, Hv=2, dk=32, dv=32, s0_std=0.1, seed=13)
    x, y = gi.make_prefill_inputs(w), gi.make_backward_inputs(w)
    t = {n: torch.tensor(x[n], dtype=torch.float64, requires_grad=True) for n in ("q", "k", "v", "g", "beta", "S0")}
    S = t["S0"][0].clone()
    outs = []
    for i in range(w.T):
        Ss = []
        for h in range(w.Hv):
            a = torch.exp(t["g"][0, i, h])
            kk, qq = t["k"][0, i, 0], t["q"][0, i, 0]
            u = t["beta"][0, i, h] * (t["v"][0, i, h] - a * (S[h].T @ kk))
            Ss.append(a * S[h] + torch.outer(kk, u))
        S = torch.stack(Ss)
        outs.append(torch.stack([S[h].T @ t["q"][0, i, 0] for h in range(w.Hv)]))
    loss = (torch.stack(outs)[None] * torch.tensor(y["dout"], dtype=torch.float64)).sum() + \
        (S[None] * torch.tensor(y["dSf"], dtype=torch.float64)).sum()
    loss.backward()
    got = gdn.gdn_recurrent_bwd(*(up(x[n], torch.float32) for n in ("q", "k", "v", "g", "beta")),
                                up(x["S0"], torch.float32), up(y["dout"], torch.float32), up(y["dSf"], torch.float32))
    torch.cuda.synchronize()
    for n, gg in zip(NAMES, got):
        assert rel_err(t[n].grad.numpy(), gg.cpu().numpy()) <= TOL, n


@pytest.mark.slow
def test_backward_prefill_gqa_8k_full_sampled():
    """The full 8k workload on the GPU; the oracle checks sequence 0, value heads 16 and 17 (both
    readers of query/key head 8, so that head's dq and dk are complete)."""
    w = gi.WORKLOADS["prefill_gqa_8k"]
    x, y = gi.make_prefill_inputs(w), gi.make_backward_inputs(w)
    dt = torch.bfloat16
    got = gdn.gdn_recurrent_bwd(*(up(x[n], dt) for n in ("q", "k", "v", "g", "beta")), up(x["S0"], torch.float32),
                                up(y["dout"], dt), up(y["dSf"], torch.float32))
    torch.cuda.synchronize()
    got = [gg.cpu().numpy() for gg in got]
    heads = [16, 17]
    sub = lambda a, ax: np.take(a[:1], heads, axis=ax)
    ref = ob.backward(x["q"][:1, :, 8:9], x["k"][:1, :, 8:9], sub(x["v"], 2), sub(x["g"], 2), sub(x["beta"], 2),
                      sub(y["dout"], 2), S0=sub(x["S0"], 1), dS_final=sub(y["dSf"], 1))
    mine = [got[0][:1, :, 8:9], got[1][:1, :, 8:9], sub(got[2], 2), sub(got[3], 2), sub(got[4], 2), sub(got[5], 1)]
    errs = {n: rel_err(r, m) for n, r, m in zip(NAMES, ref, mine)}
    assert all(e <= TOL for e in errs.values()), errs


def test_backward_no_tokens_passes_the_final_state_gradient_through():
    """T = 0: the state is never touched, so dL/dS0 = dL/dS_final."""
    dSf = torch.randn(2, 2, 32, 32, device="cuda")
    e = torch.empty(2, 0, 1, 32, dtype=torch.bfloat16, device="cuda")
    ev = torch.empty(2, 0, 2, 32, dtype=torch.bfloat16, device="cuda")
    eg = torch.empty(2, 0, 2, dtype=torch.bfloat16, device="cuda")
    S0 = torch.randn(2, 2, 32, 32, device="cuda")
    got = gdn.gdn_recurrent_bwd(e, e, ev, eg, eg, S0, ev, dSf)
    torch.cuda.synchronize()
    assert torch.equal(got[5], dSf)
    assert all(t.numel() == 0 for t in got[:5])
