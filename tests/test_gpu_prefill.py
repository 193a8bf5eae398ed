"""GPU prefill (gdn_chunk_fwd through the C ABI) against the fp64 oracle on the same seeded inputs.

Tolerance: max|out - ref| / max|ref| <= 1e-4 for fp32 inputs and <= 2e-2 for bf16 inputs, for the
outputs and for the final states alike.
"""
import numpy as np
import pytest

import gdn_inputs as gi
from oracle import recurrence as orc

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from gpu_util import TOL, prefill_on_gpu, rel_err, up  # noqa: E402
import gated_deltanet_recurrence_03_gb300 as gdn  # noqa: E402


def check(w, x, **kw):
    got_o, got_s = prefill_on_gpu(x, w.dtype, chunk=w.chunk, **kw)
    ref_o, ref_s = orc.forward(x["q"], x["k"], x["v"], x["g"], x["beta"], S0=x.get("S0"),
                               cu_seqlens=x.get("cu_seqlens"), scale=kw.get("scale", 1.0),
                               normalize_qk=kw.get("normalize_qk", False))
    eo, es = rel_err(ref_o, got_o), rel_err(ref_s, got_s)
    assert eo <= TOL[w.dtype] and es <= TOL[w.dtype], f"{w.name}: out {eo:.3e} state {es:.3e}"
    return eo, es


def test_tiny_f32_full():
    w = gi.WORKLOADS["tiny_f32"]
    check(w, gi.make_prefill_inputs(w))


def test_charlm_bf16_full():
    w = gi.WORKLOADS["charlm_bf16"]
    check(w, gi.make_prefill_inputs(w))


@pytest.mark.parametrize("T", [1, 63, 64, 65, 200])
def test_gqa_d128_ragged(T):
    """The shape of the 8k GQA workload (d = 128, 2 V heads per QK head, random S0), shortened."""
    w = gi.scaled(gi.WORKLOADS["prefill_gqa_8k"], B=2, T=T, Hqk=2, Hv=4)
    check(w, gi.make_prefill_inputs(w))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(32, 128), (128, 64), (64, 32)])
def test_mixed_head_dims(dtype, dk, dv):
    w = gi.Workload("mixed", "prefill", dtype, B=2, T=70, Hqk=1, Hv=4, dk=dk, dv=dv, chunk=32, s0_std=0.1, seed=3)
    check(w, gi.make_prefill_inputs(w))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_packed_sequences_with_empty_and_short(dtype):
    lens = (0, 1, 64, 130, 0, 77)
    w = gi.Workload("packed", "prefill", dtype, B=1, T=sum(lens), Hqk=2, Hv=4, dk=128, dv=128, chunk=64,
                    s0_std=0.1, seqlens=lens, seed=4)
    check(w, gi.make_prefill_inputs(w))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_scale_and_normalize(dtype):
    w = gi.Workload("norm", "prefill", dtype, B=1, T=90, Hqk=2, Hv=2, dk=64, dv=64, chunk=32, seed=5)
    x = gi.make_prefill_inputs(w)
    x["q"] = gi.round_to_dtype(x["q"] * 3.0, dtype)   # no longer unit length
    x["k"] = gi.round_to_dtype(x["k"] * 0.5, dtype)
    check(w, x, scale=64 ** -0.5, normalize_qk=True)


def test_zero_tokens_copies_state():
    w = gi.scaled(gi.WORKLOADS["prefill_gqa_8k"], B=2, T=0, Hqk=2, Hv=4)
    S0 = gi.make_prefill_inputs(gi.scaled(w, T=1))["S0"]
    e = lambda *s: torch.empty(*s, dtype=torch.bfloat16, device="cuda")
    S0d = up(S0, torch.float32)
    out, sf = gdn.gdn_chunk_fwd(e(2, 0, 2, 128), e(2, 0, 2, 128), e(2, 0, 4, 128), e(2, 0, 4), e(2, 0, 4), S0d)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(sf.cpu().numpy(), S0)
    _, sf0 = gdn.gdn_chunk_fwd(e(2, 0, 2, 128), e(2, 0, 2, 128), e(2, 0, 4, 128), e(2, 0, 4), e(2, 0, 4), None)
    torch.cuda.synchronize()
    assert not sf0.any()


def test_final_state_in_place_and_resume():
    """S_final may alias S0; splitting a sequence and carrying the state equals one call."""
    w = gi.scaled(gi.WORKLOADS["prefill_gqa_8k"], B=1, T=150, Hqk=2, Hv=4)
    x = gi.make_prefill_inputs(w)
    dt = torch.bfloat16
    q, k, v, g, b = (up(x[n], dt) for n in ("q", "k", "v", "g", "beta"))
    o_full, s_full = gdn.gdn_chunk_fwd(q, k, v, g, b, up(x["S0"], torch.float32))
    S = up(x["S0"], torch.float32)
    cut = 100
    o1, _ = gdn.gdn_chunk_fwd(q[:, :cut].contiguous(), k[:, :cut].contiguous(), v[:, :cut].contiguous(),
                              g[:, :cut].contiguous(), b[:, :cut].contiguous(), S, S_final=S)
    o2, _ = gdn.gdn_chunk_fwd(q[:, cut:].contiguous(), k[:, cut:].contiguous(), v[:, cut:].contiguous(),
                              g[:, cut:].contiguous(), b[:, cut:].contiguous(), S, S_final=S)
    torch.cuda.synchronize()
    assert rel_err(o_full.float().cpu().numpy(), torch.cat([o1, o2], 1).float().cpu().numpy()) <= 2e-2
    assert rel_err(s_full.cpu().numpy(), S.cpu().numpy()) <= 2e-2


def test_deterministic():
    w = gi.scaled(gi.WORKLOADS["prefill_gqa_8k"], B=1, T=333, Hqk=2, Hv=4)
    x = gi.make_prefill_inputs(w)
    a = prefill_on_gpu(x, "bf16")
    b = prefill_on_gpu(x, "bf16")
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_chain_launch_order_does_not_change_the_bits():
    """Without an event between them the chain kernel follows the prep by programmatic dependent launch
    (its set-up overlapping the prep's last CTAs, its workspace reads after the prep grid completed);
    with one it starts after the prep.  Both orders give the same bits, packed sequences included."""
    lens = (300, 0, 1, 129, 64)
    w = gi.scaled(gi.WORKLOADS["prefill_gqa_8k"], B=1, T=sum(lens), Hqk=2, Hv=4, seqlens=lens)
    x = gi.make_prefill_inputs(w)
    dt = torch.bfloat16
    q, k, v, g, beta = (up(x[n], dt) for n in ("q", "k", "v", "g", "beta"))
    S0 = up(x["S0"], torch.float32)
    cu = torch.from_numpy(np.asarray(x["cu_seqlens"], dtype=np.int32)).cuda()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    for e in ev:
        e.record()
    o1, s1 = gdn.gdn_chunk_fwd(q, k, v, g, beta, S0, cu_seqlens=cu)
    o2, s2 = gdn.gdn_chunk_fwd(q, k, v, g, beta, S0, cu_seqlens=cu, events=[e.cuda_event for e in ev])
    torch.cuda.synchronize()
    gdn.check_device_status()
    assert torch.equal(o1, o2) and torch.equal(s1, s2)
    assert rel_err(orc.forward(x["q"], x["k"], x["v"], x["g"], x["beta"], S0=x["S0"],
                               cu_seqlens=x["cu_seqlens"])[0], o1.float().cpu().numpy()) <= TOL["bf16"]


@pytest.mark.parametrize("name,dtype,d", [("tc", "bf16", 128), ("split_tf32", "f32", 32)])
def test_chunk_option_gives_the_same_result(name, dtype, d):
    """opts.chunk 16, 32 and 64 run the same 64-token blocking: bit-identical results, each within
    the tolerance of the oracle (configs asking for chunk 16 or 32 get the fast path, not a fallback)."""
    w = gi.Workload("chunks_" + name, "prefill", dtype, B=2, T=150, Hqk=2, Hv=4, dk=d, dv=d, chunk=16,
                    s0_std=0.1, seed=21)
    x = gi.make_prefill_inputs(w)
    ref_o, ref_s = orc.forward(x["q"], x["k"], x["v"], x["g"], x["beta"], S0=x.get("S0"))
    res = {c: prefill_on_gpu(x, dtype, chunk=c) for c in (16, 32, 64)}
    for c in (16, 32):
        np.testing.assert_array_equal(res[c][0], res[64][0])
        np.testing.assert_array_equal(res[c][1], res[64][1])
    assert rel_err(ref_o, res[16][0]) <= TOL[dtype] and rel_err(ref_s, res[16][1]) <= TOL[dtype]


# ---------------------------------------------------------------- full sizes, sampled heads
def _sampled(w, heads, seqs=None):
    x = gi.make_prefill_inputs(w)
    got_o, got_s = prefill_on_gpu(x, w.dtype, chunk=w.chunk)
    G = w.Hv // w.Hqk
    hk = sorted({h // G for h in heads})
    hmap = [hk.index(h // G) for h in heads]
    cu = x.get("cu_seqlens")
    # oracle on the sampled value heads only (their query/key heads regrouped)
    q, k = x["q"][:, :, hk], x["k"][:, :, hk]
    sub_v = x["v"][:, :, heads]
    sub_g, sub_b = x["g"][:, :, heads], x["beta"][:, :, heads]
    # rebuild GQA so that sampled head i reads sampled QK head hmap[i]
    q = q[:, :, hmap]
    k = k[:, :, hmap]
    S0 = None if x.get("S0") is None else x["S0"][:, heads]
    ref_o, ref_s = orc.forward(q, k, sub_v, sub_g, sub_b, S0=S0, cu_seqlens=cu)
    eo = rel_err(ref_o, got_o[:, :, heads])
    es = rel_err(ref_s, got_s[:, heads])
    assert eo <= TOL[w.dtype] and es <= TOL[w.dtype], f"{w.name}: out {eo:.3e} state {es:.3e}"


@pytest.mark.slow
def test_prefill_gqa_8k_full_sampled():
    _sampled(gi.WORKLOADS["prefill_gqa_8k"], heads=[0, 1, 17, 31])


@pytest.mark.slow
def test_prefill_varlen_128k_full_sampled():
    _sampled(gi.WORKLOADS["prefill_varlen_128k"], heads=[0, 21])


@pytest.mark.parametrize("normalize", [False, True])
def test_strong_decay_takes_the_exact_decay_path(normalize):
    """Heads 0 and 3 decay by about e^-3 per token (the log-decay span of a chunk, ~190, is too wide
    to factorise exp(G_r - G_s) = exp(G_r - G_0) exp(G_0 - G_s) in fp32), heads 1 and 2 decay weakly:
    both branches of the decay/Gram epilogue run in one launch, on the tensor-core path."""
    w = gi.scaled(gi.WORKLOADS["prefill_gqa_8k"], B=2, T=150, Hqk=2, Hv=4)
    x = gi.make_prefill_inputs(w)
    g = np.array(x["g"], dtype=np.float64)
    g[:, :, [0, 3]] = g[:, :, [0, 3]] * 60.0 - 0.5          # ~ -3.5 per token
    x["g"] = gi.round_to_dtype(g, "bf16")
    if normalize:
        x["q"] = gi.round_to_dtype(x["q"] * 2.0, "bf16")
        x["k"] = gi.round_to_dtype(x["k"] * 0.7, "bf16")
    check(w, x, normalize_qk=normalize)


@pytest.mark.parametrize("Hqk,Hv", [(2, 2), (1, 3), (2, 6)])
def test_tensor_core_path_any_head_grouping(Hqk, Hv):
    """One value head per query/key head (no GQA) and odd groupings run on the tensor-core path too:
    the last value head of an odd group pairs with itself in the prep kernel."""
    w = gi.Workload("groups", "prefill", "bf16", B=2, T=150, Hqk=Hqk, Hv=Hv, dk=128, dv=128, chunk=64,
                    s0_std=0.1, seed=7 + Hv)
    assert gdn.workspace_size(w.B, w.T, Hqk, Hv, 128, 128) > 0   # the tensor-core path is selected
    check(w, gi.make_prefill_inputs(w))


def test_tensor_core_path_odd_grouping_packed():
    lens = (70, 0, 129)
    w = gi.Workload("groups_packed", "prefill", "bf16", B=1, T=sum(lens), Hqk=1, Hv=3, dk=128, dv=128, chunk=64,
                    s0_std=0.1, seqlens=lens, seed=12)
    check(w, gi.make_prefill_inputs(w))
