"""A seeded sweep over shapes and options: prefill, decode and the backward pass on the GPU against
the fp64 oracle, at the same bounds as the targeted tests (1e-4 for fp32 inputs, 2e-2 for bf16 on
the forward; 1e-4 on the fp32 gradients).  Each case draws, from its own seed, the dtype, head dims,
query/key heads and value heads per group, chunk length, scale, in-kernel l2 norm, initial state and
either a batch or a packed set of sequences (empty ones included); about a third of the forward
cases take the tensor-core shape (bf16, d = 128, chunk 64)."""
import numpy as np
import pytest

import gdn_inputs as gi
from oracle import backward as ob
from oracle import recurrence as orc

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from gpu_util import TOL, prefill_on_gpu, rel_err, up  # noqa: E402
import gated_deltanet_recurrence_03_gb300 as gdn  # noqa: E402


def draw_case(i, max_len=150):
    rng = np.random.default_rng(9000 + i)
    tc = i % 3 == 0
    dtype = "bf16" if tc else str(rng.choice(["f32", "bf16"]))
    dk = 128 if tc else int(rng.choice([32, 64, 128]))
    dv = 128 if tc else int(rng.choice([32, 64, 128]))
    chunk = 64 if tc else int(rng.choice([16, 32, 64]))
    Hqk = int(rng.integers(1, 4))
    Hv = Hqk * int(rng.integers(1, 4))
    scale = float(rng.choice([1.0, dk ** -0.5, 0.7]))
    normalize = bool(rng.integers(0, 2))
    s0 = float(rng.choice([0.0, 0.1]))
    if rng.integers(0, 2):
        lens = tuple(int(x) for x in rng.integers(0, max_len, size=int(rng.integers(1, 5))))
        if sum(lens) == 0:
            lens = lens + (1,)
        w = gi.Workload(f"sweep{i}", "prefill", dtype, B=1, T=sum(lens), Hqk=Hqk, Hv=Hv, dk=dk, dv=dv, chunk=chunk,
                        s0_std=s0, seqlens=lens, seed=9000 + i)
    else:
        w = gi.Workload(f"sweep{i}", "prefill", dtype, B=int(rng.integers(1, 4)), T=int(rng.integers(1, max_len)),
                        Hqk=Hqk, Hv=Hv, dk=dk, dv=dv, chunk=chunk, s0_std=s0, seed=9000 + i)
    x = gi.make_prefill_inputs(w)
    if normalize:   # rows off the unit sphere, so the in-kernel norm matters
        x["q"] = gi.round_to_dtype(x["q"] * 1.7, dtype)
        x["k"] = gi.round_to_dtype(x["k"] * 0.6, dtype)
    return w, x, scale, normalize


@pytest.mark.parametrize("i", range(24))
def test_prefill_sweep(i):
    w, x, scale, normalize = draw_case(i)
    got_o, got_s = prefill_on_gpu(x, w.dtype, chunk=w.chunk, scale=scale, normalize_qk=normalize)
    ref_o, ref_s = orc.forward(x["q"], x["k"], x["v"], x["g"], x["beta"], S0=x.get("S0"),
                               cu_seqlens=x.get("cu_seqlens"), scale=scale, normalize_qk=normalize)
    eo, es = rel_err(ref_o, got_o), rel_err(ref_s, got_s)
    assert eo <= TOL[w.dtype] and es <= TOL[w.dtype], (w, scale, normalize, eo, es)


@pytest.mark.parametrize("i", range(8))
def test_decode_sweep(i):
    rng = np.random.default_rng(9100 + i)
    dtype = str(rng.choice(["f32", "bf16"]))
    dk, dv = int(rng.choice([32, 64, 128])), int(rng.choice([32, 64, 128]))
    Hqk = int(rng.integers(1, 4))
    Hv = Hqk * int(rng.integers(1, 4))
    N, steps = int(rng.integers(1, 6)), int(rng.integers(1, 5))
    scale, normalize = float(rng.choice([1.0, 0.5])), bool(rng.integers(0, 2))
    w = gi.Workload(f"dsweep{i}", "decode", dtype, B=N, T=steps, Hqk=Hqk, Hv=Hv, dk=dk, dv=dv, s0_std=0.1,
                    seed=9100 + i)
    x = gi.make_decode_inputs(w)
    S = up(x["S0"], torch.float32)
    S_ref = np.array(x["S0"], dtype=np.float64)
    for t in range(steps):
        out = gdn.gdn_recurrent_step(up(x["q"][t], dtype), up(x["k"][t], dtype), up(x["v"][t], dtype),
                                     up(x["g"][t], dtype), up(x["beta"][t], dtype), S, scale=scale,
                                     normalize_qk=normalize)
        torch.cuda.synchronize()
        ref_o, S_ref = orc.decode_step(x["q"][t], x["k"][t], x["v"][t], x["g"][t], x["beta"][t], S_ref, scale=scale,
                                       normalize_qk=normalize)
        eo = rel_err(ref_o, out.float().cpu().numpy())
        assert eo <= TOL[dtype], (w, t, eo)
    es = rel_err(S_ref, S.cpu().numpy())
    assert es <= TOL[dtype], (w, es)
    gdn.check_device_status()


@pytest.mark.parametrize("i", range(8))
def test_backward_sweep(i):
    w, x, scale, _ = draw_case(100 + i, max_len=140)
    y = gi.make_backward_inputs(w)
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    cu = x.get("cu_seqlens")
    got = gdn.gdn_recurrent_bwd(*(up(x[n], dt) for n in ("q", "k", "v", "g", "beta")),
                                None if x.get("S0") is None else up(x["S0"], torch.float32), up(y["dout"], dt),
                                up(y["dSf"], torch.float32), scale=scale,
                                cu_seqlens=None if cu is None else torch.from_numpy(np.asarray(cu, np.int32)).cuda())
    torch.cuda.synchronize()
    gdn.check_device_status()
    ref = ob.backward(x["q"], x["k"], x["v"], x["g"], x["beta"], y["dout"], S0=x.get("S0"), dS_final=y["dSf"],
                      cu_seqlens=cu, scale=scale)
    names = ("q", "k", "v", "g", "beta", "S0")
    errs = {}
    for n_, r, gg in zip(names, ref, got):
        if n_ == "S0" and gg is None:
            continue
        errs[n_] = rel_err(r, gg.cpu().numpy())
    assert all(e <= 1e-4 for e in errs.values()), (w, scale, errs)
