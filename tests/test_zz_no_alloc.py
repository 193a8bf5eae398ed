"""gdn_chunk_fwd_noalloc, the prefill entry point for callers that cannot allocate device memory.

Some callers may not call cudaMalloc where they run the prefill (a host framework that owns all
device memory, a fixed budget, code that must not synchronise the device).  This entry point takes
its scratch from an array built into the library.  Here it is called through the C ABI twice in a
row, on different inputs, the larger problem first so that the second call starts on a scratch
array still holding the first call's data.  Each result must be bit-identical to gdn_chunk_fwd
(caller workspace) on the same inputs -- the kernels are deterministic, so any difference would be
stale or shared scratch -- and within the bf16 parity tolerance of the fp64 oracle.  A problem too
large for the built-in array must be refused before anything runs.

This file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest

import gdn_inputs as gi

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from gated_deltanet_recurrence_03_gb300 import _lib as L  # noqa: E402
from gated_deltanet_recurrence_03_gb300 import build as gbuild  # noqa: E402

TOL = 2e-2


@pytest.fixture(scope="module")
def lib():
    gbuild.build()
    return L.load()


def _device_inputs(seed, T):
    w = gi.Workload("noalloc", "prefill", "bf16", B=2, T=T, Hqk=2, Hv=4, dk=128, dv=128, chunk=64,
                    s0_std=0.1, seed=seed)
    x = gi.make_prefill_inputs(w)
    d = {n: torch.from_numpy(np.ascontiguousarray(x[n])).cuda().to(torch.bfloat16)
         for n in ("q", "k", "v", "g", "beta")}
    d["S0"] = torch.from_numpy(x["S0"]).cuda()
    return w, d


def _call(lib, fn, w, d, workspace=None, dtype=None, flags=0):
    out = torch.empty_like(d["v"])
    sf = torch.empty((w.B, w.Hv, w.dk, w.dv), dtype=torch.float32, device="cuda")
    o = L.default_opts(lib)
    o.stream = torch.cuda.current_stream().cuda_stream
    if dtype is not None:
        o.dtype = dtype
    o.flags = flags
    if workspace is not None:
        o.workspace = workspace.data_ptr()
        o.workspace_bytes = workspace.numel()
    st = fn(d["q"].data_ptr(), d["k"].data_ptr(), d["v"].data_ptr(), d["g"].data_ptr(), d["beta"].data_ptr(),
            d["S0"].data_ptr(), out.data_ptr(), sf.data_ptr(), w.B, w.T, w.Hqk, w.Hv, w.dk, w.dv, ctypes.byref(o))
    return st, out, sf


def _rel(ref, got):
    ref, got = ref.double(), got.double()
    return float((got - ref).abs().max() / ref.abs().max())


def test_noalloc_matches_workspace_entry_point_twice(lib):
    from oracle import recurrence as orc
    # two calls in a row, different inputs; the larger first, so the second call's scratch still
    # holds the first call's data beyond the part it overwrites
    for seed, T in ((22, 333), (21, 200)):
        w, d = _device_inputs(seed, T)
        o = L.default_opts(lib)
        need = lib.gdn_chunk_fwd_workspace_size(w.B, w.T, w.Hqk, w.Hv, w.dk, w.dv, ctypes.byref(o))
        assert need > 0, "this shape must take the tensor-core path, which uses scratch"
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        st_ref, out_ref, sf_ref = _call(lib, lib.gdn_chunk_fwd, w, d, workspace=ws)
        assert st_ref == L.GDN_OK, lib.gdn_last_error()
        st, out, sf = _call(lib, lib.gdn_chunk_fwd_noalloc, w, d)
        assert st == L.GDN_OK, lib.gdn_last_error()
        torch.cuda.synchronize()
        assert lib.gdn_check_device_status(None) == L.GDN_OK
        assert torch.isfinite(out.float()).all() and torch.isfinite(sf).all()
        # deterministic kernels on the same inputs: any difference at all is a scratch bug
        assert torch.equal(out, out_ref), "outputs differ from the caller-workspace entry point"
        assert torch.equal(sf, sf_ref), "final states differ from the caller-workspace entry point"
        x = {n: d[n].float().cpu().numpy() for n in ("q", "k", "v", "g", "beta", "S0")}
        o_ref, s_ref = orc.forward(x["q"], x["k"], x["v"], x["g"], x["beta"], S0=x["S0"])
        assert _rel(torch.from_numpy(o_ref), out.float().cpu()) <= TOL
        assert _rel(torch.from_numpy(s_ref), sf.cpu()) <= TOL


def test_noalloc_refuses_problems_larger_than_its_scratch(lib):
    # 32 value heads of dim 128 over 4096 tokens need ~100 MB of scratch: more than the 64 MiB array.
    # The buffers are real and sized for the call, but the call must return before any launch.
    w = gi.Workload("big", "prefill", "bf16", B=1, T=4096, Hqk=16, Hv=32, dk=128, dv=128)
    e = lambda *s: torch.zeros(*s, dtype=torch.bfloat16, device="cuda")
    d = dict(q=e(1, 4096, 16, 128), k=e(1, 4096, 16, 128), v=e(1, 4096, 32, 128), g=e(1, 4096, 32),
             beta=e(1, 4096, 32), S0=torch.zeros(1, 32, 128, 128, device="cuda"))
    st, _, _ = _call(lib, lib.gdn_chunk_fwd_noalloc, w, d)
    assert st == L.GDN_ERR_WORKSPACE
    assert b"64 MiB" in lib.gdn_last_error()


@pytest.mark.parametrize("T", [300, 4096], ids=["chunked_from_scratch", "token_serial_fallback"])
def test_noalloc_off_the_tensor_core_tile(lib, T):
    # fp32, head dim 128, in-kernel l2 norm: a short call runs the chunked kernels on the built-in
    # scratch; at 32 value heads x 4096 tokens their workspace exceeds 64 MiB and the call falls back
    # to the token-serial kernel, which needs none.  Either must match the workspace entry point.
    w = gi.Workload("noalloc_f32", "prefill", "f32", B=1, T=T, Hqk=16, Hv=32, dk=128, dv=128, s0_std=0.1,
                    seed=23)
    x = gi.make_prefill_inputs(w)
    d = {n: torch.from_numpy(np.ascontiguousarray(x[n])).cuda().float() for n in ("q", "k", "v", "g", "beta")}
    d["q"], d["k"] = 2.0 * d["q"], 0.5 * d["k"]   # off the unit sphere, so the norm matters
    d["S0"] = torch.from_numpy(x["S0"]).cuda()
    o = L.default_opts(lib)
    o.dtype, o.flags = L.GDN_F32, L.GDN_NORMALIZE_QK
    need = lib.gdn_chunk_fwd_workspace_size(w.B, w.T, w.Hqk, w.Hv, w.dk, w.dv, ctypes.byref(o))
    assert (need <= 64 << 20) == (T == 300)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    st_ref, out_ref, sf_ref = _call(lib, lib.gdn_chunk_fwd, w, d, workspace=ws, dtype=L.GDN_F32,
                                    flags=L.GDN_NORMALIZE_QK)
    assert st_ref == L.GDN_OK, lib.gdn_last_error()
    st, out, sf = _call(lib, lib.gdn_chunk_fwd_noalloc, w, d, dtype=L.GDN_F32, flags=L.GDN_NORMALIZE_QK)
    assert st == L.GDN_OK, lib.gdn_last_error()
    torch.cuda.synchronize()
    assert lib.gdn_check_device_status(None) == L.GDN_OK
    # both paths are within 1e-4 of the fp64 oracle, so within 2e-4 of each other
    assert _rel(out_ref, out) <= 2e-4 and _rel(sf_ref, sf) <= 2e-4
