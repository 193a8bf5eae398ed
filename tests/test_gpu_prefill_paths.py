"""Both prefill paths for shapes off the tensor-core tile (fp32 inputs, head dims 32 / 64), called
through the C ABI on the same inputs: without a workspace (the token-serial kernel) and with
gdn_chunk_fwd_workspace_size() bytes (the chunked kernels on split-tf32 MMAs), each plain and with the
in-kernel front end (gates from raw projections, l2 norm of q and k off the unit sphere).  Each is
compared with the fp64 oracle at the parity bound of its input dtype (1e-4 fp32, 2e-2 bf16), outputs
and final states."""
import ctypes

import numpy as np
import pytest

import gdn_inputs as gi
from oracle import gates as ogates
from oracle import recurrence as orc

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from gpu_util import TOL, TORCH_DT, rel_err  # noqa: E402
from gated_deltanet_recurrence_03_gb300 import _lib as L  # noqa: E402
from gated_deltanet_recurrence_03_gb300 import build as gbuild  # noqa: E402


@pytest.fixture(scope="module")
def lib():
    gbuild.build()
    return L.load()


CASES = [
    gi.Workload("paths_f32_d32", "prefill", "f32", B=2, T=150, Hqk=2, Hv=4, dk=32, dv=32, s0_std=0.1, seed=31),
    gi.Workload("paths_f32_d128_packed", "prefill", "f32", B=1, T=300, Hqk=1, Hv=2, dk=128, dv=128, s0_std=0.1,
                seqlens=(0, 130, 1, 169), seed=32),
    gi.Workload("paths_bf16_d64", "prefill", "bf16", B=3, T=97, Hqk=2, Hv=6, dk=64, dv=32, s0_std=0.0, seed=33),
]


def _run(lib, w, x, scale, with_workspace, raw=None, normalize=False):
    dt = TORCH_DT[w.dtype]
    d = {n: torch.from_numpy(np.ascontiguousarray(x[n])).cuda().to(dt) for n in ("q", "k", "v", "g", "beta")}
    keep = []
    S0 = None if x.get("S0") is None else torch.from_numpy(x["S0"]).cuda()
    out = torch.empty_like(d["v"])
    sf = torch.empty((w.num_seqs, w.Hv, w.dk, w.dv), dtype=torch.float32, device="cuda")
    o = L.default_opts(lib)
    o.dtype = L.GDN_BF16 if w.dtype == "bf16" else L.GDN_F32
    o.scale = scale
    o.stream = torch.cuda.current_stream().cuda_stream
    if normalize:
        o.flags |= L.GDN_NORMALIZE_QK
    if raw is not None:   # g and beta hold the raw projections a and b
        d["g"] = torch.from_numpy(raw["a"]).cuda().to(dt)
        d["beta"] = torch.from_numpy(raw["b"]).cuda().to(dt)
        keep = [torch.from_numpy(raw[n]).cuda().float() for n in ("A_log", "dt_bias")]
        o.flags |= L.GDN_RAW_GATES
        o.A_log, o.dt_bias = keep[0].data_ptr(), keep[1].data_ptr()
    cu = None
    if x.get("cu_seqlens") is not None:
        cu = torch.from_numpy(np.asarray(x["cu_seqlens"], np.int32)).cuda()
        o.cu_seqlens = cu.data_ptr()
        o.num_seqs = w.num_seqs
    need = lib.gdn_chunk_fwd_workspace_size(w.B, w.T, w.Hqk, w.Hv, w.dk, w.dv, ctypes.byref(o))
    assert need > 0, "shapes off the tensor-core tile take the chunked path when given a workspace"
    ws = None
    if with_workspace:
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        o.workspace = ws.data_ptr()
        o.workspace_bytes = need
    st = lib.gdn_chunk_fwd(d["q"].data_ptr(), d["k"].data_ptr(), d["v"].data_ptr(), d["g"].data_ptr(),
                           d["beta"].data_ptr(), 0 if S0 is None else S0.data_ptr(), out.data_ptr(),
                           sf.data_ptr(), w.B, w.T, w.Hqk, w.Hv, w.dk, w.dv, ctypes.byref(o))
    assert st == L.GDN_OK, lib.gdn_last_error()
    torch.cuda.synchronize()
    assert lib.gdn_check_device_status(None) == L.GDN_OK
    return out.float().cpu().numpy(), sf.cpu().numpy()


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
@pytest.mark.parametrize("with_workspace", [False, True], ids=["token_serial", "chunked"])
@pytest.mark.parametrize("front", [False, True], ids=["plain", "front_end"])
def test_prefill_paths_off_the_tensor_core_tile(lib, w, with_workspace, front):
    x = gi.make_prefill_inputs(w)
    scale = w.dk ** -0.5
    raw = None
    g, beta = x["g"], x["beta"]
    if front:   # rows off the unit sphere, so the norm matters; gates formed from a, b
        x["q"] = gi.round_to_dtype(x["q"] * 2.5, w.dtype)
        x["k"] = gi.round_to_dtype(x["k"] * 0.45, w.dtype)
        raw = gi.make_raw_gates(w)
        g, beta = ogates.gates_from_raw(raw["a"], raw["b"], raw["A_log"], raw["dt_bias"])
    got_o, got_s = _run(lib, w, x, scale, with_workspace, raw=raw, normalize=front)
    ref_o, ref_s = orc.forward(x["q"], x["k"], x["v"], g, beta, S0=x.get("S0"),
                               cu_seqlens=x.get("cu_seqlens"), scale=scale, normalize_qk=front)
    eo, es = rel_err(ref_o, got_o), rel_err(ref_s, got_s)
    assert eo <= TOL[w.dtype] and es <= TOL[w.dtype], (w.name, eo, es)
