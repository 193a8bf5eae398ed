"""Helpers shared by the GPU parity tests: device upload of the shared synthetic inputs and the
parity metric max|got - ref| / max|ref|."""
import numpy as np
import torch

import gdn_inputs as gi

TOL = {"f32": 1e-4, "bf16": 2e-2}
TORCH_DT = {"f32": torch.float32, "bf16": torch.bfloat16}


def dev():
    return torch.device("cuda", torch.cuda.current_device())


def up(a, dtype):
    """Upload a float32 array holding exactly-representable values, narrowing to ``dtype``."""
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev()).to(TORCH_DT[dtype] if isinstance(dtype, str) else dtype)


def rel_err(ref, got):
    ref = np.asarray(ref, dtype=np.float64)
    got = np.asarray(got, dtype=np.float64)
    assert ref.shape == got.shape, (ref.shape, got.shape)
    assert np.all(np.isfinite(got)), "non-finite values in GPU result"
    den = np.abs(ref).max()
    return float(np.abs(got - ref).max() / (den if den > 0 else 1.0))


def prefill_on_gpu(x, dtype, chunk=64, scale=1.0, normalize_qk=False, with_s0=True, out_final=True):
    import gated_deltanet_recurrence_03_gb300 as gdn
    cu = None if x.get("cu_seqlens") is None else torch.from_numpy(x["cu_seqlens"]).to(dev())
    S0 = up(x["S0"], torch.float32) if (with_s0 and x.get("S0") is not None) else None
    out, sf = gdn.gdn_chunk_fwd(up(x["q"], dtype), up(x["k"], dtype), up(x["v"], dtype), up(x["g"], dtype),
                                up(x["beta"], dtype), S0, chunk=chunk, scale=scale, normalize_qk=normalize_qk,
                                cu_seqlens=cu, output_final_state=out_final)
    torch.cuda.synchronize()
    gdn.check_device_status()
    return out.float().cpu().numpy(), (None if sf is None else sf.cpu().numpy())
