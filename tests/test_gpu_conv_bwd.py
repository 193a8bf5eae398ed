"""GPU backward of the causal short convolution + SiLU (gdn_causal_conv1d_bwd through the C ABI)
against the fp64 oracle (oracle.conv.causal_conv1d_backward).  The gradients are fp32 from the same
rounded inputs on both sides: max|d - ref| / max|ref| <= 1e-4 for each of grad_x, grad_w, grad_cache_in."""
import numpy as np
import pytest

import gdn_inputs as gi
from oracle import conv as oconv

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from gpu_util import rel_err, up  # noqa: E402
import gated_deltanet_recurrence_03_gb300 as gdn  # noqa: E402

TOL = 1e-4


def _case(seed, lead, C, K, dtype, nseq):
    n = int(np.prod(lead)) * C
    x = gi.round_to_dtype(gi.normals(seed, 0, n).reshape(*lead, C), dtype)
    w = gi.round_to_dtype(0.5 * gi.normals(seed, 1, C * K).reshape(C, K), "f32")
    cache = gi.round_to_dtype(gi.normals(seed, 2, nseq * (K - 1) * C).reshape(nseq, K - 1, C), dtype)
    dy = gi.round_to_dtype(gi.normals(seed, 3, n).reshape(*lead, C), dtype)
    dco = gi.round_to_dtype(gi.normals(seed, 4, nseq * (K - 1) * C).reshape(nseq, K - 1, C), dtype)
    return x, w, cache, dy, dco


def _check(x, w, cache, dy, dco, dtype, cu=None):
    cut = None if cu is None else torch.from_numpy(np.asarray(cu, np.int32)).cuda()
    gx, gw, gc = gdn.gdn_causal_conv1d_bwd(up(x, dtype), up(w, torch.float32), up(dy, dtype),
                                           None if cache is None else up(cache, dtype),
                                           grad_cache_out=None if dco is None else up(dco, dtype), cu_seqlens=cut)
    torch.cuda.synchronize()
    rx, rw, rc = oconv.causal_conv1d_backward(x, w, dy, cache, cu_seqlens=cu, dcache_out=dco)
    errs = {"x": rel_err(rx, gx.cpu().numpy()), "w": rel_err(rw, gw.cpu().numpy())}
    if gc is not None:
        errs["cache"] = rel_err(rc, gc.cpu().numpy())
    assert max(errs.values()) <= TOL, errs
    return gx, gw, gc


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("K", [1, 2, 3, 4])
@pytest.mark.parametrize("with_cache", [False, True])
def test_conv_bwd_batched(dtype, K, with_cache):
    B, T, C = 3, 150, 96
    x, w, cache, dy, dco = _case(60 + K, (B, T), C, K, dtype, B)
    _check(x, w, cache if with_cache else None, dy, dco if with_cache else None, dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_conv_bwd_packed_with_empty_and_short(dtype):
    """Sequences of 0, 1, 2 tokens (shorter than the cache: the outgoing cache still holds incoming
    entries), one across two slots and a ragged one."""
    lens = (0, 1, 2, 65, 0, 130, 3)
    K, C = 4, 64
    x, w, cache, dy, dco = _case(70, (1, sum(lens)), C, K, dtype, len(lens))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    _check(x, w, cache, dy, dco, dtype, cu=cu)


def test_conv_bwd_packed_qkv_width_and_strided_x():
    """The layer's packed q | k | v projection width (8192 channels at 16 / 32 heads would be large;
    here 3 x 256), x a channel slice of a wider tensor (evenly strided rows)."""
    B, T, C, K = 2, 200, 768, 4
    x, w, cache, dy, dco = _case(71, (B, T), C, K, "bf16", B)
    wide = np.zeros((B, T, C + 64), dtype=np.float32)
    wide[:, :, 32:32 + C] = x
    xt = up(wide, torch.bfloat16)[:, :, 32:32 + C]
    gx, gw, gc = gdn.gdn_causal_conv1d_bwd(xt, up(w, torch.float32), up(dy, torch.bfloat16), up(cache, torch.bfloat16),
                                           grad_cache_out=up(dco, torch.bfloat16))
    torch.cuda.synchronize()
    rx, rw, rc = oconv.causal_conv1d_backward(x, w, dy, cache, dcache_out=dco)
    assert max(rel_err(rx, gx.cpu().numpy()), rel_err(rw, gw.cpu().numpy()), rel_err(rc, gc.cpu().numpy())) <= TOL


def test_conv_bwd_deterministic_and_optional_outputs():
    B, T, C, K = 2, 300, 256, 4
    x, w, cache, dy, dco = _case(72, (B, T), C, K, "bf16", B)
    bf = torch.bfloat16
    args = (up(x, bf), up(w, torch.float32), up(dy, bf), up(cache, bf))
    r1 = gdn.gdn_causal_conv1d_bwd(*args, grad_cache_out=up(dco, bf))
    r2 = gdn.gdn_causal_conv1d_bwd(*args, grad_cache_out=up(dco, bf))
    r3 = gdn.gdn_causal_conv1d_bwd(*args, grad_cache_out=up(dco, bf), want_grad_w=False, want_grad_cache_in=False)
    torch.cuda.synchronize()
    for a, b in zip(r1, r2):
        assert torch.equal(a, b)
    assert r3[1] is None and r3[2] is None and torch.equal(r3[0], r1[0])
