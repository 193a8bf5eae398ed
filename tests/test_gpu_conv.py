"""GPU causal short convolution (gdn_causal_conv1d_fwd / _step through the C ABI) against the oracle."""
import numpy as np
import pytest

import gdn_inputs as gi
from oracle import conv as oconv

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from gpu_util import TOL, rel_err, up  # noqa: E402
import gated_deltanet_recurrence_03_gb300 as gdn  # noqa: E402


def _inputs(seed, lead, C, K, dtype, nseq):
    x = gi.round_to_dtype(gi.normals(seed, 0, int(np.prod(lead)) * C).reshape(*lead, C), dtype)
    w = gi.round_to_dtype(0.5 * gi.normals(seed, 1, C * K).reshape(C, K), "f32")
    cache = gi.round_to_dtype(gi.normals(seed, 2, nseq * (K - 1) * C).reshape(nseq, K - 1, C), dtype)
    return x, w, cache


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("K", [4, 2])
@pytest.mark.parametrize("with_cache", [False, True])
def test_conv_fwd_batched(dtype, K, with_cache):
    B, T, C = 3, 150, 96
    x, w, cache = _inputs(40 + K, (B, T), C, K, dtype, B)
    y, co = gdn.gdn_causal_conv1d_fwd(up(x, dtype), up(w, torch.float32), up(cache, dtype) if with_cache else None)
    torch.cuda.synchronize()
    ry, rc = oconv.causal_conv1d(x, w, cache if with_cache else None)
    assert rel_err(ry, y.float().cpu().numpy()) <= TOL[dtype]
    np.testing.assert_array_equal(co.float().cpu().numpy(), rc)   # the cache holds inputs: bit-exact


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_conv_fwd_packed_with_empty_and_short(dtype):
    lens = (0, 1, 2, 65, 0, 130, 3)
    K, C = 4, 64
    x, w, cache = _inputs(50, (1, sum(lens)), C, K, dtype, len(lens))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    y, co = gdn.gdn_causal_conv1d_fwd(up(x, dtype), up(w, torch.float32), up(cache, dtype),
                                      cu_seqlens=torch.from_numpy(cu).cuda())
    torch.cuda.synchronize()
    ry, rc = oconv.causal_conv1d(x, w, cache, cu_seqlens=cu)
    assert rel_err(ry, y.float().cpu().numpy()) <= TOL[dtype]
    np.testing.assert_array_equal(co.float().cpu().numpy(), rc)


def test_conv_on_a_channel_slice_of_the_packed_projection():
    """q, k and v come from one packed projection: convolving each channel slice in place gives the
    slices of the full convolution (the convolution is per channel)."""
    B, T, Cq, Cv, K = 2, 80, 64, 128, 4
    C = 2 * Cq + Cv
    x, w, _ = _inputs(60, (B, T), C, K, "bf16", B)
    xd, wd = up(x, "bf16"), up(w, torch.float32)
    full, _ = gdn.gdn_causal_conv1d_fwd(xd, wd)
    parts = []
    for c0, c1 in ((0, Cq), (Cq, 2 * Cq), (2 * Cq, C)):
        yp, _ = gdn.gdn_causal_conv1d_fwd(xd[:, :, c0:c1], wd[c0:c1].contiguous())
        parts.append(yp)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(torch.cat(parts, -1).float().cpu().numpy(), full.float().cpu().numpy())


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_conv_step_equals_fwd(dtype):
    N, T, C, K = 5, 9, 128, 4
    x, w, cache = _inputs(70, (N, T), C, K, dtype, N)
    wd = up(w, torch.float32)
    cd = up(cache, dtype)
    ys = [gdn.gdn_causal_conv1d_step(up(np.ascontiguousarray(x[:, t]), dtype), wd, cd) for t in range(T)]
    torch.cuda.synchronize()
    ry, rc = oconv.causal_conv1d(x, w, cache)
    assert rel_err(ry, torch.stack(ys, 1).float().cpu().numpy()) <= TOL[dtype]
    np.testing.assert_array_equal(cd.float().cpu().numpy(), rc)


def test_conv_fwd_more_token_blocks_than_grid_rows():
    """More than 65535 blocks of 64 tokens: the token-block loop strides over the grid.  The oracle
    checks the last tokens, starting from the inputs that precede them (cache continuity is pinned)."""
    T, C, K = 65535 * 64 + 200, 8, 4
    x = gi.round_to_dtype(gi.normals(80, 0, T * C).reshape(1, T, C), "bf16")
    w = gi.round_to_dtype(0.5 * gi.normals(80, 1, C * K).reshape(C, K), "f32")
    y, co = gdn.gdn_causal_conv1d_fwd(up(x, "bf16"), up(w, torch.float32))
    torch.cuda.synchronize()
    tail = 300
    ry, rc = oconv.causal_conv1d(x[:, -tail:], w, x[:, -tail - (K - 1):-tail])
    assert rel_err(ry, y[:, -tail:].float().cpu().numpy()) <= TOL["bf16"]
    np.testing.assert_array_equal(co.float().cpu().numpy(), rc)
    hy, _ = oconv.causal_conv1d(x[:, :tail], w)
    assert rel_err(hy, y[:, :tail].float().cpu().numpy()) <= TOL["bf16"]


def test_conv_step_more_rows_than_grid_rows():
    N, C, K = 70000, 8, 4
    x, w, cache = _inputs(81, (N,), C, K, "bf16", N)
    cd = up(cache, "bf16")
    y = gdn.gdn_causal_conv1d_step(up(x, "bf16"), up(w, torch.float32), cd)
    torch.cuda.synchronize()
    sel = np.r_[0:50, N - 50:N]
    ry, rc = oconv.causal_conv1d(x[sel][:, None], w, cache[sel])
    assert rel_err(ry[:, 0], y[sel].float().cpu().numpy()) <= TOL["bf16"]
    np.testing.assert_array_equal(cd[sel].float().cpu().numpy(), rc)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("K", [1, 3])
def test_conv_fwd_short_kernels(dtype, K):
    """Kernel widths 1 and 3 (K - 1 = 0 and 2 history rows), with and without a cache."""
    B, T, C = 2, 70, 64
    x, w, cache = _inputs(90 + K, (B, T), C, K, dtype, B)
    for cache_in in (None, cache):
        y, co = gdn.gdn_causal_conv1d_fwd(up(x, dtype), up(w, torch.float32),
                                          None if cache_in is None else up(cache_in, dtype))
        torch.cuda.synchronize()
        ry, rc = oconv.causal_conv1d(x, w, cache_in)
        assert rel_err(ry, y.float().cpu().numpy()) <= TOL[dtype]
        np.testing.assert_array_equal(co.float().cpu().numpy(), rc)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("K", [2, 3, 4])
def test_conv_step_kernel_widths(dtype, K):
    N, T, C = 9, 5, 96
    x, w, cache = _inputs(95 + K, (N, T), C, K, dtype, N)
    wd, cd = up(w, torch.float32), up(cache, dtype)
    ys = [gdn.gdn_causal_conv1d_step(up(np.ascontiguousarray(x[:, t]), dtype), wd, cd) for t in range(T)]
    torch.cuda.synchronize()
    ry, rc = oconv.causal_conv1d(x, w, cache)
    assert rel_err(ry, torch.stack(ys, 1).float().cpu().numpy()) <= TOL[dtype]
    np.testing.assert_array_equal(cd.float().cpu().numpy(), rc)


def test_conv_fwd_misaligned_weights_use_scalar_taps():
    """Weights [C, K=2] starting one float into an allocation (4-byte but not 8-byte aligned): the
    kernel cannot load a channel's taps as one vector, falls back to scalar loads and gives the
    same result."""
    B, T, C, K = 1, 40, 64, 2
    x, w, _ = _inputs(99, (B, T), C, K, "bf16", B)
    big = np.zeros((C * K + 1,), dtype=np.float32)
    big[1:] = w.reshape(-1)
    wt = torch.from_numpy(big).cuda()[1:].view(C, K)   # 4-byte aligned, not 8-byte aligned
    assert wt.data_ptr() % 8 != 0
    y, _ = gdn.gdn_causal_conv1d_fwd(up(x, "bf16"), wt, None)
    torch.cuda.synchronize()
    ry, _ = oconv.causal_conv1d(x, w)
    assert rel_err(ry, y.float().cpu().numpy()) <= TOL["bf16"]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("packed", [False, True])
def test_conv_fwd_qkv_is_the_split_of_one_convolution(dtype, packed):
    """The packed q | k | v projection in one launch, written to three dense tensors: bit-identical to
    the single-output convolution of the whole projection split by channel, and within the parity
    tolerance of the oracle (caches over all channels, in and out)."""
    widths = (64, 64, 128)
    C, K = sum(widths), 4
    if packed:
        lens = (0, 3, 130, 1, 70)
        B, T, nseq = 1, sum(lens), len(lens)
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    else:
        B, T, nseq, cu = 2, 150, 2, None
    x, w, cache = _inputs(110, (B, T), C, K, dtype, nseq)
    xd, wd, cd = up(x, dtype), up(w, torch.float32), up(cache, dtype)
    cu_d = None if cu is None else torch.from_numpy(cu).cuda()
    (yq, yk, yv), co = gdn.gdn_causal_conv1d_fwd_qkv(xd, wd, widths, cd, cu_seqlens=cu_d)
    full, co_full = gdn.gdn_causal_conv1d_fwd(xd, wd, cd, cu_seqlens=cu_d)
    torch.cuda.synchronize()
    assert torch.equal(torch.cat([yq, yk, yv], -1), full)
    assert torch.equal(co, co_full)
    ry, rc = oconv.causal_conv1d(x, w, cache, cu_seqlens=cu)
    assert rel_err(ry, torch.cat([yq, yk, yv], -1).float().cpu().numpy()) <= TOL[dtype]
    np.testing.assert_array_equal(co.float().cpu().numpy(), rc)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_conv_step_qkv_is_the_split_of_one_step(dtype):
    """Decode steps of the packed projection in one launch each, against the single-output step on a
    copy of the cache (bit-identical outputs and caches) and the oracle over all steps."""
    widths = (32, 32, 64)
    N, T, C, K = 7, 5, sum(widths), 4
    x, w, cache = _inputs(120, (N, T), C, K, dtype, N)
    wd = up(w, torch.float32)
    c_split, c_one = up(cache, dtype), up(cache, dtype)
    ys = []
    for t in range(T):
        xt = up(np.ascontiguousarray(x[:, t]), dtype)
        yq, yk, yv = gdn.gdn_causal_conv1d_step_qkv(xt, wd, c_split, widths)
        y1 = gdn.gdn_causal_conv1d_step(xt, wd, c_one)
        torch.cuda.synchronize()
        assert torch.equal(torch.cat([yq, yk, yv], -1), y1)
        ys.append(y1)
    assert torch.equal(c_split, c_one)
    ry, rc = oconv.causal_conv1d(x, w, cache)
    assert rel_err(ry, torch.stack(ys, 1).float().cpu().numpy()) <= TOL[dtype]
    np.testing.assert_array_equal(c_split.float().cpu().numpy(), rc)
