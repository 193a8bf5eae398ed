"""The shared seeded input generator: published SplitMix64 outputs, Box-Muller moments,
counter-based slicing, rounding to bf16, and the workload recipes."""
import numpy as np
import pytest

import gdn_inputs as gi


def _splitmix_python(seed, i):
    """SplitMix64 written out with Python integers (the published 64-bit finaliser)."""
    M = (1 << 64) - 1
    z = (seed + (i + 1) * 0x9E3779B97F4A7C15) & M
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M
    return z ^ (z >> 31)


def test_splitmix_published_first_output():
    # first output of SplitMix64 seeded with 0
    assert int(gi.splitmix64(0, np.array([0], dtype=np.uint64))[0]) == 0xE220A8397B1DCDAF


@pytest.mark.parametrize("seed", [0, 1, 0xDEADBEEF, (1 << 64) - 1])
def test_splitmix_matches_integer_reference(seed):
    idx = np.array([0, 1, 2, 1000, (1 << 40) + 7, (1 << 45) + 3], dtype=np.uint64)
    got = gi.splitmix64(seed, idx)
    for i, x in zip(idx.tolist(), got.tolist()):
        assert x == _splitmix_python(seed, i)


def test_normals_moments_and_slicing():
    z = gi.normals(0, 2, 1_000_001)
    assert abs(z.mean()) < 5e-3 and abs(z.std() - 1) < 5e-3
    assert abs(np.mean(z ** 4) - 3) < 3e-2            # Gaussian kurtosis
    part = np.concatenate([gi.normals(0, 2, 333, start=0), gi.normals(0, 2, 1000, start=333)])
    np.testing.assert_array_equal(part, z[:1333])
    assert not np.array_equal(gi.normals(0, 3, 100), z[:100])   # streams differ


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    x = gi.normals(4, 0, 100_000) * 7.0
    mine = gi.round_to_dtype(x, "bf16")
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(mine, ref)
    assert np.array_equal(gi.round_to_dtype(x, "f32"), x.astype(np.float32))


def test_small_workload_recipe():
    w = gi.WORKLOADS["charlm_bf16"]
    d = gi.make_prefill_inputs(w)
    assert d["q"].shape == (4, 512, 4, 32) and d["v"].shape == (4, 512, 4, 32)
    assert d["g"].shape == (4, 512, 4) and d["S0"] is None
    norms = np.linalg.norm(d["k"].astype(np.float64), axis=-1)
    assert np.all(np.abs(norms - 1) < 1e-2)               # unit rows up to bf16 rounding
    alpha = np.exp(d["g"].astype(np.float64))
    assert 0 < alpha.min() and alpha.max() < 1
    assert abs(alpha.mean() - 0.93) < 0.01                # E[sigmoid(N(3,1))] ~ 0.93
    assert 0 < d["beta"].min() and d["beta"].max() < 1 and abs(d["beta"].mean() - 0.5) < 0.01
    # every value is exactly a bf16 number
    for key in ("q", "k", "v", "g", "beta"):
        a = d[key]
        assert np.array_equal(gi.round_to_dtype(a.astype(np.float64), "bf16"), a)
    again = gi.make_prefill_inputs(w)
    assert all(np.array_equal(d[x], again[x]) for x in ("q", "k", "v", "g", "beta"))


def test_packed_workload_offsets():
    w = gi.WORKLOADS["prefill_varlen_128k"]
    assert list(w.cu_seqlens) == [0, 65536, 98304, 122880, 131072]
    assert w.num_seqs == 4 and w.B == 1
