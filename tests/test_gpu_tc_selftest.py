"""GPU: the tcgen05 operand layouts and descriptors of the tensor-core prefill, one product at a time.

D = A B with A 128 x K and B K x N in every (A, B) major-ness the kernels use, against a float64
matmul of the same bf16 values (fp32 accumulation: relative error ~1e-6).
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest

from conftest import ROOT

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

SRC = os.path.join(ROOT, "tests", "cuda", "tc_selftest.cu")
LIB = os.path.join(ROOT, "_build", "libtc_selftest.so")


@pytest.fixture(scope="module")
def lib():
    from gated_deltanet_recurrence_03_gb300 import build as b
    os.makedirs(os.path.dirname(LIB), exist_ok=True)
    if not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        subprocess.check_call([b._nvcc(), *b.NVCC_FLAGS, "-shared", "-o", LIB, SRC])
    L = ctypes.CDLL(LIB)
    L.tc_selftest_mma.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 4 + [ctypes.c_void_p]
    L.tc_selftest_mma_tmem_a.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 3 + [ctypes.c_void_p]
    L.tc_selftest_wait_runs_out.argtypes = [ctypes.c_void_p, ctypes.c_ulonglong, ctypes.c_void_p]
    return L


@pytest.mark.parametrize("a_mn,b_mn,K,N", [
    (0, 0, 128, 64),    # [K; Q] K^T
    (0, 1, 64, 128),    # T D K
    (0, 1, 128, 192),   # blockdiag(P) [-W | Tb]
    (0, 1, 192, 64),    # A1 [S; V]
    (1, 1, 64, 64),     # K^T (b U)
    (1, 0, 64, 128),
])
def test_mma_layout(lib, a_mn, b_mn, K, N):
    rng = np.random.default_rng(K * 7 + N + 100 * a_mn + 10 * b_mn)
    A = torch.from_numpy(rng.normal(size=(128, K)).astype(np.float32)).bfloat16()
    B = torch.from_numpy(rng.normal(size=(K, N)).astype(np.float32)).bfloat16()
    Ad, Bd = A.cuda(), B.cuda()
    D = torch.zeros(128, N, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert lib.tc_selftest_mma(Ad.data_ptr(), Bd.data_ptr(), D.data_ptr(), K, N, a_mn, b_mn, status.data_ptr()) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0, "bounded wait ran out"
    ref = A.double().numpy() @ B.double().numpy()
    got = D.cpu().numpy()
    err = np.abs(got - ref).max() / np.abs(ref).max()
    assert err < 1e-5, f"max rel err {err:.3e}"


@pytest.mark.parametrize("K,N,b_mn", [(64, 128, 1), (128, 128, 1), (128, 64, 1), (128, 128, 0), (64, 128, 0)])
def test_mma_a_from_tmem(lib, K, N, b_mn):
    """A operand held in TMEM (as the prefill's P and T diag(beta gamma) operands and the chain's
    transposed state are), B from shared memory MN-major or K-major."""
    rng = np.random.default_rng(K + 3 * N)
    A = torch.from_numpy(rng.normal(size=(128, K)).astype(np.float32)).bfloat16()
    B = torch.from_numpy(rng.normal(size=(K, N)).astype(np.float32)).bfloat16()
    Ad, Bd = A.cuda(), B.cuda()
    D = torch.zeros(128, N, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert lib.tc_selftest_mma_tmem_a(Ad.data_ptr(), Bd.data_ptr(), D.data_ptr(), K, N, b_mn, status.data_ptr()) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0, "bounded wait ran out"
    ref = A.double().numpy() @ B.double().numpy()
    err = np.abs(D.cpu().numpy() - ref).max() / np.abs(ref).max()
    assert err < 1e-5, f"max rel err {err:.3e}"


def test_bounded_wait_runs_out_sets_status_and_returns(lib):
    """Failure detection without a GPU fault: an mbarrier wait that nothing completes gives up after
    its limit (50 ms here), sets the status flag, every thread returns, and the context still runs
    work afterwards."""
    import time
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    returned = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.time()
    assert lib.tc_selftest_wait_runs_out(status.data_ptr(), 50_000_000, returned.data_ptr()) == 0
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    assert int(status.item()) == 1, "the status flag was not set"
    assert int(returned.item()) == 1, "the wait did not report failure"
    assert elapsed < 5.0
    x = torch.arange(1024, device="cuda", dtype=torch.float32)
    assert float((x * 2).sum().item()) == 1023 * 1024   # the context is still usable
