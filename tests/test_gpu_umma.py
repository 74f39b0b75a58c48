"""GPU self-test of the tcgen05 primitives the tensor-core prefill is built from:
shared-memory descriptors (128-byte swizzle, K-major and MN-major), the bf16
instruction descriptor, TMEM allocation, tcgen05.mma / commit / ld / st and the
A-negate bit, against a torch fp32 matmul of the same bf16 values."""
import ctypes
import os
import subprocess

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def selftest(tmp_path_factory):
    out = str(tmp_path_factory.mktemp("umma") / "umma_selftest.so")
    src = os.path.join(ROOT, "tests", "csrc", "umma_selftest.cu")
    inc = os.path.join(ROOT, "linear_attention_serving_chunkwise_gb300", "csrc")
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17", "-shared",
                    "-Xcompiler", "-fPIC", "-I", inc, src, "-o", out], check=True)
    lib = ctypes.CDLL(out)
    lib.umma_selftest.restype = ctypes.c_int
    lib.umma_selftest.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    lib.umma_tf32_selftest.restype = ctypes.c_int
    lib.umma_tf32_selftest.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    return lib


def _run(selftest, A, Bm, C, K, mode, b_kmajor):
    a_store = A.t().contiguous() if mode == 2 else A.contiguous()
    b_store = Bm.t().contiguous() if b_kmajor else Bm.contiguous()
    D = torch.full((128, 128), float("nan"), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = selftest.umma_selftest(a_store.data_ptr(), b_store.data_ptr(), C.data_ptr(), D.data_ptr(), K, mode,
                                err.data_ptr())
    assert rc == 0 and int(err.item()) == 0
    return D


@pytest.mark.parametrize("K", [64, 128])
def test_umma_a_from_tmem(selftest, K):
    g = torch.Generator(device="cuda").manual_seed(7 + K)
    A = torch.randn((128, K), generator=g, device="cuda").to(torch.bfloat16)
    Bm = torch.randn((K, 128), generator=g, device="cuda").to(torch.bfloat16)
    C = torch.zeros((128, 128), device="cuda")
    D = _run(selftest, A, Bm, C, K, 4, False)
    ref = A.float() @ Bm.float()
    rel = ((D - ref).abs().max() / ref.abs().max()).item()
    assert rel < 1e-5, f"A from TMEM, K {K}: rel err {rel:.3e}"


def test_umma_m64_lane_layout(selftest):
    """M = 64 accumulator layout: result row i sits in TMEM lane (i % 16) + 32 * (i // 16)."""
    K = 64
    g = torch.Generator(device="cuda").manual_seed(3)
    A = torch.randn((128, K), generator=g, device="cuda").to(torch.bfloat16)
    A[64:] = 0
    Bm = torch.randn((K, 128), generator=g, device="cuda").to(torch.bfloat16)
    C = torch.zeros((128, 128), device="cuda")
    D = _run(selftest, A, Bm, C, K, 5, False)
    ref = (A[:64].float() @ Bm.float())
    lanes = []
    for i in range(64):
        diff = (D - ref[i][None, :]).abs().max(dim=1).values
        lane = int(torch.argmin(diff).item())
        assert diff[lane].item() < 1e-3 * ref.abs().max().item(), f"row {i} not found"
        lanes.append(lane)
    assert lanes == [(i % 16) + 32 * (i // 16) for i in range(64)]


@pytest.mark.parametrize("mode", [0, 1, 2, 3])
@pytest.mark.parametrize("K", [64, 128])
def test_umma_tile(selftest, mode, K):
    g = torch.Generator(device="cuda").manual_seed(100 * mode + K)
    A = torch.randn((128, K), generator=g, device="cuda").to(torch.bfloat16)   # math A [M, K]
    Bm = torch.randn((K, 128), generator=g, device="cuda").to(torch.bfloat16)  # math B [K, N]
    C = torch.randn((128, 128), generator=g, device="cuda")
    a_store = A.t().contiguous() if mode == 2 else A.contiguous()
    b_store = Bm.t().contiguous() if mode == 0 else Bm.contiguous()
    D = torch.full((128, 128), float("nan"), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = selftest.umma_selftest(a_store.data_ptr(), b_store.data_ptr(), C.data_ptr(), D.data_ptr(), K, mode,
                                err.data_ptr())
    assert rc == 0 and int(err.item()) == 0
    ref = A.float() @ Bm.float()
    if mode == 3:
        ref = C - ref
    assert torch.isfinite(D).all()
    rel = ((D - ref).abs().max() / ref.abs().max()).item()
    assert rel < 1e-5, f"mode {mode} K {K}: rel err {rel:.3e}"


@pytest.mark.parametrize("a_tmem", [0, 1])
@pytest.mark.parametrize("K", [32, 128])
def test_umma_tf32(selftest, K, a_tmem):
    """kind::tf32 with fp32 operands: A from shared memory or TMEM, B K-major; the
    result must carry tf32 (10-bit mantissa) precision, far better than bf16."""
    g = torch.Generator(device="cuda").manual_seed(31 + K + a_tmem)
    A = torch.randn((128, K), generator=g, device="cuda")
    B = torch.randn((128, K), generator=g, device="cuda")
    D = torch.full((128, 128), float("nan"), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = selftest.umma_tf32_selftest(A.data_ptr(), B.data_ptr(), D.data_ptr(), K, a_tmem, err.data_ptr())
    assert rc == 0 and int(err.item()) == 0
    ref = (A.double() @ B.double().t()).float()
    rel = ((D - ref).abs().max() / ref.abs().max()).item()
    assert rel < 2e-3, f"tf32 K {K} a_tmem {a_tmem}: rel err {rel:.3e}"
