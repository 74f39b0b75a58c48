"""GPU test of the bounded waits that every kernel of the library uses: a wait on an
mbarrier that nothing arrives on gives up after its time limit and reports it, the GPU
context stays usable afterwards, and the same wait after an arrival succeeds at once.  This
is the failure the kernels map to KDA_ERR_TIMEOUT; it is made here without any fault."""
import ctypes
import os
import subprocess

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def selftest(tmp_path_factory):
    out = str(tmp_path_factory.mktemp("wait") / "wait_selftest.so")
    src = os.path.join(ROOT, "tests", "csrc", "wait_selftest.cu")
    inc = os.path.join(ROOT, "linear_attention_serving_chunkwise_gb300", "csrc")
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17", "-shared",
                    "-Xcompiler", "-fPIC", "-I", inc, src, "-o", out], check=True)
    lib = ctypes.CDLL(out)
    lib.wait_selftest.restype = ctypes.c_int
    lib.wait_selftest.argtypes = [ctypes.c_ulonglong, ctypes.c_int, ctypes.c_void_p]
    return lib


def _wait(selftest, limit_ns, arrive):
    out = torch.zeros(2, dtype=torch.int64, device="cuda")
    assert selftest.wait_selftest(limit_ns, arrive, ctypes.c_void_p(out.data_ptr())) == 0
    ok, ns = (int(x) for x in out.cpu())
    return ok, ns


def test_wait_gives_up_after_its_limit(selftest):
    limit = 20_000_000   # 20 ms
    ok, ns = _wait(selftest, limit, 0)
    assert ok == 0
    assert limit <= ns < 2_000_000_000, ns
    # the context is still usable: device work after the timeout runs and is right
    x = torch.arange(1024, device="cuda", dtype=torch.float32)
    assert float((x * 2).sum().item()) == 2 * 1023 * 1024 / 2


def test_wait_after_an_arrival_succeeds_at_once(selftest):
    ok, ns = _wait(selftest, 1_000_000_000, 1)
    assert ok == 1 and ns < 1_000_000_000
