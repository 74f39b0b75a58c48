"""GPU tests of kda_prefill_host_static, the entry point for callers that cannot allocate
device memory when a request arrives (their device memory already belongs to their own pool,
or their loop cannot take a cudaMalloc's synchronisation): the host-buffer prefill with its
device staging in the library's own fixed scratch array, no workspace from the caller and no
device allocation.  Its results must equal those of kda_prefill_host with a workspace, on
consecutive calls too.  Collected last (the file sorts last) so that a run stopping at the
first failure has run every other test first; it also passes alone in a fresh process."""
import numpy as np
import pytest
import torch

import kda_workloads as W
from _parity import check, oracle_full, tol_for

pytestmark = pytest.mark.gpu


def _pinned(d):
    return {k: (None if v is None else v.contiguous().pin_memory()) for k, v in d.items()}


def test_static_scratch_equals_workspace_path(cuda_lib):
    cfg = W.random_prefill_config([300, 0, 641, 129], 3, 128, torch.bfloat16, init="normal")
    h = _pinned(W.make_prefill_inputs(cfg, seed=41))
    ref_out, ref_fin = cuda_lib.prefill_host(h["q"], h["k"], h["v"], h["g"], h["beta"], h["cu_seqlens"],
                                             h["init_state"], segment_tokens=128)
    out, fin = cuda_lib.prefill_host_static(h["q"], h["k"], h["v"], h["g"], h["beta"], h["cu_seqlens"],
                                            h["init_state"], segment_tokens=128)
    torch.cuda.synchronize()
    assert cuda_lib.last_device_status() == cuda_lib.KDA_OK
    assert torch.equal(out, ref_out) and torch.equal(fin, ref_fin)
    o, s = oracle_full({k: v for k, v in h.items()})
    check("static-scratch out vs oracle", out, o, tol_for(torch.bfloat16))
    check("static-scratch final vs oracle", fin, s, tol_for(torch.bfloat16))


def test_static_scratch_allocates_nothing(cuda_lib):
    cfg = W.random_prefill_config([700, 260], 4, 64, torch.float32, init="normal")
    h = _pinned(W.make_prefill_inputs(cfg, seed=42))
    out = torch.empty((cfg.total_tokens, 4, 64), dtype=torch.float32).pin_memory()
    fin = torch.empty((2, 4, 64, 64), dtype=torch.float32).pin_memory()
    args = (h["q"], h["k"], h["v"], h["g"], h["beta"], h["cu_seqlens"], h["init_state"], out, fin)
    cuda_lib.prefill_host_static(*args, segment_tokens=256)   # first call maps the scratch
    torch.cuda.synchronize()
    first = out.clone()
    free0, _ = torch.cuda.mem_get_info()
    alloc0 = torch.cuda.memory_allocated()
    for _ in range(3):
        cuda_lib.prefill_host_static(*args, segment_tokens=256)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_allocated() == alloc0
    assert free1 == free0, f"device free memory moved by {free0 - free1} bytes"
    assert torch.equal(out, first)


def test_static_scratch_orders_calls_on_different_streams(cuda_lib):
    """Two calls on two streams share the scratch: the second runs after the first."""
    cfgs = [W.random_prefill_config([900], 4, 128, torch.bfloat16, init="normal"),
            W.random_prefill_config([400, 333], 4, 128, torch.bfloat16, init="zero")]
    hs = [_pinned(W.make_prefill_inputs(c, seed=43 + i)) for i, c in enumerate(cfgs)]
    refs = [cuda_lib.prefill_host(h["q"], h["k"], h["v"], h["g"], h["beta"], h["cu_seqlens"], h["init_state"],
                                  segment_tokens=64) for h in hs]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    res = [cuda_lib.prefill_host_static(h["q"], h["k"], h["v"], h["g"], h["beta"], h["cu_seqlens"],
                                        h["init_state"], segment_tokens=64, stream=s) for h, s in zip(hs, streams)]
    for s in streams:
        s.synchronize()
    for (o, f), (ro, rf) in zip(res, refs):
        assert torch.equal(o, ro) and torch.equal(f, rf)


def test_static_scratch_rejects_oversize(cuda_lib):
    """The bench-size problem in 1024-token rounds needs more than the scratch: rejected
    before anything is enqueued; in 128-token rounds it fits."""
    desc = cuda_lib.make_desc(1, 8192, 96, 128, 128, cuda_lib.KDA_BF16)
    assert cuda_lib.prefill_host_workspace_bytes(desc, 1024) > cuda_lib.KDA_STATIC_SCRATCH_BYTES
    assert cuda_lib.prefill_host_workspace_bytes(desc, 128) <= cuda_lib.KDA_STATIC_SCRATCH_BYTES
    t = lambda *s: torch.zeros(*s, dtype=torch.bfloat16).pin_memory()
    f = lambda *s: torch.zeros(*s, dtype=torch.float32).pin_memory()
    q = t(8192, 96, 128)
    with pytest.raises(cuda_lib.KDAError) as e:
        cuda_lib.prefill_host_static(q, q, q, f(8192, 96, 128), f(8192, 96), segment_tokens=1024)
    assert e.value.status == cuda_lib.KDA_ERR_WORKSPACE
