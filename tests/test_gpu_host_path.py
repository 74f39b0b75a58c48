"""GPU tests of kda_prefill_host (host buffers, pipelined copies): its results equal one
kda_prefill call on the same inputs bit for bit (same chunk boundaries), and the oracle
within the bar."""
import numpy as np
import pytest
import torch

import kda_workloads as W
from _parity import check, oracle_full, to_device, tol_for

pytestmark = pytest.mark.gpu


def _pinned(d):
    return {k: (None if v is None else v.contiguous().pin_memory()) for k, v in d.items()}


@pytest.mark.parametrize("seg", [64, 192, 4096])
@pytest.mark.parametrize("dtype,dim", [(torch.bfloat16, 128), (torch.float32, 64)], ids=["bf16-128", "fp32-64"])
def test_host_path_equals_device_path(cuda_lib, dtype, dim, seg):
    lens = [300, 0, 641, 64, 1000]
    cfg = W.random_prefill_config(lens, 3, dim, dtype, init="normal")
    inp = W.make_prefill_inputs(cfg, seed=31)
    g = to_device(inp)
    ref_out, ref_fin = cuda_lib.prefill(g["q"], g["k"], g["v"], g["g"], g["beta"], g["cu_seqlens"], g["init_state"])
    h = _pinned(inp)
    out, fin = cuda_lib.prefill_host(h["q"], h["k"], h["v"], h["g"], h["beta"], h["cu_seqlens"], h["init_state"],
                                     segment_tokens=seg)
    torch.cuda.synchronize()
    assert cuda_lib.last_device_status() == cuda_lib.KDA_OK
    assert torch.equal(out, ref_out.cpu()), "host-path output differs from one kda_prefill call"
    assert torch.equal(fin, ref_fin.cpu()), "host-path final state differs from one kda_prefill call"
    if seg == 192:
        o, s = oracle_full(inp)
        check("host-path out vs oracle", out, o, tol_for(dtype))
        check("host-path final vs oracle", fin, s, tol_for(dtype))


def test_host_path_in_place_state_and_zero_init(cuda_lib):
    """final_state may be the host init_state buffer; no init_state means zero."""
    cfg = W.random_prefill_config([500, 260], 2, 128, torch.bfloat16, init="normal")
    inp = W.make_prefill_inputs(cfg, seed=32)
    g = to_device(inp)
    ref_out, ref_fin = cuda_lib.prefill(g["q"], g["k"], g["v"], g["g"], g["beta"], g["cu_seqlens"], g["init_state"])
    h = _pinned(inp)
    state = h["init_state"].clone().pin_memory()
    out, fin = cuda_lib.prefill_host(h["q"], h["k"], h["v"], h["g"], h["beta"], h["cu_seqlens"], state,
                                     final_state=state, segment_tokens=128)
    torch.cuda.synchronize()
    assert fin.data_ptr() == state.data_ptr()
    assert torch.equal(out, ref_out.cpu()) and torch.equal(state, ref_fin.cpu())
    z_out, z_fin = cuda_lib.prefill(g["q"], g["k"], g["v"], g["g"], g["beta"], g["cu_seqlens"], None)
    out0, fin0 = cuda_lib.prefill_host(h["q"], h["k"], h["v"], h["g"], h["beta"], h["cu_seqlens"], None,
                                       segment_tokens=256)
    torch.cuda.synchronize()
    assert torch.equal(out0, z_out.cpu()) and torch.equal(fin0, z_fin.cpu())


def test_host_path_no_tokens_passes_state_through(cuda_lib):
    H, D = 2, 64
    init = torch.randn(3, H, D, D, generator=torch.Generator().manual_seed(5)).pin_memory()
    empty = lambda *s: torch.empty(*s, dtype=torch.float32).pin_memory()
    cu = torch.zeros(4, dtype=torch.int32).pin_memory()
    out, fin = cuda_lib.prefill_host(empty(0, H, D), empty(0, H, D), empty(0, H, D), empty(0, H, D), empty(0, H),
                                     cu, init, segment_tokens=64)
    torch.cuda.synchronize()
    assert torch.equal(fin, init)


def test_host_path_full_size_matches_device(cuda_lib):
    """The bench workload (B=1, H=96, T=8192, bf16) through the host path with the bench's
    segment size: bit-identical to the device call."""
    cfg = W.prefill_config()
    inp = W.make_prefill_inputs(cfg, seed=0, device="cuda")
    ref_out, ref_fin = cuda_lib.prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["cu_seqlens"],
                                        inp["init_state"])
    h = {k: (None if v is None else v.cpu().pin_memory()) for k, v in inp.items()}
    out, fin = cuda_lib.prefill_host(h["q"], h["k"], h["v"], h["g"], h["beta"], h["cu_seqlens"], h["init_state"],
                                     segment_tokens=1024)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out.cpu()) and torch.equal(fin, ref_fin.cpu())
