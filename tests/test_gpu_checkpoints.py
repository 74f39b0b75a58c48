"""GPU parity of state checkpoints and of resuming a prefill from one (through the C ABI)."""
import numpy as np
import pytest
import torch

import kda_workloads as W
import oracle
from _parity import check, to_device, tol_for

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.float32, 64)], ids=["bf16-128", "fp32-64"])
def test_checkpoints_equal_prefix_states(cuda_lib, dtype, d):
    lens = [300, 640, 100, 0, 1030]
    interval, slots = 128, 6
    cfg = W.random_prefill_config(lens, 2, d, dtype, init="normal")
    inp = W.make_prefill_inputs(cfg, seed=21)
    g = to_device(inp)
    out, fin, ck = cuda_lib.prefill(g["q"], g["k"], g["v"], g["g"], g["beta"], g["cu_seqlens"], g["init_state"],
                                    checkpoint_interval=interval, checkpoint_slots=slots)
    torch.cuda.synchronize()
    assert cuda_lib.last_device_status() == cuda_lib.KDA_OK
    ck = ck.cpu()
    cu = cfg.cu_seqlens()
    tol = tol_for(dtype)
    for n, L in enumerate(lens):
        b = int(cu[n])
        for j in range(slots):
            end = (j + 1) * interval
            if end > L:
                assert torch.count_nonzero(ck[n, :, j]) == 0, (n, j)   # never written
                continue
            sl = lambda x: x[b:b + end].contiguous()
            _, ref_s = oracle.recurrent(sl(inp["q"]), sl(inp["k"]), sl(inp["v"]), sl(inp["g"]), sl(inp["beta"]),
                                        np.array([0, end], dtype=np.int32), inp["init_state"][n:n + 1])
            check(f"checkpoint seq {n} slot {j}", ck[n, :, j], ref_s[0], tol)


def test_resume_from_checkpoint_matches_full_run(cuda_lib):
    """Prefill 1024 tokens with a snapshot every 512; resume the last 512 from the
    snapshot: outputs and final state equal the one-shot oracle."""
    cfg = W.random_prefill_config([1024], 3, 128, torch.bfloat16, init="normal")
    inp = W.make_prefill_inputs(cfg, seed=22)
    ref_o, ref_s = oracle.recurrent(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["cu_seqlens"],
                                    inp["init_state"])
    g = to_device(inp)
    _, _, ck = cuda_lib.prefill(g["q"][:512].contiguous(), g["k"][:512].contiguous(), g["v"][:512].contiguous(),
                                g["g"][:512].contiguous(), g["beta"][:512].contiguous(),
                                torch.tensor([0, 512], dtype=torch.int32, device="cuda"), g["init_state"],
                                checkpoint_interval=512, checkpoint_slots=1)
    s0 = ck[:, :, 0].contiguous()
    out, fin = cuda_lib.prefill(g["q"][512:].contiguous(), g["k"][512:].contiguous(), g["v"][512:].contiguous(),
                                g["g"][512:].contiguous(), g["beta"][512:].contiguous(),
                                torch.tensor([0, 512], dtype=torch.int32, device="cuda"), s0)
    torch.cuda.synchronize()
    check("resumed out", out, ref_o[512:], 2e-2)
    check("resumed final", fin, ref_s, 2e-2)


def test_multi_token_decode_through_prefill(cuda_lib):
    """k draft tokens per sequence in one call: the batch packed as B sequences of k tokens,
    the decode state passed as init_state and final_state (updated in place)."""
    B, H, D, K = 16, 4, 128, 5
    cfg = W.DecodeConfig("drafts", B, H, D, D, torch.bfloat16, K)
    inp = W.make_decode_inputs(cfg, seed=23)
    # sequence b = tokens (b, 0..K-1): [S, B, H, .] -> [B * K, H, .]
    pack = lambda x: x.transpose(0, 1).reshape(B * K, *x.shape[2:]).contiguous()
    q, k, v, g, beta = (pack(inp[n]) for n in ("q", "k", "v", "g", "beta"))
    cu = np.arange(0, B * K + 1, K, dtype=np.int32)
    ref_o, ref_s = oracle.recurrent(q, k, v, g, beta, cu, inp["state0"])
    state = inp["state0"].cuda()
    out, _ = cuda_lib.prefill(q.cuda(), k.cuda(), v.cuda(), g.cuda(), beta.cuda(),
                              torch.from_numpy(cu).cuda(), state, final_state=state)
    torch.cuda.synchronize()
    assert cuda_lib.last_device_status() == cuda_lib.KDA_OK
    check("draft outputs", out, ref_o, 2e-2)
    check("state after drafts", state, ref_s, 2e-2)


def test_draft_verify_then_accept_prefix(cuda_lib):
    """Speculative verification: K drafts per sequence run from the current state into a
    separate buffer (the current state is untouched, so rejecting is free); accepting
    a_b <= K drafts of sequence b is one more call over those tokens, a_b = 0 included."""
    B, H, D, K = 12, 4, 128, 4
    cfg = W.DecodeConfig("drafts", B, H, D, D, torch.bfloat16, K)
    inp = W.make_decode_inputs(cfg, seed=24)
    pack = lambda x: x.transpose(0, 1).reshape(B * K, *x.shape[2:]).contiguous()
    q, k, v, g, beta = (pack(inp[n]) for n in ("q", "k", "v", "g", "beta"))
    cu = np.arange(0, B * K + 1, K, dtype=np.int32)
    ref_o, _ = oracle.recurrent(q, k, v, g, beta, cu, inp["state0"])
    state = inp["state0"].cuda()
    scratch = torch.full_like(state, float("nan"))
    out, _ = cuda_lib.prefill(q.cuda(), k.cuda(), v.cuda(), g.cuda(), beta.cuda(),
                              torch.from_numpy(cu).cuda(), state, final_state=scratch)
    torch.cuda.synchronize()
    check("draft outputs", out, ref_o, 2e-2)
    assert torch.equal(state.cpu(), inp["state0"]), "the current state must not change while verifying"
    # accept a_b tokens of sequence b
    acc = [b % (K + 1) for b in range(B)]
    rows = np.concatenate([np.arange(b * K, b * K + a) for b, a in enumerate(acc)]).astype(np.int64)
    cu_a = np.concatenate([[0], np.cumsum(acc)]).astype(np.int32)
    sel = lambda x: x[torch.from_numpy(rows)].contiguous()
    qa, ka, va, ga, ba = (sel(x) for x in (q, k, v, g, beta))
    _, ref_s = oracle.recurrent(qa, ka, va, ga, ba, cu_a, inp["state0"])
    cuda_lib.prefill(qa.cuda(), ka.cuda(), va.cuda(), ga.cuda(), ba.cuda(), torch.from_numpy(cu_a).cuda(), state,
                     final_state=state)
    torch.cuda.synchronize()
    assert cuda_lib.last_device_status() == cuda_lib.KDA_OK
    check("state after accepted drafts", state, ref_s, 2e-2)
    for b, a in enumerate(acc):
        if a == 0:
            assert torch.equal(state[b].cpu(), inp["state0"][b]), b
