"""GPU parity of kda_decode_multi (K tokens per sequence in one pass over the state) against
the oracle, and its apply-count semantics for verifying draft tokens.  Up to 8 tokens the
library runs its persistent kernel (resident CTAs walking the (sequence, head) units, the next
unit's state prefetched into shared memory); longer drafts run one CTA per unit."""
import numpy as np
import pytest
import torch

import kda_workloads as W
import oracle
from _parity import check, tol_for

pytestmark = pytest.mark.gpu


def _inputs(B, H, D, dtype, K, seed):
    inp = W.make_decode_inputs(W.DecodeConfig("multi", B, H, D, D, dtype, K), seed=seed)
    bk = lambda x: x.transpose(0, 1).contiguous()          # [K, B, ...] -> [B, K, ...]
    return {n: bk(inp[n]) for n in ("q", "k", "v", "g", "beta")}, inp["state0"]


def _oracle(x, state0, lens):
    """Oracle over sequence b's first lens[b] tokens (packed [sum(lens), H, .])."""
    B = x["q"].shape[0]
    pick = lambda t: torch.cat([t[b, :lens[b]] for b in range(B)]).contiguous()
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    return oracle.recurrent(pick(x["q"]), pick(x["k"]), pick(x["v"]), pick(x["g"]), pick(x["beta"]), cu, state0)


@pytest.mark.parametrize("K", [1, 3, 8, 12])
@pytest.mark.parametrize("dtype,D", [(torch.bfloat16, 128), (torch.float32, 64), (torch.float32, 128)],
                         ids=["bf16-128", "fp32-64", "fp32-128"])
def test_decode_multi_matches_oracle(cuda_lib, K, dtype, D):
    B, H = 8, 3
    x, s0 = _inputs(B, H, D, dtype, K, seed=60 + K)
    ref_o, ref_s = _oracle(x, s0, [K] * B)
    state = s0.cuda()
    out = cuda_lib.decode_multi(*(x[n].cuda() for n in ("q", "k", "v", "g", "beta")), state)
    torch.cuda.synchronize()
    assert cuda_lib.last_device_status() == cuda_lib.KDA_OK
    tol = tol_for(dtype)
    check("multi-token out", out.reshape(B * K, H, D), ref_o, tol)
    check("multi-token state", state, ref_s, tol)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "fp32"])
def test_decode_multi_apply_counts(cuda_lib, dtype):
    """Outputs for all K tokens; the state advanced by n_apply[b] tokens (0 = untouched)."""
    B, H, D, K = 10, 2, 128, 4
    x, s0 = _inputs(B, H, D, dtype, K, seed=70)
    n_apply = [b % (K + 1) for b in range(B)]
    ref_o, _ = _oracle(x, s0, [K] * B)
    _, ref_s = _oracle(x, s0, n_apply)
    state = s0.cuda()
    out = cuda_lib.decode_multi(*(x[n].cuda() for n in ("q", "k", "v", "g", "beta")), state,
                                n_apply=torch.tensor(n_apply, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert cuda_lib.last_device_status() == cuda_lib.KDA_OK
    tol = tol_for(dtype)
    check("outputs of all drafts", out.reshape(B * K, H, D), ref_o, tol)
    check("state after the applied prefix", state, ref_s, tol)
    for b in range(B):
        if n_apply[b] == 0:
            assert torch.equal(state[b].cpu(), s0[b])


def test_decode_multi_verify_then_apply(cuda_lib):
    """The verification pattern: a read-only pass (n_apply = 0) for the outputs of K drafts,
    then an apply pass with the accepted counts and no outputs."""
    B, H, D, K = 6, 4, 128, 5
    x, s0 = _inputs(B, H, D, torch.bfloat16, K, seed=71)
    dev = {n: x[n].cuda() for n in x}
    state = s0.cuda()
    out = cuda_lib.decode_multi(*(dev[n] for n in ("q", "k", "v", "g", "beta")), state,
                                n_apply=torch.zeros(B, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(state.cpu(), s0)
    accepted = [3, 0, 5, 1, 2, 4]
    res = cuda_lib.decode_multi(*(dev[n] for n in ("q", "k", "v", "g", "beta")), state,
                                n_apply=torch.tensor(accepted, dtype=torch.int32, device="cuda"), want_out=False)
    torch.cuda.synchronize()
    assert res is None and cuda_lib.last_device_status() == cuda_lib.KDA_OK
    ref_o, _ = _oracle(x, s0, [K] * B)
    _, ref_s = _oracle(x, s0, accepted)
    check("verify outputs", out.reshape(B * K, H, D), ref_o, 2e-2)
    check("state after accepting", state, ref_s, 2e-2)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "fp32"])
@pytest.mark.parametrize("D", [64, 128])
def test_decode_multi_single_token_equals_decode(cuda_lib, dtype, D):
    """K = 1 is the single-token decode step up to fp32 summation order (the two kernels
    split the dk sums differently: per-lane rows then shuffles here, row groups there)."""
    B, H = 16, 4
    x, s0 = _inputs(B, H, D, dtype, 1, seed=72)
    dev = {n: x[n].cuda() for n in x}
    s_multi, s_one = s0.cuda(), s0.cuda()
    o_multi = cuda_lib.decode_multi(*(dev[n] for n in ("q", "k", "v", "g", "beta")), s_multi)
    o_one = cuda_lib.decode(*(dev[n][:, 0].contiguous() for n in ("q", "k", "v", "g", "beta")), s_one)
    torch.cuda.synchronize()
    rel = lambda x, y: ((x - y).abs().max() / y.pow(2).mean().sqrt()).item()
    assert rel(o_multi[:, 0], o_one) < 2e-6 and rel(s_multi, s_one) < 2e-6


def test_decode_multi_bad_count_leaves_state(cuda_lib):
    B, H, D, K = 3, 2, 64, 2
    x, s0 = _inputs(B, H, D, torch.float32, K, seed=73)
    state = s0.cuda()
    cuda_lib.decode_multi(*(x[n].cuda() for n in ("q", "k", "v", "g", "beta")), state,
                          n_apply=torch.tensor([1, K + 1, -1], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert cuda_lib.last_device_status() == cuda_lib.KDA_ERR_INVALID_ARG
    assert torch.equal(state[1].cpu(), s0[1]) and torch.equal(state[2].cpu(), s0[2])
    _, ref_s = _oracle(x, s0, [1, 0, 0])
    check("valid sequence advanced", state[:1], ref_s[:1], 1e-4)


def test_decode_multi_serving_size(cuda_lib):
    """B = 256 sequences, H = 96, K = 4 drafts, bf16: sampled (sequence, head) units."""
    B, H, D, K = 256, 96, 128, 4
    cfg = W.DecodeConfig("drafts", B, H, D, D, torch.bfloat16, K)
    inp = W.make_decode_inputs(cfg, seed=74, device="cuda")
    x = {n: inp[n].transpose(0, 1).contiguous() for n in ("q", "k", "v", "g", "beta")}
    s0 = inp["state0"].clone()
    state = inp["state0"]
    out = cuda_lib.decode_multi(x["q"], x["k"], x["v"], x["g"], x["beta"], state)
    torch.cuda.synchronize()
    rng = np.random.default_rng(74)
    for b in rng.choice(B, size=4, replace=False).tolist():
        hs = rng.choice(H, size=3, replace=False).tolist()
        sub = {n: x[n][b, :, hs].cpu().contiguous() for n in x}
        ro, rs = oracle.recurrent(sub["q"], sub["k"], sub["v"], sub["g"], sub["beta"],
                                  np.array([0, K], dtype=np.int32), s0[b:b + 1, hs].cpu().contiguous())
        check(f"seq {b} out", out[b][:, hs].cpu(), ro, 2e-2)
        check(f"seq {b} state", state[b, hs].cpu(), rs[0], 2e-2)


@pytest.mark.parametrize("dtype,D", [(torch.bfloat16, 128), (torch.float32, 64)], ids=["bf16-128", "fp32-64"])
def test_decode_multi_units_beyond_resident_ctas(cuda_lib, dtype, D):
    """More (sequence, head) units than resident CTAs, not a multiple of them: every CTA walks
    several units, so every unit after the first comes from the prefetched copy; all checked."""
    B, H, K = 97, 7, 4                       # 679 units
    x, s0 = _inputs(B, H, D, dtype, K, seed=75)
    n_apply = [(3 * b) % (K + 1) for b in range(B)]
    ref_o, _ = _oracle(x, s0, [K] * B)
    _, ref_s = _oracle(x, s0, n_apply)
    state = s0.cuda()
    out = cuda_lib.decode_multi(*(x[n].cuda() for n in ("q", "k", "v", "g", "beta")), state,
                                n_apply=torch.tensor(n_apply, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert cuda_lib.last_device_status() == cuda_lib.KDA_OK
    tol = tol_for(dtype)
    check("outputs", out.reshape(B * K, H, D), ref_o, tol)
    check("state", state, ref_s, tol)
    for b in range(B):
        if n_apply[b] == 0:
            assert torch.equal(state[b].cpu(), s0[b])


def test_decode_multi_persistent_equals_per_unit_arithmetic(cuda_lib):
    """The two kernels run the same per-token arithmetic: the first 8 tokens of a 9-token call
    (per-unit kernel) and an 8-token call (persistent kernel) give bit-identical outputs."""
    B, H, D = 40, 12, 128
    x, s0 = _inputs(B, H, D, torch.bfloat16, 9, seed=76)
    dev = {n: x[n].cuda() for n in x}
    s9, s8 = s0.cuda(), s0.cuda()
    o9 = cuda_lib.decode_multi(*(dev[n] for n in ("q", "k", "v", "g", "beta")), s9,
                               n_apply=torch.full((B,), 8, dtype=torch.int32, device="cuda"))
    o8 = cuda_lib.decode_multi(*(dev[n][:, :8].contiguous() for n in ("q", "k", "v", "g", "beta")), s8)
    torch.cuda.synchronize()
    assert torch.equal(o9[:, :8], o8) and torch.equal(s9, s8)
