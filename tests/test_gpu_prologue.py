"""GPU tests of the input prologue (the KDA_PROLOGUE_* bits): raw q, k, g and beta go in,
and the workloads' recipe -- q and k L2-normalised per (token, head), g = -5 sigmoid(z),
beta = sigmoid(y) -- runs inside the kernels' loads.  Every path is compared with the oracle
run on the oracle's own prologue of the same raw inputs, the two tensor-core prefill forms
with each other bit for bit, and every bit on its own as well as all three together."""
import numpy as np
import pytest
import torch

import kda_workloads as W
import oracle
from _parity import check, oracle_full, to_device, tol_for

pytestmark = pytest.mark.gpu

ALL = 7


def _mixed(raw, cooked, pro):
    """Inputs for prologue bits `pro`: raw where a bit is set, the recipe's values elsewhere."""
    d = dict(cooked)
    if pro & 1:
        d["q"], d["k"] = raw["q"], raw["k"]
    if pro & 2:
        d["g"] = raw["g"]
    if pro & 4:
        d["beta"] = raw["beta"]
    return d


def _prefill(kda, d, pro):
    g = to_device(d)
    out, fin = kda.prefill(g["q"], g["k"], g["v"], g["g"], g["beta"], g["cu_seqlens"], g["init_state"], prologue=pro)
    torch.cuda.synchronize()
    assert kda.last_device_status() == kda.KDA_OK
    return out.cpu(), fin.cpu()


@pytest.mark.parametrize("pro", [ALL, 1, 2, 4], ids=["all", "qk", "g", "beta"])
@pytest.mark.parametrize("dtype,d,lens,H", [
    (torch.bfloat16, 128, [300, 0, 641, 129], 3),   # tensor cores, chunk-parallel
    (torch.float32, 64, [256], 2),                   # the tiny workload's shape: CUDA cores, fp32
    (torch.bfloat16, 64, [200, 65], 2),              # CUDA cores, bf16
    (torch.float32, 128, [130, 64], 2),              # CUDA cores, fp32, dk = 128
], ids=["tc-bf16-128", "simt-fp32-64", "simt-bf16-64", "simt-fp32-128"])
def test_prefill_prologue_matches_oracle(cuda_lib, dtype, d, lens, H, pro):
    cfg = W.random_prefill_config(lens, H, d, dtype, init="normal")
    seed = sum(lens) + d + pro
    src = _mixed(W.make_prefill_inputs(cfg, seed=seed, raw=True), W.make_prefill_inputs(cfg, seed=seed), pro)
    out, fin = _prefill(cuda_lib, src, pro)
    ref_o, ref_s = oracle_full(oracle.prologue(src, pro))
    tol = tol_for(dtype)
    check("prologue out", out, ref_o, tol)
    check("prologue final state", fin, ref_s, tol)


def test_prologue_on_both_tensor_core_forms_bitwise(cuda_lib):
    """kda_prefill (chunk-parallel here) and kda_prefill_host (one CTA per unit, in rounds)
    apply the same prologue code to the same raw inputs: identical bits."""
    H = 4
    cfg = W.random_prefill_config([300, 0, 641, 129], H, 128, torch.bfloat16, init="normal")
    raw = W.make_prefill_inputs(cfg, seed=71, raw=True)
    desc = cuda_lib.make_desc(4, cfg.total_tokens, H, 128, 128, cuda_lib.KDA_BF16, ALL)
    assert cuda_lib.prefill_query(desc)["kernel_launches"] >= 2
    o_split, s_split = _prefill(cuda_lib, raw, ALL)
    host = {n: (None if t is None else t.contiguous().pin_memory()) for n, t in raw.items()}
    o_host, s_host = cuda_lib.prefill_host(host["q"], host["k"], host["v"], host["g"], host["beta"],
                                           host["cu_seqlens"], host["init_state"], prologue=ALL)
    torch.cuda.synchronize()
    assert cuda_lib.last_device_status() == cuda_lib.KDA_OK
    assert torch.equal(o_split, o_host) and torch.equal(s_split, s_host)


def test_prologue_without_bits_is_the_plain_call(cuda_lib):
    """prologue = 0 is the plain call, bit for bit.  (The raw inputs with all bits set are not
    compared with the recipe's inputs here: the recipe rounds q and k to bf16 after
    normalising in fp64, the prologue normalises the bf16 draws, so the two are different
    inputs one bf16 step apart, which the recurrence amplifies.)"""
    cfg = W.random_prefill_config([257, 64], 3, 128, torch.bfloat16, init="normal")
    cooked = W.make_prefill_inputs(cfg, seed=72)
    o0, s0 = _prefill(cuda_lib, cooked, 0)
    g = to_device(cooked)
    o1, s1 = cuda_lib.prefill(g["q"], g["k"], g["v"], g["g"], g["beta"], g["cu_seqlens"], g["init_state"])
    torch.cuda.synchronize()
    assert torch.equal(o0, o1.cpu()) and torch.equal(s0, s1.cpu())


@pytest.mark.parametrize("dtype,D", [(torch.bfloat16, 128), (torch.float32, 64), (torch.float32, 128),
                                     (torch.bfloat16, 64)], ids=["bf16-128", "fp32-64", "fp32-128", "bf16-64"])
def test_decode_prologue_matches_oracle(cuda_lib, dtype, D):
    B, H = 6, 3
    cfg = W.DecodeConfig("pro", B, H, D, D, dtype, 1)
    raw = W.make_decode_inputs(cfg, seed=73, raw=True)
    x = {n: raw[n][0] for n in ("q", "k", "v", "g", "beta")}
    state = raw["state0"].cuda()
    out = cuda_lib.decode(*(x[n].cuda() for n in ("q", "k", "v", "g", "beta")), state, prologue=ALL)
    torch.cuda.synchronize()
    p = oracle.prologue(x, ALL)
    cu = np.arange(B + 1, dtype=np.int32)
    ref_o, ref_s = oracle.recurrent(p["q"], p["k"], p["v"], p["g"], p["beta"], cu, raw["state0"])
    tol = tol_for(dtype)
    check("decode prologue out", out, ref_o, tol)
    check("decode prologue state", state, ref_s, tol)


@pytest.mark.parametrize("K", [3, 12], ids=["persistent", "per-unit"])
@pytest.mark.parametrize("dtype,D", [(torch.bfloat16, 128), (torch.float32, 64)], ids=["bf16-128", "fp32-64"])
def test_decode_multi_prologue_matches_oracle(cuda_lib, K, dtype, D):
    B, H = 5, 2
    raw = W.make_decode_inputs(W.DecodeConfig("pro", B, H, D, D, dtype, K), seed=74 + K, raw=True)
    bk = lambda t: t.transpose(0, 1).contiguous()                      # [K, B, ...] -> [B, K, ...]
    x = {n: bk(raw[n]) for n in ("q", "k", "v", "g", "beta")}
    state = raw["state0"].cuda()
    out = cuda_lib.decode_multi(*(x[n].cuda() for n in ("q", "k", "v", "g", "beta")), state, prologue=ALL)
    torch.cuda.synchronize()
    assert cuda_lib.last_device_status() == cuda_lib.KDA_OK
    flat = {n: t.reshape(B * K, *t.shape[2:]).contiguous() for n, t in x.items()}
    p = oracle.prologue(flat, ALL)
    cu = (np.arange(B + 1) * K).astype(np.int32)
    ref_o, ref_s = oracle.recurrent(p["q"], p["k"], p["v"], p["g"], p["beta"], cu, raw["state0"])
    tol = tol_for(dtype)
    check("multi-token prologue out", out.reshape(B * K, H, D), ref_o, tol)
    check("multi-token prologue state", state, ref_s, tol)
