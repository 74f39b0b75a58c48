"""GPU parity of the output gate (kda_prefill_gated, kda_decode_gated, kda_decode_multi_gated)
against the CPU oracle, through the C ABI.

The gate is read as out = o * sigmoid(z) elementwise over the read-out channels, with the
logits z supplied by the caller (llm-atlas "K3_RESEARCH.md", Q08: an input-dependent,
full-rank output gate; its formula is not given).  The oracle applies it in fp64 to its own
recurrence output.  Every path is checked against that; the gate must leave the state (and,
for z = 0, everything but a factor of one half) exactly as the ungated call has it."""
import numpy as np
import pytest
import torch

import kda_workloads as W
import oracle
from _parity import check, oracle_full, to_device, tol_for

pytestmark = pytest.mark.gpu


def _prefill_cfg(path):
    if path == "split":         # bf16, dk = dv = 128, few units: the chunk-parallel path
        return W.random_prefill_config([300, 0, 641, 129], 3, 128, torch.bfloat16, init="normal")
    if path == "one_cta":       # 152 units: one CTA per (sequence, head)
        return W.random_prefill_config([70, 131], 76, 128, torch.bfloat16, init="normal")
    if path == "simt_fp32":
        return W.random_prefill_config([130, 67], 2, 64, torch.float32, init="normal")
    return W.random_prefill_config([130, 67], 2, 64, torch.bfloat16, init="normal")   # simt_bf16


@pytest.mark.parametrize("path", ["split", "one_cta", "simt_fp32", "simt_bf16"])
def test_prefill_gated_matches_oracle(cuda_lib, path):
    cfg = _prefill_cfg(path)
    plan = cuda_lib.prefill_query(cuda_lib.make_desc(cfg.num_seqs, cfg.total_tokens, cfg.num_heads, cfg.dk,
                                                     cfg.dv, cuda_lib.KDA_BF16 if cfg.qkv_dtype == torch.bfloat16
                                                     else cuda_lib.KDA_F32))
    expect = {"split": (1, True), "one_cta": (1, False), "simt_fp32": (0, False), "simt_bf16": (0, False)}[path]
    assert plan["tensor_cores"] == expect[0] and (plan["kernel_launches"] >= 2) == expect[1]
    d = W.make_prefill_inputs(cfg, seed=71)
    z = W.make_gate_logits((cfg.total_tokens, cfg.num_heads, cfg.dv), seed=71)
    ref_o, ref_s = oracle_full(d)
    g = to_device(d)
    zc = z.cuda()
    out, fin = cuda_lib.prefill(g["q"], g["k"], g["v"], g["g"], g["beta"], g["cu_seqlens"], g["init_state"], gate=zc)
    out0, fin0 = cuda_lib.prefill(g["q"], g["k"], g["v"], g["g"], g["beta"], g["cu_seqlens"], g["init_state"])
    half, _ = cuda_lib.prefill(g["q"], g["k"], g["v"], g["g"], g["beta"], g["cu_seqlens"], g["init_state"],
                               gate=torch.zeros_like(zc))
    torch.cuda.synchronize()
    assert cuda_lib.last_device_status() == cuda_lib.KDA_OK
    tol = tol_for(cfg.qkv_dtype)
    check(f"{path} gated out", out, oracle.output_gate(ref_o, z), tol)
    check(f"{path} final state", fin, ref_s, tol)
    assert torch.equal(fin, fin0)                 # the gate never touches the state
    assert torch.equal(half, 0.5 * out0)          # sigmoid(0) = 1/2 exactly


def test_prefill_gated_large_logits(cuda_lib):
    """z = +-30: the gate passes the output through or closes it, without overflow."""
    cfg = _prefill_cfg("split")
    d = to_device(W.make_prefill_inputs(cfg, seed=72))
    out0, _ = cuda_lib.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], d["init_state"])
    z = torch.full_like(out0, 30.0)
    z[:, :, 1::2] = -30.0
    out, _ = cuda_lib.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], d["init_state"], gate=z)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    ref = oracle.output_gate(out0.cpu().double().numpy(), z.cpu().double().numpy())
    assert np.max(np.abs(out.cpu().double().numpy() - ref)) <= 1e-6 * float(out0.abs().max())


def test_prefill_gated_rejects_overlap(cuda_lib):
    cfg = _prefill_cfg("split")
    d = to_device(W.make_prefill_inputs(cfg, seed=73))
    out = torch.empty((cfg.total_tokens, cfg.num_heads, cfg.dv), device="cuda")
    with pytest.raises(cuda_lib.KDAError):
        cuda_lib.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], d["init_state"], out=out,
                         gate=out)


@pytest.mark.parametrize("dtype,D", [(torch.bfloat16, 128), (torch.float32, 64)], ids=["bf16-128", "fp32-64"])
def test_decode_gated_matches_oracle(cuda_lib, dtype, D):
    B, H, S = 5, 3, 4
    cfg = W.DecodeConfig("gate", B, H, D, D, dtype, S)
    inp = W.make_decode_inputs(cfg, seed=74)
    z = W.make_gate_logits((S, B, H, D), seed=74)
    g = {k: v.cuda() for k, v in inp.items()}
    state, state0 = g["state0"].clone(), g["state0"].clone()
    outs, outs0 = [], []
    for s in range(S):
        outs.append(cuda_lib.decode(g["q"][s], g["k"][s], g["v"][s], g["g"][s], g["beta"][s], state,
                                    gate=z[s].cuda()))
        outs0.append(cuda_lib.decode(g["q"][s], g["k"][s], g["v"][s], g["g"][s], g["beta"][s], state0))
    torch.cuda.synchronize()
    assert torch.equal(state, state0)
    # the oracle over B*H one-unit sequences of S tokens (unit-major rows)
    units = [(b, h) for b in range(B) for h in range(H)]
    sel = lambda x: torch.stack([x[:, b, h] for b, h in units], 0)          # [U, S, ...]
    flat = lambda x: x.reshape(len(units) * S, 1, -1).contiguous()
    cu = np.arange(0, len(units) * S + 1, S, dtype=np.int32)
    s0 = torch.stack([inp["state0"][b, h] for b, h in units])[:, None].contiguous()
    ref_o, ref_s = oracle.recurrent(flat(sel(inp["q"])), flat(sel(inp["k"])), flat(sel(inp["v"])),
                                    flat(sel(inp["g"])), sel(inp["beta"]).reshape(-1, 1).contiguous(), cu, s0)
    got = sel(torch.stack(outs, 0).cpu()).reshape(-1, D)
    tol = tol_for(dtype)
    check("decode gated out", got, oracle.output_gate(ref_o.reshape(-1, D), sel(z).reshape(-1, D).numpy()), tol)


@pytest.mark.parametrize("K", [3, 12], ids=["persistent", "per_unit"])
def test_decode_multi_gated_matches_oracle(cuda_lib, K):
    B, H, D = 6, 3, 128
    inp = W.make_decode_inputs(W.DecodeConfig("gate_multi", B, H, D, D, torch.bfloat16, K), seed=75)
    x = {n: inp[n].transpose(0, 1).contiguous() for n in ("q", "k", "v", "g", "beta")}   # [B, K, ...]
    z = W.make_gate_logits((B, K, H, D), seed=75)
    pick = lambda t: t.reshape(B * K, *t.shape[2:]).contiguous()
    cu = np.arange(0, B * K + 1, K, dtype=np.int32)
    ref_o, ref_s = oracle.recurrent(pick(x["q"]), pick(x["k"]), pick(x["v"]), pick(x["g"]), pick(x["beta"]), cu,
                                    inp["state0"])
    state, state0 = inp["state0"].cuda(), inp["state0"].cuda()
    xc = [x[n].cuda() for n in ("q", "k", "v", "g", "beta")]
    out = cuda_lib.decode_multi(*xc, state, gate=z.cuda())
    out0 = cuda_lib.decode_multi(*xc, state0)
    torch.cuda.synchronize()
    assert cuda_lib.last_device_status() == cuda_lib.KDA_OK
    assert torch.equal(state, state0)
    check("multi-token gated out", out.reshape(B * K, H, D), oracle.output_gate(ref_o, z.reshape(B * K, H, D).numpy()),
          2e-2)
    check("multi-token state", state, ref_s, 2e-2)
