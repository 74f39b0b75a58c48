"""GPU parity of kda_prefill against the CPU oracle (through the C ABI)."""
import numpy as np
import pytest
import torch

import kda_workloads as W
from _parity import check, oracle_full, oracle_heads, sampled_units, to_device, tol_for

pytestmark = pytest.mark.gpu


def _run_small(kda, cfg, seed, **kw):
    d = W.make_prefill_inputs(cfg, seed=seed)
    ref_o, ref_s = oracle_full(d)
    g = to_device(d)
    out, fin = kda.prefill(g["q"], g["k"], g["v"], g["g"], g["beta"], g["cu_seqlens"], g["init_state"], **kw)
    torch.cuda.synchronize()
    assert kda.last_device_status() == kda.KDA_OK
    tol = tol_for(cfg.qkv_dtype)
    return check("out", out, ref_o, tol), check("final_state", fin, ref_s, tol)


def test_tiny_fp32_workload(cuda_lib):
    """H=2, T=256, dk=dv=64, fp32 inputs, zero initial state: bar 1e-4."""
    e_o, e_s = _run_small(cuda_lib, W.tiny_config(), seed=0)
    assert e_o <= 1e-4 and e_s <= 1e-4


@pytest.mark.parametrize("T", [1, 15, 16, 17, 63, 64, 65, 200])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["fp32", "bf16"])
def test_single_sequence_sweep(cuda_lib, T, d, dtype):
    cfg = W.random_prefill_config([T], 3, d, dtype, init="normal")
    _run_small(cuda_lib, cfg, seed=T * 7 + d)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["fp32", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
def test_varlen_with_empty_and_ragged_sequences(cuda_lib, dtype, d):
    rng = np.random.default_rng(d)
    lens = [int(x) for x in rng.integers(1, 301, size=5)]
    lens.insert(2, 0)          # an empty sequence in the middle
    lens.append(64)            # exactly one chunk
    cfg = W.random_prefill_config(lens, 2, d, dtype, init="normal")
    _run_small(cuda_lib, cfg, seed=11)


def test_zero_initial_state_and_no_final(cuda_lib):
    cfg = W.random_prefill_config([130, 7], 2, 128, torch.bfloat16, init="zero")
    d = W.make_prefill_inputs(cfg, seed=3)
    ref_o, _ = oracle_full(d)
    g = to_device(d)
    out, fin = cuda_lib.prefill(g["q"], g["k"], g["v"], g["g"], g["beta"], g["cu_seqlens"], None,
                                want_final=False)
    assert fin is None
    check("out", out, ref_o, 2e-2)


def test_equal_split_without_cu_seqlens(cuda_lib):
    cfg = W.random_prefill_config([96, 96, 96], 2, 64, torch.float32, init="normal")
    d = W.make_prefill_inputs(cfg, seed=4)
    ref_o, ref_s = oracle_full(d)
    g = to_device(d)
    out, fin = cuda_lib.prefill(g["q"], g["k"], g["v"], g["g"], g["beta"], None, g["init_state"], num_seqs=3)
    check("out", out, ref_o, 1e-4)
    check("final_state", fin, ref_s, 1e-4)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["fp32", "bf16"])
def test_in_place_chaining_equals_one_shot(cuda_lib, dtype):
    """init_state and final_state the same buffer; three chained calls vs the one-shot oracle."""
    cfg = W.random_prefill_config([300], 2, 128, dtype, init="normal")
    d = W.make_prefill_inputs(cfg, seed=5)
    ref_o, ref_s = oracle_full(d)
    g = to_device(d)
    state = g["init_state"].clone()
    outs = []
    for b, e in ((0, 100), (100, 101), (101, 300)):
        cu = torch.tensor([0, e - b], dtype=torch.int32, device="cuda")
        o, _ = cuda_lib.prefill(g["q"][b:e].contiguous(), g["k"][b:e].contiguous(), g["v"][b:e].contiguous(),
                                g["g"][b:e].contiguous(), g["beta"][b:e].contiguous(), cu, state,
                                final_state=state)
        outs.append(o)
    tol = tol_for(dtype)
    check("out", torch.cat(outs), ref_o, tol)
    check("final_state", state, ref_s, tol)


def test_bad_cu_seqlens_reported_on_device(cuda_lib):
    cfg = W.random_prefill_config([40, 40], 2, 64, torch.float32, init="zero")
    g = to_device(W.make_prefill_inputs(cfg, seed=6))
    bad = torch.tensor([0, 50, 40], dtype=torch.int32, device="cuda")   # decreasing
    cuda_lib.prefill(g["q"], g["k"], g["v"], g["g"], g["beta"], bad, None)
    assert cuda_lib.last_device_status() == cuda_lib.KDA_ERR_INVALID_ARG
    assert cuda_lib.last_device_status() == cuda_lib.KDA_OK          # cleared
    past_end = torch.tensor([0, 40, 99], dtype=torch.int32, device="cuda")
    cuda_lib.prefill(g["q"], g["k"], g["v"], g["g"], g["beta"], past_end, None)
    assert cuda_lib.last_device_status() == cuda_lib.KDA_ERR_INVALID_ARG


# ------------------------------------------------ full-size workloads, sampled outputs
def _sampled_check(kda, cfg, d, out, fin, units, tol):
    cu = cfg.cu_seqlens()
    by_seq = {}
    for n, h in units:
        by_seq.setdefault(n, []).append(h)
    for n, heads in by_seq.items():
        ref_o, ref_s = oracle_heads(d, n, heads, cu)
        b, e = int(cu[n]), int(cu[n + 1])
        check(f"out seq {n} heads {heads}", out[b:e][:, heads], ref_o, tol)
        if fin is not None:
            check(f"final seq {n} heads {heads}", fin[n][heads], ref_s, tol)


def test_prefill_workload_h96_t8192_sampled(cuda_lib):
    cfg = W.prefill_config()
    d = W.make_prefill_inputs(cfg, seed=0, device="cuda")
    out, fin = cuda_lib.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], d["init_state"])
    torch.cuda.synchronize()
    assert cuda_lib.last_device_status() == cuda_lib.KDA_OK
    assert torch.isfinite(out).all() and torch.isfinite(fin).all()
    units = sampled_units(1, 96, 6, seed=1, must=[(0, 0), (0, 95)])
    _sampled_check(cuda_lib, cfg, d, out, fin, units, 2e-2)


def test_prefill_workload_fp32_h96_t8192_sampled(cuda_lib):
    """The bench workload with fp32 q/k/v: the CUDA-core path, whose dv slices of a head share
    A, P and Wk as a thread-block cluster; sampled heads against the oracle at the 1e-4 bar."""
    base = W.prefill_config()
    cfg = W.PrefillConfig(base.name.replace("bf16", "fp32"), base.seqlens, base.num_heads, base.dk, base.dv,
                          torch.float32, base.init_state)
    d = W.make_prefill_inputs(cfg, seed=3, device="cuda")
    out, fin = cuda_lib.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], d["init_state"])
    torch.cuda.synchronize()
    assert cuda_lib.last_device_status() == cuda_lib.KDA_OK
    assert torch.isfinite(out).all() and torch.isfinite(fin).all()
    units = sampled_units(1, 96, 4, seed=3, must=[(0, 0), (0, 95)])
    _sampled_check(cuda_lib, cfg, d, out, fin, units, 1e-4)


def test_varlen_workload_32_seqs_sampled(cuda_lib):
    cfg = W.varlen_config(0)
    d = W.make_prefill_inputs(cfg, seed=0, device="cuda")
    out, fin = cuda_lib.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], None)
    torch.cuda.synchronize()
    assert cuda_lib.last_device_status() == cuda_lib.KDA_OK
    longest = int(np.argmax(cfg.seqlens))
    shortest = int(np.argmin(cfg.seqlens))
    units = sampled_units(cfg.num_seqs, 96, 6, seed=2, must=[(longest, 7), (shortest, 90), (31, 0)])
    _sampled_check(cuda_lib, cfg, d, out, fin, units, 2e-2)


def test_long_context_chained_calls_sampled(cuda_lib):
    """T=131072 as 16 chained 8192-token calls carrying final_state into init_state,
    against the one-shot oracle over all 131072 tokens."""
    cfg = W.long_config()
    d = W.make_prefill_inputs(cfg, seed=0, device="cuda")
    L = cfg.total_tokens // W.LONG_CALLS
    state = torch.zeros((1, 96, 128, 128), dtype=torch.float32, device="cuda")
    out = torch.empty((cfg.total_tokens, 96, 128), dtype=torch.float32, device="cuda")
    cu = torch.tensor([0, L], dtype=torch.int32, device="cuda")
    for i in range(W.LONG_CALLS):
        s = slice(i * L, (i + 1) * L)
        cuda_lib.prefill(d["q"][s], d["k"][s], d["v"][s], d["g"][s], d["beta"][s], cu, state,
                         out=out[s], final_state=state)
    torch.cuda.synchronize()
    assert cuda_lib.last_device_status() == cuda_lib.KDA_OK
    _sampled_check(cuda_lib, cfg, d, out, state, [(0, 3), (0, 50), (0, 95)], 2e-2)


@pytest.mark.parametrize("case", ["g_at_bound", "no_decay_beta_one", "beta_zero", "channel_extremes"])
@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.float32, 64)], ids=["bf16-128", "fp32-64"])
def test_decay_and_beta_extremes(cuda_lib, case, dtype, d):
    """The degenerate corners of the recurrence against the oracle: every g at the bound
    g_min = -5 (the largest in-tile factors, e^75 within a 16-token sub-tile), no decay with
    beta = 1 (pure overwrite), beta = 0 (the state only decays; decay scaled down so that it
    stays within fp32's range), and channels alternating between -5 and 0."""
    cfg = W.random_prefill_config([200, 77], 3, d, dtype, init="normal")
    inp = W.make_prefill_inputs(cfg, seed=51)
    g, beta = inp["g"], inp["beta"]
    if case == "g_at_bound":
        g = torch.full_like(g, -5.0)
    elif case == "no_decay_beta_one":
        g, beta = torch.zeros_like(g), torch.ones_like(beta)
    elif case == "beta_zero":
        # the state only decays: keep the total decay over 200 tokens (~e^-25) inside
        # fp32's range, or both sides would compare values the GPU cannot represent
        g, beta = 0.05 * g, torch.zeros_like(beta)
    else:
        g = torch.zeros_like(g)
        g[..., 0::2] = -5.0
    inp = dict(inp, g=g.contiguous(), beta=beta.contiguous())
    ref_o, ref_s = oracle_full(inp)
    dv = to_device(inp)
    out, fin = cuda_lib.prefill(dv["q"], dv["k"], dv["v"], dv["g"], dv["beta"], dv["cu_seqlens"], dv["init_state"])
    torch.cuda.synchronize()
    assert cuda_lib.last_device_status() == cuda_lib.KDA_OK
    tol = tol_for(dtype)
    check(f"{case} out", out, ref_o, tol)
    check(f"{case} final_state", fin, ref_s, tol)
