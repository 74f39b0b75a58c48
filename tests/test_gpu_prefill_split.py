"""GPU tests of the chunk-parallel prefill path: per-chunk operands for every (sequence, head,
chunk) at once, then the state scan (one cooperative launch when at least 32 CTAs are left
over to produce, else separate prep and scan launches).  kda_prefill picks it for bf16, dk = dv = 128 calls by a
cost estimate from the shape (few units, or a partial second wave of one CTA per unit).  The two
issue the same tensor-core instructions on the same operands, so their results are compared
bit for bit, and each is compared with the oracle."""
import numpy as np
import pytest
import torch

import kda_workloads as W
from _parity import check, oracle_full, oracle_heads, to_device, tol_for

pytestmark = pytest.mark.gpu


def _plan(kda, N, T, H):
    return kda.prefill_query(kda.make_desc(N, T, H, 128, 128, kda.KDA_BF16))


def _run(kda, d):
    g = to_device(d)
    out, fin = kda.prefill(g["q"], g["k"], g["v"], g["g"], g["beta"], g["cu_seqlens"], g["init_state"])
    torch.cuda.synchronize()
    assert kda.last_device_status() == kda.KDA_OK
    return out.cpu(), fin.cpu()


def _padded(d, extra_lens, seed):
    """d with extra sequences appended (their own random inputs): same leading tokens and states."""
    H = d["q"].shape[1]
    cfg = W.random_prefill_config(extra_lens, H, 128, torch.bfloat16, init="normal")
    e = W.make_prefill_inputs(cfg, seed=seed)
    cat = lambda n: torch.cat([d[n], e[n]])
    cu = torch.cat([d["cu_seqlens"], e["cu_seqlens"][1:] + d["cu_seqlens"][-1]])
    return {"q": cat("q"), "k": cat("k"), "v": cat("v"), "g": cat("g"), "beta": cat("beta"),
            "cu_seqlens": cu, "init_state": cat("init_state")}


def test_plan_selects_the_path(cuda_lib):
    split = _plan(cuda_lib, 1, 8192, 96)
    assert split["kernel_launches"] == 2 and split["tensor_cores"] == 1   # offsets + prep-and-scan
    assert split["workspace_bytes"] >= (8192 // 64) * 96 * 115200
    one = _plan(cuda_lib, 2, 8192, 76)          # 152 units: one full wave of one CTA per unit
    assert one["kernel_launches"] == 1 and one["workspace_bytes"] == 0
    assert _plan(cuda_lib, 1, 8192, 112)["kernel_launches"] >= 2
    assert _plan(cuda_lib, 1, 8192, 124)["kernel_launches"] == 3
    assert _plan(cuda_lib, 1, 8192, 128)["kernel_launches"] == 3
    assert _plan(cuda_lib, 1, 8192, 136)["kernel_launches"] == 3
    assert _plan(cuda_lib, 1, 8192, 144)["kernel_launches"] == 1
    assert _plan(cuda_lib, 2, 8192, 96)["kernel_launches"] >= 2   # 192 units: a second wave of 40
    long = _plan(cuda_lib, 1, 64 * 400, 96)     # 38,496 items: over the workspace cap
    assert long["kernel_launches"] == 1 and long["workspace_bytes"] == 0


@pytest.mark.parametrize("lens", [[300, 0, 641, 129], [64], [1], [0, 0, 100, 0, 64, 1], [17, 64, 65, 128, 191]],
                         ids=["ragged", "one-chunk", "one-token", "empties", "boundaries"])
def test_split_matches_oracle(cuda_lib, lens):
    cfg = W.random_prefill_config(lens, 3, 128, torch.bfloat16, init="normal")
    assert _plan(cuda_lib, len(lens), cfg.total_tokens, 3)["kernel_launches"] >= 2
    d = W.make_prefill_inputs(cfg, seed=sum(lens) + 5)
    out, fin = _run(cuda_lib, d)
    ref_o, ref_s = oracle_full(d)
    check("split out", out, ref_o, tol_for(torch.bfloat16))
    check("split final state", fin, ref_s, tol_for(torch.bfloat16))


def test_split_and_one_cta_per_head_agree_bitwise(cuda_lib):
    H = 4
    lens = [300, 0, 641, 129]
    cfg = W.random_prefill_config(lens, H, 128, torch.bfloat16, init="normal")
    d = W.make_prefill_inputs(cfg, seed=90)
    extra = [64 + 3 * i for i in range(30)]                       # 34 x 4 = 136 short units
    p = _padded(d, extra, seed=91)
    T0 = cfg.total_tokens
    assert _plan(cuda_lib, len(lens), T0, H)["kernel_launches"] >= 2
    assert _plan(cuda_lib, len(lens) + len(extra), p["q"].shape[0], H)["kernel_launches"] == 1
    o_split, s_split = _run(cuda_lib, d)
    o_one, s_one = _run(cuda_lib, p)
    diff_o = (o_split - o_one[:T0]).abs().max().item()
    diff_s = (s_split - s_one[:len(lens)]).abs().max().item()
    assert torch.equal(o_split, o_one[:T0]) and torch.equal(s_split, s_one[:len(lens)]), (diff_o, diff_s)
    # and the one-CTA-per-head run against the oracle, padding sequences included
    ref_o, ref_s = oracle_full(p)
    check("one-CTA-per-head out", o_one, ref_o, tol_for(torch.bfloat16))
    check("one-CTA-per-head final state", s_one, ref_s, tol_for(torch.bfloat16))


def test_split_checkpoints_and_in_place_state(cuda_lib):
    """Checkpoints from the state scan equal the state after each prefix; in-place chaining."""
    H, L = 2, 512
    cfg = W.random_prefill_config([L], H, 128, torch.bfloat16, init="normal")
    d = W.make_prefill_inputs(cfg, seed=92)
    g = to_device(d)
    state = g["init_state"].clone()
    out, fin, ck = cuda_lib.prefill(g["q"], g["k"], g["v"], g["g"], g["beta"], g["cu_seqlens"], state,
                                    final_state=state, checkpoint_interval=128, checkpoint_slots=4)
    torch.cuda.synchronize()
    assert cuda_lib.last_device_status() == cuda_lib.KDA_OK and fin.data_ptr() == state.data_ptr()
    for j in range(4):
        sub = {n: d[n][:128 * (j + 1)] for n in ("q", "k", "v", "g", "beta")}
        sub["cu_seqlens"] = torch.tensor([0, 128 * (j + 1)], dtype=torch.int32)
        sub["init_state"] = d["init_state"]
        _, ref_s = oracle_full(sub)
        check(f"checkpoint {j}", ck[:, :, j].cpu(), ref_s, tol_for(torch.bfloat16))
    _, ref_final = oracle_full(d)
    check("in-place final", state.cpu(), ref_final, tol_for(torch.bfloat16))


def test_split_workspace_rules(cuda_lib):
    cfg = W.random_prefill_config([200], 2, 128, torch.bfloat16, init="zero")
    g = to_device(W.make_prefill_inputs(cfg, seed=93))
    desc = cuda_lib.make_desc(1, 200, 2, 128, 128, cuda_lib.KDA_BF16)
    need = cuda_lib.prefill_workspace_bytes(desc)
    assert need > 0
    small = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(cuda_lib.KDAError) as e:
        cuda_lib.prefill(g["q"], g["k"], g["v"], g["g"], g["beta"], g["cu_seqlens"], None, workspace=small)
    assert e.value.status == cuda_lib.KDA_ERR_WORKSPACE
    ws = torch.empty(need + 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(cuda_lib.KDAError) as e:   # not 16-byte aligned
        cuda_lib.prefill(g["q"], g["k"], g["v"], g["g"], g["beta"], g["cu_seqlens"], None, workspace=ws[8:])
    assert e.value.status == cuda_lib.KDA_ERR_INVALID_ARG
    # a reused workspace gives the same bits
    o1, _ = cuda_lib.prefill(g["q"], g["k"], g["v"], g["g"], g["beta"], g["cu_seqlens"], None, workspace=ws)
    o2, _ = cuda_lib.prefill(g["q"], g["k"], g["v"], g["g"], g["beta"], g["cu_seqlens"], None, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)


def test_split_many_sequences(cuda_lib):
    """30 sequences x 2 heads, lengths 0..400 with empties: every chunk's (first token,
    sequence end) comes from the chunk table."""
    rng = np.random.default_rng(94)
    lens = [int(x) for x in rng.integers(0, 401, size=30)]
    lens[5] = lens[17] = 0
    lens[23] = 64
    cfg = W.random_prefill_config(lens, 2, 128, torch.bfloat16, init="normal")
    assert _plan(cuda_lib, 30, cfg.total_tokens, 2)["kernel_launches"] >= 2
    d = W.make_prefill_inputs(cfg, seed=95)
    out, fin = _run(cuda_lib, d)
    ref_o, ref_s = oracle_full(d)
    check("many-sequence split out", out, ref_o, tol_for(torch.bfloat16))
    check("many-sequence split final state", fin, ref_s, tol_for(torch.bfloat16))


def test_split_at_the_item_cap_sampled(cuda_lib):
    """T = 32704, H = 64: (511 + 1) x 64 = 32768 items, the most the split takes (64 more
    tokens would take the one-CTA-per-unit kernel).  Sampled heads against the oracle."""
    H, T = 64, 32704
    assert _plan(cuda_lib, 1, T, H)["kernel_launches"] >= 2
    assert _plan(cuda_lib, 1, T + 64, H)["kernel_launches"] == 1
    cfg = W.PrefillConfig("cap", (T,), H, 128, 128, torch.bfloat16, "normal")
    d = W.make_prefill_inputs(cfg, seed=96, device="cuda")
    out, fin = cuda_lib.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], d["init_state"])
    torch.cuda.synchronize()
    assert cuda_lib.last_device_status() == cuda_lib.KDA_OK
    heads = [0, 37, 63]
    host = {k: (None if v is None else v.cpu()) for k, v in d.items()}
    ro, rs = oracle_heads(host, 0, heads, host["cu_seqlens"].numpy())
    check("cap split out", out[:, heads].cpu(), ro, tol_for(torch.bfloat16))
    check("cap split final state", fin[0, heads].cpu(), rs, tol_for(torch.bfloat16))


def test_split_separate_launches_sampled(cuda_lib):
    """160 heads x 1024 tokens: the split runs (one CTA per unit would need a second wave) as
    separate prep and scan launches (160 units leave no CTAs over for a single launch)."""
    H, T = 160, 1024
    assert _plan(cuda_lib, 1, T, H)["kernel_launches"] == 3
    cfg = W.PrefillConfig("two_waves", (T,), H, 128, 128, torch.bfloat16, "normal")
    d = W.make_prefill_inputs(cfg, seed=97, device="cuda")
    out, fin = cuda_lib.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], d["init_state"])
    torch.cuda.synchronize()
    assert cuda_lib.last_device_status() == cuda_lib.KDA_OK
    heads = [0, 77, 151, 152, 159]
    host = {k: (None if v is None else v.cpu()) for k, v in d.items()}
    ro, rs = oracle_heads(host, 0, heads, host["cu_seqlens"].numpy())
    check("separate-launch split out", out[:, heads].cpu(), ro, tol_for(torch.bfloat16))
    check("separate-launch split final state", fin[0, heads].cpu(), rs, tol_for(torch.bfloat16))


@pytest.mark.parametrize("gated", [False, True], ids=["plain", "gated"])
def test_split_separate_launches_uneven_sequences(cuda_lib, gated):
    """5 uneven sequences x 32 heads = 160 units: separate prep and scan launches, whose scan
    CTAs take their sequences longest first; every unit against the oracle (the state scan's
    ragged last chunks, one-chunk sequences, and with the gate its logits loaded into the O
    staging buffers a chunk ahead)."""
    import oracle
    lens = [700, 64, 1300, 200, 900]
    H = 32
    cfg = W.random_prefill_config(lens, H, 128, torch.bfloat16, init="normal")
    assert _plan(cuda_lib, len(lens), cfg.total_tokens, H)["kernel_launches"] == 3
    d = W.make_prefill_inputs(cfg, seed=99)
    g = to_device(d)
    z = W.make_gate_logits((cfg.total_tokens, H, 128), seed=100, device="cuda") if gated else None
    out, fin = cuda_lib.prefill(g["q"], g["k"], g["v"], g["g"], g["beta"], g["cu_seqlens"], g["init_state"], gate=z)
    torch.cuda.synchronize()
    assert cuda_lib.last_device_status() == cuda_lib.KDA_OK
    ref_o, ref_s = oracle_full(d)
    if gated:
        ref_o = oracle.output_gate(ref_o, z.cpu())
    check("separate-launch varlen out", out.cpu(), ref_o, tol_for(torch.bfloat16))
    check("separate-launch varlen final state", fin.cpu(), ref_s, tol_for(torch.bfloat16))


def test_concurrent_calls_on_two_streams(cuda_lib):
    """Two single-launch prefills on two streams with their own workspaces, and a decode on a
    third stream, in flight together: each equals its run alone, bit for bit (cooperative
    launches take the whole GPU, so the runtime orders them; nothing waits across calls)."""
    runs = []
    for i, (lens, H) in enumerate([([700, 333], 8), ([1024], 12)]):
        cfg = W.random_prefill_config(lens, H, 128, torch.bfloat16, init="normal")
        assert _plan(cuda_lib, len(lens), cfg.total_tokens, H)["kernel_launches"] == 2
        runs.append(to_device(W.make_prefill_inputs(cfg, seed=98 + i)))
    solo = []
    for g in runs:
        o, f = cuda_lib.prefill(g["q"], g["k"], g["v"], g["g"], g["beta"], g["cu_seqlens"], g["init_state"])
        solo.append((o.clone(), f.clone()))
    torch.cuda.synchronize()
    dcfg = W.DecodeConfig("side", 64, 16, 128, 128, torch.bfloat16, 1)
    di = W.make_decode_inputs(dcfg, seed=99, device="cuda")
    dstate, dstate_ref = di["state0"].clone(), di["state0"].clone()
    dref = cuda_lib.decode(di["q"][0], di["k"][0], di["v"][0], di["g"][0], di["beta"][0], dstate_ref)
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in range(3)]
    outs = []
    for _ in range(3):   # several rounds, so that the calls overlap in different ways
        outs.clear()
        for g, s in zip(runs, streams):
            outs.append(cuda_lib.prefill(g["q"], g["k"], g["v"], g["g"], g["beta"], g["cu_seqlens"], g["init_state"],
                                         stream=s))
        dstate.copy_(di["state0"])
        dout = cuda_lib.decode(di["q"][0], di["k"][0], di["v"][0], di["g"][0], di["beta"][0], dstate, stream=streams[2])
        torch.cuda.synchronize()
        assert cuda_lib.last_device_status() == cuda_lib.KDA_OK
        for (o, f), (ro, rf) in zip(outs, solo):
            assert torch.equal(o, ro) and torch.equal(f, rf)
        assert torch.equal(dout, dref) and torch.equal(dstate, dstate_ref)


def test_single_launch_uneven_sequences_near_the_limit(cuda_lib):
    """112 units of uneven sequences (7 sequences x 16 heads, one of a single token): items are
    claimed and published across all CTAs, and the scans of the long sequences run well past
    the short ones'."""
    rng = np.random.default_rng(100)
    lens = [int(x) for x in rng.integers(700, 2200, size=7)]
    lens[3] = 1
    cfg = W.random_prefill_config(lens, 16, 128, torch.bfloat16, init="normal")
    assert _plan(cuda_lib, 7, cfg.total_tokens, 16)["kernel_launches"] == 2
    d = W.make_prefill_inputs(cfg, seed=101)
    out, fin = _run(cuda_lib, d)
    ref_o, ref_s = oracle_full(d)
    check("near-limit out", out, ref_o, tol_for(torch.bfloat16))
    check("near-limit final state", fin, ref_s, tol_for(torch.bfloat16))


def test_beta_zero_read_out_on_both_paths(cuda_lib):
    """beta = 0: every output is the history read-out Q' S of the decaying initial state, and
    the first tokens of a sequence, which see the undecayed state, dominate the output's RMS
    over many near-zero outputs.  Both tensor-core forms meet the tensor-wide bar there."""
    H = 4
    lens = [200, 77]
    cfg = W.random_prefill_config(lens, H, 128, torch.bfloat16, init="normal")
    d = W.make_prefill_inputs(cfg, seed=52)
    # total decay over 200 tokens ~e^-25, inside fp32's range
    d = dict(d, g=(0.05 * d["g"]).contiguous(), beta=torch.zeros_like(d["beta"]))
    ref_o, ref_s = oracle_full(d)
    p = _padded(d, [64 + 3 * i for i in range(32)], seed=93)   # 136 units: one CTA per unit
    T0 = cfg.total_tokens
    assert _plan(cuda_lib, len(lens), T0, H)["kernel_launches"] >= 2
    assert _plan(cuda_lib, len(lens) + 32, p["q"].shape[0], H)["kernel_launches"] == 1
    o_split, s_split = _run(cuda_lib, d)
    o_one, s_one = _run(cuda_lib, p)
    tol = tol_for(torch.bfloat16)
    check("split out", o_split, ref_o, tol)
    check("split final state", s_split, ref_s, tol)
    check("one CTA per unit out", o_one[:T0], ref_o, tol)
    check("one CTA per unit final state", s_one[:len(lens)], ref_s, tol)


@pytest.mark.parametrize("launches", [2, 3], ids=["single-launch", "separate-launches"])
def test_split_repeated_calls_are_deterministic(cuda_lib, launches):
    """The chunk-parallel path, gated, 40 times over on uneven sequences: every call completes
    (no bounded wait runs out) and gives the same bits as the first, whatever order its CTAs
    claimed the items and however its roles interleaved (the state scan's barriers are waited
    for with parity, so a signaller two phases ahead of its waiter would hang the waiter)."""
    lens, H = ([700, 64, 1300, 200, 900], 32) if launches == 3 else ([700, 64, 1300, 200, 900], 16)
    cfg = W.random_prefill_config(lens, H, 128, torch.bfloat16, init="normal")
    assert _plan(cuda_lib, len(lens), cfg.total_tokens, H)["kernel_launches"] == launches
    g = to_device(W.make_prefill_inputs(cfg, seed=101))
    z = W.make_gate_logits((cfg.total_tokens, H, 128), seed=102, device="cuda")
    first = None
    for i in range(40):
        out, fin = cuda_lib.prefill(g["q"], g["k"], g["v"], g["g"], g["beta"], g["cu_seqlens"], g["init_state"],
                                    gate=z)
        torch.cuda.synchronize()
        assert cuda_lib.last_device_status() == cuda_lib.KDA_OK, f"call {i}"
        if first is None:
            first = (out.clone(), fin.clone())
        else:
            assert torch.equal(out, first[0]) and torch.equal(fin, first[1]), f"call {i} differs from the first"
