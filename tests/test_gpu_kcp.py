"""GPU tests of context-parallel prefill of one sequence (token ranges run independently, one
fold of (transition, zero-start state) pairs, then a rerun from the folded states), with the
ranks emulated as ranges of one sequence on one GPU, and of its fold step kda_state_combine.
Every result is compared with the one-shot oracle over the whole sequence."""
import numpy as np
import pytest
import torch

import kda_workloads as W
import oracle
from _parity import check, oracle_full, to_device, tol_for
from linear_attention_serving_chunkwise_gb300 import kcp

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d", [64, 128])
def test_state_combine_matches_definition(cuda_lib, d):
    """out = M in + add per (sequence, head), against the product in fp64; None operands are
    zero; in place over add."""
    rng = np.random.default_rng(d)
    n = 5
    M = torch.from_numpy(rng.standard_normal((n, d, d)).astype(np.float32))
    S = torch.from_numpy(rng.standard_normal((n, d, d)).astype(np.float32))
    A = torch.from_numpy(rng.standard_normal((n, d, d)).astype(np.float32))
    ref = M.double().numpy() @ S.double().numpy() + A.double().numpy()
    Mc, Sc, Ac = M.cuda(), S.cuda(), A.cuda()
    out = cuda_lib.state_combine(Mc, Sc, Ac)
    only_add = cuda_lib.state_combine(None, None, Ac)
    no_add = cuda_lib.state_combine(Mc, Sc, None)
    in_place = Ac.clone()
    cuda_lib.state_combine(Mc, Sc, in_place, out=in_place)
    torch.cuda.synchronize()
    scale = np.sqrt(d) * 1e-6   # fp32 dot products of length d
    assert np.max(np.abs(out.cpu().double().numpy() - ref)) < scale * 10
    assert torch.equal(only_add, Ac)
    assert np.max(np.abs(no_add.cpu().double().numpy() - (ref - A.double().numpy()))) < scale * 10
    assert torch.equal(in_place, out)
    with pytest.raises(cuda_lib.KDAError):
        cuda_lib.state_combine(Mc, Sc, Ac, out=Sc)          # out over in: rejected


def _one_sequence(T, H, d, dtype, seed, g_scale):
    cfg = W.random_prefill_config([T], H, d, dtype, init="normal")
    x = W.make_prefill_inputs(cfg, seed=seed)
    x["g"] = (g_scale * x["g"]).contiguous()
    return x


@pytest.mark.parametrize("ranks", [2, 3, 4])
@pytest.mark.parametrize("g_scale", [0.05, 1.0], ids=["mild_decay", "workload_decay"])
def test_virtual_ranks_match_one_shot_bf16(cuda_lib, ranks, g_scale):
    x = _one_sequence(1000, 4, 128, torch.bfloat16, seed=82 + ranks, g_scale=g_scale)
    ref_o, ref_s = oracle_full(x)
    g = to_device(x)
    out, fin, (Ms, Ss) = kcp.virtual_ranks_prefill(g["q"], g["k"], g["v"], g["g"], g["beta"], g["init_state"],
                                                   ranks=ranks)
    torch.cuda.synchronize()
    assert cuda_lib.last_device_status() == cuda_lib.KDA_OK
    tol = tol_for(torch.bfloat16)
    check("context-parallel out", out, ref_o, tol)
    check("context-parallel final state", fin, ref_s, tol)
    # each range's affine map, as the fold uses it: M_r S_in + S_r, with S_in the oracle's state
    # entering the range, against the oracle's state after it.  (M_r alone is compared only
    # through this: from the identity its entries shrink to e^-60 and below over a range, so
    # its error relative to its own RMS measures cancellation, not anything the fold uses.)
    s0 = x["init_state"]
    for r in range(ranks):
        t0, t1 = kcp.range_bounds(1000, ranks, r)
        pre = {n: x[n][:t1].contiguous() for n in ("q", "k", "v", "g", "beta")}
        cu = lambda n: np.array([0, n], dtype=np.int32)
        _, S_after = oracle.recurrent(pre["q"], pre["k"], pre["v"], pre["g"], pre["beta"], cu(t1), s0)
        if t0 > 0:
            _, S_in = oracle.recurrent(pre["q"][:t0], pre["k"][:t0], pre["v"][:t0], pre["g"][:t0],
                                       pre["beta"][:t0], cu(t0), s0)
        else:
            S_in = s0.double().numpy()
        got = Ms[r].cpu().double().numpy() @ S_in + Ss[r].cpu().double().numpy()
        check(f"range {r} map M S_in + S_r", got, S_after, tol)


def test_virtual_ranks_match_one_shot_fp32(cuda_lib):
    """The fp32 path (CUDA-core prefill, dk = dv = 64) holds the 1e-4 bar through the fold."""
    x = _one_sequence(700, 3, 64, torch.float32, seed=86, g_scale=0.05)
    ref_o, ref_s = oracle_full(x)
    g = to_device(x)
    out, fin, _ = kcp.virtual_ranks_prefill(g["q"], g["k"], g["v"], g["g"], g["beta"], g["init_state"], ranks=3)
    torch.cuda.synchronize()
    check("context-parallel out (fp32)", out, ref_o, 1e-4)
    check("context-parallel final state (fp32)", fin, ref_s, 1e-4)


def test_local_pass_and_fold_of_two_ranges(cuda_lib):
    """The per-rank entry points one rank of a real multi-GPU run calls: local_pass on each
    range, fold, then the rerun, here for two ranges in one process."""
    x = _one_sequence(640, 2, 128, torch.bfloat16, seed=87, g_scale=0.05)
    ref_o, ref_s = oracle_full(x)
    g = to_device(x)
    b = [kcp.range_bounds(640, 2, r) for r in range(2)]
    parts = [{n: g[n][t0:t1].contiguous() for n in ("q", "k", "v", "g", "beta")} for t0, t1 in b]
    pairs = [kcp.local_pass(p["q"], p["k"], p["v"], p["g"], p["beta"]) for p in parts]
    Ms, Ss = [p[0] for p in pairs], [p[1] for p in pairs]
    outs, fin = [], None
    for r, p in enumerate(parts):
        S_in = kcp.fold(Ms, Ss, r, g["init_state"])
        o, fin = cuda_lib.prefill(p["q"], p["k"], p["v"], p["g"], p["beta"], None, S_in)
        outs.append(o)
    torch.cuda.synchronize()
    tol = tol_for(torch.bfloat16)
    check("two-range out", torch.cat(outs), ref_o, tol)
    check("two-range final state", fin, ref_s, tol)
