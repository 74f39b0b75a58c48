"""Host logic of context-parallel prefill (one sequence split over ranks in token order) on
CPU: world sizes 2 and 3 over gloo.  Each rank holds its token range; the per-range work
(transition M_r and zero-start state S_r, then the rerun from the folded state) is done by the
fp64 oracle standing in for the GPU, the fold's step M S + A in fp64 numpy, and the exchange
and fold are the package's own.  The gathered outputs and the last rank's state must equal
the one-shot oracle over the whole sequence."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from linear_attention_serving_chunkwise_gb300.kcp import range_bounds


def test_range_bounds_cover_in_whole_chunks():
    for T in (0, 1, 63, 64, 65, 1000, 8192):
        for world in (1, 2, 3, 8):
            spans = [range_bounds(T, world, r) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == T
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
            assert all(a % 64 == 0 or a == T for a, _ in spans)
            chunks = [(b - a + 63) // 64 for a, b in spans]
            assert max(chunks) - min(chunks) <= 1


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, result_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import kda_workloads as W
    import oracle
    from linear_attention_serving_chunkwise_gb300 import kcp
    dist.init_process_group("gloo", rank=rank, world_size=world)
    H, d, T = 3, 8, 200
    cfg = W.random_prefill_config([T], H, d, torch.float32, init="normal")
    full = W.make_prefill_inputs(cfg, seed=81)
    full["g"] = (0.1 * full["g"]).contiguous()          # mild decay: the ranges' states matter
    t0, t1 = kcp.range_bounds(T, world, rank)
    mine = {n: full[n][t0:t1].contiguous() for n in ("q", "k", "v", "g", "beta")}

    def run(q, k, v, g, beta, s0):
        o, f = oracle.recurrent(q, k, v, g, beta, np.array([0, q.shape[0]], dtype=np.int32),
                                None if s0 is None else s0.to(torch.float32), threads=1)
        return torch.from_numpy(o), torch.from_numpy(f)

    def local(q, k, v, g, beta):
        eye = torch.eye(d, dtype=torch.float32).expand(1, H, d, d).contiguous()
        _, M = run(q, k, torch.zeros_like(v), g, beta, eye)
        _, S = run(q, k, v, g, beta, None)
        return M, S

    def combine(M, S, A):
        prod = 0.0 if S is None else torch.from_numpy(M.double().numpy() @ S.double().numpy())
        return prod + A.double()

    out, fin = kcp.context_parallel_prefill(mine["q"], mine["k"], mine["v"], mine["g"], mine["beta"],
                                            full["init_state"], local=local, combine=combine, run=run)
    parts = [None] * world
    dist.all_gather_object(parts, (rank, out.numpy(), fin.numpy()))
    if rank == 0:
        ref_o, ref_f = oracle.recurrent(full["q"], full["k"], full["v"], full["g"], full["beta"],
                                        full["cu_seqlens"], full["init_state"], threads=1)
        parts.sort(key=lambda p: p[0])
        got_o = np.concatenate([p[1] for p in parts], axis=0)
        err_o = oracle.rel_err(got_o, ref_o)
        err_f = oracle.rel_err(parts[-1][2], ref_f)
        result_q.put((err_o, err_f))
    dist.destroy_process_group()


def _spawn(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    err_o, err_f = q.get(timeout=240)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    # the range states re-enter the oracle as fp32 (its init_state type): fp32 rounding only
    assert err_o < 1e-6 and err_f < 1e-6, (err_o, err_f)


def test_two_ranks_match_one_shot():
    _spawn(2)


def test_three_ranks_match_one_shot():
    _spawn(3)
