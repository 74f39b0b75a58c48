"""Multi-rank host logic on CPU: world size 2 over gloo.  Each rank takes its share of
(sequence, head) units, runs the oracle on it, and the gathered shares must equal the
single-process result; the bench's barrier and max-over-ranks helpers run too."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from linear_attention_serving_chunkwise_gb300.sharding import shard_heads, shard_sequences


def test_shard_heads_covers_exactly():
    for H in (1, 2, 95, 96):
        for world in (1, 2, 3, 8):
            spans = [shard_heads(H, world, r) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == H
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
            sizes = [b - a for a, b in spans]
            assert max(sizes) - min(sizes) <= 1


def test_shard_sequences_partition_and_balance():
    rng = np.random.default_rng(0)
    lens = [int(x) for x in rng.integers(512, 16385, size=32)]
    for world in (1, 2, 4):
        parts = [shard_sequences(lens, world, r) for r in range(world)]
        assert sorted(i for p in parts for i in p) == list(range(32))
        loads = [sum(lens[i] for i in p) for p in parts]
        assert max(loads) - min(loads) <= max(lens)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, result_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import bench
    import kda_workloads as W
    import oracle
    w, r, _ = bench._dist_setup(world)
    assert (w, r) == (world, rank)
    cfg = W.random_prefill_config([40, 9, 70], 5, 8, torch.float32, init="normal")
    d = W.make_prefill_inputs(cfg, seed=3)
    h0, h1 = shard_heads(cfg.num_heads, world, rank)
    sl = lambda x: x[:, h0:h1].contiguous()
    o, f = oracle.recurrent(sl(d["q"]), sl(d["k"]), sl(d["v"]), sl(d["g"]), sl(d["beta"]), d["cu_seqlens"],
                            d["init_state"][:, h0:h1].contiguous(), threads=1)
    parts = [None] * world
    dist.all_gather_object(parts, (h0, h1, o, f))
    bench._barrier(world)
    m = bench._max_over_ranks(float(rank + 1), world)
    if rank == 0:
        full_o, full_f = oracle.recurrent(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                                          d["init_state"], threads=1)
        go = np.concatenate([p[2] for p in sorted(parts, key=lambda p: p[0])], axis=1)
        gf = np.concatenate([p[3] for p in sorted(parts, key=lambda p: p[0])], axis=1)
        result_q.put((bool(np.array_equal(go, full_o) and np.array_equal(gf, full_f)), m))
    dist.destroy_process_group()


def test_two_rank_head_sharding_matches_one_process():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    ok, m = q.get(timeout=240)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert ok and m == 2.0
