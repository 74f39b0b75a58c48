"""The seeded input generators: shapes, ranges, determinism (CPU)."""
import numpy as np
import torch

import kda_workloads as W


def test_tiny_config_shapes_and_ranges():
    cfg = W.tiny_config()
    d = W.make_prefill_inputs(cfg, seed=0)
    assert d["q"].shape == (256, 2, 64) and d["q"].dtype == torch.float32
    assert d["beta"].shape == (256, 2)
    assert d["init_state"] is None
    assert float(d["g"].min()) >= W.G_MIN and float(d["g"].max()) <= 0.0
    assert float(d["beta"].min()) > 0.0 and float(d["beta"].max()) < 1.0
    n = torch.linalg.vector_norm(d["k"].double(), dim=-1)
    assert torch.allclose(n, torch.ones_like(n), atol=1e-6)
    assert d["cu_seqlens"].tolist() == [0, 256]


def test_seeded_determinism():
    cfg = W.random_prefill_config([33, 7], 3, 16, torch.bfloat16)
    a = W.make_prefill_inputs(cfg, seed=5)
    b = W.make_prefill_inputs(cfg, seed=5)
    c = W.make_prefill_inputs(cfg, seed=6)
    for key in ("q", "k", "v", "g", "beta", "init_state"):
        assert torch.equal(a[key], b[key])
    assert not torch.equal(a["v"], c["v"])
    assert a["q"].dtype == torch.bfloat16 and a["init_state"].shape == (2, 3, 16, 16)


def test_varlen_lengths_in_range():
    cfg = W.varlen_config(0)
    assert cfg.num_seqs == 32
    assert all(512 <= s <= 16384 for s in cfg.seqlens)
    cu = cfg.cu_seqlens()
    assert cu[0] == 0 and np.all(np.diff(cu) == np.asarray(cfg.seqlens))


def test_decode_inputs_shapes():
    cfg = W.decode_config()
    small = W.DecodeConfig("d", 4, 2, 8, 8, torch.bfloat16, 3)
    d = W.make_decode_inputs(small, seed=1)
    assert d["q"].shape == (3, 4, 2, 8) and d["beta"].shape == (3, 4, 2)
    assert d["state0"].shape == (4, 2, 8, 8) and d["state0"].dtype == torch.float32
    assert cfg.steps == 64 and cfg.batch == 256
