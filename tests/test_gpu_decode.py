"""GPU parity of kda_decode against the CPU oracle (through the C ABI).

A decode step is the recurrence on a one-token sequence, so S decode steps of
batch B equal the oracle over B sequences of S tokens each."""
import numpy as np
import pytest
import torch

import kda_workloads as W
import oracle
from _parity import check, tol_for

pytestmark = pytest.mark.gpu


def _as_sequences(d, b_idx, h_idx):
    """Step-major decode inputs [S, B, H, .] of the chosen (b, h) units as packed
    sequences [S * U, 1, .] (one sequence per unit), on the host."""
    sel = lambda x: torch.stack([x[:, b, h] for b, h in zip(b_idx, h_idx)], dim=0).cpu()  # [U, S, ...]
    q, k, v, g = (sel(d[n]) for n in ("q", "k", "v", "g"))
    beta = sel(d["beta"])
    U, S = beta.shape
    flat = lambda x: x.reshape(U * S, 1, -1).contiguous()
    s0 = torch.stack([d["state0"][b, h] for b, h in zip(b_idx, h_idx)]).cpu()[:, None].contiguous()
    cu = np.arange(0, U * S + 1, S, dtype=np.int32)
    return flat(q), flat(k), flat(v), flat(g), beta.reshape(U * S, 1).contiguous(), cu, s0


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["fp32", "bf16"])
def test_decode_small_all_units(cuda_lib, d, dtype):
    cfg = W.DecodeConfig("small", 5, 3, d, d, dtype, 6)
    inp = W.make_decode_inputs(cfg, seed=d)
    g = {k: v.cuda() for k, v in inp.items()}
    state = g["state0"].clone()
    outs = [cuda_lib.decode(g["q"][s], g["k"][s], g["v"][s], g["g"][s], g["beta"][s], state)
            for s in range(cfg.steps)]
    torch.cuda.synchronize()
    B, H = cfg.batch, cfg.num_heads
    bs, hs = zip(*[(b, h) for b in range(B) for h in range(H)])
    q, k, v, gg, beta, cu, s0 = _as_sequences(inp, bs, hs)
    ref_o, ref_s = oracle.recurrent(q, k, v, gg, beta, cu, s0.reshape(-1, 1, d, d))
    # ref_o rows: unit-major (unit u, step s) -> compare per step
    got = torch.stack(outs, 0).cpu()                                   # [S, B, H, dv]
    got_units = torch.stack([got[:, b, h] for b, h in zip(bs, hs)], 0)  # [U, S, dv]
    tol = tol_for(dtype)
    check("decode out", got_units.reshape(-1, d), ref_o.reshape(-1, d), tol)
    got_s = torch.stack([state[b, h] for b, h in zip(bs, hs)], 0)
    check("decode state", got_s, ref_s[:, 0], tol)


def test_decode_workload_b256_h96_64_steps_sampled(cuda_lib):
    cfg = W.decode_config()
    d = W.make_decode_inputs(cfg, seed=0, device="cuda")
    state = d["state0"].clone()
    out = torch.empty((cfg.steps, cfg.batch, cfg.num_heads, cfg.dv), dtype=torch.float32, device="cuda")
    for s in range(cfg.steps):
        cuda_lib.decode(d["q"][s], d["k"][s], d["v"][s], d["g"][s], d["beta"][s], state, out=out[s])
    torch.cuda.synchronize()
    assert torch.isfinite(out).all() and torch.isfinite(state).all()
    rng = np.random.default_rng(3)
    units = [(0, 0), (255, 95)] + [(int(rng.integers(256)), int(rng.integers(96))) for _ in range(14)]
    bs, hs = zip(*units)
    q, k, v, g, beta, cu, s0 = _as_sequences(d, bs, hs)
    ref_o, ref_s = oracle.recurrent(q, k, v, g, beta, cu, s0.reshape(-1, 1, 128, 128))
    got = torch.stack([out[:, b, h] for b, h in units], 0).cpu()
    check("decode out", got.reshape(-1, 128), ref_o.reshape(-1, 128), 2e-2)
    got_s = torch.stack([state[b, h] for b, h in units], 0)
    check("decode state", got_s, ref_s[:, 0], 2e-2)


def test_decode_empty_batch_is_noop(cuda_lib):
    z = torch.empty((0, 2, 64), device="cuda")
    st = torch.empty((0, 2, 64, 64), device="cuda")
    out = cuda_lib.decode(z, z, z, z, torch.empty((0, 2), device="cuda"), st)
    assert out.shape == (0, 2, 64)
