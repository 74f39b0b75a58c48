"""Shared helpers of the GPU parity tests: run the CUDA path and the CPU oracle on the
same seeded inputs and compare.

Error measure: max |x - ref| / RMS(ref) over the compared tensor.  Bars: 1e-4 for
fp32 q/k/v, 2e-2 for bf16 q/k/v (fp32 state, fp32 output), for outputs and final
states alike.
"""
import numpy as np
import torch

import oracle

TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}


def tol_for(dtype):
    return TOL[dtype]


def to_device(d, device="cuda"):
    return {k: (None if v is None else v.to(device)) for k, v in d.items()}


def oracle_full(d):
    """Oracle over a whole (small) packed workload held on any device."""
    return oracle.recurrent(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], d.get("init_state"))


def check(name, got, ref, tol):
    got = got.detach().to("cpu", torch.float64).numpy() if isinstance(got, torch.Tensor) else got
    err = oracle.rel_err(got, ref)
    assert np.isfinite(got).all(), f"{name}: non-finite values"
    assert err <= tol, f"{name}: rel err {err:.3e} > {tol:.1e}"
    return err


def sampled_units(num_seqs, num_heads, count, seed, must=()):
    """A seeded sample of (seq, head) pairs, always including ``must``."""
    rng = np.random.default_rng(seed)
    units = list(must)
    while len(units) < count:
        u = (int(rng.integers(num_seqs)), int(rng.integers(num_heads)))
        if u not in units:
            units.append(u)
    return units


def oracle_heads(d, seq, heads, cu_host, threads=None):
    """Oracle for several heads of one sequence at once (threads over heads)."""
    b, e = int(cu_host[seq]), int(cu_host[seq + 1])
    hs = list(heads)
    pick = lambda x: x[b:e][:, hs].contiguous() if isinstance(x, torch.Tensor) else x[b:e][:, hs]
    s0 = d.get("init_state")
    s0 = None if s0 is None else s0[seq:seq + 1][:, hs].contiguous()
    o, f = oracle.recurrent(pick(d["q"]), pick(d["k"]), pick(d["v"]), pick(d["g"]), pick(d["beta"]),
                            np.array([0, e - b], dtype=np.int32), s0, threads=threads or len(hs))
    return o, f[0]
