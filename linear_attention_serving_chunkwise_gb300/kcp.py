"""Context-parallel prefill of one long sequence: consecutive token ranges on different ranks.

The pages list KCP among the pretraining mechanisms of Kimi K3's KDA (llm-atlas
"K3_RESEARCH.md", section 8 system-state table, pretraining row); Q07 gives the chunkwise form
in which the state is the only thing passed from one stretch of tokens to the next.  Read as
context parallelism for KDA, it rests on the recurrence being affine in its initial state:
a token range r maps the state entering it as

    S_after = M_r S_before + S_r,

where M_r (dk x dk) is the product of the range's chunk transitions Diag(e^{Gamma_C}) -
K~^T Wk and S_r is the state the range reaches from a zero start.  So every rank can run its
range without waiting for the ranks before it, and one exchange fixes the states:

1. local pass: M_r = the state after the range from initial state I with v = 0, and S_r =
   the state after it from a zero state with the real v (two kda_prefill calls);
2. exchange: all ranks gather every (M_j, S_j) (one all-gather of 2 x H x dk x dv fp32 per
   rank; no TMA multicast, no library GEMM on a peer's memory);
3. fold: the state entering range r is S <- M_j S + S_j over j < r, from the sequence's
   initial state (kda_state_combine, one call per step);
4. rerun: kda_prefill on the range from that state gives its outputs and the state after
   it (the last rank's is the sequence's final state).

All arithmetic runs in the CUDA library; this module only allocates the zero v, the identity
initial state and scratch outputs, and moves tensors between ranks.  The exchange and the fold
take their collective and their combine step as arguments, so that the host logic can be
tested over gloo on CPU with the oracle standing in for the GPU.
"""
from __future__ import annotations

from typing import Callable, List, Optional, Sequence, Tuple

import torch

from . import _lib as kda


def range_bounds(total_tokens: int, world: int, rank: int, align: int = 64) -> Tuple[int, int]:
    """Token range [t0, t1) of `rank`: whole `align`-token chunks, split as evenly as the chunk
    count allows (earlier ranks take the extra chunk); the last range ends at total_tokens."""
    if not (0 <= rank < world) or total_tokens < 0 or align < 1:
        raise ValueError("bad rank/world/total_tokens/align")
    chunks = (total_tokens + align - 1) // align
    base, extra = divmod(chunks, world)
    c0 = rank * base + min(rank, extra)
    c1 = c0 + base + (1 if rank < extra else 0)
    return min(c0 * align, total_tokens), min(c1 * align, total_tokens)


def local_pass(q, k, v, g, beta, *, stream=None, prologue: int = 0):
    """(M_r, S_r) of one token range of one sequence, all heads: M_r [1, H, dk, dk] is the
    state after the range from the identity with v = 0, S_r [1, H, dk, dv] the state after it
    from zero.  q, k, v, g, beta are the range's tokens ([L, H, .], device tensors)."""
    L, H, dk = q.shape
    dv = v.shape[2]
    if dk != dv:
        raise ValueError("context-parallel prefill needs dk == dv (the transition is square)")
    scratch = torch.empty((L, H, dv), dtype=torch.float32, device=q.device)
    _, S_r = kda.prefill(q, k, v, g, beta, None, None, out=scratch, stream=stream, prologue=prologue)
    eye = torch.eye(dk, dtype=torch.float32, device=q.device).expand(1, H, dk, dk).contiguous()
    zero_v = torch.zeros_like(v)
    M_r = torch.empty_like(eye)
    kda.prefill(q, k, zero_v, g, beta, None, eye, out=scratch, final_state=M_r, stream=stream, prologue=prologue)
    for t in (scratch, eye, zero_v):
        kda._keep_until_done(t, stream)
    return M_r, S_r


def fold(Ms: Sequence[torch.Tensor], Ss: Sequence[torch.Tensor], rank: int, init_state: Optional[torch.Tensor],
         combine: Optional[Callable] = None):
    """The state entering range `rank`: S <- M_j S + S_j for j = 0 .. rank-1, from init_state
    (None = zero).  `combine(M, S_in, S_add)` returns M S_in + S_add (None entries are zero);
    by default the library's kda_state_combine."""
    combine = combine or (lambda M, S, A: kda.state_combine(M, S, A))
    S = init_state
    for j in range(rank):
        S = combine(Ms[j], S, Ss[j])
    return S


def exchange(M_r: torch.Tensor, S_r: torch.Tensor, group=None) -> Tuple[List[torch.Tensor], List[torch.Tensor]]:
    """All-gather every rank's (M_j, S_j) over `group` (torch.distributed; NCCL for device
    tensors, gloo for host ones).  Returns the lists in rank order."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    both = torch.cat([M_r.reshape(-1), S_r.reshape(-1)])
    parts = [torch.empty_like(both) for _ in range(world)]
    dist.all_gather(parts, both, group=group)
    n = M_r.numel()
    return ([p[:n].reshape(M_r.shape) for p in parts], [p[n:].reshape(S_r.shape) for p in parts])


def context_parallel_prefill(q, k, v, g, beta, init_state=None, *, group=None, stream=None, prologue: int = 0,
                             local: Optional[Callable] = None, combine: Optional[Callable] = None,
                             run: Optional[Callable] = None):
    """This rank's part of a prefill of one sequence split over the ranks of `group` in token
    order (rank r holds the r-th range: q, k, v, g, beta [L_r, H, .]).  init_state [1, H, dk,
    dv] is the sequence's initial state, the same on every rank (None = zero).  Returns (out
    [L_r, H, dv], state after the range); the last rank's state is the sequence's final state.
    `local`, `combine` and `run` replace the library calls (tests on CPU)."""
    import torch.distributed as dist
    rank = dist.get_rank(group)
    local = local or (lambda *a: local_pass(*a, stream=stream, prologue=prologue))
    run = run or (lambda q_, k_, v_, g_, b_, s0: kda.prefill(q_, k_, v_, g_, b_, None, s0, stream=stream,
                                                              prologue=prologue))
    M_r, S_r = local(q, k, v, g, beta)
    Ms, Ss = exchange(M_r, S_r, group)
    S_in = fold(Ms, Ss, rank, init_state, combine)
    return run(q, k, v, g, beta, S_in)


def virtual_ranks_prefill(q, k, v, g, beta, init_state=None, *, ranks: int = 2, stream=None, prologue: int = 0):
    """The same scheme on one GPU with `ranks` ranges of one sequence held in one process (no
    collective): the local passes of all ranges run as one varlen kda_prefill call each, then
    the fold, then one call that reruns every range from its entering state.  q, k, v, g,
    beta [T, H, .] of one sequence; init_state [1, H, dk, dv] or None.  Returns (out [T, H, dv],
    final state [1, H, dk, dv]) and the per-range (M_r, S_r)."""
    T, H, dk = q.shape
    dv = v.shape[2]
    if dk != dv:
        raise ValueError("context-parallel prefill needs dk == dv (the transition is square)")
    dev = q.device
    bounds = [range_bounds(T, ranks, r) for r in range(ranks)]
    cu = torch.tensor([b[0] for b in bounds] + [T], dtype=torch.int32, device=dev)
    scratch = torch.empty((T, H, dv), dtype=torch.float32, device=dev)
    _, S_all = kda.prefill(q, k, v, g, beta, cu, None, out=scratch, stream=stream, prologue=prologue)
    eye = torch.eye(dk, dtype=torch.float32, device=dev).expand(ranks, H, dk, dk).contiguous()
    zero_v = torch.zeros_like(v)
    M_all = torch.empty_like(eye)
    kda.prefill(q, k, zero_v, g, beta, cu, eye, out=scratch, final_state=M_all, stream=stream, prologue=prologue)
    Ms = [M_all[r:r + 1] for r in range(ranks)]
    Ss = [S_all[r:r + 1] for r in range(ranks)]
    S_in = torch.zeros((ranks, H, dk, dv), dtype=torch.float32, device=dev)
    if init_state is not None:
        S_in[0:1].copy_(init_state)
    for r in range(ranks - 1):   # the fold, each step straight into the next range's slot
        kda.state_combine(Ms[r], S_in[r:r + 1], Ss[r], out=S_in[r + 1:r + 2], stream=stream)
    out, fin = kda.prefill(q, k, v, g, beta, cu, S_in, stream=stream, prologue=prologue)
    for t in (scratch, eye, zero_v, S_in):
        kda._keep_until_done(t, stream)
    return out, fin[ranks - 1:ranks], (Ms, Ss)
