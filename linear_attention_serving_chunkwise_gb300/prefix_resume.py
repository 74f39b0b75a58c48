"""Where a request can resume from a cached prefix (host-side arithmetic).

The serving layer keys its prefix cache on fixed hash blocks and keeps sparse KDA state
snapshots (llm-atlas K3_RESEARCH.md, Q31: unified page pool, 512-token hash boundary
inside a 6144-token physical block, sparse KDA checkpoints, a hit needs both the KDA
state and the MLA KV; Lab H: matched prefix, physical block, hash block and checkpoint
boundary give the longest reusable boundary and the tokens to recompute).  A KDA state
exists only at checkpoint boundaries, and the cache can only match whole hash blocks,
so the reusable boundary is the largest common multiple of both that does not exceed
the matched prefix.  The physical block size decides page allocation, not where KDA can
resume.
"""
from __future__ import annotations

import math
from typing import NamedTuple


class ResumePlan(NamedTuple):
    boundary: int          # tokens covered by the reused prefix (0 = no reuse)
    checkpoint_slot: int   # snapshot index to load (-1 = none)
    recompute: int         # prompt tokens that still go through prefill


def plan_resume(matched_prefix: int, prompt_len: int, hash_block: int = 512, checkpoint_interval: int = 512,
                checkpoint_slots: int | None = None) -> ResumePlan:
    """Longest reusable boundary <= matched_prefix that is both a whole number of hash
    blocks and a checkpoint position (and, if given, within the kept slots); the rest of
    the prompt is recomputed.  At least one token is always recomputed so the request
    produces its last position's output."""
    if min(hash_block, checkpoint_interval) <= 0 or checkpoint_interval % 64:
        raise ValueError("hash_block > 0 and checkpoint_interval a positive multiple of 64")
    if not (0 <= matched_prefix <= prompt_len):
        raise ValueError("0 <= matched_prefix <= prompt_len")
    step = hash_block * checkpoint_interval // math.gcd(hash_block, checkpoint_interval)
    b = (min(matched_prefix, prompt_len - 1) // step) * step if prompt_len > 0 else 0
    if checkpoint_slots is not None:
        b = min(b, (checkpoint_slots * checkpoint_interval // step) * step)
    slot = b // checkpoint_interval - 1 if b > 0 else -1
    return ResumePlan(b, slot, prompt_len - b)
