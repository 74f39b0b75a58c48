"""CPU oracle for Kimi Delta Attention -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The CUDA library never imports, links or calls
it, and the two share no code.
"""
from .kda_ref import (  # noqa: F401
    build_oracle,
    recurrent,
    unrolled_bruteforce,
    chunkwise_naive,
    delta_invariant_keys,
    rel_err,
    prologue,
    output_gate,
    sigmoid64,
    l2_normalise64,
    PROLOGUE_QK_L2NORM,
    PROLOGUE_G_LOGITS,
    PROLOGUE_BETA_LOGITS,
)
