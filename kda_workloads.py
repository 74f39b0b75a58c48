"""Seeded synthetic inputs for Kimi Delta Attention (KDA) prefill and decode.

This module only draws random numbers and lays them out; it holds none of the
KDA arithmetic.  Both the CPU oracle (under ``oracle/``) and the CUDA library
are fed from it, and neither imports the other.

Input recipe (the five workloads named by the library's headline benchmark):

* q, k ~ N(0, 1), then L2-normalised per (token, head) over the key channels
  (fp64, divisor max(||x||, 1e-12)), then stored in the input dtype;
* v ~ N(0, 1);
* beta = sigmoid(N(0, 1)), one per (token, head), fp32;
* g = -5 * sigmoid(N(0, 1)), one per (token, head, key channel), fp32, so
  g lies in (-5, 0): the bounded log-decay g_min = -5 of the Kimi K3 report
  (llm-atlas "K3_RESEARCH.md", question ledger Q06 and Figure 3);
* initial state ~ N(0, 0.02) (standard deviation 0.02) where the workload has
  one, zero otherwise;
* varlen lengths uniform in [512, 16384] inclusive;
* output-gate logits z ~ N(0, 1) per output element, fp32 (for the gated entry points:
  out = o * sigmoid(z)).

Random draws come from a ``torch.Generator`` seeded per tensor with
``seed * 1000 + stream`` on the device the tensors are made on, so a large
workload can be drawn directly in GPU memory.  The oracle always reads host
copies of the stored tensors, so CPU and GPU draws need not agree bit for bit.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional

import numpy as np
import torch

G_MIN = -5.0

# stream ids: one independent generator per tensor kind
_S_Q, _S_K, _S_V, _S_G, _S_B, _S_S0, _S_LEN, _S_Z = 1, 2, 3, 4, 5, 6, 7, 8


@dataclasses.dataclass(frozen=True)
class PrefillConfig:
    """Shape of one prefill workload."""
    name: str
    seqlens: tuple            # tokens of each packed sequence
    num_heads: int
    dk: int
    dv: int
    qkv_dtype: torch.dtype    # torch.float32 or torch.bfloat16
    init_state: str           # "zero" or "normal"

    @property
    def num_seqs(self) -> int:
        return len(self.seqlens)

    @property
    def total_tokens(self) -> int:
        return int(sum(self.seqlens))

    def cu_seqlens(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(np.asarray(self.seqlens, dtype=np.int64))]).astype(np.int32)


@dataclasses.dataclass(frozen=True)
class DecodeConfig:
    """Shape of one decode workload: ``steps`` single-token steps over ``batch`` states."""
    name: str
    batch: int
    num_heads: int
    dk: int
    dv: int
    qkv_dtype: torch.dtype
    steps: int


def varlen_lengths(num_seqs: int, lo: int, hi: int, seed: int) -> tuple:
    """Integers uniform in [lo, hi] inclusive, drawn with numpy's PCG64 from ``seed``."""
    rng = np.random.default_rng(seed * 1000 + _S_LEN)
    return tuple(int(x) for x in rng.integers(lo, hi + 1, size=num_seqs))


def tiny_config() -> PrefillConfig:
    """B=1, H=2, T=256, dk=dv=64, fp32 inputs, zero initial state."""
    return PrefillConfig("tiny_fp32_h2_t256_d64", (256,), 2, 64, 64, torch.float32, "zero")


def prefill_config() -> PrefillConfig:
    """B=1, H=96, T=8192, dk=dv=128, bf16 q/k/v, N(0,0.02) initial state."""
    return PrefillConfig("prefill_bf16_h96_t8192_d128", (8192,), 96, 128, 128, torch.bfloat16, "normal")


def varlen_config(seed: int = 0) -> PrefillConfig:
    """32 packed sequences, lengths uniform in [512, 16384], H=96, dk=dv=128, bf16, zero init."""
    return PrefillConfig("varlen32_bf16_h96_d128", varlen_lengths(32, 512, 16384, seed), 96, 128, 128,
                         torch.bfloat16, "zero")


def decode_config() -> DecodeConfig:
    """B=256, H=96, dk=dv=128, bf16 q/k/v, 64 consecutive single-token steps."""
    return DecodeConfig("decode_bf16_b256_h96_d128", 256, 96, 128, 128, torch.bfloat16, 64)


def long_config() -> PrefillConfig:
    """B=1, H=96, T=131072, dk=dv=128, bf16, zero init (run as 16 chained 8192-token calls)."""
    return PrefillConfig("long_bf16_h96_t131072_d128", (131072,), 96, 128, 128, torch.bfloat16, "zero")


LONG_CALLS = 16


def _gen(seed: int, stream: int, device) -> torch.Generator:
    gen = torch.Generator(device=device)
    gen.manual_seed(seed * 1000 + stream)
    return gen


def _normal(shape, seed, stream, device, std=1.0, dtype=torch.float32):
    x = torch.randn(shape, generator=_gen(seed, stream, device), device=device, dtype=dtype)
    return x * std if std != 1.0 else x


def _l2_normalised(shape, seed, stream, device, out_dtype):
    x = _normal(shape, seed, stream, device, dtype=torch.float64)
    n = torch.linalg.vector_norm(x, dim=-1, keepdim=True).clamp_min(1e-12)
    return (x / n).to(out_dtype)


def _qkgb(shape_qk, shape_b, seed, device, dtype, raw):
    """q, k, g, beta of the recipe, or with ``raw`` the same draws before it: q and k not
    normalised (the N(0,1) draws in the storage type), g and beta as the N(0,1) logits."""
    if raw:
        q = _normal(shape_qk, seed, _S_Q, device, dtype=torch.float64).to(dtype)
        k = _normal(shape_qk, seed, _S_K, device, dtype=torch.float64).to(dtype)
        return q, k, _normal(shape_qk, seed, _S_G, device), _normal(shape_b, seed, _S_B, device)
    q = _l2_normalised(shape_qk, seed, _S_Q, device, dtype)
    k = _l2_normalised(shape_qk, seed, _S_K, device, dtype)
    g = (G_MIN * torch.sigmoid(_normal(shape_qk, seed, _S_G, device))).contiguous()
    return q, k, g, torch.sigmoid(_normal(shape_b, seed, _S_B, device)).contiguous()


def make_prefill_inputs(cfg: PrefillConfig, seed: int = 0, device="cpu", raw: bool = False) -> dict:
    """Seeded prefill inputs in the library layouts.

    q, k: [T, H, dk]; v: [T, H, dv] (cfg.qkv_dtype); g: [T, H, dk] fp32;
    beta: [T, H] fp32; cu_seqlens: [N+1] int32; init_state: [N, H, dk, dv]
    fp32 or None.  All tensors are contiguous on ``device``.  With ``raw`` q, k, g and
    beta are the draws before the recipe (for the library's input prologue).
    """
    T, H, dk, dv = cfg.total_tokens, cfg.num_heads, cfg.dk, cfg.dv
    d = {}
    d["q"], d["k"], d["g"], d["beta"] = _qkgb((T, H, dk), (T, H), seed, device, cfg.qkv_dtype, raw)
    d["v"] = _normal((T, H, dv), seed, _S_V, device).to(cfg.qkv_dtype)
    d["cu_seqlens"] = torch.from_numpy(cfg.cu_seqlens()).to(device)
    if cfg.init_state == "normal":
        d["init_state"] = _normal((cfg.num_seqs, H, dk, dv), seed, _S_S0, device, std=0.02)
    else:
        d["init_state"] = None
    return d


def make_decode_inputs(cfg: DecodeConfig, seed: int = 0, device="cpu", steps: Optional[int] = None,
                       raw: bool = False) -> dict:
    """Seeded decode inputs: per step q,k [S,B,H,dk], v [S,B,H,dv], g [S,B,H,dk], beta [S,B,H];
    state0 [B,H,dk,dv] ~ N(0, 0.02).  ``raw`` as for make_prefill_inputs."""
    S = cfg.steps if steps is None else steps
    B, H, dk, dv = cfg.batch, cfg.num_heads, cfg.dk, cfg.dv
    d = {}
    d["q"], d["k"], d["g"], d["beta"] = _qkgb((S, B, H, dk), (S, B, H), seed, device, cfg.qkv_dtype, raw)
    d["v"] = _normal((S, B, H, dv), seed, _S_V, device).to(cfg.qkv_dtype)
    d["state0"] = _normal((B, H, dk, dv), seed, _S_S0, device, std=0.02)
    return d


def make_gate_logits(shape, seed: int = 0, device="cpu") -> torch.Tensor:
    """Seeded output-gate logits z ~ N(0, 1), fp32, of the output's shape ([T, H, dv] for
    prefill, [B, H, dv] or [B, K, H, dv] for decode)."""
    return _normal(tuple(shape), seed, _S_Z, device).contiguous()


def random_prefill_config(seqlens: List[int], num_heads: int, d: int, qkv_dtype, init: str = "normal",
                          dv: Optional[int] = None) -> PrefillConfig:
    """A small ad-hoc workload for parity sweeps (ragged lengths, several chunks)."""
    return PrefillConfig(f"rand_n{len(seqlens)}_h{num_heads}_d{d}", tuple(int(s) for s in seqlens),
                         num_heads, d, d if dv is None else dv, qkv_dtype, init)


def named_prefill_configs(seed: int = 0) -> dict:
    return {"tiny": tiny_config(), "prefill": prefill_config(), "varlen": varlen_config(seed),
            "long": long_config()}
