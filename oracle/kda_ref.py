"""Python side of the KDA CPU oracle -- test infrastructure only.

* ``recurrent``: ctypes wrapper over the plain-C fp64 token-by-token recurrence
  in ``kda_oracle.c`` (the definition of KDA; see that file's header).
* ``unrolled_bruteforce``: the same quantity written as explicit products of
  dk x dk transition matrices, for tiny T (an independent formulation used to
  pin the recurrence).
* ``chunkwise_naive``: the chunkwise-parallel rewrite in plain fp64 numpy, with
  every intra-chunk decay taken directly as exp(Gamma_r - Gamma_i) and the
  triangular system solved by an explicit matrix inverse -- no sub-tiling, no
  factoring, no blocking.  It pins the recurrence from another direction and
  states the chunk algebra the GPU path follows.

Sources: llm-atlas "K3_RESEARCH.md" question ledger Q04-Q07 (recurrent state,
delta-rule write, bounded decay, chunkwise parallel form with state passed
between chunks and parallel matrix work inside a chunk); agihunt digest page
(FlashKDA chunkwise parallel form with 16-token tiles).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIBS = {}


def build_oracle(mutant: int = 0, out_dir: Optional[str] = None, force: bool = False) -> str:
    """Compile kda_oracle.c with gcc into a shared library and return its path.

    ``mutant`` != 0 plants one of the deliberate mistakes (tests only) and
    builds into ``out_dir`` (a temporary directory by default)."""
    if mutant:
        out_dir = out_dir or tempfile.mkdtemp(prefix="kda_oracle_mutant_")
    else:
        out_dir = out_dir or _BUILD_DIR
    os.makedirs(out_dir, exist_ok=True)
    so = os.path.join(out_dir, f"libkda_oracle_m{mutant}.so")
    if force or not os.path.exists(so) or os.path.getmtime(so) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-pthread", "-shared", "-fPIC",
               f"-DKDA_ORACLE_MUTANT={int(mutant)}", _SRC, "-o", so + ".tmp", "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(so + ".tmp", so)
    return so


def _lib(mutant: int = 0, path: Optional[str] = None):
    key = path or mutant
    if key not in _LIBS:
        lib = ctypes.CDLL(path or build_oracle(mutant))
        f = lib.kda_oracle_recurrent
        f.restype = ctypes.c_int
        f.argtypes = [ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                      ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                      ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32]
        lib.kda_oracle_mutant.restype = ctypes.c_int
        _LIBS[key] = lib
    return _LIBS[key]


def _host(x):
    """A contiguous host numpy array holding x's stored values; bf16 is kept as uint16 bits."""
    if x is None:
        return None, False
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().to("cpu").contiguous()
            if x.dtype == torch.bfloat16:
                return x.view(torch.int16).numpy().view(np.uint16), True
            return x.numpy(), False
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(x)
    return a, a.dtype == np.uint16


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def recurrent(q, k, v, g, beta, cu_seqlens, init_state=None, threads: Optional[int] = None,
              want_final: bool = True, mutant: int = 0, lib_path: Optional[str] = None):
    """fp64 KDA over packed sequences.

    q, k [T,H,dk]; v [T,H,dv] (fp32 or bf16); g [T,H,dk] fp32; beta [T,H] fp32;
    cu_seqlens [N+1]; init_state [N,H,dk,dv] fp32 or None.  Accepts torch
    tensors (any device; copied to host) or numpy arrays.
    Returns (out [T,H,dv] float64, final_state [N,H,dk,dv] float64 or None)."""
    qh, qb = _host(q)
    kh, kb = _host(k)
    vh, vb = _host(v)
    if not (qb == kb == vb):
        raise ValueError("q, k, v must share one storage type")
    if not qb and qh.dtype != np.float32:
        raise ValueError("q/k/v must be fp32 or bf16")
    gh = np.ascontiguousarray(_host(g)[0], dtype=np.float32)
    bh = np.ascontiguousarray(_host(beta)[0], dtype=np.float32)
    cu = np.ascontiguousarray(_host(cu_seqlens)[0], dtype=np.int32)
    s0 = None if init_state is None else np.ascontiguousarray(_host(init_state)[0], dtype=np.float32)
    T, H, dk = qh.shape
    dv = vh.shape[2]
    N = cu.shape[0] - 1
    out = np.zeros((T, H, dv), dtype=np.float64)
    fin = np.zeros((N, H, dk, dv), dtype=np.float64) if want_final else None
    nthr = threads if threads is not None else (os.cpu_count() or 1)
    rc = _lib(mutant, lib_path).kda_oracle_recurrent(N, _ptr(cu), H, dk, dv, int(qb), _ptr(qh), _ptr(kh), _ptr(vh),
                                                     _ptr(gh), _ptr(bh), _ptr(s0), _ptr(out), _ptr(fin), nthr)
    if rc != 0:
        raise ValueError(f"kda_oracle_recurrent rejected its arguments (rc={rc})")
    return out, fin


def _f64(x):
    if x is None:
        return None
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


def unrolled_bruteforce(q, k, v, g, beta, S0=None):
    """KDA for one (sequence, head) as explicit products of transition matrices.

    With M_t = (I - beta_t k_t k_t^T) Diag(exp g_t), the recurrence unrolls to
    S_t = M_t...M_1 S_0 + sum_{i<=t} M_t...M_{i+1} beta_i k_i v_i^T, and
    o_t = S_t^T q_t.  Every S_t is rebuilt from scratch from the products, so no
    state is carried from one token to the next.  Meant for T <= 8.
    Shapes: q, k, g [T, dk]; v [T, dv]; beta [T]; S0 [dk, dv] or None."""
    q, k, v, g, beta = map(_f64, (q, k, v, g, beta))
    T, dk = k.shape
    dv = v.shape[1]
    S0 = np.zeros((dk, dv)) if S0 is None else _f64(S0)
    I = np.eye(dk)
    M = [(I - beta[t] * np.outer(k[t], k[t])) @ np.diag(np.exp(g[t])) for t in range(T)]

    def prod(t, i):  # M_t ... M_{i+1} (1-based t; i < t), identity when i == t
        P = I.copy()
        for j in range(i + 1, t + 1):
            P = M[j - 1] @ P
        return P

    out = np.zeros((T, dv))
    S = S0
    for t in range(1, T + 1):
        S = prod(t, 0) @ S0
        for i in range(1, t + 1):
            S = S + prod(t, i) @ (beta[i - 1] * np.outer(k[i - 1], v[i - 1]))
        out[t - 1] = S.T @ q[t - 1]
    return out, S


def chunkwise_naive(q, k, v, g, beta, S0=None, chunk: int = 64):
    """Chunkwise-parallel KDA for one (sequence, head), plain fp64 numpy.

    Within a chunk of n tokens with state S on entry and Gamma_r the inclusive
    prefix sum of g over the chunk (per key channel):
      A[r,i]  = beta_r sum_c k_r[c] k_i[c] exp(Gamma_r[c] - Gamma_i[c]),  i < r
      P[r,i]  =        sum_c q_r[c] k_i[c] exp(Gamma_r[c] - Gamma_i[c]),  i <= r
      Tinv    = (I + A)^-1
      U       = Tinv diag(beta) V,   Wk = Tinv diag(beta) (K * exp Gamma)
      W       = U - Wk S
      O       = (Q * exp Gamma) S + P W
      S_next  = Diag(exp Gamma_n) S + (K * exp(Gamma_n - Gamma))^T W
    The decay between two tokens is taken directly as one exponential of the
    difference, and the inverse is numpy's dense inverse.  The last chunk of a
    sequence may be shorter than ``chunk``.
    Returns (out [T, dv], S_final [dk, dv])."""
    q, k, v, g, beta = map(_f64, (q, k, v, g, beta))
    T, dk = k.shape
    dv = v.shape[1]
    S = np.zeros((dk, dv)) if S0 is None else _f64(S0).copy()
    out = np.zeros((T, dv))
    for s in range(0, T, chunk):
        e = min(T, s + chunk)
        n = e - s
        Gam = np.cumsum(g[s:e], axis=0)
        diff = Gam[:, None, :] - Gam[None, :, :]                    # [r, i, c]
        lower = np.tril(np.ones((n, n), dtype=bool))                 # i <= r
        dec = np.exp(np.where(lower[:, :, None], diff, -np.inf))     # 0 above the diagonal
        kk = np.einsum("rc,ic,ric->ri", k[s:e], k[s:e], dec)
        A = beta[s:e, None] * np.tril(kk, -1)
        P = np.einsum("rc,ic,ric->ri", q[s:e], k[s:e], dec)
        Tinv = np.linalg.inv(np.eye(n) + A)
        U = Tinv @ (beta[s:e, None] * v[s:e])
        Wk = Tinv @ (beta[s:e, None] * (k[s:e] * np.exp(Gam)))
        W = U - Wk @ S
        out[s:e] = (q[s:e] * np.exp(Gam)) @ S + P @ W
        S = np.exp(Gam[-1])[:, None] * S + (k[s:e] * np.exp(Gam[-1][None, :] - Gam)).T @ W
    return out, S


# Input prologue bits, as in the C ABI's KDA_PROLOGUE_* (restated here: the oracle shares
# no header with the library).
PROLOGUE_QK_L2NORM = 1
PROLOGUE_G_LOGITS = 2
PROLOGUE_BETA_LOGITS = 4
G_MIN = -5.0          # the bound on the log-decay (llm-atlas Q06 and Figure 3)
L2_EPS = 1e-12


def sigmoid64(y) -> np.ndarray:
    """1 / (1 + e^-y) in fp64, without overflow for large |y|."""
    y = np.asarray(y, dtype=np.float64)
    e = np.exp(-np.abs(y))
    return np.where(y >= 0, 1.0 / (1.0 + e), e / (1.0 + e))


def l2_normalise64(x) -> np.ndarray:
    """x / max(||x||_2, 1e-12) over the last axis, in fp64."""
    x = np.asarray(x, dtype=np.float64)
    n = np.sqrt(np.sum(x * x, axis=-1, keepdims=True))
    return x / np.maximum(n, L2_EPS)


def prologue(inputs: dict, flags: int) -> dict:
    """The workloads' input recipe applied to raw inputs, as the library's prologue bits ask:
    q and k L2-normalised per (token, head) over dk in fp64 and rounded to their storage
    type (bf16 stays bf16, fp32 stays fp32); g = g_min * sigmoid(z); beta = sigmoid(y), both
    in fp64 and then stored as fp32 like every g and beta.  Returns a new dict of CPU torch
    tensors in the storage types.  The recipe is the benchmark workloads' (q, k ~ N(0,1)
    then L2-normalised per (token, head), beta = sigmoid(N(0,1)), g = -5 sigmoid(N(0,1)));
    -5 is the pages' bound on the log-decay.  Test infrastructure: the oracle side of the
    prologue parity tests."""
    import torch
    out = dict(inputs)
    if flags & PROLOGUE_QK_L2NORM:
        for name in ("q", "k"):
            t = inputs[name].detach().to("cpu")
            n64 = l2_normalise64(t.to(torch.float64).numpy())
            out[name] = torch.from_numpy(n64).to(t.dtype)
    if flags & PROLOGUE_G_LOGITS:
        z = inputs["g"].detach().to("cpu", torch.float64).numpy()
        out["g"] = torch.from_numpy(G_MIN * sigmoid64(z)).to(torch.float32)
    if flags & PROLOGUE_BETA_LOGITS:
        y = inputs["beta"].detach().to("cpu", torch.float64).numpy()
        out["beta"] = torch.from_numpy(sigmoid64(y)).to(torch.float32)
    return out


def output_gate(out, z) -> np.ndarray:
    """The output gate: o * sigmoid(z) elementwise over the read-out channels, in fp64.

    llm-atlas "K3_RESEARCH.md", question ledger Q08: KDA's output gate is input-dependent and
    full-rank over the read-out channels; the pages give no formula.  Read here as an
    elementwise sigmoid gate on the fp32 attention output o (the recurrence's o_t = S_t^T q_t),
    with the logits z of the same shape supplied by the caller (their projection is outside
    the attention).  The state is not touched."""
    return _f64(out) * sigmoid64(_f64(z))


def delta_invariant_keys(dk: int, n: int, seed: int = 0) -> np.ndarray:
    """n <= dk orthonormal keys (rows), from a QR factorisation of a seeded Gaussian matrix."""
    rng = np.random.default_rng(seed)
    Qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    return Qm.T[:n].copy()


def rel_err(x, ref) -> float:
    """max |x - ref| / RMS(ref), the error measure of the parity bar."""
    x = _f64(x)
    ref = _f64(ref)
    if ref.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(ref * ref)))
    if rms == 0.0:
        return float(np.max(np.abs(x - ref))) if x.size else 0.0
    return float(np.max(np.abs(x - ref)) / rms) if x.size else 0.0
