"""ctypes binding of the KDA C ABI (include/kda.h).

Argument marshalling only: every step of prefill and decode runs in the CUDA
library ``libkda_gb300.so``.  PyTorch supplies device memory and streams.  There
is no fallback: if the library is missing or fails to load, calls raise.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkda_gb300.so")

KDA_OK = 0
KDA_ERR_INVALID_ARG = -1
KDA_ERR_UNSUPPORTED = -2
KDA_ERR_WORKSPACE = -3
KDA_ERR_CUDA = -4
KDA_ERR_TIMEOUT = -5
KDA_F32 = 0
KDA_BF16 = 1
KDA_ABI_VERSION = 3
# input prologue bits (include/kda.h): q/k L2 normalisation, g = -5 sigmoid(z), beta = sigmoid(y)
KDA_PROLOGUE_QK_L2NORM = 1
KDA_PROLOGUE_G_LOGITS = 2
KDA_PROLOGUE_BETA_LOGITS = 4
KDA_PROLOGUE_ALL = 7

# Every symbol include/kda.h declares.
EXPORTED = ("kda_abi_version", "kda_status_string", "kda_prefill_workspace_bytes", "kda_prefill_query",
            "kda_prefill", "kda_prefill_gated", "kda_prefill_checkpointed", "kda_prefill_host_workspace_bytes",
            "kda_prefill_host", "kda_prefill_host_static", "kda_decode", "kda_decode_gated", "kda_decode_multi",
            "kda_decode_multi_gated", "kda_state_combine", "kda_last_device_status")
KDA_DECODE_MULTI_MAX_TOKENS = 64
KDA_STATIC_SCRATCH_BYTES = 64 << 20


class KDAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


class PrefillDesc(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("total_tokens", ctypes.c_int32), ("num_heads", ctypes.c_int32),
                ("dk", ctypes.c_int32), ("dv", ctypes.c_int32), ("qkv_dtype", ctypes.c_int32),
                ("prologue", ctypes.c_int32)]


class PrefillPlan(ctypes.Structure):
    _fields_ = [("kernel_launches", ctypes.c_int32), ("tensor_cores", ctypes.c_int32),
                ("workspace_bytes", ctypes.c_size_t)]


_lib = None


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load the CUDA library (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"KDA CUDA library not built ({p} missing): run "
                           "`python -m linear_attention_serving_chunkwise_gb300.build`")
    lib = ctypes.CDLL(p)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    lib.kda_abi_version.restype = i32
    lib.kda_abi_version.argtypes = []
    lib.kda_status_string.restype = ctypes.c_char_p
    lib.kda_status_string.argtypes = [ctypes.c_int]
    lib.kda_prefill_workspace_bytes.restype = sz
    lib.kda_prefill_workspace_bytes.argtypes = [ctypes.POINTER(PrefillDesc)]
    lib.kda_prefill_query.restype = ctypes.c_int
    lib.kda_prefill_query.argtypes = [ctypes.POINTER(PrefillDesc), ctypes.POINTER(PrefillPlan)]
    lib.kda_prefill.restype = ctypes.c_int
    lib.kda_prefill.argtypes = [ctypes.POINTER(PrefillDesc), vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.kda_prefill_gated.restype = ctypes.c_int
    lib.kda_prefill_gated.argtypes = [ctypes.POINTER(PrefillDesc), vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.kda_prefill_checkpointed.restype = ctypes.c_int
    lib.kda_prefill_checkpointed.argtypes = [ctypes.POINTER(PrefillDesc), vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                             i32, i32, vp, vp, sz, vp]
    lib.kda_prefill_host_workspace_bytes.restype = sz
    lib.kda_prefill_host_workspace_bytes.argtypes = [ctypes.POINTER(PrefillDesc), i32]
    lib.kda_prefill_host.restype = ctypes.c_int
    lib.kda_prefill_host.argtypes = [ctypes.POINTER(PrefillDesc), vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, sz,
                                     vp]
    lib.kda_prefill_host_static.restype = ctypes.c_int
    lib.kda_prefill_host_static.argtypes = [ctypes.POINTER(PrefillDesc), vp, vp, vp, vp, vp, vp, vp, vp, vp, i32,
                                            vp]
    lib.kda_decode.restype = ctypes.c_int
    lib.kda_decode.argtypes = [i32, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.kda_decode_gated.restype = ctypes.c_int
    lib.kda_decode_gated.argtypes = [i32, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.kda_decode_multi.restype = ctypes.c_int
    lib.kda_decode_multi.argtypes = [i32, i32, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.kda_decode_multi_gated.restype = ctypes.c_int
    lib.kda_decode_multi_gated.argtypes = [i32, i32, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                           vp]
    lib.kda_state_combine.restype = ctypes.c_int
    lib.kda_state_combine.argtypes = [i32, i32, i32, vp, vp, vp, vp, vp]
    lib.kda_last_device_status.restype = ctypes.c_int
    lib.kda_last_device_status.argtypes = [vp]
    if path is None:
        _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().kda_status_string(int(status)).decode()


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return KDA_BF16
    if t.dtype == torch.float32:
        return KDA_F32
    raise TypeError(f"q/k/v must be float32 or bfloat16, got {t.dtype}")


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("KDA tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr()) if t.numel() > 0 else None


def _stream_handle(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _keep_until_done(tensor: torch.Tensor, stream) -> None:
    """A scratch tensor this module allocated on the current stream and the library uses on
    ``stream``: tell the caching allocator, so that the memory is not handed to another
    allocation before that stream's work is done."""
    if stream is not None and stream != torch.cuda.current_stream(tensor.device):
        tensor.record_stream(stream)


def make_desc(num_seqs: int, total_tokens: int, num_heads: int, dk: int, dv: int, qkv_dtype: int,
              prologue: int = 0) -> PrefillDesc:
    return PrefillDesc(int(num_seqs), int(total_tokens), int(num_heads), int(dk), int(dv), int(qkv_dtype),
                       int(prologue))


def prefill_workspace_bytes(desc: PrefillDesc) -> int:
    return int(load().kda_prefill_workspace_bytes(ctypes.byref(desc)))


def prefill_query(desc: PrefillDesc) -> dict:
    """What one kda_prefill call for ``desc`` will launch (host only)."""
    plan = PrefillPlan()
    st = load().kda_prefill_query(ctypes.byref(desc), ctypes.byref(plan))
    if st != KDA_OK:
        raise KDAError(st, "kda_prefill_query")
    return {"kernel_launches": plan.kernel_launches, "tensor_cores": plan.tensor_cores,
            "workspace_bytes": plan.workspace_bytes}


def prefill(q, k, v, g, beta, cu_seqlens=None, init_state=None, out=None, final_state=None, *,
            num_seqs: Optional[int] = None, want_final: bool = True, workspace=None, stream=None, check=True,
            checkpoint_interval: int = 0, checkpoint_slots: int = 0, checkpoints=None, prologue: int = 0,
            gate=None):
    """KDA prefill through ``kda_prefill`` (``kda_prefill_gated`` when ``gate`` is given).

    q, k [T,H,dk], v [T,H,dv] (fp32 or bf16); g [T,H,dk] fp32; beta [T,H] fp32;
    cu_seqlens [N+1] int32 on the device, or None with ``num_seqs`` equal
    sequences (default 1); init_state [N,H,dk,dv] fp32 or None.
    ``out``/``final_state`` are allocated if not given (``final_state`` may be
    ``init_state`` for in-place chaining).  ``prologue``: KDA_PROLOGUE_* bits (q, k, g and
    beta then hold the raw values of the input recipe).  ``gate``: output gate logits
    [T,H,dv] fp32 (out = o * sigmoid(gate)), not combined with checkpoints.  Returns
    (out, final_state)."""
    T, H, dk = q.shape
    dv = v.shape[2]
    N = (cu_seqlens.numel() - 1) if cu_seqlens is not None else (1 if num_seqs is None else int(num_seqs))
    desc = make_desc(N, T, H, dk, dv, _dtype_code(q), prologue)
    if out is None:
        out = torch.empty((T, H, dv), dtype=torch.float32, device=q.device)
        _keep_until_done(out, stream)
    if final_state is None and want_final:
        final_state = torch.empty((N, H, dk, dv), dtype=torch.float32, device=q.device)
        _keep_until_done(final_state, stream)
    need = prefill_workspace_bytes(desc)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        _keep_until_done(workspace, stream)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if checkpoint_interval:
        if gate is not None:
            raise ValueError("the output gate is not offered with checkpoints")
        if checkpoints is None:
            checkpoints = torch.zeros((N, H, checkpoint_slots, dk, dv), dtype=torch.float32, device=q.device)
            _keep_until_done(checkpoints, stream)
        st = load().kda_prefill_checkpointed(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                             _ptr(cu_seqlens), _ptr(init_state), _ptr(out), _ptr(final_state),
                                             int(checkpoint_interval), int(checkpoint_slots), _ptr(checkpoints),
                                             _ptr(workspace), ws_bytes, _stream_handle(stream))
        if check and st != KDA_OK:
            raise KDAError(st, "kda_prefill_checkpointed")
        return out, final_state, checkpoints
    if gate is not None:
        st = load().kda_prefill_gated(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(gate),
                                      _ptr(cu_seqlens), _ptr(init_state), _ptr(out), _ptr(final_state),
                                      _ptr(workspace), ws_bytes, _stream_handle(stream))
        if check and st != KDA_OK:
            raise KDAError(st, "kda_prefill_gated")
        return out, final_state
    st = load().kda_prefill(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu_seqlens),
                            _ptr(init_state), _ptr(out), _ptr(final_state), _ptr(workspace), ws_bytes,
                            _stream_handle(stream))
    if check and st != KDA_OK:
        raise KDAError(st, "kda_prefill")
    return out, final_state


def prefill_host_workspace_bytes(desc: PrefillDesc, segment_tokens: int) -> int:
    return int(load().kda_prefill_host_workspace_bytes(ctypes.byref(desc), int(segment_tokens)))


def prefill_host(q, k, v, g, beta, cu_seqlens=None, init_state=None, out=None, final_state=None, *,
                 segment_tokens: int = 1024, num_seqs: Optional[int] = None, want_final: bool = True,
                 workspace=None, stream=None, check=True, device=None, prologue: int = 0):
    """KDA prefill through ``kda_prefill_host``: every tensor is a CPU tensor (pinned for
    the copies to overlap the kernels); ``workspace`` is a CUDA uint8 tensor, allocated if
    not given.  Asynchronous like the other entry points: the results are in ``out`` /
    ``final_state`` once ``stream`` (default: the current stream) has been synchronised.
    Returns (out, final_state)."""
    T, H, dk = q.shape
    dv = v.shape[2]
    N = (cu_seqlens.numel() - 1) if cu_seqlens is not None else (1 if num_seqs is None else int(num_seqs))
    desc = make_desc(N, T, H, dk, dv, _dtype_code(q), prologue)
    pin = q.is_pinned()
    if out is None:
        out = torch.empty((T, H, dv), dtype=torch.float32, pin_memory=pin)
    if final_state is None and want_final:
        final_state = torch.empty((N, H, dk, dv), dtype=torch.float32, pin_memory=pin)
    if workspace is None:
        need = prefill_host_workspace_bytes(desc, segment_tokens)
        dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
        _keep_until_done(workspace, stream)
    ws_bytes = workspace.numel() * workspace.element_size()
    st = load().kda_prefill_host(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                 _ptr(cu_seqlens), _ptr(init_state), _ptr(out), _ptr(final_state),
                                 int(segment_tokens), ctypes.c_void_p(workspace.data_ptr()), ws_bytes,
                                 _stream_handle(stream))
    if check and st != KDA_OK:
        raise KDAError(st, "kda_prefill_host")
    return out, final_state


def prefill_host_static(q, k, v, g, beta, cu_seqlens=None, init_state=None, out=None, final_state=None, *,
                        segment_tokens: int = 128, num_seqs: Optional[int] = None, want_final: bool = True,
                        stream=None, check=True, prologue: int = 0):
    """``prefill_host`` through ``kda_prefill_host_static``: the device staging is the
    library's own scratch (no workspace, no device allocation).  Returns (out, final_state)."""
    T, H, dk = q.shape
    dv = v.shape[2]
    N = (cu_seqlens.numel() - 1) if cu_seqlens is not None else (1 if num_seqs is None else int(num_seqs))
    desc = make_desc(N, T, H, dk, dv, _dtype_code(q), prologue)
    pin = q.is_pinned()
    if out is None:
        out = torch.empty((T, H, dv), dtype=torch.float32, pin_memory=pin)
    if final_state is None and want_final:
        final_state = torch.empty((N, H, dk, dv), dtype=torch.float32, pin_memory=pin)
    st = load().kda_prefill_host_static(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                        _ptr(cu_seqlens), _ptr(init_state), _ptr(out), _ptr(final_state),
                                        int(segment_tokens), _stream_handle(stream))
    if check and st != KDA_OK:
        raise KDAError(st, "kda_prefill_host_static")
    return out, final_state


def decode(q, k, v, g, beta, state, out=None, *, stream=None, check=True, prologue: int = 0, gate=None):
    """One KDA decode step through ``kda_decode`` (``kda_decode_gated`` with ``gate``);
    ``state`` [B,H,dk,dv] fp32 is updated in place.

    q, k [B,H,dk], v [B,H,dv] (fp32 or bf16); g [B,H,dk] fp32; beta [B,H] fp32;
    ``prologue``: KDA_PROLOGUE_* bits; ``gate``: output gate logits [B,H,dv] fp32.
    Returns out [B,H,dv] fp32."""
    B, H, dk = q.shape
    dv = v.shape[2]
    if out is None:
        out = torch.empty((B, H, dv), dtype=torch.float32, device=q.device)
        _keep_until_done(out, stream)
    if gate is not None:
        st = load().kda_decode_gated(B, H, dk, dv, _dtype_code(q), int(prologue), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                     _ptr(beta), _ptr(gate), _ptr(state), _ptr(out), _stream_handle(stream))
        if check and st != KDA_OK:
            raise KDAError(st, "kda_decode_gated")
        return out
    st = load().kda_decode(B, H, dk, dv, _dtype_code(q), int(prologue), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                           _ptr(state), _ptr(out), _stream_handle(stream))
    if check and st != KDA_OK:
        raise KDAError(st, "kda_decode")
    return out


def decode_multi(q, k, v, g, beta, state, out=None, n_apply=None, *, want_out=True, stream=None, check=True,
                 prologue: int = 0, gate=None):
    """K tokens per sequence through ``kda_decode_multi``: q, k [B,K,H,dk], v [B,K,H,dv]
    (fp32 or bf16); g [B,K,H,dk] fp32; beta [B,K,H] fp32; ``state`` [B,H,dk,dv] fp32 is
    replaced by the state after the first ``n_apply[b]`` tokens (int32 [B] on the device;
    None = all K); ``prologue``: KDA_PROLOGUE_* bits.  Returns out [B,K,H,dv] fp32 (None
    when ``want_out`` is False).  ``gate``: output gate logits [B,K,H,dv] fp32 (through
    ``kda_decode_multi_gated``)."""
    B, K, H, dk = q.shape
    dv = v.shape[3]
    if out is None and want_out:
        out = torch.empty((B, K, H, dv), dtype=torch.float32, device=q.device)
        _keep_until_done(out, stream)
    if gate is not None:
        st = load().kda_decode_multi_gated(B, K, H, dk, dv, _dtype_code(q), int(prologue), _ptr(q), _ptr(k), _ptr(v),
                                           _ptr(g), _ptr(beta), _ptr(gate), _ptr(n_apply), _ptr(state), _ptr(out),
                                           _stream_handle(stream))
        if check and st != KDA_OK:
            raise KDAError(st, "kda_decode_multi_gated")
        return out
    st = load().kda_decode_multi(B, K, H, dk, dv, _dtype_code(q), int(prologue), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                 _ptr(beta),
                                 _ptr(n_apply), _ptr(state), _ptr(out), _stream_handle(stream))
    if check and st != KDA_OK:
        raise KDAError(st, "kda_decode_multi")
    return out


def state_combine(transition, state_in, state_add, out=None, *, stream=None, check=True):
    """out = transition @ state_in + state_add per (sequence, head), through
    ``kda_state_combine``: transition [..., dk, dk], states [..., dk, dv] fp32 on the device
    (state_in or state_add may be None = zero; ``out`` may be ``state_add``).  Returns out."""
    ref = state_add if state_add is not None else state_in
    dk, dv = ref.shape[-2], ref.shape[-1]
    count = ref.numel() // (dk * dv)
    if out is None:
        out = torch.empty_like(ref)
        _keep_until_done(out, stream)
    st = load().kda_state_combine(count, dk, dv, _ptr(transition), _ptr(state_in), _ptr(state_add), _ptr(out),
                                  _stream_handle(stream))
    if check and st != KDA_OK:
        raise KDAError(st, "kda_state_combine")
    return out


def last_device_status(stream=None) -> int:
    return int(load().kda_last_device_status(_stream_handle(stream)))
