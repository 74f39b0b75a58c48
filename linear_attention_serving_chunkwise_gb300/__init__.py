"""Kimi Delta Attention (KDA) on one GB300: chunkwise prefill and fused decode.

The compute lives in the CUDA library ``libkda_gb300.so`` behind the C ABI in
``include/kda.h``; this package is the thin ctypes binding over it.
"""
from ._lib import (  # noqa: F401
    EXPORTED,
    KDA_ABI_VERSION,
    KDA_BF16,
    KDA_DECODE_MULTI_MAX_TOKENS,
    KDA_ERR_CUDA,
    KDA_ERR_INVALID_ARG,
    KDA_ERR_TIMEOUT,
    KDA_ERR_UNSUPPORTED,
    KDA_ERR_WORKSPACE,
    KDA_F32,
    KDA_OK,
    KDA_PROLOGUE_ALL,
    KDA_PROLOGUE_BETA_LOGITS,
    KDA_PROLOGUE_G_LOGITS,
    KDA_PROLOGUE_QK_L2NORM,
    KDA_STATIC_SCRATCH_BYTES,
    KDAError,
    LIB_PATH,
    PrefillDesc,
    decode,
    decode_multi,
    last_device_status,
    load,
    make_desc,
    prefill,
    prefill_host,
    prefill_host_static,
    prefill_host_workspace_bytes,
    prefill_query,
    prefill_workspace_bytes,
    state_combine,
    status_string,
)
