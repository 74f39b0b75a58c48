"""The C-ABI library loads and exports every symbol include/kda.h declares; host-side
argument checks return their codes before anything reaches a GPU (CPU only)."""
import ctypes
import os
import re

import pytest

import linear_attention_serving_chunkwise_gb300 as kda
from linear_attention_serving_chunkwise_gb300 import _lib
from linear_attention_serving_chunkwise_gb300.build import LIB, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build()
    return kda.load()


def _declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(kda_[a-z0-9_]+)\s*\(", src))
    return names


def test_every_declared_symbol_is_exported(lib):
    declared = _declared_functions()
    assert {"kda_prefill", "kda_decode", "kda_prefill_workspace_bytes"} <= declared
    for name in declared:
        assert hasattr(lib, name), name
    assert set(_lib.EXPORTED) == declared


def test_abi_version_and_status_strings(lib):
    assert lib.kda_abi_version() == kda.KDA_ABI_VERSION == 3
    for code in (0, -1, -2, -3, -4, -5):
        assert kda.status_string(code).startswith("KDA")
    assert "unknown" in kda.status_string(-99)


def _fake(addr):
    # host-side validation never dereferences these
    return ctypes.c_void_p(addr)


def _prefill(lib, desc, q=0x10000, k=0x20000, v=0x30000, g=0x40000, beta=0x50000, cu=None, s0=None,
             out=0x60000, fin=None, ws=None, ws_bytes=0):
    p = lambda a: None if a is None else _fake(a)
    return lib.kda_prefill(ctypes.byref(desc) if desc is not None else None, p(q), p(k), p(v), p(g), p(beta),
                           p(cu), p(s0), p(out), p(fin), p(ws), ws_bytes, None)


def test_prefill_rejects_bad_arguments_on_host(lib):
    d = kda.make_desc(1, 64, 2, 64, 64, kda.KDA_F32)
    assert _prefill(lib, None) == kda.KDA_ERR_INVALID_ARG
    assert _prefill(lib, kda.make_desc(1, 64, 2, 96, 96, kda.KDA_F32)) == kda.KDA_ERR_UNSUPPORTED
    assert _prefill(lib, kda.make_desc(1, 64, 2, 128, 64, kda.KDA_F32)) == kda.KDA_ERR_UNSUPPORTED
    assert _prefill(lib, kda.make_desc(1, 64, 2, 64, 64, 7)) == kda.KDA_ERR_UNSUPPORTED
    assert _prefill(lib, kda.make_desc(-1, 64, 2, 64, 64, 0)) == kda.KDA_ERR_INVALID_ARG
    assert _prefill(lib, kda.make_desc(1, 64, 0, 64, 64, 0)) == kda.KDA_ERR_INVALID_ARG
    assert _prefill(lib, kda.make_desc(0, 64, 2, 64, 64, 0)) == kda.KDA_ERR_INVALID_ARG
    # equal split needs T % N == 0
    assert _prefill(lib, kda.make_desc(3, 64, 2, 64, 64, 0)) == kda.KDA_ERR_INVALID_ARG
    # null required pointer
    assert _prefill(lib, d, q=None) == kda.KDA_ERR_INVALID_ARG
    assert _prefill(lib, d, out=None) == kda.KDA_ERR_INVALID_ARG
    # misaligned pointer
    assert _prefill(lib, d, k=0x20008) == kda.KDA_ERR_INVALID_ARG
    # out aliasing an input
    assert _prefill(lib, d, out=0x10000) == kda.KDA_ERR_INVALID_ARG
    # final_state overlapping out
    assert _prefill(lib, d, fin=0x60000 + 64) == kda.KDA_ERR_INVALID_ARG
    # nothing to do: zero sequences
    assert _prefill(lib, kda.make_desc(0, 0, 2, 64, 64, 0)) == kda.KDA_OK
    # the input prologue: any of its three bits, nothing else
    assert _prefill(lib, kda.make_desc(0, 0, 2, 64, 64, 0, kda.KDA_PROLOGUE_ALL)) == kda.KDA_OK
    assert _prefill(lib, kda.make_desc(1, 64, 2, 64, 64, 0, 8)) == kda.KDA_ERR_INVALID_ARG
    assert _prefill(lib, kda.make_desc(1, 64, 2, 64, 64, 0, -1)) == kda.KDA_ERR_INVALID_ARG
    with pytest.raises(kda.KDAError):
        kda.prefill_query(kda.make_desc(1, 64, 2, 64, 64, 0, 16))
    # the prologue does not change the plan
    for dt, d in ((kda.KDA_BF16, 128), (kda.KDA_F32, 64)):
        assert kda.prefill_query(kda.make_desc(1, 8192, 96, d, d, dt)) == \
            kda.prefill_query(kda.make_desc(1, 8192, 96, d, d, dt, kda.KDA_PROLOGUE_ALL))


def test_workspace_query(lib):
    d = kda.make_desc(4, 1000, 8, 128, 128, kda.KDA_BF16)
    n = kda.prefill_workspace_bytes(d)
    assert n >= 0
    assert kda.prefill_workspace_bytes(kda.make_desc(4, 1000, 8, 96, 96, kda.KDA_BF16)) == 0
    if n > 0:
        assert _prefill(lib, d, ws=0x70000, ws_bytes=n - 1) == kda.KDA_ERR_WORKSPACE


def test_prefill_query(lib):
    plan = kda.prefill_query(kda.make_desc(1, 8192, 96, 128, 128, kda.KDA_BF16))
    assert plan["kernel_launches"] >= 1 and plan["workspace_bytes"] >= 0
    assert kda.prefill_query(kda.make_desc(0, 0, 4, 64, 64, kda.KDA_F32))["kernel_launches"] == 0
    with pytest.raises(kda.KDAError):
        kda.prefill_query(kda.make_desc(1, 10, 4, 96, 96, kda.KDA_F32))


def test_prefill_path_selection_and_split_workspace(lib):
    """bf16, dk = dv = 128: the three-launch chunk-parallel path where its cost estimate beats
    one CTA per (sequence, head) and its items fit the workspace cap (32768); its workspace
    holds the chunk offsets, the chunk table and 115,200 bytes of operands per item.
    Otherwise one launch, no workspace."""
    def plan(N, T, H, dt=kda.KDA_BF16, d=128):
        return kda.prefill_query(kda.make_desc(N, T, H, d, d, dt))
    p = plan(1, 8192, 96)
    items = (8192 // 64 + 1) * 96
    assert p["kernel_launches"] == 2 and p["tensor_cores"] == 1   # offsets + one cooperative launch
    assert items * 115200 <= p["workspace_bytes"] <= items * 115200 + items * 4 + 4096
    assert plan(1, 8192, 112)["kernel_launches"] == 2
    assert plan(1, 8192, 120)["kernel_launches"] == 2                # the last single launch
    assert plan(1, 8192, 124)["kernel_launches"] == 3                # split, separate launches
    assert plan(1, 8192, 128)["kernel_launches"] == 3                # split, separate launches
    assert plan(1, 8192, 136)["kernel_launches"] == 3                # split, separate launches
    assert plan(1, 8192, 144)["kernel_launches"] == 1 and plan(1, 8192, 144)["workspace_bytes"] == 0
    assert plan(2, 8192, 64)["kernel_launches"] == 3                 # 128 units of 4096 tokens
    assert plan(1, 8192, 152)["kernel_launches"] == 1                # one full wave
    assert plan(1, 8192, 160)["kernel_launches"] == 3                # a second wave of 8: separate launches
    assert plan(1, 8192, 240)["kernel_launches"] == 3                # a second wave of 88
    assert plan(2, 8192, 76)["kernel_launches"] == 1                 # one full wave
    assert plan(40, 8000, 3)["kernel_launches"] == 1                 # 120 short sequences
    assert plan(1, 64 * 400, 96)["kernel_launches"] == 1             # 38,496 items: over the cap
    assert plan(1, 8192, 96, kda.KDA_F32)["kernel_launches"] == 1    # fp32 inputs: CUDA-core kernel
    assert plan(1, 8192, 96, d=64)["kernel_launches"] == 1


def test_split_workspace_rejected_on_host(lib):
    d = kda.make_desc(1, 200, 2, 128, 128, kda.KDA_BF16)
    n = kda.prefill_workspace_bytes(d)
    assert n > 0
    assert _prefill(lib, d, ws=None, ws_bytes=n) == kda.KDA_ERR_INVALID_ARG           # missing
    assert _prefill(lib, d, ws=0x1000008, ws_bytes=n) == kda.KDA_ERR_INVALID_ARG      # misaligned
    assert _prefill(lib, d, ws=0x10000, ws_bytes=n) == kda.KDA_ERR_INVALID_ARG        # over q
    assert _prefill(lib, d, ws=0x60000 - 256, ws_bytes=n) == kda.KDA_ERR_INVALID_ARG  # over out


def test_decode_rejects_bad_arguments_on_host(lib):
    f = _fake
    args = lambda **kw: [kw.get(n, f(a)) for n, a in
                         (("q", 0x10000), ("k", 0x20000), ("v", 0x30000), ("g", 0x40000), ("beta", 0x50000),
                          ("state", 0x100000), ("out", 0x60000))]
    assert lib.kda_decode(2, 2, 96, 96, 0, 0, *args(), None) == kda.KDA_ERR_UNSUPPORTED
    assert lib.kda_decode(2, 2, 64, 64, 5, 0, *args(), None) == kda.KDA_ERR_UNSUPPORTED
    assert lib.kda_decode(-1, 2, 64, 64, 0, 0, *args(), None) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_decode(2, 2, 64, 64, 0, 0, *args(q=None), None) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_decode(2, 2, 64, 64, 0, 0, *args(out=f(0x100000)), None) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_decode(2, 2, 64, 64, 0, 0, *args(g=f(0x40004)), None) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_decode(0, 2, 64, 64, 0, 0, *args(), None) == kda.KDA_OK
    assert lib.kda_decode(2, 2, 64, 64, 0, 8, *args(), None) == kda.KDA_ERR_INVALID_ARG   # unknown prologue bit
    assert lib.kda_decode(0, 2, 64, 64, 0, kda.KDA_PROLOGUE_ALL, *args(), None) == kda.KDA_OK


def test_library_is_in_tree():
    assert os.path.dirname(LIB) == os.path.dirname(_lib.__file__)


def _host_call(lib, desc, seg, cu=None, ws=0x100000, ws_bytes=1 << 40, init=None, fin=None):
    import numpy as np
    T, H, dk, dv = desc.total_tokens, desc.num_heads, desc.dk, desc.dv
    arrs = {n: np.zeros(max(T, 1) * H * d, dtype=np.float32) for n, d in
            (("q", dk), ("k", dk), ("v", dv), ("g", dk), ("out", dv))}
    beta = np.zeros(max(T, 1) * H, dtype=np.float32)
    p = lambda a: None if a is None else a.ctypes.data_as(ctypes.c_void_p)
    return lib.kda_prefill_host(ctypes.byref(desc), p(arrs["q"]), p(arrs["k"]), p(arrs["v"]), p(arrs["g"]), p(beta),
                                p(cu), p(init), p(arrs["out"]), p(fin), seg, _fake(ws), ws_bytes, None)


def test_prefill_host_rejects_bad_arguments_on_host(lib):
    """kda_prefill_host checks everything on the host before its first CUDA call."""
    import numpy as np
    d = kda.make_desc(2, 256, 2, 64, 64, kda.KDA_F32)
    need = kda.prefill_host_workspace_bytes(d, 128)
    assert need > 0
    for seg in (0, -64, 100, 65):
        assert _host_call(lib, d, seg, ws_bytes=need) == kda.KDA_ERR_INVALID_ARG
    assert _host_call(lib, d, 128, ws_bytes=need - 1) == kda.KDA_ERR_WORKSPACE
    assert _host_call(lib, d, 128, ws=0x100010, ws_bytes=need) == kda.KDA_ERR_INVALID_ARG   # misaligned
    bad_cu = [np.array([0, 200, 100], dtype=np.int32), np.array([1, 100, 256], dtype=np.int32),
              np.array([0, 100, 255], dtype=np.int32)]
    for cu in bad_cu:
        assert _host_call(lib, d, 128, cu=cu, ws_bytes=need) == kda.KDA_ERR_INVALID_ARG
    assert _host_call(lib, kda.make_desc(3, 256, 2, 64, 64, kda.KDA_F32), 128, ws_bytes=1 << 40) == \
        kda.KDA_ERR_INVALID_ARG   # equal split needs T % N == 0
    assert _host_call(lib, kda.make_desc(1, 64, 2, 96, 96, kda.KDA_F32), 128) == kda.KDA_ERR_UNSUPPORTED
    # final_state overlapping the initial state (but not identical) is rejected
    st = np.zeros(2 * 2 * 64 * 64 + 16, dtype=np.float32)
    init = st[:2 * 2 * 64 * 64]
    fin = st[16:]
    assert _host_call(lib, d, 128, ws_bytes=need, init=init, fin=fin) == kda.KDA_ERR_INVALID_ARG
    assert _host_call(lib, kda.make_desc(0, 0, 2, 64, 64, kda.KDA_F32), 128) == kda.KDA_OK
    # unknown prologue bits are rejected before any copy; the known ones pass the checks
    assert _host_call(lib, kda.make_desc(2, 256, 2, 64, 64, kda.KDA_F32, 8), 128, ws_bytes=need) == \
        kda.KDA_ERR_INVALID_ARG
    assert kda.prefill_host_workspace_bytes(kda.make_desc(2, 256, 2, 64, 64, kda.KDA_F32, kda.KDA_PROLOGUE_ALL),
                                            128) == need
    assert _host_call(lib, kda.make_desc(0, 0, 2, 64, 64, kda.KDA_F32, kda.KDA_PROLOGUE_ALL), 128) == kda.KDA_OK


def test_prefill_host_workspace_bytes():
    d = kda.make_desc(2, 1000, 4, 128, 128, kda.KDA_BF16)
    state = 2 * 4 * 128 * 128 * 4
    per_token = 4 * (2 * 128 * 2 + 128 * 2 + 128 * 4 + 4 + 128 * 4)
    w64, w128, w4k = (kda.prefill_host_workspace_bytes(d, s) for s in (64, 128, 4096))
    assert w64 >= state + 2 * 128 * per_token and w128 >= state + 2 * 256 * per_token
    assert w64 < w128 < w4k
    assert w4k >= state + 2 * 1000 * per_token          # a round never holds more than all tokens
    assert w4k < state + 2 * 1000 * per_token + 64 * 1024
    assert kda.prefill_host_workspace_bytes(d, 100) == 0


def test_decode_multi_rejects_bad_arguments_on_host(lib):
    f = _fake
    base = dict(q=f(0x10000), k=f(0x20000), v=f(0x30000), g=f(0x40000), beta=f(0x50000), n=None,
                state=f(0x100000), out=f(0x60000))
    call = lambda B=2, K=2, H=2, d=64, dt=0, pro=0, **kw: lib.kda_decode_multi(
        B, K, H, d, d, dt, pro, *[kw.get(n, base[n]) for n in ("q", "k", "v", "g", "beta", "n", "state", "out")],
        None)
    assert call(K=0) == kda.KDA_ERR_INVALID_ARG
    assert call(K=kda.KDA_DECODE_MULTI_MAX_TOKENS + 1) == kda.KDA_ERR_INVALID_ARG
    assert call(d=96) == kda.KDA_ERR_UNSUPPORTED
    assert call(dt=5) == kda.KDA_ERR_UNSUPPORTED
    assert call(q=None) == kda.KDA_ERR_INVALID_ARG
    assert call(n=f(0x70002)) == kda.KDA_ERR_INVALID_ARG          # misaligned counts
    assert call(out=f(0x100000)) == kda.KDA_ERR_INVALID_ARG       # out over the state
    assert call(state=f(0x10000 + 64)) == kda.KDA_ERR_INVALID_ARG  # state over q
    assert call(B=0) == kda.KDA_OK
    assert call(pro=-1) == kda.KDA_ERR_INVALID_ARG                 # unknown prologue bits
    assert call(B=0, pro=kda.KDA_PROLOGUE_ALL) == kda.KDA_OK


def test_gated_entry_points_reject_bad_gates_on_host(lib):
    """The output gate's pointer is checked like the other inputs before anything runs:
    16-byte alignment, and no overlap with out, final_state or the state."""
    d = kda.make_desc(1, 64, 2, 64, 64, kda.KDA_F32)
    p = _fake
    args = lambda gate, out=0x60000, fin=None: (ctypes.byref(d), p(0x10000), p(0x20000), p(0x30000), p(0x40000),
                                                 p(0x50000), None if gate is None else p(gate), None, None, p(out),
                                                 None if fin is None else p(fin), None, 0, None)
    assert lib.kda_prefill_gated(*args(0x70008)) == kda.KDA_ERR_INVALID_ARG            # misaligned
    assert lib.kda_prefill_gated(*args(0x60000 + 256)) == kda.KDA_ERR_INVALID_ARG      # inside out
    assert lib.kda_prefill_gated(*args(0x80000, fin=0x80000)) == kda.KDA_ERR_INVALID_ARG
    # decode: B=2, H=2, d=64 fp32; out at 0x60000 (1 KB), state at 0x90000 (64 KB)
    dec = lambda gate: lib.kda_decode_gated(2, 2, 64, 64, kda.KDA_F32, 0, p(0x10000), p(0x20000), p(0x30000),
                                            p(0x40000), p(0x50000), p(gate), p(0x90000), p(0x60000), None)
    assert dec(0x70004) == kda.KDA_ERR_INVALID_ARG
    assert dec(0x60000) == kda.KDA_ERR_INVALID_ARG
    assert dec(0x90000 + 4096) == kda.KDA_ERR_INVALID_ARG
    mul = lambda gate: lib.kda_decode_multi_gated(2, 3, 2, 64, 64, kda.KDA_F32, 0, p(0x10000), p(0x20000),
                                                  p(0x30000), p(0x40000), p(0x50000), p(gate), None, p(0x90000),
                                                  p(0x60000), None)
    assert mul(0x70004) == kda.KDA_ERR_INVALID_ARG
    assert mul(0x60000 + 512) == kda.KDA_ERR_INVALID_ARG
