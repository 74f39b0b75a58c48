"""Per-phase cycle tables of the tensor-core prefill kernels, from an instrumented build.

``python -m linear_attention_serving_chunkwise_gb300.phase_clocks`` builds
``libkda_gb300_clocks.so`` (the library with KDA_PHASE_CLOCKS defined: thread 0 of CTA 0
adds clock64() cycles between marks in its loop to a device array), runs a prefill shape on
each tensor-core path twice (``--prologue``: also the chunk-parallel path's prologue
instances on raw draws), and prints the cycles of each span per item (chunk prep), per
chunk (state scan) and per chunk (one CTA per (sequence, head)), averaged over what CTA 0 ran
in the second call.  CTA 0 of the single cooperative launch preps items, then scans its unit,
so both of its tables come from one CTA.  The instrumented library is a measuring tool only;
the marks cost a few cycles each, and everything else loads the uninstrumented library.
"""
from __future__ import annotations

import ctypes
import sys

import torch

from . import _lib
from .build import build

TC_SPANS = ["inputs in (loop top)", "phase 1: token rows, off-diagonal rows (the first chunk: cumsum, factors)",
            "A/P tf32 MMA, K~ alongside", "A/P read-out", "solve (state operand and seed alongside)",
            "Tb operands, M = P Tb, [Tb; M] hi/lo", "[Wk; -Q'] MMA, the next chunk's cumsum alongside",
            "[-Wk; Q'] hi/lo operands", "S half of D1 (state lo and decay, the next chunk's factors alongside)", "W hi/lo",
            "state update, O staged",
            "checkpoint, O stores issued"]
PREP_SPANS = ["loop top: claims, beta", "off-diagonal rows", "A/P tf32 MMA, K~ staged alongside", "A/P read-out",
              "solve (seed, image stores, publication alongside)", "Tb operands", "M = P Tb, Tb rows",
              "M rows, [Tb; M] staged", "next item's phase 1 under the [Wk; -Q'] MMA", "wait for that MMA",
              "[-Wk; Q'] hi, Q' lo staged"]
SCAN_SPANS = ["waited for the last update", "S^T_hi into tensor memory", "gamma_C waited for, S^T_lo and the decay",
              "waited for D1", "W^T split into tensor memory", "O read out and stored"]


def _measure(lib, reader, seqlens, heads, prologue=0):
    """The marks of the second of two calls on one shape (with `prologue`, on the recipe's raw
    draws and the kernels' prologue instances)."""
    import kda_workloads as W
    cfg = W.PrefillConfig("clocks", tuple(seqlens), heads, 128, 128, torch.bfloat16, "normal")
    d = W.make_prefill_inputs(cfg, seed=0, device="cuda", raw=bool(prologue))
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], d["init_state"])
    out, fin = _lib.prefill(*args, prologue=prologue)
    torch.cuda.synchronize()
    _read(lib, reader)
    _lib.prefill(*args, out=out, final_state=fin, prologue=prologue)
    torch.cuda.synchronize()
    if _lib.last_device_status() != _lib.KDA_OK:
        raise RuntimeError("the instrumented prefill reported a device error")
    return _read(lib, reader)


def _read(lib, name):
    buf = (ctypes.c_ulonglong * 32)()
    if getattr(lib, name)(buf) != 0:
        raise RuntimeError(f"{name} failed")
    return list(buf)


def _table(title, vals, spans, first, count_slot):
    n = vals[count_slot]
    if n == 0:
        print(f"{title}: nothing ran on CTA 0")
        return
    print(f"{title} (cycles per unit of work, {n} on CTA 0)")
    total = 0
    for i, name in enumerate(spans):
        c = vals[first + i] / n
        total += c
        print(f"  {name:60s} {c / 1e3:6.2f} K")
    print(f"  {'total':60s} {total / 1e3:6.2f} K")


def main(argv=None):
    sys.path.insert(0, __import__("os").path.dirname(__import__("os").path.dirname(__file__)))
    lib_path = build(phase_clocks=True)
    _lib.LIB_PATH = lib_path
    lib = _lib.load()
    for n in ("kda_phase_clocks_tc", "kda_phase_clocks_split"):
        getattr(lib, n).restype = ctypes.c_int
        getattr(lib, n).argtypes = [ctypes.c_void_p]
    # the chunk-parallel path: B=1, H=96, T=8192 (one cooperative launch)
    v = _measure(lib, "kda_phase_clocks_split", [8192], 96)
    print("chunk-parallel path, B=1 H=96 T=8192, dk=dv=128 bf16 (single cooperative launch, CTA 0)")
    _table("chunk prep, per item", v, PREP_SPANS, 0, 31)
    _table("state scan, per chunk", v, SCAN_SPANS, 16, 30)
    if "--prologue" in (argv if argv is not None else sys.argv[1:]):
        v = _measure(lib, "kda_phase_clocks_split", [8192], 96, prologue=_lib.KDA_PROLOGUE_ALL)
        print("the same with the input prologue (raw draws, every prologue bit)")
        _table("chunk prep, per item", v, PREP_SPANS, 0, 31)
        _table("state scan, per chunk", v, SCAN_SPANS, 16, 30)
    # the same path as separate prep and scan launches (124 units): the scan's table without
    # waits on items still being prepared
    v = _measure(lib, "kda_phase_clocks_split", [8192], 124)
    print("chunk-parallel path, B=1 H=124 T=8192 (separate prep and scan launches, CTA 0 of each)")
    _table("state scan, per chunk", v, SCAN_SPANS, 16, 30)
    # one CTA per unit: 4 sequences x 2048 tokens, H=38 (152 units, one wave)
    v = _measure(lib, "kda_phase_clocks_tc", [2048] * 4, 38)
    print("one CTA per (sequence, head), 4 x 2048 tokens, H=38, dk=dv=128 bf16 (CTA 0)")
    _table("per chunk", v, TC_SPANS, 0, 31)


if __name__ == "__main__":
    main()
