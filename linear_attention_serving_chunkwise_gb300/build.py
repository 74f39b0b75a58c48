"""Build the KDA CUDA library in-tree for sm_103a with nvcc (no cmake, no torch extension).

``python -m linear_attention_serving_chunkwise_gb300.build`` or ``build()`` compiles each
``csrc/*.cu`` translation unit in parallel and links ``libkda_gb300.so`` beside this file.
``build(phase_clocks=True)`` builds a separate instrumented library,
``libkda_gb300_clocks.so``, with the per-phase cycle marks compiled in (see phase_clocks.py);
the library everything else loads never has them.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
OBJ = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libkda_gb300.so")
OBJ_CLOCKS = os.path.join(PKG, "_build_clocks")
LIB_CLOCKS = os.path.join(PKG, "libkda_gb300_clocks.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the KDA library needs the CUDA 13 toolkit to build")


def _cuda_lib_dir(nvcc: str) -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "lib64")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        [os.path.join(os.path.dirname(PKG), "include", "kda.h")]


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(force: bool = False, verbose: bool = False, ptxas_v: bool = False, phase_clocks: bool = False) -> str:
    lib_path, obj_dir = (LIB_CLOCKS, OBJ_CLOCKS) if phase_clocks else (LIB, OBJ)
    if not force and up_to_date(lib_path):
        return lib_path
    nvcc = _nvcc()
    os.makedirs(obj_dir, exist_ok=True)
    common = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
                     "--expt-relaxed-constexpr", "-I", os.path.join(os.path.dirname(PKG), "include")]
    if phase_clocks:
        common += ["-DKDA_PHASE_CLOCKS"]
    if ptxas_v:
        common += ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(obj_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc] + common + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0 or verbose or ptxas_v:
            sys.stderr.write(r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}")
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(8, len(_sources()))) as ex:
        objs = list(ex.map(compile_one, _sources()))
    libdir = _cuda_lib_dir(nvcc)
    cmd = [nvcc] + ARCH + ["-shared", "-cudart", "shared", "-o", lib_path + ".tmp"] + objs + \
        ["-Xlinker", f"-rpath,{libdir}", "-L", libdir]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError(f"linking {os.path.basename(lib_path)} failed")
    os.replace(lib_path + ".tmp", lib_path)
    return lib_path


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv, ptxas_v="--ptxas-v" in sys.argv)
    print(LIB)
