"""Builds the layer's shared library (libmoe.so) in-tree with nvcc for sm_103a.

    python -m mixture_experts_layer_gb300.build [--force]

Each .cu file compiles in parallel to an object under csrc/_build/, then nvcc
links them into mixture_experts_layer_gb300/libmoe.so with the CUDA runtime
linked statically and only the C ABI exported.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(CSRC, "_build")
LIB = os.path.join(PKG, "libmoe.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["plan.cu", "rows.cu", "gemm.cu", "moe_abi.cu"]
HEADERS = ["common.cuh", "kernels.cuh"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmoe.so")


def _inputs() -> list[str]:
    return ([os.path.join(CSRC, s) for s in SOURCES + HEADERS]
            + [os.path.join(ROOT, "include", "moe.h"), os.path.abspath(__file__)])


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _inputs())


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("command failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    return r.stdout + r.stderr


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False, defines=(), out: str = LIB) -> str:
    """Compiles the library (libmoe.so by default) if any source is newer than it; returns its path.

    defines: extra preprocessor macros, for diagnosis builds written to another
    file (e.g. MOE_TIMELINE into libmoe_timeline.so); the product build has none."""
    if not force and up_to_date(out):
        return out
    bdir = BUILD if not defines else BUILD + "_" + "_".join(d.lower() for d in defines)
    os.makedirs(bdir, exist_ok=True)
    cc = nvcc()
    common = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden",
                     "-I" + os.path.join(ROOT, "include")] + ["-D" + d for d in defines]
    if ptxas_info:
        common += ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(bdir, src.replace(".cu", ".o"))
        out = _run([cc] + common + ["-c", os.path.join(CSRC, src), "-o", obj])
        return obj, out

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose or ptxas_info:
        for obj, out in results:
            if out.strip():
                print(f"== {os.path.basename(obj)}\n{out}")
    tmp = out + ".tmp"
    _run([cc] + ARCH + ["-shared", "-cudart", "static", "-Xlinker", "--exclude-libs,ALL", "-o", tmp]
         + [o for o, _ in results])
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv)
    print(LIB)
