"""Builds libpa.so, the CUDA library behind the C ABI in include/pa.h, in-tree.

nvcc compiles each translation unit for sm_103a in parallel (one -gencode, no other
architectures), then links a shared library with the static CUDA runtime.  The
library lands next to this file; build objects go to ``_build/``.
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
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libpa.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = [
    "pa_decode_bf16_d128.cu",
    "pa_decode_f16_d128.cu",
    "pa_decode_bf16_d64.cu",
    "pa_decode_f16_d64.cu",
    "pa_decode_fp8.cu",
    "pa_decode_mq_f16.cu",
    "pa_decode_mq_bf16.cu",
    "pa_decode_tc.cu",
    "pa_aux.cu",
    "pa_noalloc.cu",
    "pa_host.cpp",
    "pa_alloc.cpp",
]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpa.so")


def _newest_input() -> float:
    paths = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    paths += [os.path.join(ROOT, "include", "pa.h"), os.path.abspath(__file__)]
    return max(os.path.getmtime(p) for p in paths if os.path.exists(p))


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False,
          defines: tuple = (), out: str | None = None) -> str:
    """Compile (if stale) and return the path of libpa.so.

    ``defines`` (e.g. ``("PA_CORE_CONSUMERS=4",)``) and ``out`` build a variant of the
    library elsewhere for tuning sweeps; the default build ignores both."""
    lib = out or LIB
    build_dir = BUILD if not defines else os.path.join(BUILD, "variant_" + "_".join(defines))
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= _newest_input():
        return lib
    nvcc = _nvcc()
    os.makedirs(build_dir, exist_ok=True)
    common = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                     "-I", os.path.join(ROOT, "include"), "-I", CSRC]
    common += ["-D" + d for d in defines]
    if ptxas_info:
        common += ["-Xptxas", "-v"]

    def compile_one(src: str) -> str:
        obj = os.path.join(build_dir, src + ".o")
        cmd = [nvcc] + common + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0 or verbose or ptxas_info:
            sys.stderr.write(r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}")
        return obj

    with ThreadPoolExecutor(max_workers=min(len(SOURCES), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs + ["-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError("nvcc link of libpa.so failed")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv))
