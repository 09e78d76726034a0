"""Builds libpagedkv.so (the C-ABI library) in-tree with nvcc for sm_103a.

Each .cu translation unit compiles in parallel to an object file under
csrc/_build/, then nvcc links them into paged_kv_cache_fill_gb300/libpagedkv.so
(CUDA runtime linked statically; the driver's tensor-map encoder is fetched at
run time, so no libcuda link is needed). Rebuilds only what changed.

build(debug=True) makes the bounds-checking library instead: the same
sources compiled with PAGEDKV_DEBUG_BOUNDS into csrc/_build_debug/ and
linked as libpagedkv_debug.so (load it with
paged_kv_cache_fill_gb300.use_library before the first call).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(CSRC, "_build")
LIB = os.path.join(HERE, "libpagedkv.so")
OUT_DIR_DEBUG = os.path.join(CSRC, "_build_debug")
LIB_DEBUG = os.path.join(HERE, "libpagedkv_debug.so")
SOURCES = ["abi.cu", "kv_write.cu", "fused_k.cu", "decode.cu", "prefill.cu", "static_scratch.cu"]
HEADERS = ["common.cuh", "internal.h", "rope_tables.h", os.path.join("..", "..", "include", "pagedkv.h")]

NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "-prec-div=true", "-prec-sqrt=true", "-ftz=false"]


def _mtime(p: str) -> float:
    return os.path.getmtime(p) if os.path.exists(p) else -1.0


def _compile(src: str, verbose_ptxas: bool, debug: bool = False) -> str:
    obj = os.path.join(OUT_DIR_DEBUG if debug else OUT_DIR, src.replace(".cu", ".o"))
    deps = [os.path.join(CSRC, src)] + [os.path.join(CSRC, h) for h in HEADERS]
    if _mtime(obj) >= max(_mtime(d) for d in deps):
        return obj
    cmd = [NVCC, *ARCH, *FLAGS, *(["-DPAGEDKV_DEBUG_BOUNDS"] if debug else []), "-c", os.path.join(CSRC, src),
           "-o", obj]
    if verbose_ptxas:
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if verbose_ptxas:
        print(r.stderr)
    return obj


def build(verbose_ptxas: bool = False, debug: bool = False) -> str:
    out_dir, lib = (OUT_DIR_DEBUG, LIB_DEBUG) if debug else (OUT_DIR, LIB)
    os.makedirs(out_dir, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose_ptxas, debug), SOURCES))
    if _mtime(lib) < max(_mtime(o) for o in objs):
        tmp = lib + f".tmp{os.getpid()}"
        r = subprocess.run([NVCC, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    import sys
    print(build(verbose_ptxas=True, debug="--debug" in sys.argv[1:]))
