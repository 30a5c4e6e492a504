"""Build the PN CUDA library in-tree: ``bit_weight_only_pn_gb300/libpn_gb300.so``.

Each translation unit in ``csrc/`` is compiled for sm_103a in parallel, then
linked into one shared library with the CUDA runtime linked statically, so the
library loads without any other CUDA shared object.  Objects go to
``bit_weight_only_pn_gb300/_build/``.  Rebuilds only what is out of date.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIBRARY = os.path.join(HERE, "libpn_gb300.so")
SOURCES = ["pn_capi.cu", "pn_codec.cu", "pn_gemv_ffma.cu", "pn_gemv_simt.cu", "pn_gemv_stream.cu", "pn_gemv_tc.cu",
           "pn_gptq.cu", "pn_noalloc.cu", "pn_prefill.cu", "pn_probe.cu", "pn_rotate.cu"]
HEADERS = ["pn_device.cuh", "pn_internal.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _newer(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str, extra=()) -> str:
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
    deps = [os.path.join(CSRC, src)] + [os.path.join(CSRC, h) for h in HEADERS] + \
        [os.path.join(ROOT, "include", "pn.h")]
    if _newer(obj, deps):
        cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{res.stdout}\n{res.stderr}")
    return obj


def build(verbose: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as pool:
        objs = list(pool.map(_compile, SOURCES))
    if _newer(LIBRARY, objs):
        tmp = LIBRARY + ".tmp"
        cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
        os.replace(tmp, LIBRARY)
    if verbose:
        print(LIBRARY)
    return LIBRARY


if __name__ == "__main__":
    build(verbose="-q" not in sys.argv)
