"""Build libcsf.so in-tree for sm_103a (GB300).

Compiles the CUDA translation units in parallel with nvcc and links one shared
library next to this file.  `python -m lossless_nvfp4_scale_gb300.build`
rebuilds it; `ensure_built()` rebuilds only when a source is newer.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(HERE, "libcsf.so")
SOURCES = ["csf_api.cu", "csf_decode.cu", "csf_tiles.cu", "csf_tiled.cu", "csf_prepare.cu",
           "csf_prepare_static.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libcsf.so")


def _inputs():
    files = [os.path.join(CSRC, s) for s in SOURCES]
    files += [os.path.join(CSRC, "csf_internal.cuh"), os.path.join(CSRC, "csf_device.cuh"),
              os.path.join(INCLUDE, "csf.h"), os.path.join(INCLUDE, "csf_tile.cuh")]
    return files


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in _inputs())


def build(verbose: bool = False) -> str:
    cc = nvcc()
    tmpdir = tempfile.mkdtemp(prefix="csf_build_", dir=HERE)
    try:
        def compile_one(src):
            obj = os.path.join(tmpdir, src.replace(".cu", ".o"))
            cmd = [cc, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                   "-I", INCLUDE, "-c", os.path.join(CSRC, src), "-o", obj]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
            if verbose and (r.stdout or r.stderr):
                print(r.stdout + r.stderr, file=sys.stderr)
            return obj

        with cf.ThreadPoolExecutor(len(SOURCES)) as ex:
            objs = list(ex.map(compile_one, SOURCES))
        out_tmp = os.path.join(tmpdir, "libcsf.so")
        cmd = [cc, *ARCH, "-shared", "-cudart", "shared", *objs, "-o", out_tmp]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(out_tmp, LIB)
    finally:
        shutil.rmtree(tmpdir, ignore_errors=True)
    return LIB


def ensure_built() -> str:
    if stale():
        build()
    return LIB


if __name__ == "__main__":
    print(build(verbose=True))
