"""Builds the CUDA library ``_lib/libfm.so`` in-tree with nvcc for sm_103a.

Each translation unit is compiled in parallel; the CUDA runtime is linked
statically, so the library needs only the driver (libcuda) at run time and
loads on a machine without a GPU (for the ABI checks).  ``build(debug=True)``
builds the same sources with the FM_DEBUG definition (device-side checks that
report FM_ERR_DEBUG_CHECK) into ``_lib/debug/libfm_debug.so``; the binding
loads it when the FM_LIBRARY environment variable names it.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(HERE, "_lib")
LIB = os.path.join(OUT_DIR, "libfm.so")
DEBUG_DIR = os.path.join(OUT_DIR, "debug")
DEBUG_LIB = os.path.join(DEBUG_DIR, "libfm_debug.so")
SOURCES = ["fm_api.cu", "fm_classify.cu", "fm_fwd.cu", "fm_bwd.cu", "fm_fp8.cu", "fm_compress.cu", "fm_noalloc.cu", "fm_mask.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc():
    p = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(p):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libfm.so")
    return p


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "fm.h"),
                                                                 os.path.abspath(__file__)]
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    out_dir, lib = (DEBUG_DIR, DEBUG_LIB) if debug else (OUT_DIR, LIB)
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= _deps():
        return lib
    os.makedirs(out_dir, exist_ok=True)
    nvcc = _nvcc()
    common = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-fvisibility=hidden",
              "-I", INCLUDE, "-I", CSRC, *ARCH]
    if debug:
        common += ["-DFM_DEBUG"]
    if verbose:
        common += ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(out_dir, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc, *common, "-c", os.path.join(CSRC, src), "-o", obj]
        if src.endswith(".cpp"):
            cmd = [nvcc, "-x", "c++", *common, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose:
        for _, err in results:
            if err:
                print(err)
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-Xcompiler", "-fPIC", "-o", tmp, *[o for o, _ in results],
           "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    import sys
    print(build(force=True, verbose="-v" in sys.argv))
