"""Build libradixattn.so in-tree: CUDA kernels for sm_103a plus the host C++ radix tree.

    python -m prefix_cached_kv_radix_gb300.build [--force] [-v]

Translation units compile in parallel; the result is prefix_cached_kv_radix_gb300/_build/
libradixattn.so (git-ignored).  nvcc: -gencode arch=compute_103a,code=sm_103a -O3 -lineinfo.  Also
_build/_rxstep*.so, the per-step call's marshalling as a CPython extension, where the Python
headers are installed.
"""
from __future__ import annotations

import argparse
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_build")
LIB_NAME = "libradixattn.so"
LIB_PATH = os.path.join(OUT_DIR, LIB_NAME)

CU_SOURCES = ["kv_pool_write.cu", "attention_simt.cu", "extend_attention.cu", "decode_attention.cu", "step_runtime.cu",
              "wait_selftest.cu"]
CPP_SOURCES = ["radix_tree.cpp"]
GENCODE = "arch=compute_103a,code=sm_103a"
# the per-step marshalling as a CPython extension (optional: the ctypes binding does the same)
PYSTEP_SRC = "pystep.c"


def pystep_path() -> str:
    import sysconfig
    return os.path.join(OUT_DIR, "_rxstep" + (sysconfig.get_config_var("EXT_SUFFIX") or ".so"))


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libradixattn.so")


def _headers():
    hs = [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    hs += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    return hs


def _stale(obj: str, src: str) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(p) > t for p in [src, *_headers(), __file__])


def _run(cmd, verbose):
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"build failed: {' '.join(cmd)}\n{r.stdout}")
    if verbose and r.stdout.strip():
        print(r.stdout, flush=True)
    return r.stdout


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False) -> str:
    os.makedirs(OUT_DIR, exist_ok=True)
    nv = nvcc()
    jobs = []
    objs = []
    for f in CU_SOURCES:
        src = os.path.join(CSRC, f)
        obj = os.path.join(OUT_DIR, f + ".o")
        objs.append(obj)
        if force or _stale(obj, src):
            cmd = [nv, "-gencode", GENCODE, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                   "-I", INCLUDE, "-I", CSRC, "-c", src, "-o", obj]
            if ptxas_verbose:
                cmd[1:1] = ["-Xptxas", "-v"]
            jobs.append(cmd)
    for f in CPP_SOURCES:
        src = os.path.join(CSRC, f)
        obj = os.path.join(OUT_DIR, f + ".o")
        objs.append(obj)
        if force or _stale(obj, src):
            jobs.append(["g++", "-O3", "-std=c++17", "-fPIC", "-Wall", "-I", INCLUDE, "-I", CSRC,
                         "-c", src, "-o", obj])
    if jobs:
        with ThreadPoolExecutor(max_workers=len(jobs)) as ex:
            outs = list(ex.map(lambda c: _run(c, verbose), jobs))
        if ptxas_verbose:
            for o in outs:
                print(o)
    if jobs or not os.path.exists(LIB_PATH):
        tmp = LIB_PATH + f".tmp{os.getpid()}"
        _run([nv, "-shared", "-gencode", GENCODE, "-o", tmp, *objs, "-lcudart_static", "-lrt", "-lpthread",
              "-ldl"], verbose)
        os.replace(tmp, LIB_PATH)
    build_pystep(force, verbose)
    return LIB_PATH


def build_pystep(force: bool = False, verbose: bool = False) -> str | None:
    """The _rxstep extension next to the library, when the Python headers are installed."""
    import sysconfig
    inc = sysconfig.get_paths().get("include")
    if not inc or not os.path.exists(os.path.join(inc, "Python.h")):
        return None
    src, out = os.path.join(CSRC, PYSTEP_SRC), pystep_path()
    if force or _stale(out, src):
        tmp = out + f".tmp{os.getpid()}"
        _run(["gcc", "-O2", "-shared", "-fPIC", "-Wall", "-I", inc, "-I", INCLUDE, src, "-o", tmp], verbose)
        os.replace(tmp, out)
    return out


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("-v", "--verbose", action="store_true")
    ap.add_argument("--ptxas", action="store_true", help="print register/smem usage (-Xptxas -v)")
    a = ap.parse_args()
    print(build(a.force, a.verbose, a.ptxas))
    sys.exit(0)
