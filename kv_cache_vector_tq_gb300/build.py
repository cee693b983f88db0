"""Build libtq.so in-tree: nvcc for sm_103a, one object per translation unit, in parallel.

Usage: python -m kv_cache_vector_tq_gb300.build  (or call build()).
"""

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJ = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libtq.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]
SOURCES = ["tq_host.cpp", "tq_encode.cu", "tq_encode_wht.cu", "tq_encode_umma.cu", "tq_encode128.cu", "tq_scores.cu",
           "tq_decode.cu", "tq_decode_k1.cu", "tq_decode_k2.cu", "tq_decode_k3.cu", "tq_decode_k4.cu",
           "tq_decode_prod.cu", "tq_decode_mixed.cu"]


def _nvcc():
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _compile(src, verbose_ptxas=False):
    out = os.path.join(OBJ, os.path.splitext(src)[0] + ".o")
    cmd = [_nvcc(), "-c", os.path.join(CSRC, src), "-o", out] + ARCH + COMMON
    if src.endswith(".cpp"):
        cmd += ["-x", "cu"]
    if verbose_ptxas and src.endswith(".cu"):
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    return out, r.stderr


def build(verbose_ptxas=False, quiet=True):
    """Compile every CUDA/C++ source and link libtq.so (returns its path)."""
    os.makedirs(OBJ, exist_ok=True)
    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(lambda s: _compile(s, verbose_ptxas), SOURCES))
    objs = [o for o, _ in results]
    if verbose_ptxas and not quiet:
        for _, log in results:
            sys.stderr.write(log)
    tmp = LIB + ".tmp"
    cmd = [_nvcc(), "-shared", "-o", tmp] + objs + ARCH
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    v = "-v" in sys.argv
    print(build(verbose_ptxas=v, quiet=not v))
