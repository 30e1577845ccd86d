"""Build liblapl_attn.so (sm_103a) in-tree with nvcc.

Each translation unit under csrc/ is compiled in parallel to an object file, then linked into
``liblapl_attn.so`` beside this file.  Only ``-gencode arch=compute_103a,code=sm_103a`` is
emitted.  Objects live in ``_build/`` (git-ignored) and are rebuilt only when a source or
header is newer.
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
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(HERE, "liblapl_attn.so")

SOURCES = ["api.cu", "pool.cu", "ns.cu", "cdist.cu", "cdist_d32.cu", "cdist_d64.cu", "cdist_d0.cu",
           "cdist_gauss_d32.cu", "cdist_gauss_d64.cu", "cdist_gauss_d0.cu",
           "cdist_tma_f32.cu", "cdist_tma_bf16.cu", "cdist_l1.cu", "cdist_l1_bf16.cu",
           "cdist_gauss_tc.cu", "chain.cu", "bv_tc.cu", "out_tc.cu", "noalloc.cu", "ns_tc.cu", "cg.cu", "backward.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build liblapl_attn")
    return path


def _headers():
    hs = [os.path.join(INCLUDE, "lapl_attn.h")]
    hs += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    return hs


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(dp) > t for dp in deps)


def _compile(src: str, extra) -> str:
    obj = os.path.join(BUILD, os.path.basename(src) + ".o")
    if _stale(obj, [src, *_headers(), __file__]):
        cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj + ".tmp"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        os.replace(obj + ".tmp", obj)
    return obj


def build(verbose: bool = False, extra=(), force: bool = False) -> str:
    """Compile and link; return the path of liblapl_attn.so."""
    os.makedirs(BUILD, exist_ok=True)
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    if force:
        for s in srcs:
            o = os.path.join(BUILD, os.path.basename(s) + ".o")
            if os.path.exists(o):
                os.remove(o)
    with cf.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        objs = list(ex.map(lambda s: _compile(s, list(extra)), srcs))
    if _stale(LIB, objs):
        tmp = LIB + f".{os.getpid()}.tmp"
        cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
    if verbose:
        print(LIB)
    return LIB


if __name__ == "__main__":
    extra = sys.argv[1:]
    build(verbose=True, extra=extra)
