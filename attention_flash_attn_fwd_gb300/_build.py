"""Build the sm_103a shared library ``libattn_gb300.so`` in-tree with nvcc.

Each ``csrc/*.cu`` translation unit is compiled in parallel for exactly one
target, ``-gencode arch=compute_103a,code=sm_103a``, then linked with the
shared CUDA runtime.  The result lands next to this file and is git-ignored.
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libattn_gb300.so")
SOURCES = ["attn_api.cu", "prefill_sm103a.cu", "decode_sm103a.cu", "attn_noalloc.cu",
           "backward_sm103a.cu", "mqa_logits_sm103a.cu"]
HEADERS = ["sm103a_ptx.cuh", "tmap.h", "host_once.h", "prefill_sm103a.h", "decode_sm103a.h",
           "backward_sm103a.h", "mqa_logits_sm103a.h", "decode_plan.h"]
GENCODE = "arch=compute_103a,code=sm_103a"


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build")
    return cand


def _cuda_lib_dir(nvcc: str) -> str:
    root = os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    for sub in ("lib64", "lib"):
        if os.path.isdir(os.path.join(root, sub)):
            return os.path.join(root, sub)
    return os.path.join(root, "lib64")


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    deps.append(os.path.join(HERE, "..", "include", "attn_gb300.h"))
    deps.append(os.path.abspath(__file__))
    return any(os.path.getmtime(d) > t for d in deps if os.path.exists(d))


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile (if stale) and return the path of ``libattn_gb300.so``."""
    if not force and not _stale():
        return LIB
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    flags = ["-gencode", GENCODE, "-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
             "--expt-relaxed-constexpr", "-Xcompiler", "-fvisibility=hidden"]
    if verbose:
        flags += ["-Xptxas", "-v"]

    def compile_one(src: str) -> str:
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        cmd = [nvcc, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed for %s:\n%s%s" % (src, r.stdout, r.stderr))
        if verbose:
            print(r.stdout + r.stderr)
        return obj

    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + ".tmp.%d" % os.getpid()
    libdir = _cuda_lib_dir(nvcc)
    cmd = [nvcc, "-shared", "-gencode", GENCODE, "-cudart", "shared", *objs, "-o", tmp,
           "-Xlinker", "-rpath," + libdir]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s%s" % (r.stdout, r.stderr))
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
