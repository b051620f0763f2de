"""Build the sm_103a CUDA library in-tree with nvcc.

    python -m decode_context_mla_dcp_gb300.build [--force]

The library lands in decode_context_mla_dcp_gb300/_build/ (git-ignored). It is
one translation unit compiled for sm_103a only; the CUDA runtime is linked
statically so the library needs nothing beyond the driver at run time.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
SOURCES = [os.path.join(PKG, "csrc", name) for name in ("dcp_lse_reduce.cu", "mla_decode_partial.cu")]
HEADERS = [os.path.join(ROOT, "include", "dcp_lse_reduce.h"), os.path.join(ROOT, "include", "dcp_mla_decode.h")]
BUILD_DIR = os.path.join(PKG, "_build")
LIB_NAME = "libdcp_lse_reduce.so"
LIB_PATH = os.path.join(BUILD_DIR, LIB_NAME)

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC,-O2", "-shared",
    "-cudart", "static",
]


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is needed to build the sm_103a library")


def is_stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(s) > t for s in SOURCES + HEADERS + [os.path.abspath(__file__)])


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not is_stale():
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    tag = f".tmp{os.getpid()}"
    objs = [os.path.join(BUILD_DIR, os.path.basename(src) + tag + ".o") for src in SOURCES]
    compile_flags = [f for f in NVCC_FLAGS if f != "-shared"]
    procs = []
    for src, obj in zip(SOURCES, objs):
        cmd = [nvcc_path(), *compile_flags, "-I", os.path.join(ROOT, "include"), "-c", "-o", obj, src]
        if verbose:
            print(" ".join(cmd), flush=True)
        procs.append((cmd, subprocess.Popen(cmd)))
    for cmd, pr in procs:
        if pr.wait() != 0:
            raise subprocess.CalledProcessError(pr.returncode, cmd)
    tmp = LIB_PATH + tag
    cmd = [nvcc_path(), "-gencode", "arch=compute_103a,code=sm_103a", "-shared", "-cudart", "static", "-o", tmp,
           *objs]
    if verbose:
        print(" ".join(cmd), flush=True)
    subprocess.run(cmd, check=True)
    for obj in objs:
        os.remove(obj)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
