"""Build libpkv.so in-tree with nvcc for sm_103a (translation units compiled in parallel)."""
from __future__ import annotations

import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libpkv.so")
SOURCES = ["pkv_host.cu", "append_rope.cu", "decode_partial.cu", "combine.cu", "decode_noalloc.cu", "qkv_append.cu", "prefill.cu"]
ARCH = "103a"


def nvcc() -> str:
    return shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"


def compile_flags(extra=()):
    return ["-O3", "-std=c++17", f"-gencode=arch=compute_{ARCH},code=sm_{ARCH}", "-lineinfo",
            "-Xcompiler", "-fPIC", "-I", os.path.join(ROOT, "include"), *extra]


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(ROOT, "include", "pkv.h")]
    return any(os.path.getmtime(p) > t for p in deps)


def build(verbose: bool = False, extra=()) -> str:
    os.makedirs(BUILD, exist_ok=True)
    objs, procs = [], []
    for src in SOURCES:
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        objs.append(obj)
        cmd = [nvcc(), *compile_flags(extra), "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd))
        procs.append(subprocess.Popen(cmd))
    if any(p.wait() for p in procs):
        raise RuntimeError("nvcc failed while building libpkv.so")
    tmp = LIB + ".tmp"
    link = [nvcc(), "-shared", f"-gencode=arch=compute_{ARCH},code=sm_{ARCH}", "-cudart", "shared", *objs,
            "-o", tmp, "-Xlinker", "-rpath,/usr/local/cuda/lib64"]
    subprocess.run(link, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(verbose=True)
