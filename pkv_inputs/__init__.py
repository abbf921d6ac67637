"""Seeded synthetic inputs shared by the oracle side and the CUDA side.

This package holds no arithmetic of the attention method.  It provides:

* a counter-based generator (SplitMix64 words, Irwin-Hall normals rounded to
  fp16) with a host implementation (``hostgen.c``) and a bit-identical device
  implementation (``devgen.cu``) for filling multi-GB pools in HBM;
* the workload table and the construction of one decode step's inputs
  (sequence lengths, page tables, positions, the cache state before the step),
  in :mod:`pkv_inputs.workloads`.

The shared libraries are built in-tree by :func:`build`.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
HOST_LIB = os.path.join(_HERE, "libpkvgen_host.so")
DEV_LIB = os.path.join(_HERE, "libpkvgen_dev.so")

GAMMA = 0x9E3779B97F4A7C15
MASK64 = (1 << 64) - 1


def build_commands(nvcc: str = "nvcc", arch: str = "103a"):
    """Commands that build both generator libraries (run in parallel by callers)."""
    host = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
            os.path.join(_HERE, "hostgen.c"), "-o", HOST_LIB]
    dev = [nvcc, "-O3", "-std=c++17", "-shared", "-Xcompiler", "-fPIC", "-cudart", "shared",
           f"-gencode=arch=compute_{arch},code=sm_{arch}",
           os.path.join(_HERE, "devgen.cu"), "-o", DEV_LIB,
           "-Xlinker", "-rpath,/usr/local/cuda/lib64"]
    return [host, dev]


def build(nvcc: str = "nvcc") -> None:
    procs = [subprocess.Popen(c) for c in build_commands(nvcc)]
    rcs = [p.wait() for p in procs]
    if any(rcs):
        raise RuntimeError(f"pkv_inputs build failed: return codes {rcs}")


_host = None
_dev = None


def _host_lib():
    global _host
    if _host is None:
        if not os.path.exists(HOST_LIB):
            raise RuntimeError(f"{HOST_LIB} is missing: run pkv_inputs.build()")
        lib = ctypes.CDLL(HOST_LIB)
        u64, i64, f32, ip = ctypes.c_uint64, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p
        lib.pkvgen_key.restype = u64
        lib.pkvgen_key.argtypes = [u64, u64]
        lib.pkvgen_word.restype = u64
        lib.pkvgen_word.argtypes = [u64, u64]
        lib.pkvgen_fill_range.restype = None
        lib.pkvgen_fill_range.argtypes = [ip, i64, u64, i64, f32, u64, i64, ctypes.c_int]
        lib.pkvgen_fill_blocks.restype = None
        lib.pkvgen_fill_blocks.argtypes = [ip, ip, i64, i64, u64, f32, u64, i64, ctypes.c_int]
        lib.pkvgen_words.restype = None
        lib.pkvgen_words.argtypes = [ip, i64, u64, i64]
        _host = lib
    return _host


def _dev_lib():
    global _dev
    if _dev is None:
        if not os.path.exists(DEV_LIB):
            raise RuntimeError(f"{DEV_LIB} is missing: run pkv_inputs.build()")
        lib = ctypes.CDLL(DEV_LIB)
        lib.pkvgen_dev_fill_range.restype = ctypes.c_int
        lib.pkvgen_dev_fill_range.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64,
                                              ctypes.c_int64, ctypes.c_float, ctypes.c_uint64,
                                              ctypes.c_int64, ctypes.c_int, ctypes.c_void_p]
        _dev = lib
    return _dev


def key(seed: int, tag: int) -> int:
    return int(_host_lib().pkvgen_key(seed & MASK64, tag & MASK64))


def words(k: int, n: int, first: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    if n:
        _host_lib().pkvgen_words(out.ctypes.data, n, k & MASK64, first)
    return out


def fill_range(n: int, k: int, first: int = 0, scale: float = 1.0, okey: int = 0,
               row_len: int = 0, pct: int = 0) -> np.ndarray:
    """fp16 bit patterns (uint16) of value(first .. first+n-1)."""
    out = np.empty(n, dtype=np.uint16)
    if n:
        _host_lib().pkvgen_fill_range(out.ctypes.data, n, k & MASK64, first, float(np.float32(scale)),
                                      okey & MASK64, max(row_len, 1), pct)
    return out


def fill_blocks(blocks: np.ndarray, block_elems: int, k: int, scale: float = 1.0, okey: int = 0,
                row_len: int = 0, pct: int = 0) -> np.ndarray:
    """Rows value(b*block_elems .. +block_elems) for each listed block b (uint16 [n, block_elems])."""
    blocks = np.ascontiguousarray(blocks, dtype=np.int64)
    out = np.empty((blocks.size, block_elems), dtype=np.uint16)
    if blocks.size:
        _host_lib().pkvgen_fill_blocks(out.ctypes.data, blocks.ctypes.data, blocks.size, block_elems,
                                       k & MASK64, float(np.float32(scale)), okey & MASK64,
                                       max(row_len, 1), pct)
    return out


def dev_fill_range(ptr: int, n: int, k: int, first: int = 0, scale: float = 1.0, okey: int = 0,
                   row_len: int = 0, pct: int = 0, stream: int = 0) -> None:
    """Device twin of :func:`fill_range`, writing n fp16 values at device address ``ptr``."""
    rc = _dev_lib().pkvgen_dev_fill_range(ptr, n, k & MASK64, first, float(np.float32(scale)),
                                          okey & MASK64, max(row_len, 1), pct, stream)
    if rc != 0:
        raise RuntimeError(f"pkvgen_dev_fill_range failed with cudaError {rc}")
