"""Oracle for the decode-step paged-KV attention path (TEST INFRASTRUCTURE ONLY).

A plain fp64 CPU implementation (``pkv_oracle.c``) of what the path computes,
written from the Zero TVM documentation ("KV cache", "Decode loop", "How it
works", "Port to Phi-4-mini or Qwen3").  Only the tests, the smoke check and
the bench's CPU baseline load it; the product library never does, and the two
share no code.  Every function here is a thin ctypes marshaller around the C
definitions; the arithmetic lives in ``pkv_oracle.c``.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB = os.environ.get("PKV_ORACLE_LIB") or os.path.join(_HERE, "liboracle.so")

ERRORS = {1: "invalid argument", 3: "out of range", 5: "duplicate position in one sequence"}


class OracleError(RuntimeError):
    def __init__(self, code: int):
        super().__init__(f"oracle rejected the input: {ERRORS.get(code, code)}")
        self.code = code


def build_command(source=None, target=None):
    return ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
            source or os.path.join(_HERE, "pkv_oracle.c"), "-o", target or LIB, "-lm"]


def build() -> None:
    subprocess.run(build_command(), check=True)


class Geom(ctypes.Structure):
    _fields_ = [("num_pages", ctypes.c_int), ("num_qo_heads", ctypes.c_int),
                ("num_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int),
                ("max_position", ctypes.c_int), ("rope_theta", ctypes.c_double)]


_lib = None


def _L():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise RuntimeError(f"{LIB} is missing: run oracle.build()")
        lib = ctypes.CDLL(LIB)
        P = ctypes.c_void_p
        i, d = ctypes.c_int, ctypes.c_double
        lib.orc_f16_to_f64.restype = d
        lib.orc_f16_to_f64.argtypes = [ctypes.c_uint16]
        lib.orc_f64_to_f16.restype = ctypes.c_uint16
        lib.orc_f64_to_f16.argtypes = [d]
        lib.orc_f16_decode_array.argtypes = [P, P, ctypes.c_int64]
        lib.orc_f16_encode_array.argtypes = [P, P, ctypes.c_int64]
        lib.orc_rope.argtypes = [P, P, i, ctypes.c_int64, d]
        lib.orc_append.restype = i
        lib.orc_append.argtypes = [P, P, P, P, i, P, P, i, P, P, P, P]
        lib.orc_attention.restype = i
        lib.orc_attention.argtypes = [P, P, P, i, P, P, P, d, i, P, P, P]
        lib.orc_split_attention.restype = i
        lib.orc_split_attention.argtypes = [P, P, P, i, P, P, P, i, i, i, d, i, P, P]
        lib.orc_split_attention_balanced.restype = i
        lib.orc_split_attention_balanced.argtypes = [P, P, P, i, P, P, P, i, i, d, i, P, P]
        lib.orc_combine.restype = i
        lib.orc_combine.argtypes = [P, P, i, i, i, i, P, P, P, P]
        lib.orc_quantize_row.restype = None
        lib.orc_quantize_row.argtypes = [P, i, P, P]
        lib.orc_append_int8.restype = i
        lib.orc_append_int8.argtypes = [P, P, P, P, i, P, P, i, P, P, P, P]
        lib.orc_quantize_pool.restype = None
        lib.orc_quantize_pool.argtypes = [P, P, P]
        lib.orc_dequantize_pool.restype = None
        lib.orc_dequantize_pool.argtypes = [P, P, P]
        lib.orc_attention_int8.restype = i
        lib.orc_attention_int8.argtypes = [P, P, P, i, P, P, P, d, i, P, P, P]
        lib.orc_split_attention_int8.restype = i
        lib.orc_split_attention_int8.argtypes = [P, P, P, i, P, P, P, i, i, i, d, i, P, P]
        lib.orc_prefill_attention.restype = i
        lib.orc_prefill_attention.argtypes = [P, P, P, i, i, P, P, P, P, P, d, i, P, P, P]
        lib.orc_qkv_project.restype = i
        lib.orc_qkv_project.argtypes = [P, P, P, i, i, i, P]
        lib.orc_threads.restype = i
        lib.orc_threads.argtypes = []
        lib.orc_init.restype = None
        lib.orc_init()
        _lib = lib
    return _lib


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data


@dataclass
class Geometry:
    num_pages: int
    num_qo_heads: int
    num_kv_heads: int
    head_dim: int
    max_position: int
    rope_theta: float

    def c(self) -> Geom:
        return Geom(self.num_pages, self.num_qo_heads, self.num_kv_heads, self.head_dim,
                    self.max_position, self.rope_theta)


def threads() -> int:
    """OpenMP threads the oracle's parallel loops use."""
    return int(_L().orc_threads())


def f16_to_f64(bits) -> np.ndarray:
    b, pb = _c(bits, np.uint16)
    out = np.empty(b.shape, dtype=np.float64)
    _L().orc_f16_decode_array(pb, out.ctypes.data, b.size)
    return out


def f64_to_f16(x) -> np.ndarray:
    a, pa = _c(x, np.float64)
    out = np.empty(a.shape, dtype=np.uint16)
    _L().orc_f16_encode_array(pa, out.ctypes.data, a.size)
    return out


def rope(x, pos: int, theta: float) -> np.ndarray:
    a, pa = _c(x, np.float64)
    out = np.empty_like(a)
    _L().orc_rope(pa, out.ctypes.data, a.size, int(pos), float(theta))
    return out


def append(geom: Geometry, q, k, v, pos_map, append_indptr, page_indptr, page_indices, pool):
    """RoPE + KV append.  ``pool`` (uint16 [pages, 2, Hkv, 16, d]) is updated in place.

    Returns q_out (uint16 [T, Hq, d])."""
    q, pq = _c(q, np.uint16)
    k, pk = _c(k, np.uint16)
    v, pv = _c(v, np.uint16)
    pm, ppm = _c(pos_map, np.int32)
    ai, pai = _c(append_indptr, np.int32)
    pi, ppi = _c(page_indptr, np.int32)
    px, ppx = _c(page_indices, np.int32)
    assert pool.dtype == np.uint16 and pool.flags["C_CONTIGUOUS"]
    T = pm.size
    q_out = np.empty((T, geom.num_qo_heads, geom.head_dim), dtype=np.uint16)
    g = geom.c()
    rc = _L().orc_append(ctypes.byref(g), pq, pk, pv, T, ppm, pai, ai.size - 1, ppi, ppx,
                         pool.ctypes.data, q_out.ctypes.data)
    if rc:
        raise OracleError(rc)
    return q_out


def int8_block_bytes(head_dim: int) -> int:
    """Bytes of one int8 block: the 16 slots' codes (K blocks [16][d], V blocks [d][16]) and fp32
    scales [16]."""
    return 16 * head_dim + 64


def quantize_row(x):
    """Row quantizer of the int8 cache: x fp16 bits [d] -> (codes int8 [d], scale float32)."""
    x, px = _c(x, np.uint16)
    codes = np.empty(x.size, dtype=np.int8)
    sc = np.empty(1, dtype=np.float32)
    _L().orc_quantize_row(px, x.size, codes.ctypes.data, sc.ctypes.data)
    return codes, sc[0]


def append_int8(geom: Geometry, q, k, v, pos_map, append_indptr, page_indptr, page_indices, pool8):
    """Append into an int8 pool (uint8 [P, 2, Hkv, 16*d + 64], in place); returns q_out."""
    q, pq = _c(q, np.uint16)
    k, pk = _c(k, np.uint16)
    v, pv = _c(v, np.uint16)
    pm, ppm = _c(pos_map, np.int32)
    ai, pai = _c(append_indptr, np.int32)
    pi, ppi = _c(page_indptr, np.int32)
    px, ppx = _c(page_indices, np.int32)
    if not (pool8.flags["C_CONTIGUOUS"] and pool8.dtype == np.uint8):
        raise ValueError("pool8 must be a C-contiguous uint8 array")
    T = q.shape[0]
    q_out = np.empty_like(q)
    g = geom.c()
    rc = _L().orc_append_int8(ctypes.byref(g), pq, pk, pv, T, ppm, pai, ai.size - 1, ppi, ppx, pool8.ctypes.data,
                              q_out.ctypes.data)
    if rc:
        raise OracleError(rc)
    return q_out


def quantize_pool(geom: Geometry, pool):
    """Every slot row of an fp16 pool [P, 2, Hkv, 16, d] quantized: uint8 [P, 2, Hkv, 16*d + 64]."""
    p16, pp = _c(pool, np.uint16)
    out = np.empty((geom.num_pages, 2, geom.num_kv_heads, int8_block_bytes(geom.head_dim)), dtype=np.uint8)
    g = geom.c()
    _L().orc_quantize_pool(ctypes.byref(g), pp, out.ctypes.data)
    return out


def dequantize_pool(geom: Geometry, pool8):
    """fp64 values of an int8 pool, laid out like the fp16 pool [P, 2, Hkv, 16, d]."""
    p8, pp = _c(pool8, np.uint8)
    out = np.empty((geom.num_pages, 2, geom.num_kv_heads, 16, geom.head_dim), dtype=np.float64)
    g = geom.c()
    _L().orc_dequantize_pool(ctypes.byref(g), pp, out.ctypes.data)
    return out


def attention_int8(geom: Geometry, pool8, q_rope, page_indptr, page_indices, last_page_len, sm_scale=None,
                   window: int = 0, sinks=None):
    """attention() over an int8 pool."""
    sm_scale = default_scale(geom.head_dim) if sm_scale is None else sm_scale
    p8, pp = _c(pool8, np.uint8)
    q, pq = _c(q_rope, np.uint16)
    pi, ppi = _c(page_indptr, np.int32)
    px, ppx = _c(page_indices, np.int32)
    lp, plp = _c(last_page_len, np.int32)
    B = pi.size - 1
    out = np.empty((B, geom.num_qo_heads, geom.head_dim), dtype=np.float64)
    lse = np.empty((B, geom.num_qo_heads), dtype=np.float64)
    g = geom.c()
    sk, psk = _sinks(sinks, geom.num_qo_heads)
    rc = _L().orc_attention_int8(ctypes.byref(g), pp, pq, B, ppi, ppx, plp, float(sm_scale), int(window), psk,
                                 out.ctypes.data, lse.ctypes.data)
    if rc:
        raise OracleError(rc)
    return out, lse


def split_attention_int8(geom: Geometry, pool8, q_rope, page_indptr, page_indices, last_page_len,
                         num_splits: int = 0, chunk_pages: int = 0, num_out_splits: int = 1, sm_scale=None,
                         window: int = 0):
    """split_attention() over an int8 pool."""
    sm_scale = default_scale(geom.head_dim) if sm_scale is None else sm_scale
    p8, pp = _c(pool8, np.uint8)
    q, pq = _c(q_rope, np.uint16)
    pi, ppi = _c(page_indptr, np.int32)
    px, ppx = _c(page_indices, np.int32)
    lp, plp = _c(last_page_len, np.int32)
    B = pi.size - 1
    S = num_out_splits
    po = np.empty((B, geom.num_qo_heads, S, geom.head_dim), dtype=np.float64)
    pl = np.empty((B, geom.num_qo_heads, S), dtype=np.float64)
    g = geom.c()
    rc = _L().orc_split_attention_int8(ctypes.byref(g), pp, pq, B, ppi, ppx, plp, int(num_splits), int(chunk_pages),
                                       S, float(sm_scale), int(window), po.ctypes.data, pl.ctypes.data)
    if rc:
        raise OracleError(rc)
    return po, pl


def qkv_project(x, w_packed, scales):
    """Q4F16_1 projection: x fp16 bits [T, hidden], w uint32 [N, hidden/8], scales fp16 bits
    [N, hidden/32] -> y fp16 bits [T, N] (see orc_qkv_project)."""
    x, px = _c(x, np.uint16)
    w, pw = _c(w_packed, np.uint32)
    sc, ps = _c(scales, np.uint16)
    T, hidden = x.shape
    N = w.shape[0]
    if w.shape != (N, hidden // 8) or sc.shape != (N, hidden // 32):
        raise ValueError("weight / scale shapes do not match the input")
    y = np.empty((T, N), dtype=np.uint16)
    rc = _L().orc_qkv_project(px, pw, ps, T, hidden, N, y.ctypes.data)
    if rc:
        raise OracleError(rc)
    return y


def qkv_append(geom: Geometry, x, w_packed, scales, pos_map, append_indptr, page_indptr, page_indices, pool):
    """The fused step of the pages' decode loop: the Q4F16_1 QKV projection, then RoPE and the KV
    append.  Returns (y, q_out): y fp16 bits [T, (Hq + 2Hkv) d] (q, k, v rows), q_out as append()."""
    y = qkv_project(x, w_packed, scales)
    T = y.shape[0]
    hq, hkv, d = geom.num_qo_heads, geom.num_kv_heads, geom.head_dim
    q = y[:, :hq * d].reshape(T, hq, d)
    k = y[:, hq * d:(hq + hkv) * d].reshape(T, hkv, d)
    v = y[:, (hq + hkv) * d:].reshape(T, hkv, d)
    q_out = append(geom, q, k, v, pos_map, append_indptr, page_indptr, page_indices, pool)
    return y, q_out


def default_scale(head_dim: int) -> float:
    return 1.0 / math.sqrt(head_dim)


def _sinks(sinks, hq):
    if sinks is None:
        return None, None
    a = np.ascontiguousarray(np.asarray(sinks, dtype=np.float64).reshape(hq))
    return a, a.ctypes.data


def attention(geom: Geometry, pool, q_rope, page_indptr, page_indices, last_page_len, sm_scale=None,
              window: int = 0, sinks=None):
    """Unsplit decode attention: returns out (float64 [B, Hq, d]) and lse (float64 [B, Hq]).
    window: attend to the `window` most recent positions (0 = all); sinks: per query head logits
    (natural log, units of the scaled scores) joining the softmax denominator, or None."""
    sm_scale = default_scale(geom.head_dim) if sm_scale is None else sm_scale
    pool, pp = _c(pool, np.uint16)
    q, pq = _c(q_rope, np.uint16)
    pi, ppi = _c(page_indptr, np.int32)
    px, ppx = _c(page_indices, np.int32)
    lp, plp = _c(last_page_len, np.int32)
    B = pi.size - 1
    out = np.empty((B, geom.num_qo_heads, geom.head_dim), dtype=np.float64)
    lse = np.empty((B, geom.num_qo_heads), dtype=np.float64)
    g = geom.c()
    sk, psk = _sinks(sinks, geom.num_qo_heads)
    rc = _L().orc_attention(ctypes.byref(g), pp, pq, B, ppi, ppx, plp, float(sm_scale), int(window), psk,
                            out.ctypes.data, lse.ctypes.data)
    if rc:
        raise OracleError(rc)
    return out, lse


def prefill_attention(geom: Geometry, pool, q_rope, append_indptr, pos_map, page_indptr, page_indices,
                      last_page_len, sm_scale=None, window: int = 0, sinks=None):
    """Chunked-prefill attention: every token t (rows of q_rope [T, Hq, d]) attends causally to the
    positions <= pos_map[t] of its sequence.  Returns out float64 [T, Hq, d], lse float64 [T, Hq]."""
    sm_scale = default_scale(geom.head_dim) if sm_scale is None else sm_scale
    pool, pp = _c(pool, np.uint16)
    q, pq = _c(q_rope, np.uint16)
    ai, pai = _c(append_indptr, np.int32)
    pm, ppm = _c(pos_map, np.int32)
    pi, ppi = _c(page_indptr, np.int32)
    px, ppx = _c(page_indices, np.int32)
    lp, plp = _c(last_page_len, np.int32)
    T, B = q.shape[0], ai.size - 1
    out = np.empty((T, geom.num_qo_heads, geom.head_dim), dtype=np.float64)
    lse = np.empty((T, geom.num_qo_heads), dtype=np.float64)
    g = geom.c()
    sk, psk = _sinks(sinks, geom.num_qo_heads)
    rc = _L().orc_prefill_attention(ctypes.byref(g), pp, pq, T, B, pai, ppm, ppi, ppx, plp, float(sm_scale),
                                    int(window), psk, out.ctypes.data, lse.ctypes.data)
    if rc:
        raise OracleError(rc)
    return out, lse


def split_attention(geom: Geometry, pool, q_rope, page_indptr, page_indices, last_page_len,
                    num_splits: int = 0, chunk_pages: int = 0, num_out_splits: int | None = None,
                    sm_scale=None, window: int = 0):
    """Split-K partials: (partial_o float64 [B, Hq, S, d], partial_lse float64 [B, Hq, S]).
    With a window the chunks cover each sequence's visible pages (see orc_split_attention)."""
    sm_scale = default_scale(geom.head_dim) if sm_scale is None else sm_scale
    pool, pp = _c(pool, np.uint16)
    q, pq = _c(q_rope, np.uint16)
    pi, ppi = _c(page_indptr, np.int32)
    px, ppx = _c(page_indices, np.int32)
    lp, plp = _c(last_page_len, np.int32)
    B = pi.size - 1
    if num_out_splits is None:
        if chunk_pages > 0:
            n = np.diff(pi)
            num_out_splits = max(1, int(-(-n.max() // chunk_pages)) if n.size else 1)
        else:
            num_out_splits = num_splits
    S = num_out_splits
    po = np.empty((B, geom.num_qo_heads, S, geom.head_dim), dtype=np.float64)
    pl = np.empty((B, geom.num_qo_heads, S), dtype=np.float64)
    g = geom.c()
    rc = _L().orc_split_attention(ctypes.byref(g), pp, pq, B, ppi, ppx, plp, int(num_splits),
                                  int(chunk_pages), S, float(sm_scale), int(window), po.ctypes.data,
                                  pl.ctypes.data)
    if rc:
        raise OracleError(rc)
    return po, pl


def split_attention_balanced(geom: Geometry, pool, q_rope, page_indptr, page_indices, last_page_len,
                             num_warps: int, num_out_splits: int, sm_scale=None, window: int = 0):
    """Partials of the page-balanced partition into ``num_warps`` equal runs of page units (the
    visible pages under a window)."""
    sm_scale = default_scale(geom.head_dim) if sm_scale is None else sm_scale
    pool, pp = _c(pool, np.uint16)
    q, pq = _c(q_rope, np.uint16)
    pi, ppi = _c(page_indptr, np.int32)
    px, ppx = _c(page_indices, np.int32)
    lp, plp = _c(last_page_len, np.int32)
    B = pi.size - 1
    S = num_out_splits
    po = np.empty((B, geom.num_qo_heads, S, geom.head_dim), dtype=np.float64)
    pl = np.empty((B, geom.num_qo_heads, S), dtype=np.float64)
    g = geom.c()
    rc = _L().orc_split_attention_balanced(ctypes.byref(g), pp, pq, B, ppi, ppx, plp, int(num_warps), S,
                                           float(sm_scale), int(window), po.ctypes.data, pl.ctypes.data)
    if rc:
        raise OracleError(rc)
    return po, pl


def combine(partial_o, partial_lse, sinks=None):
    """LSE merge: returns (out float64 [B, Hq, d], out fp16 bits uint16, lse float64 [B, Hq]);
    sinks: per query head logits joining the denominator, or None."""
    po, ppo = _c(partial_o, np.float64)
    pl, ppl = _c(partial_lse, np.float64)
    B, Hq, S, d = po.shape
    sk, psk = _sinks(sinks, Hq)
    out = np.empty((B, Hq, d), dtype=np.float64)
    out16 = np.empty((B, Hq, d), dtype=np.uint16)
    lse = np.empty((B, Hq), dtype=np.float64)
    rc = _L().orc_combine(ppo, ppl, B, Hq, S, d, psk, out.ctypes.data, out16.ctypes.data, lse.ctypes.data)
    if rc:
        raise OracleError(rc)
    return out, out16, lse
