"""Shared helpers for the GPU parity tests: the same seeded inputs for the CUDA path and the oracle.

The CUDA side runs through the Python binding (the C ABI); the oracle side runs on host arrays.
Nothing here computes attention itself.
"""
from __future__ import annotations

import math

import numpy as np

import oracle
from pkv_inputs import workloads as W

# Tolerances.  Attention output: the stated max-abs 2e-3 and relative L2 1e-3.  LSE: the
# probabilities summed on tensor cores are fp16, whose rounding is at most 2^-11 relative per
# term, so ln(sum) is off by less than 2^-11 < 5e-4; fp32 accumulation adds far less.
OUT_MAX_ABS = 2e-3
OUT_REL_L2 = 1e-3
LSE_ABS = 5e-4


def geometry(step: W.Step) -> oracle.Geometry:
    c = step.cfg
    return oracle.Geometry(step.num_pages, c.hq, c.hkv, c.head_dim, step.max_position, c.theta)


def ulp_distance(a, b):
    """Distance in fp16 steps between arrays of finite fp16 bit patterns."""
    def ordered(x):
        x = np.asarray(x).astype(np.int32)
        return np.where(x & 0x8000, -(x & 0x7FFF), x)
    return np.abs(ordered(a) - ordered(b))


def assert_close_out(got16, ref64, what="out"):
    got = np.asarray(got16, dtype=np.uint16).view(np.float16).astype(np.float64)
    ref = np.asarray(ref64, dtype=np.float64)
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    err = np.abs(got - ref)
    max_abs = float(err.max()) if err.size else 0.0
    rel = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)) if err.size else 0.0
    assert max_abs <= OUT_MAX_ABS, f"{what}: max-abs {max_abs:.3e} > {OUT_MAX_ABS}"
    assert rel <= OUT_REL_L2, f"{what}: relative L2 {rel:.3e} > {OUT_REL_L2}"
    return max_abs, rel


def assert_close_lse(got, ref, what="lse"):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    inf_ref = np.isinf(ref)
    assert np.array_equal(np.isinf(got), inf_ref), f"{what}: -inf pattern differs"
    if (~inf_ref).any():
        d = float(np.abs(got[~inf_ref] - ref[~inf_ref]).max())
        assert d <= LSE_ABS, f"{what}: max-abs {d:.3e} > {LSE_ABS}"


def assert_close_partial_o(got, ref, lse_ref, what="partial_o"):
    mask = ~np.isinf(np.asarray(lse_ref))
    g = np.asarray(got, dtype=np.float64)[mask]
    r = np.asarray(ref, dtype=np.float64)[mask]
    err = np.abs(g - r)
    assert np.isfinite(g).all(), f"{what}: non-finite values in written chunks"
    assert float(err.max()) <= OUT_MAX_ABS, f"{what}: max-abs {float(err.max()):.3e}"
    rel = float(np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30))
    assert rel <= OUT_REL_L2, f"{what}: relative L2 {rel:.3e}"


# ------------------------------------------------------------------------------------------------
# device side


def to_dev(a, dtype=None):
    import torch

    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.cuda()


def device_tables(step: W.Step):
    import torch

    d = {
        "pos_map": to_dev(step.pos_map), "append_indptr": to_dev(step.append_indptr),
        "page_indptr": to_dev(step.page_indptr), "page_indices": to_dev(step.page_indices),
        "last_page_len": to_dev(step.last_page_len),
    }
    d["q_indptr"] = d["append_indptr"] if int(step.new_tokens.max(initial=1)) > 1 else None
    return d


def device_qkv(step: W.Step, layer: int):
    import torch

    q, k, v = W.new_qkv(step, layer)
    return to_dev(q, torch.float16), to_dev(k, torch.float16), to_dev(v, torch.float16)


def make_cache(step: W.Step, layers, pools, options=0):
    import paged_kv_decode_pkv_gb300 as pkv

    c = step.cfg
    return pkv.Cache(len(layers), step.num_pages, c.hq, c.hkv, c.head_dim, step.max_position, c.theta,
                     pools=pools, options=options)


def run_chain(cache, layer_slot, tabs, q, k, v, step: W.Step, num_splits=0, chunk_pages=0, total_pages=None):
    """append -> decode -> combine on the device; returns the device tensors."""
    q_out = cache.append_rope(layer_slot, q, k, v, tabs["pos_map"], tabs["append_indptr"], tabs["page_indptr"],
                              tabs["page_indices"])
    tp = int(step.page_indptr[-1]) if total_pages is None else total_pages
    po, pl, S = cache.decode_attention(layer_slot, q_out, tabs["page_indptr"], tabs["page_indices"],
                                       tabs["last_page_len"], step.max_pages_per_seq, q_indptr=tabs["q_indptr"],
                                       total_pages=tp, num_splits=num_splits, chunk_pages=chunk_pages)
    out, lse = cache.combine(po, pl)
    return q_out, po, pl, out, lse


def query_rows(step: W.Step) -> np.ndarray:
    """Row of q_out used as the decode query of each sequence (its last appended token)."""
    return (step.append_indptr[1:] - 1).astype(np.int64)


# ------------------------------------------------------------------------------------------------
# oracle side


def oracle_chain(step: W.Step, pool, q, k, v, num_splits=0, chunk_pages=0, window=0, sinks=None):
    """The oracle's own append on a copy of ``pool`` followed by split attention and combine
    (window / sinks: the layer's sliding window and attention-sink logits)."""
    g = geometry(step)
    pool = pool.copy()
    q_out = oracle.append(g, q, k, v, step.pos_map, step.append_indptr, step.page_indptr, step.page_indices, pool)
    qd = q_out[query_rows(step)]
    res = {"pool": pool, "q_out": q_out}
    if num_splits or chunk_pages:
        po, pl = oracle.split_attention(g, pool, qd, step.page_indptr, step.page_indices, step.last_page_len,
                                        num_splits=num_splits, chunk_pages=chunk_pages, window=window)
        res["partial_o"], res["partial_lse"] = po, pl
        res["out"], res["out16"], res["lse"] = oracle.combine(po, pl, sinks=sinks)
    else:
        res["out"], res["lse"] = oracle.attention(g, pool, qd, step.page_indptr, step.page_indices,
                                                  step.last_page_len, window=window, sinks=sinks)
    return res


def oracle_attention_on(step: W.Step, pool, q_rope_rows, window=0, sinks=None):
    g = geometry(step)
    return oracle.attention(g, pool, q_rope_rows, step.page_indptr, step.page_indices, step.last_page_len,
                            window=window, sinks=sinks)


def default_scale(step: W.Step) -> float:
    return 1.0 / math.sqrt(step.cfg.head_dim)
