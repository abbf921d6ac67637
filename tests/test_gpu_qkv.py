"""The Q4F16_1 QKV projection fused with RoPE and the KV append, on the GPU: the projection against
the oracle (fp32 against fp64 accumulation: at most one fp16 step apart), the fused call bit for bit
against the projection followed by pkv_append_rope, and the whole step (fused projection and append,
then the merged decode) against the oracle's projection, append and attention."""
import numpy as np
import pytest

import oracle
from pkv_inputs import workloads as W
from tests import harness as H
from tests.test_gpu_parity import SMALL
from tests.test_oracle_qkv import _dequantize

pytestmark = pytest.mark.gpu

CASES = ["tiny", "phi3_b1_ctx300", "ragged_d96", "gqa4_mixed_chunks", "gqa4_d64", "gqa8_d128", "gqa2_d96"]


def _bits(t):
    import torch

    return t.contiguous().view(torch.int32 if t.dtype == torch.float32 else torch.int16).cpu().numpy()


def _inputs(step, layer=0):
    import torch

    w, sc = W.qkv_weights(step, layer)
    x = W.hidden_states(step, layer)
    dev = (H.to_dev(x, torch.float16), H.to_dev(w.view(np.int32)), H.to_dev(sc, torch.float16))
    return (x, w, sc), dev


@pytest.mark.parametrize("name", CASES)
def test_projection_matches_oracle_within_one_fp16_step(name):
    import torch

    step = W.make_step(SMALL[name])
    cache = H.make_cache(step, [0], [H.to_dev(W.host_pool(step, 0), torch.float16)])
    (x, w, sc), (xd, wd, scd) = _inputs(step)
    y = cache.qkv_project(xd, wd, scd)
    torch.cuda.synchronize()
    got = _bits(y).view(np.uint16)
    ref = oracle.qkv_project(x, w, sc)
    # fp32 summation of n products is within n * 2^-24 * sum |x w| of the exact sum (the recursive
    # summation bound); the fp16 roundings of both sides add at most one step each side
    hidden = x.shape[1]
    absw = np.abs(_dequantize(w, sc, hidden))
    bound = hidden * 2.0 ** -24 * (np.abs(x.view(np.float16).astype(np.float64)) @ absw.T)
    g = got.view(np.float16).astype(np.float64)
    r = ref.view(np.float16).astype(np.float64)
    step16 = np.spacing(np.abs(r).astype(np.float16)).astype(np.float64)
    assert np.all(np.abs(g - r) <= bound + 2 * step16)
    assert float(np.mean(H.ulp_distance(got, ref) == 0)) >= 0.95


@pytest.mark.parametrize("name", CASES)
def test_fused_projection_and_append_is_bit_identical_to_project_then_append(name):
    import torch

    cfg = SMALL[name]
    step = W.make_step(cfg)
    host_pool = W.host_pool(step, 0)
    pool_a = H.to_dev(host_pool, torch.float16)
    pool_b = H.to_dev(host_pool, torch.float16)
    cache_a = H.make_cache(step, [0], [pool_a])
    cache_b = H.make_cache(step, [0], [pool_b])
    tabs = H.device_tables(step)
    _, (xd, wd, scd) = _inputs(step)
    y = cache_a.qkv_project(xd, wd, scd)
    T, hq, hkv, d = step.num_tokens, cfg.hq, cfg.hkv, cfg.head_dim
    q = y[:, :hq * d].reshape(T, hq, d).contiguous()
    k = y[:, hq * d:(hq + hkv) * d].reshape(T, hkv, d).contiguous()
    v = y[:, (hq + hkv) * d:].reshape(T, hkv, d).contiguous()
    q_out_a = cache_a.append_rope(0, q, k, v, tabs["pos_map"], tabs["append_indptr"], tabs["page_indptr"],
                                  tabs["page_indices"])
    q_out_b = cache_b.qkv_append_rope(0, xd, wd, scd, tabs["pos_map"], tabs["append_indptr"], tabs["page_indptr"],
                                      tabs["page_indices"])
    torch.cuda.synchronize()
    assert cache_a.check_status() == (0, 0) and cache_b.check_status() == (0, 0)
    assert np.array_equal(_bits(pool_a), _bits(pool_b)), "pool image"
    assert np.array_equal(_bits(q_out_a), _bits(q_out_b)), "q_out"


@pytest.mark.parametrize("name", ["tiny", "ragged_d96", "gqa4_mixed_chunks", "gqa8_d128"])
def test_projection_append_and_decode_match_the_oracle_step(name):
    import torch

    cfg = SMALL[name]
    step = W.make_step(cfg)
    host_pool = W.host_pool(step, 0)
    pool = H.to_dev(host_pool, torch.float16)
    cache = H.make_cache(step, [0], [pool])
    tabs = H.device_tables(step)
    (x, w, sc), (xd, wd, scd) = _inputs(step)
    q_out = cache.qkv_append_rope(0, xd, wd, scd, tabs["pos_map"], tabs["append_indptr"], tabs["page_indptr"],
                                  tabs["page_indices"])
    counters = torch.zeros(step.batch * cfg.hkv, dtype=torch.int32, device="cuda")
    out, lse = cache.decode_attention_merged(0, q_out, tabs["page_indptr"], tabs["page_indices"],
                                             tabs["last_page_len"], step.max_pages_per_seq, counters,
                                             q_indptr=tabs["q_indptr"], total_pages=int(step.page_indptr[-1]))
    torch.cuda.synchronize()
    assert cache.check_status() == (0, 0)
    # attention isolated: the oracle over the GPU's own cache and rotated queries
    gpool = _bits(pool).view(np.uint16)
    gq = _bits(q_out).view(np.uint16)
    ref_out, ref_lse = oracle.attention(H.geometry(step), gpool, gq[H.query_rows(step)], step.page_indptr,
                                        step.page_indices, step.last_page_len)
    H.assert_close_out(_bits(out).view(np.uint16), ref_out)
    H.assert_close_lse(lse.cpu().numpy(), ref_lse)
    # end to end: the oracle's own projection, append and attention
    opool = host_pool.copy()
    _, oq_out = oracle.qkv_append(H.geometry(step), x, w, sc, step.pos_map, step.append_indptr, step.page_indptr,
                                  step.page_indices, opool)
    e_out, e_lse = oracle.attention(H.geometry(step), opool, oq_out[H.query_rows(step)], step.page_indptr,
                                    step.page_indices, step.last_page_len)
    H.assert_close_out(_bits(out).view(np.uint16), e_out, "out (end to end)")
    H.assert_close_lse(lse.cpu().numpy(), e_lse, "lse (end to end)")
