"""Sliding window and attention sinks on the GPU against the oracle (and against each other's
launch layouts, bit for bit).

Window W: the query at position len-1 attends to [max(0, len-W), len); sink: one fp32 logit per
query head in the softmax denominator (Splash models page: sliding_window, layer_types and a
layer's attn_sinks).  Every case runs the append, then the merged decode (oracle's attention over
the GPU's own cache and q_out), the explicit-plan partials (oracle's windowed split), the partials
merged by pkv_combine with the sinks (bit-identical to the merged decode), and the one-launch step
(bit-identical to append + merged decode)."""
import numpy as np
import pytest

import oracle
from pkv_inputs import workloads as W
from tests import harness as H
from tests.test_gpu_parity import SMALL

pytestmark = pytest.mark.gpu

CASES = ["tiny", "ragged_d96", "gqa2_d96", "gqa4_d64", "gqa8_d128", "mha_d64_long"]
WINDOWS = [1, 16, 17, 100, 1 << 20]


def _bits(t):
    import torch

    return t.contiguous().view(torch.int32 if t.dtype == torch.float32 else torch.int16).cpu().numpy()


def _setup(name, window, with_sinks, seed_extra=0):
    import torch

    import paged_kv_decode_pkv_gb300 as pkv

    cfg = SMALL[name]
    step = W.make_step(cfg)
    host_pool = W.host_pool(step, 0)
    rng = np.random.default_rng(1000 + window % 997 + seed_extra)
    sinks_host = (rng.standard_normal(cfg.hq) * 2).astype(np.float32) if with_sinks else None
    sinks = torch.from_numpy(sinks_host).cuda() if with_sinks else None

    def cache_over(pool_dev, options=0):
        return pkv.Cache(1, step.num_pages, cfg.hq, cfg.hkv, cfg.head_dim, step.max_position, cfg.theta,
                         pools=[pool_dev], windows=[window], sinks=[sinks], options=options)

    return step, host_pool, sinks_host, sinks, cache_over


@pytest.mark.parametrize("name", CASES)
@pytest.mark.parametrize("window", WINDOWS)
@pytest.mark.parametrize("with_sinks", [False, True])
def test_windowed_decode_with_sinks_matches_oracle(name, window, with_sinks):
    import torch

    step, host_pool, sinks_host, sinks, cache_over = _setup(name, window, with_sinks)
    cfg = step.cfg
    pool = H.to_dev(host_pool, torch.float16)
    cache = cache_over(pool)
    tabs = H.device_tables(step)
    q, k, v = H.device_qkv(step, 0)
    tp = int(step.page_indptr[-1])
    q_out = cache.append_rope(0, q, k, v, tabs["pos_map"], tabs["append_indptr"], tabs["page_indptr"],
                              tabs["page_indices"])
    counters = torch.zeros(step.batch * cfg.hkv, dtype=torch.int32, device="cuda")
    out, lse = cache.decode_attention_merged(0, q_out, tabs["page_indptr"], tabs["page_indices"],
                                             tabs["last_page_len"], step.max_pages_per_seq, counters,
                                             q_indptr=tabs["q_indptr"], total_pages=tp)
    torch.cuda.synchronize()
    assert cache.check_status() == (0, 0)
    gpool = _bits(pool).view(np.uint16)
    gq = _bits(q_out).view(np.uint16)[H.query_rows(step)]
    ref_out, ref_lse = oracle.attention(H.geometry(step), gpool, gq, step.page_indptr, step.page_indices,
                                        step.last_page_len, window=window,
                                        sinks=None if sinks_host is None else sinks_host.astype(np.float64))
    H.assert_close_out(_bits(out).view(np.uint16), ref_out)
    H.assert_close_lse(lse.cpu().numpy(), ref_lse)


@pytest.mark.parametrize("name", ["ragged_d96", "gqa4_d64", "gqa8_d128"])
@pytest.mark.parametrize("window", [16, 17, 100])
@pytest.mark.parametrize("plan", [{"num_splits": 3}, {"chunk_pages": 2}])
def test_windowed_partials_combine_and_merged_agree(name, window, plan):
    import torch

    step, host_pool, sinks_host, sinks, cache_over = _setup(name, window, True, seed_extra=7)
    cfg = step.cfg
    pool = H.to_dev(host_pool, torch.float16)
    cache = cache_over(pool)
    tabs = H.device_tables(step)
    q, k, v = H.device_qkv(step, 0)
    tp = int(step.page_indptr[-1])
    q_out = cache.append_rope(0, q, k, v, tabs["pos_map"], tabs["append_indptr"], tabs["page_indptr"],
                              tabs["page_indices"])
    po, pl, S = cache.decode_attention(0, q_out, tabs["page_indptr"], tabs["page_indices"], tabs["last_page_len"],
                                       step.max_pages_per_seq, q_indptr=tabs["q_indptr"], total_pages=tp, **plan)
    out_c, lse_c = cache.combine(po, pl, sinks=sinks)
    counters = torch.zeros(step.batch * cfg.hkv, dtype=torch.int32, device="cuda")
    out_m, lse_m = cache.decode_attention_merged(0, q_out, tabs["page_indptr"], tabs["page_indices"],
                                                 tabs["last_page_len"], step.max_pages_per_seq, counters,
                                                 q_indptr=tabs["q_indptr"], total_pages=tp, **plan)
    torch.cuda.synchronize()
    assert cache.check_status() == (0, 0)
    assert np.array_equal(_bits(out_c), _bits(out_m)) and np.array_equal(_bits(lse_c), _bits(lse_m))
    gpool = _bits(pool).view(np.uint16)
    gq = _bits(q_out).view(np.uint16)[H.query_rows(step)]
    rpo, rpl = oracle.split_attention(H.geometry(step), gpool, gq, step.page_indptr, step.page_indices,
                                      step.last_page_len, num_out_splits=S, window=window, **plan)
    H.assert_close_lse(pl.cpu().numpy(), rpl, "partial_lse")
    H.assert_close_partial_o(po.cpu().numpy(), rpo, rpl)
    ref_out, _, ref_lse = oracle.combine(rpo, rpl, sinks=sinks_host.astype(np.float64))
    H.assert_close_out(_bits(out_c).view(np.uint16), ref_out)
    H.assert_close_lse(lse_c.cpu().numpy(), ref_lse)


@pytest.mark.parametrize("name", ["tiny", "ragged_d96", "gqa2_d96", "gqa8_d128"])
@pytest.mark.parametrize("window", [1, 17, 100])
@pytest.mark.parametrize("early", [False, True])
def test_windowed_one_launch_step_is_bit_identical(name, window, early):
    import torch

    import paged_kv_decode_pkv_gb300 as pkv

    step, host_pool, sinks_host, sinks, cache_over = _setup(name, window, True, seed_extra=11)
    cfg = step.cfg
    if int(step.new_tokens.max()) > 1:
        pytest.skip("one-launch layout needs one new token per sequence")
    pool_a = H.to_dev(host_pool, torch.float16)
    pool_b = H.to_dev(host_pool, torch.float16)
    cache_a = cache_over(pool_a)
    cache_b = cache_over(pool_b, (pkv.OPT_PDL | pkv.OPT_EARLY_PAGES) if early else 0)
    tabs = H.device_tables(step)
    q, k, v = H.device_qkv(step, 0)
    tp = int(step.page_indptr[-1])
    counters = torch.zeros(step.batch * cfg.hkv, dtype=torch.int32, device="cuda")
    q_out_a = cache_a.append_rope(0, q, k, v, tabs["pos_map"], tabs["append_indptr"], tabs["page_indptr"],
                                  tabs["page_indices"])
    out_a, lse_a = cache_a.decode_attention_merged(0, q_out_a, tabs["page_indptr"], tabs["page_indices"],
                                                   tabs["last_page_len"], step.max_pages_per_seq, counters,
                                                   q_indptr=tabs["append_indptr"], total_pages=tp)
    q_out_b, out_b, lse_b = cache_b.append_decode_attention(
        0, q, k, v, tabs["pos_map"], tabs["append_indptr"], tabs["page_indptr"], tabs["page_indices"],
        tabs["last_page_len"], step.max_pages_per_seq, counters, total_pages=tp)
    torch.cuda.synchronize()
    assert cache_a.check_status() == (0, 0) and cache_b.check_status() == (0, 0)
    assert np.array_equal(_bits(pool_a), _bits(pool_b)), "pool image"
    assert np.array_equal(_bits(q_out_a), _bits(q_out_b)), "q_out"
    assert np.array_equal(_bits(out_a), _bits(out_b)), "out"
    assert np.array_equal(_bits(lse_a), _bits(lse_b)), "lse"


@pytest.mark.parametrize("name", ["tiny", "ragged_d96", "gqa4_d64", "gqa8_d128", "mha_d64_long"])
@pytest.mark.parametrize("window", [1, 17, 100])
def test_windowed_balanced_partials_match_oracle(name, window):
    """The automatic plan of a windowed layer: the page-balanced partition of the visible pages,
    every piece compared."""
    import torch

    step, host_pool, sinks_host, sinks, cache_over = _setup(name, window, True, seed_extra=13)
    pool = H.to_dev(host_pool, torch.float16)
    cache = cache_over(pool)
    tabs = H.device_tables(step)
    q, k, v = H.device_qkv(step, 0)
    q_out = cache.append_rope(0, q, k, v, tabs["pos_map"], tabs["append_indptr"], tabs["page_indptr"],
                              tabs["page_indices"])
    po, pl, S = cache.decode_attention(0, q_out, tabs["page_indptr"], tabs["page_indices"], tabs["last_page_len"],
                                       step.max_pages_per_seq, q_indptr=tabs["q_indptr"],
                                       total_pages=int(step.page_indptr[-1]))
    out_c, lse_c = cache.combine(po, pl, sinks=sinks)
    torch.cuda.synchronize()
    assert cache.check_status() == (0, 0)
    sms, warps = cache.device_info(step.batch)
    L = step.seq_len
    visible = int(sum(-(-int(x) // 16) - max(0, int(x) - window) // 16 for x in L)) * step.cfg.hkv
    gpool = _bits(pool).view(np.uint16)
    gq = _bits(q_out).view(np.uint16)[H.query_rows(step)]
    rpo, rpl = oracle.split_attention_balanced(H.geometry(step), gpool, gq, step.page_indptr, step.page_indices,
                                               step.last_page_len, min(sms * warps, visible), S, window=window)
    H.assert_close_lse(pl.cpu().numpy(), rpl, "partial_lse")
    H.assert_close_partial_o(po.cpu().numpy(), rpo, rpl)
    ref_out, _, ref_lse = oracle.combine(rpo, rpl, sinks=sinks_host.astype(np.float64))
    H.assert_close_out(_bits(out_c).view(np.uint16), ref_out)
    H.assert_close_lse(lse_c.cpu().numpy(), ref_lse)
