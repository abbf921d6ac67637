"""The one-launch layer step (pkv_append_decode_attention) against the two-launch path
(pkv_append_rope + pkv_decode_attention_merged): the same pool image, rotated queries, outputs and
LSEs bit for bit, for every split plan, chunked appends of more than 32 tokens, and GQA groups."""
import numpy as np
import pytest

from pkv_inputs import workloads as W
from tests import harness as H
from tests.test_gpu_parity import SMALL

pytestmark = pytest.mark.gpu


def _bits(t):
    import torch

    return t.contiguous().view(torch.int32 if t.dtype == torch.float32 else torch.int16).cpu().numpy()


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("plan,early", [({}, False), ({"num_splits": 3}, False), ({"chunk_pages": 2}, False),
                                        ({}, True)])
def test_fused_step_is_bit_identical_to_append_then_merged_decode(name, plan, early):
    import torch

    import paged_kv_decode_pkv_gb300 as pkv

    cfg = SMALL[name]
    if cfg.num_splits and not plan:
        plan = {"num_splits": cfg.num_splits}
    step = W.make_step(cfg)
    host_pool = W.host_pool(step, 0)
    pool_a = H.to_dev(host_pool, torch.float16)
    pool_b = H.to_dev(host_pool, torch.float16)
    cache_a = H.make_cache(step, [0], [pool_a])
    # early pages: the one-launch kernel copies the cache before its launch wait (with PDL)
    cache_b = H.make_cache(step, [0], [pool_b], options=(pkv.OPT_PDL | pkv.OPT_EARLY_PAGES) if early else 0)
    tabs = H.device_tables(step)
    q, k, v = H.device_qkv(step, 0)
    tp = int(step.page_indptr[-1])
    counters = torch.zeros(step.batch * cfg.hkv, dtype=torch.int32, device="cuda")
    q_out_a = cache_a.append_rope(0, q, k, v, tabs["pos_map"], tabs["append_indptr"], tabs["page_indptr"],
                                  tabs["page_indices"])
    out_a, lse_a = cache_a.decode_attention_merged(0, q_out_a, tabs["page_indptr"], tabs["page_indices"],
                                                   tabs["last_page_len"], step.max_pages_per_seq, counters,
                                                   q_indptr=tabs["append_indptr"], total_pages=tp, **plan)
    q_out_b, out_b, lse_b = cache_b.append_decode_attention(
        0, q, k, v, tabs["pos_map"], tabs["append_indptr"], tabs["page_indptr"], tabs["page_indices"],
        tabs["last_page_len"], step.max_pages_per_seq, counters, total_pages=tp, **plan)
    torch.cuda.synchronize()
    assert cache_a.check_status()[0] == 0 and cache_b.check_status()[0] == 0
    assert np.array_equal(_bits(pool_a), _bits(pool_b)), "pool image"
    assert np.array_equal(_bits(q_out_a), _bits(q_out_b)), "q_out"
    assert np.array_equal(_bits(out_a), _bits(out_b)), "out"
    assert np.array_equal(_bits(lse_a), _bits(lse_b)), "lse"
    assert int(counters.abs().sum()) == 0
    # and against the oracle end to end
    qh, kh, vh = W.new_qkv(step, 0)
    ref = H.oracle_chain(step, host_pool, qh, kh, vh)
    H.assert_close_out(_bits(out_b).view(np.uint16), ref["out"])
    H.assert_close_lse(lse_b.cpu().numpy(), ref["lse"])


def test_fused_step_reports_positions_out_of_range():
    import torch

    import paged_kv_decode_pkv_gb300 as pkv

    cfg = SMALL["gqa4_mixed_chunks"]
    step = W.make_step(cfg)
    pool = H.to_dev(W.host_pool(step, 0), torch.float16)
    cache = H.make_cache(step, [0], [pool])
    tabs = H.device_tables(step)
    q, k, v = H.device_qkv(step, 0)
    bad = tabs["pos_map"].clone()
    chunk_seq = int(np.flatnonzero(step.new_tokens > 1)[0])
    bad[int(step.append_indptr[chunk_seq])] = 1 << 30  # not the query token of that sequence
    counters = torch.zeros(step.batch * cfg.hkv, dtype=torch.int32, device="cuda")
    cache.append_decode_attention(0, q, k, v, bad, tabs["append_indptr"], tabs["page_indptr"], tabs["page_indices"],
                                  tabs["last_page_len"], step.max_pages_per_seq, counters,
                                  total_pages=int(step.page_indptr[-1]))
    code, flags = cache.check_status()
    assert code == pkv.ERR_OUT_OF_RANGE and flags & pkv.FLAG_BAD_POSITION


def _single_token_case():
    import torch

    cfg = SMALL["phi3_b1_ctx300"]
    cfg = W.scaled(cfg, batch=3, lengths=("uniform", 40, 300), pool_pages=60)
    step = W.make_step(cfg)
    assert int(step.new_tokens.max()) == 1
    pool = H.to_dev(W.host_pool(step, 0), torch.float16)
    cache = H.make_cache(step, [0], [pool])
    tabs = H.device_tables(step)
    q, k, v = H.device_qkv(step, 0)
    counters = torch.zeros(step.batch * cfg.hkv, dtype=torch.int32, device="cuda")
    return step, cache, tabs, (q, k, v), counters


def test_one_launch_reports_a_position_past_the_pages():
    import paged_kv_decode_pkv_gb300 as pkv

    step, cache, tabs, (q, k, v), counters = _single_token_case()
    bad = tabs["pos_map"].clone()
    n_pages = int(step.page_indptr[1] - step.page_indptr[0])
    bad[0] = n_pages * 16  # inside the RoPE table, past sequence 0's pages
    cache.append_decode_attention(0, q, k, v, bad, tabs["append_indptr"], tabs["page_indptr"], tabs["page_indices"],
                                  tabs["last_page_len"], step.max_pages_per_seq, counters,
                                  total_pages=int(step.page_indptr[-1]))
    code, flags = cache.check_status()
    assert code == pkv.ERR_OUT_OF_RANGE and flags & pkv.FLAG_BAD_POSITION


def test_one_launch_reports_a_sequence_without_exactly_one_token():
    import paged_kv_decode_pkv_gb300 as pkv

    step, cache, tabs, (q, k, v), counters = _single_token_case()
    indptr = tabs["append_indptr"].clone()
    indptr[1] = 2  # sequence 0 takes two tokens, sequence 1 none: still batch tokens in total
    cache.append_decode_attention(0, q, k, v, tabs["pos_map"], indptr, tabs["page_indptr"], tabs["page_indices"],
                                  tabs["last_page_len"], step.max_pages_per_seq, counters,
                                  total_pages=int(step.page_indptr[-1]))
    code, flags = cache.check_status()
    assert code == pkv.ERR_OUT_OF_RANGE and flags & pkv.FLAG_BAD_SEQUENCE
