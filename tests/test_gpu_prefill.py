"""Chunked-prefill attention on the GPU (pkv_prefill_attention) against the oracle: every appended
token attends causally over its sequence, checked on the GPU's own cache and rotated queries
(attention isolated) for all head dims and GQA groups, with windows and sinks, and the one-token
case against the merged decode."""
import numpy as np
import pytest

import oracle
from pkv_inputs import workloads as W
from tests import harness as H
from tests.test_gpu_parity import SMALL

pytestmark = pytest.mark.gpu

CASES = {
    "mixed_chunks_g4_d128": SMALL["gqa4_mixed_chunks"],
    "chunks_g1_d96": W.scaled(W.CONFIGS[3], batch=5, lengths=("uniform", 60, 700), pool_pages=600,
                              chunk_seqs=3, chunk_tokens=37),
    "chunks_g2_d128": W.scaled(W.CONFIGS[4], layers=1, batch=3, lengths=("fixed", 300), pool_pages=80,
                               chunk_seqs=2, chunk_tokens=50),
    "chunks_g8_d128": W.scaled(W.CONFIGS[5], hq=32, hkv=4, batch=4, lengths=("uniform", 40, 500), pool_pages=300,
                               chunk_seqs=2, chunk_tokens=33),
    "chunks_g4_d64": W.scaled(W.CONFIGS[3], hq=16, hkv=4, head_dim=64, batch=4, lengths=("uniform", 20, 400),
                              pool_pages=300, chunk_seqs=4, chunk_tokens=17),
    "long_chunk_g2_d96": W.scaled(W.CONFIGS[3], hq=16, hkv=8, batch=2, lengths=("fixed", 2100), pool_pages=300,
                                  chunk_seqs=1, chunk_tokens=200),
}


def _bits(t):
    import torch

    return t.contiguous().view(torch.int32 if t.dtype == torch.float32 else torch.int16).cpu().numpy()


def _run(cfg, window=0, with_sinks=False):
    import torch

    import paged_kv_decode_pkv_gb300 as pkv

    step = W.make_step(cfg)
    pool = H.to_dev(W.host_pool(step, 0), torch.float16)
    rng = np.random.default_rng(77 + window)
    sinks_host = (rng.standard_normal(cfg.hq) * 2).astype(np.float32) if with_sinks else None
    sinks = torch.from_numpy(sinks_host).cuda() if with_sinks else None
    cache = pkv.Cache(1, step.num_pages, cfg.hq, cfg.hkv, cfg.head_dim, step.max_position, cfg.theta, pools=[pool],
                      windows=[window], sinks=[sinks])
    tabs = H.device_tables(step)
    q, k, v = H.device_qkv(step, 0)
    q_out = cache.append_rope(0, q, k, v, tabs["pos_map"], tabs["append_indptr"], tabs["page_indptr"],
                              tabs["page_indices"])
    out, lse = cache.prefill_attention(0, q_out, tabs["append_indptr"], tabs["pos_map"], tabs["page_indptr"],
                                       tabs["page_indices"], tabs["last_page_len"])
    torch.cuda.synchronize()
    assert cache.check_status() == (0, 0)
    gpool = _bits(pool).view(np.uint16)
    gq = _bits(q_out).view(np.uint16)
    ref_out, ref_lse = oracle.prefill_attention(H.geometry(step), gpool, gq, step.append_indptr, step.pos_map,
                                                step.page_indptr, step.page_indices, step.last_page_len,
                                                window=window,
                                                sinks=None if sinks_host is None else sinks_host.astype(np.float64))
    return step, cache, tabs, q_out, out, lse, ref_out, ref_lse


@pytest.mark.parametrize("name", list(CASES))
def test_prefill_matches_oracle(name):
    step, cache, tabs, q_out, out, lse, ref_out, ref_lse = _run(CASES[name])
    assert step.num_tokens > step.batch
    H.assert_close_out(_bits(out).view(np.uint16), ref_out)
    H.assert_close_lse(lse.cpu().numpy(), ref_lse)


@pytest.mark.parametrize("name", ["chunks_g1_d96", "chunks_g2_d128", "chunks_g4_d64", "long_chunk_g2_d96"])
@pytest.mark.parametrize("window", [1, 16, 45])
def test_prefill_with_window_and_sinks_matches_oracle(name, window):
    step, cache, tabs, q_out, out, lse, ref_out, ref_lse = _run(CASES[name], window=window, with_sinks=True)
    H.assert_close_out(_bits(out).view(np.uint16), ref_out)
    H.assert_close_lse(lse.cpu().numpy(), ref_lse)


@pytest.mark.parametrize("name", ["ragged_d96", "gqa2_d96", "gqa8_d128", "tiny"])
def test_one_token_prefill_agrees_with_the_merged_decode(name):
    import torch

    cfg = SMALL[name]
    step, cache, tabs, q_out, out, lse, ref_out, ref_lse = _run(cfg)
    counters = torch.zeros(step.batch * cfg.hkv, dtype=torch.int32, device="cuda")
    d_out, d_lse = cache.decode_attention_merged(0, q_out, tabs["page_indptr"], tabs["page_indices"],
                                                 tabs["last_page_len"], step.max_pages_per_seq, counters,
                                                 q_indptr=tabs["q_indptr"], total_pages=int(step.page_indptr[-1]))
    torch.cuda.synchronize()
    H.assert_close_out(_bits(out).view(np.uint16), ref_out)
    a = _bits(out).view(np.uint16).view(np.float16).astype(np.float64)
    b = _bits(d_out).view(np.uint16).view(np.float16).astype(np.float64)
    assert np.abs(a - b).max() <= 2e-3
    assert np.abs(lse.cpu().numpy() - d_lse.cpu().numpy()).max() <= 5e-4


@pytest.mark.parametrize("name", ["mixed_chunks_g4_d128", "chunks_g1_d96"])
def test_back_to_back_prefill_launches_share_the_work_counter(name):
    """Three prefill launches on one stream with no host synchronisation between them, under
    programmatic dependent launch: the CTAs of each take their work items from the cache's device
    counter, which the previous launch's last CTA resets.  Every launch computes every row: the
    three outputs are bit-identical and match the oracle."""
    import torch

    import paged_kv_decode_pkv_gb300 as pkv

    cfg = CASES[name]
    step = W.make_step(cfg)
    pool = H.to_dev(W.host_pool(step, 0), torch.float16)
    cache = pkv.Cache(1, step.num_pages, cfg.hq, cfg.hkv, cfg.head_dim, step.max_position, cfg.theta, pools=[pool],
                      options=pkv.OPT_PDL)
    tabs = H.device_tables(step)
    q, k, v = H.device_qkv(step, 0)
    q_out = cache.append_rope(0, q, k, v, tabs["pos_map"], tabs["append_indptr"], tabs["page_indptr"],
                              tabs["page_indices"])
    T = step.num_tokens
    outs = []
    for _ in range(3):  # NaN-filled outputs: a row no launch wrote stays NaN
        o = torch.full((T, cfg.hq, cfg.head_dim), float("nan"), dtype=torch.float16, device="cuda")
        l = torch.full((T, cfg.hq), float("nan"), dtype=torch.float32, device="cuda")
        outs.append(cache.prefill_attention(0, q_out, tabs["append_indptr"], tabs["pos_map"], tabs["page_indptr"],
                                            tabs["page_indices"], tabs["last_page_len"], out=o, lse=l))
    torch.cuda.synchronize()
    assert cache.check_status() == (0, 0)
    for o, l in outs[1:]:
        assert np.array_equal(_bits(o), _bits(outs[0][0])) and np.array_equal(_bits(l), _bits(outs[0][1]))
    ref_out, ref_lse = oracle.prefill_attention(H.geometry(step), _bits(pool).view(np.uint16),
                                                _bits(q_out).view(np.uint16), step.append_indptr, step.pos_map,
                                                step.page_indptr, step.page_indices, step.last_page_len)
    H.assert_close_out(_bits(outs[2][0]).view(np.uint16), ref_out)
    H.assert_close_lse(outs[2][1].cpu().numpy(), ref_lse)
