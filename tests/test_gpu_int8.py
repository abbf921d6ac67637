"""int8 KV cache (PKV_OPT_INT8_KV) on the GPU against the oracle: the quantizing append (V codes and
scales bit for bit; K, whose fp16 rotation may differ by one step from the oracle's, within one
code), attention over the GPU's own int8 cache (merged decode and explicit-plan partials), end to
end against the oracle's own int8 append, and the one-token step entry point against the two
launches it runs."""
import numpy as np
import pytest

import oracle
from pkv_inputs import workloads as W
from tests import harness as H
from tests.test_gpu_parity import SMALL

pytestmark = pytest.mark.gpu

# group sizes 1 (one query head per KV head), 2, 4 and 8; head dims 64, 96 and 128
CASES = ["gqa2_d128_outliers", "gqa4_mixed_chunks", "gqa2_d96", "gqa4_d64", "gqa8_d128", "tiny", "ragged_d96",
         "phi3_b1_ctx300"]


def _bits(t):
    import torch

    return t.contiguous().view(torch.int32 if t.dtype == torch.float32 else torch.int16).cpu().numpy()


def _setup(name):
    import torch

    import paged_kv_decode_pkv_gb300 as pkv

    cfg = SMALL[name]
    step = W.make_step(cfg)
    g = H.geometry(step)
    host16 = W.host_pool(step, 0)
    host8 = oracle.quantize_pool(g, host16)
    pool8 = torch.from_numpy(host8).cuda()
    cache = pkv.Cache(1, step.num_pages, cfg.hq, cfg.hkv, cfg.head_dim, step.max_position, cfg.theta,
                      pools=[pool8], options=pkv.OPT_INT8_KV)
    return step, g, host16, host8, pool8, cache


@pytest.mark.parametrize("name", CASES)
def test_int8_append_matches_oracle(name):
    import torch

    step, g, host16, host8, pool8, cache = _setup(name)
    tabs = H.device_tables(step)
    q, k, v = H.device_qkv(step, 0)
    q_out = cache.append_rope(0, q, k, v, tabs["pos_map"], tabs["append_indptr"], tabs["page_indptr"],
                              tabs["page_indices"])
    torch.cuda.synchronize()
    assert cache.check_status() == (0, 0)
    qh, kh, vh = W.new_qkv(step, 0)
    ref8 = host8.copy()
    ref_q = oracle.append_int8(g, qh, kh, vh, step.pos_map, step.append_indptr, step.page_indptr,
                               step.page_indices, ref8)
    got8 = pool8.cpu().numpy()
    d = step.cfg.head_dim
    # q_out: the fp16 append's rotation, within one fp16 step of the oracle's
    assert int(H.ulp_distance(_bits(q_out).view(np.uint16), ref_q).max()) <= 1
    # V blocks bit for bit; K codes within one step and scales within the fp16 rounding of K
    assert np.array_equal(got8[:, 1], ref8[:, 1]), "V blocks"
    kc_got = got8[:, 0, :, :16 * d].astype(np.int32)  # stored code + 128: differences are code differences
    kc_ref = ref8[:, 0, :, :16 * d].astype(np.int32)
    assert int(np.abs(kc_got - kc_ref).max()) <= 1
    ks_got = got8[:, 0, :, 16 * d:].copy().view(np.float32)
    ks_ref = ref8[:, 0, :, 16 * d:].copy().view(np.float32)
    assert np.allclose(ks_got, ks_ref, rtol=2e-3, atol=0)


@pytest.mark.parametrize("name", CASES)
def test_int8_decode_matches_oracle(name):
    import torch

    step, g, host16, host8, pool8, cache = _setup(name)
    cfg = step.cfg
    tabs = H.device_tables(step)
    q, k, v = H.device_qkv(step, 0)
    q_out = cache.append_rope(0, q, k, v, tabs["pos_map"], tabs["append_indptr"], tabs["page_indptr"],
                              tabs["page_indices"])
    counters = torch.zeros(step.batch * cfg.hkv, dtype=torch.int32, device="cuda")
    out, lse = cache.decode_attention_merged(0, q_out, tabs["page_indptr"], tabs["page_indices"],
                                             tabs["last_page_len"], step.max_pages_per_seq, counters,
                                             q_indptr=tabs["q_indptr"], total_pages=int(step.page_indptr[-1]))
    po, pl, S = cache.decode_attention(0, q_out, tabs["page_indptr"], tabs["page_indices"], tabs["last_page_len"],
                                       step.max_pages_per_seq, q_indptr=tabs["q_indptr"],
                                       total_pages=int(step.page_indptr[-1]), num_splits=3)
    torch.cuda.synchronize()
    assert cache.check_status() == (0, 0)
    gpool8 = pool8.cpu().numpy()
    gq = _bits(q_out).view(np.uint16)[H.query_rows(step)]
    # attention isolated: the oracle over the GPU's own int8 cache and rotated queries
    ref_out, ref_lse = oracle.attention_int8(g, gpool8, gq, step.page_indptr, step.page_indices,
                                             step.last_page_len)
    H.assert_close_out(_bits(out).view(np.uint16), ref_out)
    H.assert_close_lse(lse.cpu().numpy(), ref_lse)
    rpo, rpl = oracle.split_attention_int8(g, gpool8, gq, step.page_indptr, step.page_indices,
                                           step.last_page_len, num_splits=3, num_out_splits=S)
    H.assert_close_lse(pl.cpu().numpy(), rpl, "partial_lse")
    H.assert_close_partial_o(po.cpu().numpy(), rpo, rpl)
    # end to end: the oracle's own int8 append and attention
    qh, kh, vh = W.new_qkv(step, 0)
    ref8 = host8.copy()
    oq = oracle.append_int8(g, qh, kh, vh, step.pos_map, step.append_indptr, step.page_indptr, step.page_indices,
                            ref8)
    e_out, e_lse = oracle.attention_int8(g, ref8, oq[H.query_rows(step)], step.page_indptr, step.page_indices,
                                         step.last_page_len)
    H.assert_close_out(_bits(out).view(np.uint16), e_out, "out (end to end)")
    H.assert_close_lse(lse.cpu().numpy(), e_lse, "lse (end to end)")


@pytest.mark.parametrize("name", ["gqa2_d128_outliers", "gqa8_d128"])
def test_int8_step_entry_point_runs_append_then_merged_decode(name):
    import torch

    step, g, host16, host8, pool_a, cache_a = _setup(name)
    _, _, _, _, pool_b, cache_b = _setup(name)
    cfg = step.cfg
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
    assert np.array_equal(pool_a.cpu().numpy(), pool_b.cpu().numpy())
    assert np.array_equal(_bits(out_a), _bits(out_b)) and np.array_equal(_bits(lse_a), _bits(lse_b))


@pytest.mark.parametrize("name", ["gqa2_d128_outliers", "ragged_d96", "gqa4_d64", "gqa8_d128", "tiny"])
@pytest.mark.parametrize("window", [1, 17, 100])
@pytest.mark.parametrize("with_sinks", [False, True])
def test_int8_window_and_sinks_match_oracle(name, window, with_sinks):
    """A windowed int8 layer (the first visible page may start inside a two-page stage's first page)
    with and without sink logits: merged decode against the oracle over the GPU's own int8 pool."""
    import torch

    import paged_kv_decode_pkv_gb300 as pkv

    cfg = SMALL[name]
    step = W.make_step(cfg)
    g = H.geometry(step)
    pool8 = torch.from_numpy(oracle.quantize_pool(g, W.host_pool(step, 0))).cuda()
    rng = np.random.default_rng(300 + window)
    sinks_host = (rng.standard_normal(cfg.hq) * 2).astype(np.float32) if with_sinks else None
    sinks = torch.from_numpy(sinks_host).cuda() if with_sinks else None
    cache = pkv.Cache(1, step.num_pages, cfg.hq, cfg.hkv, cfg.head_dim, step.max_position, cfg.theta,
                      pools=[pool8], options=pkv.OPT_INT8_KV, windows=[window], sinks=[sinks])
    tabs = H.device_tables(step)
    q, k, v = H.device_qkv(step, 0)
    q_out = cache.append_rope(0, q, k, v, tabs["pos_map"], tabs["append_indptr"], tabs["page_indptr"],
                              tabs["page_indices"])
    counters = torch.zeros(step.batch * cfg.hkv, dtype=torch.int32, device="cuda")
    out, lse = cache.decode_attention_merged(0, q_out, tabs["page_indptr"], tabs["page_indices"],
                                             tabs["last_page_len"], step.max_pages_per_seq, counters,
                                             q_indptr=tabs["q_indptr"], total_pages=int(step.page_indptr[-1]))
    torch.cuda.synchronize()
    assert cache.check_status() == (0, 0)
    gq = _bits(q_out).view(np.uint16)[H.query_rows(step)]
    ref_out, ref_lse = oracle.attention_int8(g, pool8.cpu().numpy(), gq, step.page_indptr, step.page_indices,
                                             step.last_page_len, window=window,
                                             sinks=None if sinks_host is None else sinks_host.astype(np.float64))
    H.assert_close_out(_bits(out).view(np.uint16), ref_out)
    H.assert_close_lse(lse.cpu().numpy(), ref_lse)


@pytest.mark.parametrize("which", [0, 1])
def test_int8_bad_page_in_a_stage_sets_status_and_masks_it(which):
    """A page id out of range as the first (which = 0) or second (which = 1) page of a two-page
    stage: the status word reports it, the page is masked out, the other sequences are unchanged."""
    import torch

    import paged_kv_decode_pkv_gb300 as pkv

    step, g, host16, host8, pool8, cache = _setup("ragged_d96")
    cfg = step.cfg
    tabs = H.device_tables(step)
    q, k, v = H.device_qkv(step, 0)
    q_out = cache.append_rope(0, q, k, v, tabs["pos_map"], tabs["append_indptr"], tabs["page_indptr"],
                              tabs["page_indices"])

    def run(pages):
        counters = torch.zeros(step.batch * cfg.hkv, dtype=torch.int32, device="cuda")
        out, lse = cache.decode_attention_merged(0, q_out, tabs["page_indptr"], pages, tabs["last_page_len"],
                                                 step.max_pages_per_seq, counters, q_indptr=tabs["q_indptr"],
                                                 num_splits=1)
        torch.cuda.synchronize()
        return out, lse, cache.check_status()

    good_out, good_lse, st = run(tabs["page_indices"])
    assert st == (0, 0)
    s = int(np.argmax(np.diff(step.page_indptr)))  # the longest sequence: one chunk, pages in pairs
    assert int(step.page_indptr[s + 1] - step.page_indptr[s]) >= 4
    bad = tabs["page_indices"].clone()
    bad[int(step.page_indptr[s]) + 2 + which] = step.num_pages + 5
    out, lse, (code, flags) = run(bad)
    assert code == pkv.ERR_OUT_OF_RANGE and flags & pkv.FLAG_BAD_PAGE
    others = [i for i in range(step.batch) if i != s]
    assert np.array_equal(_bits(out)[others], _bits(good_out)[others])
    assert np.all(np.isfinite(out.float().cpu().numpy()[s]))
