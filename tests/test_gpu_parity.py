"""Parity of the CUDA path (through the C ABI) with the oracle, on the same seeded inputs.

Small cases compare every output element: the whole pool image after the append (placement
bit-exact, V bit-exact, K and q_out within one fp16 step), the partials of explicit split plans,
and the combined output and LSE, both (i) against the oracle's attention over the GPU's own
cache and rotated queries and (ii) end to end against the oracle's own append.  The full-size
workloads run the chain exactly as the bench launches it (automatic split plan) and compare
sampled sequences, regenerated on the host, one by one.
"""
import numpy as np
import pytest

from pkv_inputs import workloads as W
from tests import harness as H

pytestmark = pytest.mark.gpu

SMALL = {
    "tiny": W.CONFIGS[1],
    "phi3_b1_ctx300": W.scaled(W.CONFIGS[2], layers=2, lengths=("fixed", 300), pool_pages=24),
    "ragged_d96": W.scaled(W.CONFIGS[3], batch=9, pool_pages=3000),
    "gqa2_d128_outliers": W.scaled(W.CONFIGS[4], layers=2, batch=3, lengths=("fixed", 1000), pool_pages=260),
    "gqa4_mixed_chunks": W.scaled(W.CONFIGS[5], batch=12, lengths=("loguniform", 16, 3000), pool_pages=3000,
                                  chunk_seqs=3, chunk_tokens=40),
    "gqa2_d96": W.scaled(W.CONFIGS[3], hq=16, hkv=8, batch=5, lengths=("uniform", 1, 700), pool_pages=600),
    "gqa4_d64": W.scaled(W.CONFIGS[3], hq=16, hkv=4, head_dim=64, batch=5, lengths=("uniform", 1, 500),
                         pool_pages=400),
    "gqa8_d128": W.scaled(W.CONFIGS[5], hq=32, hkv=4, batch=4, lengths=("uniform", 20, 900), pool_pages=300,
                          chunk_seqs=0, chunk_tokens=0),
    "mha_d64_long": W.scaled(W.CONFIGS[1], batch=2, lengths=("fixed", 2100), pool_pages=400,
                             page_table="permuted", num_splits=0),
}


def _gpu_pool_after(case_cfg, layer=0, plan=None):
    import torch

    step = W.make_step(case_cfg)
    host_pool = W.host_pool(step, layer)
    pool_dev = H.to_dev(host_pool, torch.float16)
    cache = H.make_cache(step, [0], [pool_dev])
    tabs = H.device_tables(step)
    q, k, v = H.device_qkv(step, layer)
    plan = plan or {}
    q_out, po, pl, out, lse = H.run_chain(cache, 0, tabs, q, k, v, step, **plan)
    torch.cuda.synchronize()
    code, flags = cache.check_status()
    assert code == 0 and flags == 0, f"device status {code} flags {flags:#x}"
    return step, host_pool, cache, tabs, dict(
        pool=pool_dev.view(torch.int16).cpu().numpy().view(np.uint16), q_out=q_out.view(torch.int16).cpu().numpy().view(np.uint16),
        po=po.cpu().numpy(), pl=pl.cpu().numpy(), out=out.view(torch.int16).cpu().numpy().view(np.uint16),
        lse=lse.cpu().numpy())


def _check_placement(step, gpu_pool, gpu_qout, ref):
    nan_ref = (ref["pool"] & 0x7C00) == 0x7C00
    nan_gpu = (gpu_pool & 0x7C00) == 0x7C00
    assert np.array_equal(nan_ref, nan_gpu), "written slot set differs from the oracle"
    assert np.array_equal(gpu_pool[:, 1], ref["pool"][:, 1]), "V must be bit-exact"
    kmask = ~nan_ref[:, 0]
    d = H.ulp_distance(gpu_pool[:, 0][kmask], ref["pool"][:, 0][kmask])
    assert d.max(initial=0) <= 1, f"K differs by {d.max()} fp16 steps"
    dq = H.ulp_distance(gpu_qout, ref["q_out"])
    assert dq.max(initial=0) <= 1, f"q_out differs by {dq.max()} fp16 steps"


@pytest.mark.parametrize("name", list(SMALL))
def test_chain_parity_small(name):
    cfg = SMALL[name]
    plan = {"num_splits": cfg.num_splits} if cfg.num_splits else {}
    step, host_pool, cache, tabs, g = _gpu_pool_after(cfg, plan=plan)
    q, k, v = W.new_qkv(step, 0)
    ref = H.oracle_chain(step, host_pool, q, k, v)
    _check_placement(step, g["pool"], g["q_out"], ref)
    # (ii) end to end from the oracle's own append
    H.assert_close_out(g["out"], ref["out"], "out vs oracle end to end")
    H.assert_close_lse(g["lse"], ref["lse"], "lse vs oracle end to end")
    # (i) the oracle's attention over the GPU's own cache and rotated queries
    out_i, lse_i = H.oracle_attention_on(step, g["pool"], g["q_out"][H.query_rows(step)])
    H.assert_close_out(g["out"], out_i, "out vs oracle on the GPU cache")
    H.assert_close_lse(g["lse"], lse_i, "lse vs oracle on the GPU cache")


@pytest.mark.parametrize("name", ["tiny", "ragged_d96", "gqa4_mixed_chunks", "gqa2_d96", "gqa4_d64"])
@pytest.mark.parametrize("plan", [{"num_splits": 1}, {"num_splits": 3}, {"num_splits": 7}, {"chunk_pages": 1},
                                  {"chunk_pages": 5}, {"chunk_pages": 64}])
def test_partials_parity_explicit_plans(name, plan):
    import oracle

    step, host_pool, cache, tabs, g = _gpu_pool_after(SMALL[name], plan=plan)
    gq = g["q_out"][H.query_rows(step)]
    po, pl = oracle.split_attention(H.geometry(step), g["pool"], gq, step.page_indptr, step.page_indices,
                                    step.last_page_len, num_out_splits=g["pl"].shape[2], **plan)
    H.assert_close_lse(g["pl"], pl, "partial_lse")
    H.assert_close_partial_o(g["po"], po, pl)
    out, out16, lse = oracle.combine(po, pl)
    H.assert_close_out(g["out"], out)
    H.assert_close_lse(g["lse"], lse)


@pytest.mark.parametrize("name", ["tiny", "phi3_b1_ctx300", "ragged_d96", "gqa4_mixed_chunks", "gqa2_d96",
                                  "gqa4_d64", "gqa8_d128", "mha_d64_long"])
def test_partials_parity_balanced_partition(name):
    """The automatic plan with the exact page total: every piece of the page-balanced partition."""
    import oracle

    step, host_pool, cache, tabs, g = _gpu_pool_after(SMALL[name], plan={})
    S, chunk = cache.plan_decode(step.batch, step.max_pages_per_seq, int(step.page_indptr[-1]))
    assert chunk == -1 and g["pl"].shape[2] == S
    sms, warps = cache.device_info(step.batch)
    W = min(sms * warps, step.cfg.hkv * int(step.page_indptr[-1]))
    gq = g["q_out"][H.query_rows(step)]
    po, pl = oracle.split_attention_balanced(H.geometry(step), g["pool"], gq, step.page_indptr, step.page_indices,
                                             step.last_page_len, W, S)
    H.assert_close_lse(g["pl"], pl, "partial_lse")
    H.assert_close_partial_o(g["po"], po, pl)


@pytest.mark.parametrize("name", ["tiny", "phi3_b1_ctx300", "ragged_d96", "gqa4_mixed_chunks", "gqa8_d128",
                                  "gqa2_d96", "mha_d64_long"])
@pytest.mark.parametrize("plan", [{}, {"num_splits": 3}, {"chunk_pages": 2}])
def test_merged_decode_is_bit_identical_to_decode_then_combine(name, plan):
    import torch

    step, host_pool, cache, tabs, g = _gpu_pool_after(SMALL[name], plan=plan)
    cfg = step.cfg
    counters = torch.zeros(step.batch * cfg.hkv, dtype=torch.int32, device="cuda")
    q_out = torch.from_numpy(g["q_out"]).view(torch.float16).cuda()
    tp = int(step.page_indptr[-1])
    for _ in range(2):  # the second call checks that the counters were left at zero
        out, lse = cache.decode_attention_merged(0, q_out, tabs["page_indptr"], tabs["page_indices"],
                                                 tabs["last_page_len"], step.max_pages_per_seq, counters,
                                                 q_indptr=tabs["q_indptr"], total_pages=tp, **plan)
        torch.cuda.synchronize()
        assert cache.check_status()[0] == 0
        assert np.array_equal(out.view(torch.int16).cpu().numpy().view(np.uint16), g["out"])
        assert np.array_equal(lse.cpu().numpy().view(np.uint32), g["lse"].view(np.uint32))
        assert int(counters.abs().sum()) == 0


def test_device_generator_matches_host():
    import torch

    import pkv_inputs

    k = pkv_inputs.key(11, 22)
    okey = pkv_inputs.key(11, 23)
    n = 3_000_017
    t = torch.empty(n, dtype=torch.float16, device="cuda")
    pkv_inputs.dev_fill_range(t.data_ptr(), n, k, 12345, 0.1020620726, okey, 128, 1)
    torch.cuda.synchronize()
    host = pkv_inputs.fill_range(n, k, 12345, 0.1020620726, okey, 128, 1)
    assert np.array_equal(t.view(torch.int16).cpu().numpy().view(np.uint16), host)


# ------------------------------------------------------------------------------------------------
# full-size workloads, sampled


def _full_size_check(cid, layers_to_check, seqs_fn):
    """The workload at its full size, launched as bench.py launches it (pkv_append_decode_attention
    per layer, programmatic dependent launch with early page copies, the planner's automatic split),
    checked on sampled sequences regenerated on the host."""
    import torch

    import paged_kv_decode_pkv_gb300 as pkv

    cfg = W.CONFIGS[cid]
    step = W.make_step(cfg)
    tabs = H.device_tables(step)
    layers = list(range(cfg.layers))
    pools = [W.device_pool(step, l) for l in layers]
    sinks_host = [W.sink_logits(step, l) for l in layers] if cfg.sinks else None
    sinks = [torch.from_numpy(x).cuda() for x in sinks_host] if cfg.sinks else None
    cache = pkv.Cache(cfg.layers, step.num_pages, cfg.hq, cfg.hkv, cfg.head_dim, step.max_position, cfg.theta,
                      pools=pools, options=pkv.OPT_PDL | pkv.OPT_EARLY_PAGES,
                      windows=[cfg.window] * cfg.layers if cfg.window else None,
                      sinks=sinks)
    tp = int(step.page_indptr[-1])
    counters = torch.zeros(step.batch * cfg.hkv, dtype=torch.int32, device="cuda")
    outs = {}
    for l in layers:
        q, k, v = H.device_qkv(step, l)
        q_out, out, lse = cache.append_decode_attention(
            l, q, k, v, tabs["pos_map"], tabs["append_indptr"], tabs["page_indptr"], tabs["page_indices"],
            tabs["last_page_len"], step.max_pages_per_seq, counters, total_pages=tp)
        if l in layers_to_check:
            outs[l] = (q_out, out, lse)
    torch.cuda.synchronize()
    code, flags = cache.check_status()
    assert code == 0 and flags == 0
    seqs = seqs_fn(step)
    sub = W.substep(step, seqs)
    rows = W.token_rows(step, seqs)
    for l in layers_to_check:
        q_out, out, lse = outs[l]
        sk = None if sinks_host is None else sinks_host[l].astype(np.float64)
        pool_sub = W.host_pool_pages(sub, l, np.arange(sub.num_pages))
        q, k, v = W.new_qkv(step, l, rows=rows)
        ref = H.oracle_chain(sub, pool_sub, q, k, v, window=cfg.window, sinks=sk)
        origin = torch.from_numpy(sub.page_origin).cuda()
        gpu_pages = pools[l].index_select(0, origin).view(torch.int16).cpu().numpy().view(np.uint16)
        gpu_qout = q_out.view(torch.int16)[torch.from_numpy(rows).cuda()].cpu().numpy().view(np.uint16)
        _check_placement(sub, gpu_pages, gpu_qout, ref)
        sel = torch.from_numpy(np.asarray(seqs)).cuda()
        g_out = out.view(torch.int16)[sel].cpu().numpy().view(np.uint16)
        g_lse = lse[sel].cpu().numpy()
        H.assert_close_out(g_out, ref["out"], f"config {cid} layer {l} out")
        H.assert_close_lse(g_lse, ref["lse"], f"config {cid} layer {l} lse")
        out_i, lse_i = H.oracle_attention_on(sub, gpu_pages, gpu_qout[H.query_rows(sub)], window=cfg.window,
                                             sinks=sk)
        H.assert_close_out(g_out, out_i, f"config {cid} layer {l} out (GPU cache)")
    del pools, cache
    torch.cuda.empty_cache()


def test_full_size_phi3_single_stream():
    _full_size_check(2, [0, 31], lambda st: [0])


def test_full_size_ragged_batch64():
    _full_size_check(3, [0], lambda st: [0, int(np.argmax(st.seq_len)), int(np.argmin(st.seq_len)), 63])


def test_full_size_gqa_long_context():
    _full_size_check(4, [0, 27], lambda st: [0, 7])


def test_full_size_mixed_serving():
    def pick(st):
        chunk = np.flatnonzero(st.new_tokens > 1)
        return sorted({int(np.argmax(st.seq_len)), int(np.argmin(st.seq_len)), int(chunk[0]), int(chunk[-1]), 5})
    _full_size_check(5, [0], pick)


def test_full_size_sliding_window_with_sinks():
    _full_size_check(6, [0, 7], lambda st: [0, 31])
