"""Consecutive steps on one stream, as a serving loop issues them, against the oracle.

The one-launch step with programmatic dependent launch and early page copies starts copying the
cache before the previous kernels of the stream have finished.  These tests run two decode steps
back to back without a host synchronisation (step 2 appends position p + 1 right after step 1
appended p, on the same page or on a new one), on one-layer and two-layer caches (where the step-1
kernel of the same layer is one or two launches back), a chunked append followed by a decode step
of the same layer, and page tables written by an ordinary kernel right before the launch.  Step 2
is compared with the oracle's two appends and attention, and bit for bit with the same steps on a
cache without programmatic dependent launch.

The bounded waits are tested on a healthy GPU: the decode kernels' page stages are armed for more
bytes than they receive (a wait for something nothing provides), the prefill kernel's waits get a
limit shorter than a copy; the kernels report PKV_ERR_TIMEOUT, and the next call with the default
settings is checked against the oracle.
"""
import numpy as np
import pytest

import oracle
from pkv_inputs import workloads as W
from tests import harness as H

pytestmark = pytest.mark.gpu

# step-1 lengths: the step-2 token starts a new page (16, 32), lands in the last slot (31 -> 31),
# follows an empty history (1), or sits anywhere in a page
LENS = [16, 47, 1, 100, 32, 31, 250, 63]
CFGS = {
    "g1_d96": W.scaled(W.CONFIGS[2], layers=2, batch=len(LENS), pool_pages=160, page_table="permuted"),
    "g4_d128": W.scaled(W.CONFIGS[5], layers=2, batch=len(LENS), pool_pages=160, chunk_seqs=0, chunk_tokens=0),
    "g2_d128": W.scaled(W.CONFIGS[4], layers=2, batch=len(LENS), pool_pages=160, outlier_pct=1),
}


def _step(cfg, seed, lens, new, pages_of, pool_pages):
    """A Step whose sequences hold `lens` tokens after appending `new` tokens each, with page lists
    taken from the front of each sequence's reserved pages."""
    lens = np.asarray(lens, dtype=np.int64)
    new = np.asarray(new, dtype=np.int64)
    n = (lens + 15) // 16
    pages = np.concatenate([pages_of[s][: n[s]] for s in range(lens.size)])
    page_indptr = np.concatenate([[0], np.cumsum(n)])
    append_indptr = np.concatenate([[0], np.cumsum(new)])
    pos_map = np.concatenate([np.arange(lens[s] - new[s], lens[s]) for s in range(lens.size)])
    return W.Step(cfg=cfg, seed=seed, seq_len=lens, new_tokens=new, page_indptr=page_indptr.astype(np.int32),
                  page_indices=pages.astype(np.int32), last_page_len=(lens - (n - 1) * 16).astype(np.int32),
                  append_indptr=append_indptr.astype(np.int32), pos_map=pos_map.astype(np.int32),
                  num_pages=pool_pages)


def _reserved_pages(cfg, lens_max, seed):
    """Disjoint seeded page lists per sequence, long enough for `lens_max` tokens."""
    n = (np.asarray(lens_max) + 15) // 16
    order = np.random.default_rng(seed).permutation(cfg.pool_pages)
    starts = np.concatenate([[0], np.cumsum(n)])
    assert starts[-1] <= cfg.pool_pages
    return [order[starts[s]:starts[s + 1]] for s in range(len(n))]


def _steps(cfg, first_new=1):
    """Step 1 appends `first_new` tokens per sequence ending at LENS - 1; step 2 appends one more."""
    seed = W.SEED_BASE + 900 + cfg.cid
    lens = np.asarray(LENS, dtype=np.int64)
    reserved = _reserved_pages(cfg, lens + 1, seed)
    new1 = np.minimum(first_new, lens)
    s1 = _step(cfg, seed, lens, new1, reserved, cfg.pool_pages)
    s2 = _step(cfg, seed + 1, lens + 1, np.ones_like(lens), reserved, cfg.pool_pages)
    return s1, s2


def _bits(t):
    import torch

    return t.contiguous().view(torch.int32 if t.dtype == torch.float32 else torch.int16).cpu().numpy()


def _oracle_two_steps(s1, s2, layer):
    g = H.geometry(s2)  # step 2 holds the largest positions
    pool = W.host_pool(s1, layer).copy()
    q1, k1, v1 = W.new_qkv(s1, layer)
    q_out1 = oracle.append(g, q1, k1, v1, s1.pos_map, s1.append_indptr, s1.page_indptr, s1.page_indices, pool)
    out1, lse1 = oracle.attention(g, pool, q_out1[H.query_rows(s1)], s1.page_indptr, s1.page_indices,
                                  s1.last_page_len)
    q2, k2, v2 = W.new_qkv(s2, layer)
    q_out2 = oracle.append(g, q2, k2, v2, s2.pos_map, s2.append_indptr, s2.page_indptr, s2.page_indices, pool)
    out2, lse2 = oracle.attention(g, pool, q_out2[H.query_rows(s2)], s2.page_indptr, s2.page_indices,
                                  s2.last_page_len)
    return pool, (out1, lse1), (out2, lse2)


def _run_two_steps(s1, s2, layers, options, first="one_launch", tables2_by_kernel=False):
    """Both steps on one stream with no synchronisation between them; returns the pools and the
    outputs of both steps per layer."""
    import torch

    cfg = s1.cfg
    pools = [H.to_dev(W.host_pool(s1, l), torch.float16) for l in layers]
    cache = H.make_cache(s2, layers, pools, options=options)  # step 2 holds the largest positions
    t1 = H.device_tables(s1)
    t2 = H.device_tables(s2)
    if tables2_by_kernel:
        # step 2's page table and positions start out wrong and are written by ordinary (torch)
        # kernels launched right before step 2's kernels
        src = {k: t2[k].clone() for k in ("page_indices", "pos_map")}
        for k in src:
            t2[k] = torch.zeros_like(src[k])
        torch.cuda.synchronize()
    counters = torch.zeros(max(s1.batch, s2.batch) * cfg.hkv, dtype=torch.int32, device="cuda")
    qkv1 = [H.device_qkv(s1, l) for l in layers]
    qkv2 = [H.device_qkv(s2, l) for l in layers]
    res1, res2 = {}, {}
    for i, l in enumerate(layers):
        q, k, v = qkv1[i]
        if first == "one_launch":
            _, out, lse = cache.append_decode_attention(
                i, q, k, v, t1["pos_map"], t1["append_indptr"], t1["page_indptr"], t1["page_indices"],
                t1["last_page_len"], s1.max_pages_per_seq, counters, total_pages=int(s1.page_indptr[-1]))
            res1[l] = (out, lse)
        else:  # a chunked append of the layer and nothing else
            cache.append_rope(i, q, k, v, t1["pos_map"], t1["append_indptr"], t1["page_indptr"], t1["page_indices"])
    if tables2_by_kernel:
        for k in src:
            torch.add(src[k], 0, out=t2[k])
    for i, l in enumerate(layers):
        q, k, v = qkv2[i]
        _, out, lse = cache.append_decode_attention(
            i, q, k, v, t2["pos_map"], t2["append_indptr"], t2["page_indptr"], t2["page_indices"],
            t2["last_page_len"], s2.max_pages_per_seq, counters, total_pages=int(s2.page_indptr[-1]))
        res2[l] = (out, lse)
    torch.cuda.synchronize()
    code, flags = cache.check_status()
    assert code == 0 and flags == 0, f"device status {code} flags {flags:#x}"
    assert int(counters.abs().sum()) == 0
    return pools, res1, res2


def _check_against_oracle(s1, s2, layers, pools, res1, res2):
    for i, l in enumerate(layers):
        ref_pool, ref1, ref2 = _oracle_two_steps(s1, s2, l)
        gp = _bits(pools[i]).view(np.uint16)
        used = s2.page_indices
        nan_ref = (ref_pool[used] & 0x7C00) == 0x7C00
        assert np.array_equal((gp[used] & 0x7C00) == 0x7C00, nan_ref), f"layer {l}: written slot set"
        assert np.array_equal(gp[used][:, 1], ref_pool[used][:, 1]), f"layer {l}: V must be bit-exact"
        kmask = ~nan_ref[:, 0]
        assert H.ulp_distance(gp[used][:, 0][kmask], ref_pool[used][:, 0][kmask]).max(initial=0) <= 1
        if l in res1:
            H.assert_close_out(_bits(res1[l][0]).view(np.uint16), ref1[0], f"layer {l} step 1 out")
            H.assert_close_lse(res1[l][1].cpu().numpy(), ref1[1], f"layer {l} step 1 lse")
        H.assert_close_out(_bits(res2[l][0]).view(np.uint16), ref2[0], f"layer {l} step 2 out")
        H.assert_close_lse(res2[l][1].cpu().numpy(), ref2[1], f"layer {l} step 2 lse")


@pytest.mark.parametrize("name", list(CFGS))
@pytest.mark.parametrize("nlayers", [1, 2])
def test_two_decode_steps_back_to_back_with_early_pages(name, nlayers):
    import paged_kv_decode_pkv_gb300 as pkv

    s1, s2 = _steps(CFGS[name])
    layers = list(range(nlayers))
    pools, r1, r2 = _run_two_steps(s1, s2, layers, pkv.OPT_PDL | pkv.OPT_EARLY_PAGES)
    _check_against_oracle(s1, s2, layers, pools, r1, r2)
    # the same two steps with plain launches give the same bits
    pools_p, r1_p, r2_p = _run_two_steps(s1, s2, layers, 0)
    for i, l in enumerate(layers):
        assert np.array_equal(_bits(pools[i]), _bits(pools_p[i])), f"layer {l}: pool image"
        for a, b in ((r1[l], r1_p[l]), (r2[l], r2_p[l])):
            assert np.array_equal(_bits(a[0]), _bits(b[0])) and np.array_equal(_bits(a[1]), _bits(b[1]))


@pytest.mark.parametrize("name", ["g1_d96", "g4_d128"])
def test_chunked_append_then_decode_step_of_the_same_layer(name):
    """A 20-token append of each sequence (pkv_append_rope) directly followed by the one-launch
    decode step of the same layer: that step must not copy pages before its launch wait."""
    import paged_kv_decode_pkv_gb300 as pkv

    s1, s2 = _steps(CFGS[name], first_new=20)
    layers = [0]
    pools, r1, r2 = _run_two_steps(s1, s2, layers, pkv.OPT_PDL | pkv.OPT_EARLY_PAGES, first="append")
    _check_against_oracle(s1, s2, layers, pools, r1, r2)


@pytest.mark.parametrize("name", ["g1_d96", "g2_d128"])
def test_page_table_written_by_an_ordinary_kernel_right_before(name):
    """Step 2's page_indices and pos_map are written by torch kernels launched right before step 2
    (kernels without programmatic dependent launch, so they finish before the next one starts)."""
    import paged_kv_decode_pkv_gb300 as pkv

    s1, s2 = _steps(CFGS[name])
    layers = [0, 1]
    pools, r1, r2 = _run_two_steps(s1, s2, layers, pkv.OPT_PDL | pkv.OPT_EARLY_PAGES, tables2_by_kernel=True)
    _check_against_oracle(s1, s2, layers, pools, r1, r2)


# ------------------------------------------------------------------------------------------------
# bounded waits


TIMEOUT_CASES = {
    "g1_d96": W.scaled(W.CONFIGS[2], layers=1, lengths=("fixed", 600), pool_pages=40),
    "g4_d128": W.scaled(W.CONFIGS[5], batch=6, lengths=("loguniform", 16, 2000), pool_pages=400, chunk_seqs=2,
                        chunk_tokens=30),
}


@pytest.mark.parametrize("name", list(TIMEOUT_CASES))
@pytest.mark.parametrize("entry", ["merged", "one_launch", "prefill"])
def test_wait_timeout_is_reported_and_the_next_call_is_correct(name, entry):
    import torch

    import paged_kv_decode_pkv_gb300 as pkv

    cfg = TIMEOUT_CASES[name]
    if entry == "one_launch":
        cfg = W.scaled(cfg, chunk_seqs=0, chunk_tokens=0)
    if entry == "prefill" and not cfg.chunk_seqs:
        cfg = W.scaled(cfg, batch=2, chunk_seqs=1, chunk_tokens=40, pool_pages=100)
    step = W.make_step(cfg)
    host_pool = W.host_pool(step, 0)
    tabs = H.device_tables(step)
    q, k, v = H.device_qkv(step, 0)
    tp = int(step.page_indptr[-1])

    def run(cache, pool):
        counters = torch.zeros(step.batch * cfg.hkv, dtype=torch.int32, device="cuda")
        if entry == "one_launch":
            _, out, lse = cache.append_decode_attention(
                0, q, k, v, tabs["pos_map"], tabs["append_indptr"], tabs["page_indptr"], tabs["page_indices"],
                tabs["last_page_len"], step.max_pages_per_seq, counters, total_pages=tp)
            return out, lse
        q_out = cache.append_rope(0, q, k, v, tabs["pos_map"], tabs["append_indptr"], tabs["page_indptr"],
                                  tabs["page_indices"])
        torch.cuda.synchronize()
        if entry == "merged":
            return cache.decode_attention_merged(0, q_out, tabs["page_indptr"], tabs["page_indices"],
                                                 tabs["last_page_len"], step.max_pages_per_seq, counters,
                                                 q_indptr=tabs["q_indptr"], total_pages=tp)
        return cache.prefill_attention(0, q_out, tabs["append_indptr"], tabs["pos_map"], tabs["page_indptr"],
                                       tabs["page_indices"], tabs["last_page_len"])

    pool = H.to_dev(host_pool, torch.float16)
    cache = H.make_cache(step, [0], [pool], options=pkv.OPT_PDL | pkv.OPT_EARLY_PAGES)
    cache.set_wait_limit(1)  # 1 ns: the prefill kernel's waits for its copies run out
    if entry != "prefill":
        cache.set_stage_stall(True)  # the decode stages never complete: every stage wait runs out
    run(cache, pool)
    code, flags = cache.check_status()
    assert code == pkv.ERR_TIMEOUT and flags & pkv.FLAG_TIMEOUT, (code, flags)
    # the default settings again, on a fresh pool (the timed-out launch left its work unfinished)
    cache.set_wait_limit(0)
    cache.set_stage_stall(False)
    pool.copy_(H.to_dev(host_pool, torch.float16))
    out, lse = run(cache, pool)
    torch.cuda.synchronize()
    assert cache.check_status() == (0, 0)
    g = H.geometry(step)
    if entry == "prefill":
        gp = _bits(pool).view(np.uint16)
        q_out = cache.append_rope(0, q, k, v, tabs["pos_map"], tabs["append_indptr"], tabs["page_indptr"],
                                  tabs["page_indices"])  # the same bits again (no compute change)
        torch.cuda.synchronize()
        ref_out, ref_lse = oracle.prefill_attention(g, gp, _bits(q_out).view(np.uint16), step.append_indptr,
                                                    step.pos_map, step.page_indptr, step.page_indices,
                                                    step.last_page_len)
    else:
        qh, kh, vh = W.new_qkv(step, 0)
        ref = H.oracle_chain(step, host_pool, qh, kh, vh)
        ref_out, ref_lse = ref["out"], ref["lse"]
    H.assert_close_out(_bits(out).view(np.uint16), ref_out)
    H.assert_close_lse(lse.cpu().numpy(), ref_lse)
