"""Properties of the CUDA path that hold at any size (GPU): exact invariances, degenerate cases,
and device-side error reporting through the status word."""
import numpy as np
import pytest

from pkv_inputs import workloads as W
from tests import harness as H

pytestmark = pytest.mark.gpu


def _bits(t):
    import torch

    return t.contiguous().view(torch.int32 if t.dtype == torch.float32 else torch.int16).cpu().numpy()


def _run(step, host_pool, plan=None, layer=0):
    import torch

    pool = H.to_dev(host_pool, torch.float16)
    cache = H.make_cache(step, [0], [pool])
    tabs = H.device_tables(step)
    q, k, v = H.device_qkv(step, layer)
    q_out, po, pl, out, lse = H.run_chain(cache, 0, tabs, q, k, v, step, **(plan or {}))
    torch.cuda.synchronize()
    code, flags = cache.check_status()
    return dict(cache=cache, pool=pool, q_out=q_out, po=po, pl=pl, out=out, lse=lse, code=code, flags=flags)


CASES = {
    "mha_d96": W.scaled(W.CONFIGS[3], batch=6, pool_pages=2000),
    "gqa4_d128": W.scaled(W.CONFIGS[5], batch=10, lengths=("loguniform", 16, 4000), pool_pages=3000,
                          chunk_seqs=2, chunk_tokens=33),
}


@pytest.mark.parametrize("name", list(CASES))
def test_page_permutation_gives_bit_identical_output(name):
    step = W.make_step(CASES[name])
    pool = W.host_pool(step, 0)
    a = _run(step, pool)
    rng = np.random.default_rng(5)
    perm = rng.permutation(step.num_pages)        # physical page i moves to perm[i]
    pool2 = np.empty_like(pool)
    pool2[perm] = pool
    step2 = W.make_step(CASES[name])
    step2.page_indices = perm[step.page_indices].astype(np.int32)
    b = _run(step2, pool2)
    for key in ("q_out", "out", "lse", "pl"):
        assert np.array_equal(_bits(a[key]), _bits(b[key])), key


@pytest.mark.parametrize("name", list(CASES))
def test_run_to_run_bit_identical(name):
    step = W.make_step(CASES[name])
    pool = W.host_pool(step, 0)
    a, b = _run(step, pool), _run(step, pool)
    for key in ("q_out", "out", "lse", "po", "pl"):
        if key == "po":
            mask = ~np.isinf(a["pl"].cpu().numpy())
            assert np.array_equal(_bits(a["po"])[mask], _bits(b["po"])[mask])
        else:
            assert np.array_equal(_bits(a[key]), _bits(b[key])), key


@pytest.mark.parametrize("name", list(CASES))
def test_split_count_does_not_change_the_result_beyond_tolerance(name):
    step = W.make_step(CASES[name])
    pool = W.host_pool(step, 0)
    q, k, v = W.new_qkv(step, 0)
    ref = H.oracle_chain(step, pool, q, k, v)
    for plan in ({"num_splits": 1}, {"num_splits": 4}, {"chunk_pages": 2}, {}):
        r = _run(step, pool, plan)
        H.assert_close_out(_bits(r["out"]).view(np.uint16), ref["out"], f"out {plan}")
        H.assert_close_lse(r["lse"].cpu().numpy(), ref["lse"], f"lse {plan}")


@pytest.mark.parametrize("hq,hkv,d", [(4, 4, 64), (32, 32, 96), (32, 8, 128), (16, 8, 96)])
def test_length_one_returns_v_exactly(hq, hkv, d):
    cfg = W.scaled(W.CONFIGS[1], batch=5, hq=hq, hkv=hkv, head_dim=d, lengths=("fixed", 1), pool_pages=9,
                   page_table="permuted", num_splits=0)
    step = W.make_step(cfg)
    r = _run(step, W.host_pool(step, 0))
    q, k, v = W.new_qkv(step, 0)
    expect = np.repeat(v, hq // hkv, axis=1)  # query head h reads KV head h / G
    assert np.array_equal(_bits(r["out"]).view(np.uint16), expect)
    # the LSE of a single token is its scaled score
    gp = _bits(r["pool"]).view(np.uint16)
    _, lse_ref = H.oracle_attention_on(step, gp, _bits(r["q_out"]).view(np.uint16))
    H.assert_close_lse(r["lse"].cpu().numpy(), lse_ref)


def test_position_zero_rotation_is_identity():
    cfg = W.scaled(W.CONFIGS[1], batch=3, lengths=("fixed", 1), pool_pages=5, num_splits=0)
    step = W.make_step(cfg)
    r = _run(step, W.host_pool(step, 0))
    q, k, v = W.new_qkv(step, 0)
    assert np.array_equal(_bits(r["q_out"]).view(np.uint16), q)
    pool = _bits(r["pool"]).view(np.uint16)
    for s in range(3):
        page = step.page_indices[step.page_indptr[s]]
        assert np.array_equal(pool[page, 0, :, 0, :], k[s])


def test_empty_sequence_and_zero_query():
    import torch

    cfg = W.scaled(W.CONFIGS[3], batch=4, pool_pages=1200)
    step = W.make_step(cfg)
    pool = W.host_pool(step, 0)
    # sequence 1 becomes empty: no pages, no appended token
    keep = np.array([0, 2, 3])
    n = np.diff(step.page_indptr)
    n[1] = 0
    step.page_indptr = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    old = W.make_step(cfg)
    step.page_indices = np.concatenate([old.page_indices[old.page_indptr[s]:old.page_indptr[s + 1]]
                                        for s in keep]).astype(np.int32)
    new = step.new_tokens.copy()
    new[1] = 0
    step.new_tokens = new
    step.append_indptr = np.concatenate([[0], np.cumsum(new)]).astype(np.int32)
    step.pos_map = np.concatenate([old.pos_map[old.append_indptr[s]:old.append_indptr[s + 1]]
                                   for s in keep]).astype(np.int32)
    step.seq_len = step.seq_len.copy()
    step.seq_len[1] = 0
    tabs = H.device_tables(step)
    tabs["q_indptr"] = tabs["append_indptr"]
    dev_pool = H.to_dev(pool, torch.float16)
    cache = H.make_cache(step, [0], [dev_pool])
    qh, kh, vh = W.new_qkv(old, 0)
    rows = W.token_rows(old, keep)
    q, k, v = (H.to_dev(x[rows], torch.float16) for x in (qh, kh, vh))
    q_out, po, pl, out, lse = H.run_chain(cache, 0, tabs, q, k, v, step)
    torch.cuda.synchronize()
    assert cache.check_status()[0] == 0
    o = out.float().cpu().numpy()
    l = lse.cpu().numpy()
    assert np.all(o[1] == 0) and np.all(np.isinf(l[1]) & (l[1] < 0))
    assert np.isfinite(o[[0, 2, 3]]).all()
    # zero queries: the output is the mean of V over the sequence, lse = ln(len)
    zq = torch.zeros_like(q_out)
    po, pl, S = cache.decode_attention(0, zq, tabs["page_indptr"], tabs["page_indices"], tabs["last_page_len"],
                                       step.max_pages_per_seq, q_indptr=tabs["q_indptr"], num_splits=3)
    out0, lse0 = cache.combine(po, pl)
    gp = dev_pool.view(torch.int16).cpu().numpy().view(np.uint16)
    out_ref, lse_ref = H.oracle_attention_on(step, gp, np.zeros((4, cfg.hq, cfg.head_dim), np.uint16))
    H.assert_close_out(_bits(out0).view(np.uint16)[[0, 2, 3]], out_ref[[0, 2, 3]])
    np.testing.assert_allclose(lse0.cpu().numpy()[[0, 2, 3]], np.log(step.seq_len[[0, 2, 3]])[:, None] *
                               np.ones((1, cfg.hq)), atol=H.LSE_ABS)


def test_device_errors_set_status_and_skip():
    import torch

    import paged_kv_decode_pkv_gb300 as pkv

    cfg = W.scaled(W.CONFIGS[3], batch=3, pool_pages=1000)
    step = W.make_step(cfg)
    pool = W.host_pool(step, 0)
    good = _run(step, pool)
    assert good["code"] == 0
    # a page id out of range in the decode page table: flagged, that page is masked out
    tabs = H.device_tables(step)
    bad_pages = tabs["page_indices"].clone()
    bad_pages[int(step.page_indptr[1])] = step.num_pages + 7
    cache = good["cache"]
    po, pl, S = cache.decode_attention(0, good["q_out"], tabs["page_indptr"], bad_pages, tabs["last_page_len"],
                                       step.max_pages_per_seq, total_pages=int(step.page_indptr[-1]))
    code, flags = cache.check_status()
    assert code == pkv.ERR_OUT_OF_RANGE and flags & pkv.FLAG_BAD_PAGE
    out, lse = cache.combine(po, pl)
    assert np.array_equal(_bits(out)[[0, 2]], _bits(good["out"])[[0, 2]])
    # a position beyond max_position in the append: flagged, the token is skipped
    q, k, v = H.device_qkv(step, 0)
    bad_pos = tabs["pos_map"].clone()
    bad_pos[0] = 1 << 30
    before = good["pool"].clone()
    cache.append_rope(0, q, k, v, bad_pos, tabs["append_indptr"], tabs["page_indptr"], tabs["page_indices"])
    code, flags = cache.check_status()
    assert code == pkv.ERR_OUT_OF_RANGE and flags & pkv.FLAG_BAD_POSITION
    # last_page_len outside [1, 16]: flagged, the sequence is reported empty
    bad_last = tabs["last_page_len"].clone()
    bad_last[2] = 0
    po, pl, S = cache.decode_attention(0, good["q_out"], tabs["page_indptr"], tabs["page_indices"], bad_last,
                                       step.max_pages_per_seq)
    code, flags = cache.check_status()
    assert code == pkv.ERR_OUT_OF_RANGE and flags & pkv.FLAG_BAD_SEQUENCE
    assert np.all(np.isinf(pl[2].cpu().numpy()))
    # more pages than declared: flagged
    po, pl, S = cache.decode_attention(0, good["q_out"], tabs["page_indptr"], tabs["page_indices"],
                                       tabs["last_page_len"], 1, chunk_pages=1)
    code, flags = cache.check_status()
    assert code == pkv.ERR_OUT_OF_RANGE and flags & pkv.FLAG_BAD_SEQUENCE
    del before
