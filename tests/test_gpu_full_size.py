"""Parity at the sizes the benchmark measures, for the paths beyond the decode step.

* Chunked prefill on the mixed-serving workload at full size (128 sequences of log-uniform length
  in [16, 65 536], 16 of them appending 512-token chunks, a permuted 600 000-page pool): the step
  runs as the benchmark runs it (the chunked append, the merged decode, then prefill attention
  over the 16 chunk sequences), and every row of the longest, the shortest and two other chunk
  sequences is compared with the oracle's causal attention over the GPU's own cache and rotated
  queries.
* The int8 KV cache on the long-context GQA workload (8 x 32 768 tokens; two of its 28 layers,
  the per-layer work is the same for every layer), on the ragged Phi-3 batch (one query head per
  KV head) and on the mixed-serving workload at full size,
  run through the one-launch entry point as `bench.py --int8` runs it, compared on sampled
  sequences with the oracle's int8 attention over the GPU's own int8 pool.

Sampled sequences are regenerated on the host page by page (only their pages are read back).
"""
import numpy as np
import pytest

import oracle
from pkv_inputs import workloads as W
from tests import harness as H

pytestmark = pytest.mark.gpu


def _bits(t):
    import torch

    return t.contiguous().view(torch.int32 if t.dtype == torch.float32 else torch.int16).cpu().numpy()


def _chunk_tables(step, dev):
    """Page tables restricted to the sequences that appended a chunk, as the benchmark's prefill
    measurement builds them; returns (sequences, token rows, device tables)."""
    import torch

    seqs = np.flatnonzero(step.new_tokens > 1)
    ai = np.concatenate([[0], np.cumsum(step.new_tokens[seqs])]).astype(np.int32)
    rows = np.concatenate([np.arange(step.append_indptr[s], step.append_indptr[s + 1]) for s in seqs])
    pi = np.concatenate([[0], np.cumsum(np.diff(step.page_indptr)[seqs])]).astype(np.int32)
    px = np.concatenate([step.page_indices[step.page_indptr[s]:step.page_indptr[s + 1]] for s in seqs])
    tabs = {"append_indptr": ai, "pos_map": step.pos_map[rows], "page_indptr": pi, "page_indices": px,
            "last_page_len": step.last_page_len[seqs]}
    tabs = {k: torch.from_numpy(np.ascontiguousarray(v, dtype=np.int32)).to(dev) for k, v in tabs.items()}
    return seqs, rows, tabs


def test_full_size_prefill_mixed_serving():
    import torch

    import paged_kv_decode_pkv_gb300 as pkv

    cfg = W.CONFIGS[5]
    step = W.make_step(cfg)
    dev = torch.device("cuda")
    pool = W.device_pool(step, 0)
    cache = pkv.Cache(1, step.num_pages, cfg.hq, cfg.hkv, cfg.head_dim, step.max_position, cfg.theta, pools=[pool],
                      options=pkv.OPT_PDL | pkv.OPT_EARLY_PAGES)
    tabs = H.device_tables(step)
    q, k, v = H.device_qkv(step, 0)
    counters = torch.zeros(step.batch * cfg.hkv, dtype=torch.int32, device=dev)
    q_out, _, _ = cache.append_decode_attention(0, q, k, v, tabs["pos_map"], tabs["append_indptr"],
                                                tabs["page_indptr"], tabs["page_indices"], tabs["last_page_len"],
                                                step.max_pages_per_seq, counters,
                                                total_pages=int(step.page_indptr[-1]))
    seqs, rows, ct = _chunk_tables(step, dev)
    q_chunk = q_out.index_select(0, torch.from_numpy(rows.astype(np.int64)).to(dev))
    out, lse = cache.prefill_attention(0, q_chunk, ct["append_indptr"], ct["pos_map"], ct["page_indptr"],
                                       ct["page_indices"], ct["last_page_len"])
    torch.cuda.synchronize()
    assert cache.check_status() == (0, 0)
    assert seqs.size == 16 and rows.size == 16 * 512
    lens = step.seq_len[seqs]
    picks = sorted({int(np.argmax(lens)), int(np.argmin(lens)), 3, 11})
    out_bits = _bits(out).view(np.uint16)
    lse_h = lse.cpu().numpy()
    q_bits = _bits(q_out).view(np.uint16)
    ai = np.concatenate([[0], np.cumsum(step.new_tokens[seqs])])
    for i in picks:
        s = int(seqs[i])
        sub = W.substep(step, [s])
        gpu_pages = pool.index_select(0, torch.from_numpy(sub.page_origin).to(dev)).view(torch.int16)
        gpu_pages = gpu_pages.cpu().numpy().view(np.uint16)
        gq = q_bits[W.token_rows(step, [s])]
        ref_out, ref_lse = oracle.prefill_attention(H.geometry(sub), gpu_pages, gq, sub.append_indptr, sub.pos_map,
                                                    sub.page_indptr, sub.page_indices, sub.last_page_len)
        H.assert_close_out(out_bits[ai[i]:ai[i + 1]], ref_out, f"prefill rows of sequence {s} (len {lens[i]})")
        H.assert_close_lse(lse_h[ai[i]:ai[i + 1]], ref_lse, f"prefill lse of sequence {s}")


def _int8_full_size(cid, layers_of_workload, seqs_fn):
    import torch

    import paged_kv_decode_pkv_gb300 as pkv
    from bench import int8_pools

    base = W.CONFIGS[cid]
    # a cache of len(layers_of_workload) layers; layer i of the cache is layer layers_of_workload[i] of
    # the workload (its seeds), with the workload's full batch, lengths and pool
    cfg = W.scaled(base, layers=max(layers_of_workload) + 1)
    step = W.make_step(cfg)
    dev = torch.device("cuda")
    pools = int8_pools(step, cfg, layers_of_workload, dev)
    cache = pkv.Cache(len(layers_of_workload), step.num_pages, cfg.hq, cfg.hkv, cfg.head_dim, step.max_position,
                      cfg.theta, pools=pools, options=pkv.OPT_PDL | pkv.OPT_EARLY_PAGES | pkv.OPT_INT8_KV)
    tabs = H.device_tables(step)
    counters = torch.zeros(step.batch * cfg.hkv, dtype=torch.int32, device=dev)
    tp = int(step.page_indptr[-1])
    res = []
    for i, l in enumerate(layers_of_workload):
        q, k, v = H.device_qkv(step, l)
        res.append(cache.append_decode_attention(i, q, k, v, tabs["pos_map"], tabs["append_indptr"],
                                                 tabs["page_indptr"], tabs["page_indices"], tabs["last_page_len"],
                                                 step.max_pages_per_seq, counters, total_pages=tp))
    torch.cuda.synchronize()
    assert cache.check_status() == (0, 0)
    seqs = seqs_fn(step)
    sub = W.substep(step, seqs)
    rows = W.token_rows(step, seqs)
    sel = torch.from_numpy(np.asarray(seqs, dtype=np.int64)).to(dev)
    origin = torch.from_numpy(sub.page_origin).to(dev)
    for i, l in enumerate(layers_of_workload):
        q_out, out, lse = res[i]
        gpool8 = pools[i].index_select(0, origin).cpu().numpy()
        gq = _bits(q_out).view(np.uint16)[rows][H.query_rows(sub)]
        ref_out, ref_lse = oracle.attention_int8(H.geometry(sub), gpool8, gq, sub.page_indptr, sub.page_indices,
                                                 sub.last_page_len)
        H.assert_close_out(_bits(out.index_select(0, sel)).view(np.uint16), ref_out, f"layer {l} out")
        H.assert_close_lse(lse.index_select(0, sel).cpu().numpy(), ref_lse, f"layer {l} lse")


def test_full_size_int8_gqa_long_context():
    _int8_full_size(4, [0, 27], lambda st: [0, 7])


def test_full_size_int8_ragged_batch64():
    """One query head per KV head (the Phi-3 ragged batch)."""
    _int8_full_size(3, [0], lambda st: [0, int(np.argmax(st.seq_len)), int(np.argmin(st.seq_len)), 63])


def test_full_size_int8_mixed_serving():
    def pick(st):
        chunk = np.flatnonzero(st.new_tokens > 1)
        return sorted({int(np.argmax(st.seq_len)), int(np.argmin(st.seq_len)), int(chunk[0]), int(chunk[-1]), 5})
    _int8_full_size(5, [0], pick)
