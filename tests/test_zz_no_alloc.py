"""The allocation-free merged decode (pkv_decode_attention_noalloc), on a GPU.

It serves callers that cannot allocate device memory on the attention path (a framework that owns
all device memory through its own allocator, or a serving loop that must not risk an allocation
failure or an implicit synchronisation mid-step): they pass only inputs and outputs, and the
library keeps its scratch in a fixed device array.  These checks compare it, through the C ABI,
with the existing merged entry point that takes caller workspace, on two calls in a row (the
second call runs on the scratch the first one left behind), and check that requests beyond the
fixed scratch size are rejected.  This file is collected last so that a failure here does not
hide the other tests when a run stops at the first failure.
"""
import numpy as np
import pytest

from pkv_inputs import workloads as W
from tests import harness as H

pytestmark = pytest.mark.gpu

CASES = {  # workload, split plan
    "phi3_b1_ctx300": (W.scaled(W.CONFIGS[2], layers=1, lengths=("fixed", 300), pool_pages=24), {}),
    "gqa4_mixed_chunks": (W.scaled(W.CONFIGS[5], batch=12, lengths=("loguniform", 16, 3000), pool_pages=3000,
                                   chunk_seqs=3, chunk_tokens=40), {"num_splits": 6}),
}


@pytest.mark.parametrize("name", list(CASES))
def test_noalloc_matches_the_workspace_entry_point_on_two_calls(name):
    import torch

    cfg, plan = CASES[name]
    step = W.make_step(cfg)
    pool = H.to_dev(W.host_pool(step, 0), torch.float16)
    cache = H.make_cache(step, [0], [pool])
    tabs = H.device_tables(step)
    q, k, v = H.device_qkv(step, 0)
    q_out = cache.append_rope(0, q, k, v, tabs["pos_map"], tabs["append_indptr"], tabs["page_indptr"],
                              tabs["page_indices"])
    tp = int(step.page_indptr[-1])
    counters = torch.zeros(step.batch * cfg.hkv, dtype=torch.int32, device="cuda")
    ref_out, ref_lse = cache.decode_attention_merged(0, q_out, tabs["page_indptr"], tabs["page_indices"],
                                                     tabs["last_page_len"], step.max_pages_per_seq, counters,
                                                     q_indptr=tabs["q_indptr"], total_pages=tp, **plan)
    torch.cuda.synchronize()
    ref_out = ref_out.view(torch.int16).cpu().numpy().view(np.uint16)
    ref_lse = ref_lse.cpu().numpy()
    ref64 = ref_out.view(np.float16).astype(np.float64)
    for _ in range(2):
        out = torch.full((step.batch, cfg.hq, cfg.head_dim), float("nan"), dtype=torch.float16, device="cuda")
        lse = torch.full((step.batch, cfg.hq), float("nan"), dtype=torch.float32, device="cuda")
        cache.decode_attention_noalloc(0, q_out, tabs["page_indptr"], tabs["page_indices"], tabs["last_page_len"],
                                       step.max_pages_per_seq, out, lse, q_indptr=tabs["q_indptr"], total_pages=tp,
                                       **plan)
        torch.cuda.synchronize()
        assert cache.check_status()[0] == 0
        H.assert_close_out(out.view(torch.int16).cpu().numpy().view(np.uint16), ref64, "noalloc out")
        H.assert_close_lse(lse.cpu().numpy(), ref_lse, "noalloc lse")


def test_noalloc_rejects_requests_beyond_its_scratch():
    import torch

    import paged_kv_decode_pkv_gb300 as pkv

    cfg, _ = CASES["phi3_b1_ctx300"]
    step = W.make_step(cfg)
    pool = H.to_dev(W.host_pool(step, 0), torch.float16)
    cache = H.make_cache(step, [0], [pool])
    tabs = H.device_tables(step)
    out = torch.empty((1, cfg.hq, cfg.head_dim), dtype=torch.float16, device="cuda")
    # 32 heads x 4000 splits x 97 floats x 4 bytes is about 50 MB of partials: above the 32 MiB array
    with pytest.raises(pkv.PkvError) as e:
        cache.decode_attention_noalloc(0, out, tabs["page_indptr"], tabs["page_indices"], tabs["last_page_len"],
                                       4000, out, chunk_pages=1)
    assert e.value.code == pkv.ERR_UNSUPPORTED and "32 MiB" in str(e.value)
