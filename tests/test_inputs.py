"""The seeded input generator and the workload construction (CPU only)."""
import numpy as np
import pytest

import pkv_inputs
from pkv_inputs import workloads as W


def test_words_are_the_published_splitmix64_sequence():
    # SplitMix64 seeded with 1234567: the first five outputs of the public-domain reference code
    expect = [6457827717110365317, 3203168211198807973, 9817491932198370423, 4593380528125082431,
              16408922859458223821]
    assert [int(x) for x in pkv_inputs.words(1234567, 5)] == expect
    assert int(pkv_inputs.words(1234567, 1, first=3)[0]) == expect[3]


def test_normal_values_follow_the_stated_definition():
    k = pkv_inputs.key(5, 9)
    n = 4096
    w = pkv_inputs.words(k, 3 * n).reshape(n, 3)
    halves = np.stack([(w >> np.uint64(16 * j)) & np.uint64(0xFFFF) for j in range(4)], axis=-1)
    s = halves.astype(np.int64).sum(axis=(1, 2))
    x = ((s - 393210).astype(np.float32) * np.float32(2.0 ** -16))
    scale = np.float32(0.1020620726)
    expect = (x * scale).astype(np.float16).view(np.uint16)
    assert np.array_equal(pkv_inputs.fill_range(n, k, scale=float(scale)), expect)


def test_normal_moments_and_outlier_rows():
    k = pkv_inputs.key(1, 1)
    v = pkv_inputs.fill_range(1_000_000, k).view(np.float16).astype(np.float64)
    assert abs(v.mean()) < 5e-3 and abs(v.std() - 1) < 5e-3 and np.abs(v).max() <= 6
    okey = pkv_inputs.key(1, 2)
    base = pkv_inputs.fill_range(128 * 1000, k).reshape(1000, 128).view(np.float16).astype(np.float64)
    out = pkv_inputs.fill_range(128 * 1000, k, okey=okey, row_len=128, pct=1).reshape(1000, 128)
    out = out.view(np.float16).astype(np.float64)
    ratio = np.abs(out).sum(1) / np.abs(base).sum(1)
    hit = np.isclose(ratio, 8.0)
    assert np.all(hit | np.isclose(ratio, 1.0)) and 2 <= hit.sum() <= 25


def test_fill_blocks_equals_fill_range_slices():
    k = pkv_inputs.key(3, 4)
    full = pkv_inputs.fill_range(10 * 64, k)
    blocks = np.array([7, 2, 9])
    got = pkv_inputs.fill_blocks(blocks, 64, k)
    for i, b in enumerate(blocks):
        assert np.array_equal(got[i], full[b * 64:(b + 1) * 64])


@pytest.mark.parametrize("cid", [1, 2, 3, 4, 5])
def test_workload_step_is_consistent(cid):
    st = W.make_step(W.CONFIGS[cid])
    B = st.batch
    n = np.diff(st.page_indptr)
    assert np.all(n == (st.seq_len + 15) // 16)
    assert np.all((st.last_page_len >= 1) & (st.last_page_len <= 16))
    assert np.all(16 * (n - 1) + st.last_page_len == st.seq_len)
    assert st.page_indices.min() >= 0 and st.page_indices.max() < st.num_pages
    assert np.unique(st.page_indices).size == st.page_indices.size, "pages must not be shared"
    assert st.append_indptr[-1] == st.pos_map.size
    for s in range(B):
        pm = st.pos_map[st.append_indptr[s]:st.append_indptr[s + 1]]
        assert np.array_equal(pm, np.arange(st.seq_len[s] - st.new_tokens[s], st.seq_len[s]))
    cfg = W.CONFIGS[cid]
    if cfg.lengths[0] != "fixed":
        lo, hi = cfg.lengths[1], cfg.lengths[2]
        base = st.seq_len - np.where(st.new_tokens > 1, st.new_tokens, 0)
        assert base.min() >= lo and base.max() <= hi
    if cid == 5:
        assert (st.new_tokens == 512).sum() == 16 and st.max_position <= 65536 + 512


def test_config_sizes_match_the_stated_workloads():
    assert W.make_step(W.CONFIGS[1]).kv_bytes() == 102_400
    assert W.make_step(W.CONFIGS[2]).kv_bytes() == 4096 * 12_288
    assert W.make_step(W.CONFIGS[4]).kv_bytes() == 8 * 32768 * 4096
    e3 = W.make_step(W.CONFIGS[3]).seq_len.mean()
    assert 1700 < e3 < 2500


def test_cache_state_marks_only_cached_slots():
    cfg = W.scaled(W.CONFIGS[3], batch=4, pool_pages=1100)
    st = W.make_step(cfg)
    pool = W.host_pool(st, 0)
    cached = ~((pool & 0x7C00) == 0x7C00)
    per_slot = cached.all(axis=(1, 2, 4))
    assert per_slot.sum() == int(st.hist_len.sum())
    assert np.array_equal(per_slot, cached.any(axis=(1, 2, 4)))


def test_substep_regenerates_the_same_pages():
    cfg = W.scaled(W.CONFIGS[3], batch=5, pool_pages=1400)
    st = W.make_step(cfg)
    full = W.host_pool(st, 0)
    sub = W.substep(st, [3, 1])
    part = W.host_pool(sub, 0)
    assert np.array_equal(part, full[sub.page_origin])
    q, k, v = W.new_qkv(st, 0)
    q2, k2, v2 = W.new_qkv(st, 0, rows=W.token_rows(st, [3, 1]))
    assert np.array_equal(q2, q[W.token_rows(st, [3, 1])]) and np.array_equal(v2, v[W.token_rows(st, [3, 1])])


def test_gpu_test_cases_are_constructible():
    """Every scaled workload the GPU tests use builds on the host (pool large enough, valid tables)."""
    from tests import test_gpu_invariants as inv
    from tests import test_gpu_parity as par

    extra = [W.scaled(W.CONFIGS[3], batch=4, pool_pages=1200), W.scaled(W.CONFIGS[3], batch=3, pool_pages=1000)]
    for cfg in list(par.SMALL.values()) + list(inv.CASES.values()) + extra:
        st = W.make_step(cfg)
        assert st.page_indices.size <= st.num_pages
