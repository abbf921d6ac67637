"""Pins of the oracle's sliding window and attention sinks (CPU), each against something other than
the oracle itself: a dense numpy softmax over the window's positions with the sink as one more
logit of value zero, closed forms, and the split + combine = unsplit identity.

Readings (Splash models page: the families' sliding_window / layer_types and a layer's
attn_sinks; Zero TVM Documentation, "Decode loop": the unused lengthInfo fields): window W > 0
lets the query at position len-1 attend to positions [max(0, len-W), len); a sink is one logit per
query head, in the units of the scaled scores, that joins the softmax denominator and carries no
value."""
import math

import numpy as np
import pytest

import oracle
from tests.dense_ref import f16, logical_kv, random_paged_case


def _geom(pool, hq, hkv, d):
    return oracle.Geometry(pool.shape[0], hq, hkv, d, 1 << 20, 1e4)


def dense_window_sink(q, K, V, scale, window, sinks):
    """q [Hq, d], K/V [Hkv, L, d] -> out [Hq, d], lse [Hq] over the last `window` positions
    (0 = all) with per-head sink logits (None = none), written out directly."""
    Hq, Hkv, L = q.shape[0], K.shape[0], K.shape[1]
    t0 = max(0, L - window) if window > 0 else 0
    Kr = np.repeat(K[:, t0:], Hq // Hkv, axis=0)
    Vr = np.repeat(V[:, t0:], Hq // Hkv, axis=0)
    logits = scale * np.einsum("hd,hld->hl", q, Kr)
    if sinks is not None:
        logits = np.concatenate([logits, np.asarray(sinks, dtype=np.float64)[:, None]], axis=1)
        Vr = np.concatenate([Vr, np.zeros((Hq, 1, Vr.shape[2]))], axis=1)
    if logits.shape[1] == 0:
        return np.zeros_like(q), np.full(Hq, -np.inf)
    m = logits.max(axis=1, keepdims=True)
    e = np.exp(logits - m)
    out = np.einsum("hl,hld->hd", e, Vr) / e.sum(axis=1, keepdims=True)
    return out, m[:, 0] + np.log(e.sum(axis=1))


LENGTHS = [1, 15, 16, 17, 40, 100, 257]


@pytest.mark.parametrize("window", [1, 5, 16, 17, 33, 100, 1000])
@pytest.mark.parametrize("with_sinks", [False, True])
def test_window_and_sinks_match_dense_softmax(window, with_sinks):
    rng = np.random.default_rng(window * 7 + with_sinks)
    hq, hkv, d = 4, 2, 16
    pool, q, pi, px, last = random_paged_case(rng, LENGTHS, hq, hkv, d)
    sinks = rng.standard_normal(hq) * 2 if with_sinks else None
    out, lse = oracle.attention(_geom(pool, hq, hkv, d), pool, q, pi, px, last, window=window, sinks=sinks)
    for s, L in enumerate(LENGTHS):
        K = f16(logical_kv(pool, pi, px, s, L, 0))
        V = f16(logical_kv(pool, pi, px, s, L, 1))
        ro, rl = dense_window_sink(f16(q[s]), K, V, 1 / math.sqrt(d), window, sinks)
        np.testing.assert_allclose(out[s], ro, atol=1e-12, rtol=1e-12)
        np.testing.assert_allclose(lse[s], rl, atol=1e-12, rtol=1e-12)


def test_window_at_least_the_length_changes_nothing():
    rng = np.random.default_rng(31)
    pool, q, pi, px, last = random_paged_case(rng, LENGTHS, 4, 4, 8)
    g = _geom(pool, 4, 4, 8)
    ref = oracle.attention(g, pool, q, pi, px, last)
    for w in (257, 258, 10 ** 6):
        got = oracle.attention(g, pool, q, pi, px, last, window=w)
        assert np.array_equal(ref[0], got[0]) and np.array_equal(ref[1], got[1])


def test_window_one_returns_the_last_value_exactly():
    rng = np.random.default_rng(32)
    pool, q, pi, px, last = random_paged_case(rng, LENGTHS, 4, 2, 16)
    out, lse = oracle.attention(_geom(pool, 4, 2, 16), pool, q, pi, px, last, window=1)
    for s, L in enumerate(LENGTHS):
        V = f16(logical_kv(pool, pi, px, s, L, 1))[:, L - 1]
        assert np.array_equal(out[s], np.repeat(V, 2, axis=0))


def test_minus_inf_sinks_change_nothing():
    rng = np.random.default_rng(33)
    pool, q, pi, px, last = random_paged_case(rng, LENGTHS, 4, 2, 8)
    g = _geom(pool, 4, 2, 8)
    ref = oracle.attention(g, pool, q, pi, px, last, window=20)
    got = oracle.attention(g, pool, q, pi, px, last, window=20, sinks=np.full(4, -np.inf))
    assert np.array_equal(ref[0], got[0]) and np.array_equal(ref[1], got[1])


def test_sink_closed_form_with_zero_query():
    # all scores 0: out = mean(V) * n / (n + e^sink), lse = ln(n + e^sink)
    rng = np.random.default_rng(34)
    lengths = [7, 50]
    pool, q, pi, px, last = random_paged_case(rng, lengths, 2, 2, 8)
    q[:] = 0
    sinks = np.array([0.5, -1.25])
    out, lse = oracle.attention(_geom(pool, 2, 2, 8), pool, q, pi, px, last, sinks=sinks)
    for s, L in enumerate(lengths):
        V = f16(logical_kv(pool, pi, px, s, L, 1))
        for h in range(2):
            den = L + math.exp(sinks[h])
            np.testing.assert_allclose(out[s, h], V[h].sum(axis=0) / den, atol=1e-13)
            np.testing.assert_allclose(lse[s, h], math.log(den), atol=1e-13)


def test_empty_sequence_with_a_sink_has_the_sink_as_lse():
    rng = np.random.default_rng(35)
    pool, q, pi, px, last = random_paged_case(rng, [0, 3], 2, 2, 8)
    out, lse = oracle.attention(_geom(pool, 2, 2, 8), pool, q, pi, px, last, sinks=[0.25, -2.0])
    assert np.all(out[0] == 0) and np.array_equal(lse[0], [0.25, -2.0])


@pytest.mark.parametrize("window", [1, 16, 17, 60, 0])
@pytest.mark.parametrize("plan", [{"num_splits": 1}, {"num_splits": 3}, {"chunk_pages": 1}, {"chunk_pages": 2}])
def test_windowed_split_and_combine_with_sinks_equal_unsplit(window, plan):
    rng = np.random.default_rng(36 + window)
    hq, hkv, d = 4, 2, 16
    pool, q, pi, px, last = random_paged_case(rng, LENGTHS, hq, hkv, d)
    g = _geom(pool, hq, hkv, d)
    sinks = rng.standard_normal(hq)
    ref, ref_lse = oracle.attention(g, pool, q, pi, px, last, window=window, sinks=sinks)
    nmax = int(np.diff(pi).max())
    S = nmax if "chunk_pages" in plan else plan["num_splits"]
    po, pl = oracle.split_attention(g, pool, q, pi, px, last, num_out_splits=S, window=window, **plan)
    out, out16, lse = oracle.combine(po, pl, sinks=sinks)
    np.testing.assert_allclose(out, ref, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, atol=1e-12)


def test_windowed_chunks_cover_only_visible_pages():
    # chunk j of a windowed sequence starts at its first visible page: with one-page chunks, chunk 0
    # holds the positions [len - W, end of that page) and nothing before the window is read
    rng = np.random.default_rng(37)
    lengths = [100]
    pool, q, pi, px, last = random_paged_case(rng, lengths, 2, 2, 8)
    g = _geom(pool, 2, 2, 8)
    W = 40                                     # positions 60..99: pages 3 (60..63) to 6
    po, pl = oracle.split_attention(g, pool, q, pi, px, last, chunk_pages=1, num_out_splits=7, window=W)
    K = f16(logical_kv(pool, pi, px, 0, 100, 0))
    V = f16(logical_kv(pool, pi, px, 0, 100, 1))
    ro, rl = dense_window_sink(f16(q[0]), K[:, :64], V[:, :64], 1 / math.sqrt(8), 4, None)
    np.testing.assert_allclose(po[0, :, 0], ro, atol=1e-12)
    np.testing.assert_allclose(pl[0, :, 0], rl, atol=1e-12)
    assert np.all(pl[0, :, 4:] == -np.inf)      # 4 visible pages: chunks 4..6 are empty


@pytest.mark.parametrize("window", [1, 17, 60])
@pytest.mark.parametrize("warps", [1, 5, 40])
def test_windowed_balanced_partition_merges_to_unsplit(window, warps):
    rng = np.random.default_rng(38 + window + warps)
    hq, hkv, d = 4, 2, 16
    pool, q, pi, px, last = random_paged_case(rng, LENGTHS, hq, hkv, d)
    g = _geom(pool, hq, hkv, d)
    sinks = rng.standard_normal(hq)
    ref, ref_lse = oracle.attention(g, pool, q, pi, px, last, window=window, sinks=sinks)
    S = int(np.diff(pi).max()) + 1
    # runs are non-empty: at most as many as visible page units (the kernel takes the same minimum)
    visible = sum(-(-L // 16) - max(0, L - window) // 16 for L in LENGTHS) * hkv
    po, pl = oracle.split_attention_balanced(g, pool, q, pi, px, last, min(warps, visible), S, window=window)
    out, out16, lse = oracle.combine(po, pl, sinks=sinks)
    np.testing.assert_allclose(out, ref, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, atol=1e-12)
