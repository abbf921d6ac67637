"""Pins of the oracle's chunked-prefill attention (CPU): a dense numpy causal softmax over each
sequence's logical tokens, causality itself (changing later positions changes nothing), and the
one-token case (a decode step: the sequence's last position)."""
import math

import numpy as np
import pytest

import oracle
from tests.dense_ref import f16, logical_kv, random_paged_case
from tests.test_oracle_window_sinks import dense_window_sink


def _case(rng, lengths, chunks, hq, hkv, d):
    pool, _, pi, px, last = random_paged_case(rng, lengths, hq, hkv, d)
    # sequence s appended its last chunks[s] positions
    ai = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    pos = np.concatenate([np.arange(L - c, L) for L, c in zip(lengths, chunks)]).astype(np.int32)
    q = (rng.standard_normal((int(ai[-1]), hq, d))).astype(np.float16).view(np.uint16)
    return pool, q, pi, px, last, ai, pos


@pytest.mark.parametrize("window", [0, 5, 40])
@pytest.mark.parametrize("with_sinks", [False, True])
def test_prefill_matches_dense_causal_softmax(window, with_sinks):
    rng = np.random.default_rng(50 + window + with_sinks)
    lengths, chunks = [20, 70, 33], [20, 17, 1]
    hq, hkv, d = 4, 2, 16
    pool, q, pi, px, last, ai, pos = _case(rng, lengths, chunks, hq, hkv, d)
    g = oracle.Geometry(pool.shape[0], hq, hkv, d, 1 << 20, 1e4)
    sinks = rng.standard_normal(hq) if with_sinks else None
    out, lse = oracle.prefill_attention(g, pool, q, ai, pos, pi, px, last, window=window, sinks=sinks)
    for s, L in enumerate(lengths):
        K = f16(logical_kv(pool, pi, px, s, L, 0))
        V = f16(logical_kv(pool, pi, px, s, L, 1))
        for t in range(ai[s], ai[s + 1]):
            p = int(pos[t])
            ro, rl = dense_window_sink(f16(q[t]), K[:, :p + 1], V[:, :p + 1], 1 / math.sqrt(d), window, sinks)
            np.testing.assert_allclose(out[t], ro, atol=1e-12, rtol=1e-12)
            np.testing.assert_allclose(lse[t], rl, atol=1e-12, rtol=1e-12)


def test_prefill_is_causal():
    rng = np.random.default_rng(60)
    lengths, chunks = [50], [30]
    pool, q, pi, px, last, ai, pos = _case(rng, lengths, chunks, 2, 2, 8)
    g = oracle.Geometry(pool.shape[0], 2, 2, 8, 1 << 20, 1e4)
    out, lse = oracle.prefill_attention(g, pool, q, ai, pos, pi, px, last)
    pool2 = pool.copy()
    p_cut = 35                               # change every position after 35
    pages = px[pi[0]:pi[1]]
    for t in range(p_cut + 1, 50):
        pool2[pages[t // 16], :, :, t % 16, :] = f16(rng.standard_normal((2, 2, 8))).astype(np.float16).view(np.uint16)
    out2, lse2 = oracle.prefill_attention(g, pool2, q, ai, pos, pi, px, last)
    upto = pos <= p_cut
    assert np.array_equal(out[upto], out2[upto]) and np.array_equal(lse[upto], lse2[upto])
    assert not np.array_equal(out[~upto], out2[~upto])


def test_one_token_per_sequence_at_its_end_is_the_decode():
    rng = np.random.default_rng(61)
    lengths = [1, 17, 64, 100]
    pool, q, pi, px, last, ai, pos = _case(rng, lengths, [1] * 4, 4, 2, 16)
    g = oracle.Geometry(pool.shape[0], 4, 2, 16, 1 << 20, 1e4)
    out, lse = oracle.prefill_attention(g, pool, q, ai, pos, pi, px, last)
    ref, ref_lse = oracle.attention(g, pool, q, pi, px, last)
    assert np.array_equal(out, ref) and np.array_equal(lse, ref_lse)
