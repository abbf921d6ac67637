"""Pins of the oracle against things other than itself (CPU only).

Each group targets a plausible mistake: the fp16 codec against numpy's
IEEE-754 casts; RoPE against its group properties, a complex-number
formulation and frequency facts read back from its behaviour; placement
against a brute-force numpy layout; attention against dense numpy softmax,
closed-form special cases and the split/permutation invariants of the
Zero TVM documentation's paged, split-K design ("KV cache", "How it works").
"""
import math

import numpy as np
import pytest

import oracle
from tests.dense_ref import (PAGE, dense_attention, f16, logical_kv, random_paged_case, rope_complex,
                             to_f16_bits)


# ------------------------------------------------------------------------------------------------
# fp16 codec


def test_f16_decode_every_pattern_matches_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.f16_to_f64(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_f16_encode_matches_numpy_rne_on_a_million_doubles():
    rng = np.random.default_rng(7)
    n = 1_000_000
    normal = rng.standard_normal(n // 4) * np.exp2(rng.integers(-14, 16, n // 4))
    sub = rng.uniform(-2.0 ** -14, 2.0 ** -14, n // 4)
    # exact midpoints between neighbouring fp16 values (ties) and points next to them
    h = rng.integers(0, 0x7BFF, n // 8).astype(np.uint16)
    lo, hi = h.view(np.float16).astype(np.float64), (h + 1).view(np.float16).astype(np.float64)
    mid = (lo + hi) / 2
    near = np.concatenate([np.nextafter(mid, np.inf), np.nextafter(mid, -np.inf)])
    edge = np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, 65536.0, 1e300, -1e300, np.inf, -np.inf,
                     2.0 ** -24, 2.0 ** -25, 2.0 ** -25 * 1.0000001, 3 * 2.0 ** -26, 2.0 ** -14])
    x = np.concatenate([normal, sub, mid, -mid, near, edge, rng.standard_normal(n - 3 * (n // 4) - n // 8)])
    ours = oracle.f64_to_f16(x)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)
    assert np.array_equal(oracle.f64_to_f16(np.array([np.nan])) & 0x7C00, np.array([0x7C00], np.uint16))


# ------------------------------------------------------------------------------------------------
# RoPE


@pytest.mark.parametrize("d", [4, 64, 96, 128])
def test_rope_position_zero_is_identity(d):
    x = np.random.default_rng(d).standard_normal(d)
    assert np.array_equal(oracle.rope(x, 0, 1e4), x)


@pytest.mark.parametrize("d,theta", [(64, 1e4), (96, 1e4), (128, 1e6)])
def test_rope_preserves_each_pair_norm_and_composes(d, theta):
    rng = np.random.default_rng(1)
    x = rng.standard_normal(d)
    for p in [1, 17, 4095, 65535]:
        y = oracle.rope(x, p, theta)
        h = d // 2
        np.testing.assert_allclose(y[:h] ** 2 + y[h:] ** 2, x[:h] ** 2 + x[h:] ** 2, rtol=1e-12)
    # rotations compose: R(a) R(b) = R(a + b)
    a, b = 123, 4567
    np.testing.assert_allclose(oracle.rope(oracle.rope(x, a, theta), b, theta), oracle.rope(x, a + b, theta),
                               atol=1e-9)


@pytest.mark.parametrize("d,theta", [(64, 1e4), (128, 1e6)])
def test_rope_relative_position_property(d, theta):
    """<RoPE(q, p), RoPE(k, p')> = <RoPE(q, p - p'), k>: scores depend on the offset only."""
    rng = np.random.default_rng(2)
    q, k = rng.standard_normal(d), rng.standard_normal(d)
    for p, pp in [(5, 3), (100, 99), (4096, 17), (30000, 65000)]:
        lhs = oracle.rope(q, p, theta) @ oracle.rope(k, pp, theta)
        rhs = oracle.rope(q, p - pp, theta) @ k
        assert abs(lhs - rhs) < 1e-9 * (np.linalg.norm(q) * np.linalg.norm(k))


@pytest.mark.parametrize("d,theta", [(4, 1e4), (64, 1e4), (96, 1e4), (128, 1e6)])
def test_rope_matches_complex_phasor_formulation(d, theta):
    rng = np.random.default_rng(3)
    x = rng.standard_normal(d)
    for p in [1, 2, 99, 4095, 66047]:
        np.testing.assert_allclose(oracle.rope(x, p, theta), rope_complex(x, p, theta), atol=1e-9)


@pytest.mark.parametrize("d,theta", [(64, 1e4), (128, 1e6)])
def test_rope_frequencies_read_back_from_unit_vectors(d, theta):
    """Rotating e_i at p = 1 reveals the angle of pair i: pair 0 turns by exactly 1 radian,
    pairs pair i with i + d/2, and successive angles shrink by the constant ratio theta^(-2/d)."""
    h = d // 2
    ang = []
    for i in range(h):
        e = np.zeros(d)
        e[i] = 1.0
        y = oracle.rope(e, 1, theta)
        others = np.delete(y, [i, i + h])
        assert np.all(others == 0.0)
        ang.append(math.atan2(y[i + h], y[i]))
    ang = np.array(ang)
    assert abs(ang[0] - 1.0) < 1e-15
    np.testing.assert_allclose(ang[1:] / ang[:-1], theta ** (-2.0 / d), rtol=1e-12)


# ------------------------------------------------------------------------------------------------
# placement (append)


def _append_case(rng, lengths, new, hq, hkv, d, theta=1e4):
    lengths = np.asarray(lengths)
    new = np.asarray(new)
    hist = lengths - new
    pool, _, page_indptr, page_indices, last = random_paged_case(rng, hist, hq, hkv, d, extra_pages=0)
    # give every sequence the pages its new length needs (pages beyond the history are fresh)
    n_new = (lengths + PAGE - 1) // PAGE
    P0 = pool.shape[0]
    pages, nxt = [], P0
    for s in range(lengths.size):
        own = list(page_indices[page_indptr[s]:page_indptr[s + 1]])
        while len(own) < n_new[s]:
            own.append(nxt)
            nxt += 1
        pages.append(own)
    extra = nxt - P0 + 2
    pool = np.concatenate([pool, np.full((extra,) + pool.shape[1:], 0x7E00, np.uint16)])
    page_indptr = np.concatenate([[0], np.cumsum(n_new)]).astype(np.int32)
    page_indices = np.concatenate(pages).astype(np.int32)
    T = int(new.sum())
    append_indptr = np.concatenate([[0], np.cumsum(new)]).astype(np.int32)
    pos_map = np.concatenate([rng.permutation(np.arange(hist[s], lengths[s])) for s in range(lengths.size)])
    q = to_f16_bits(rng.standard_normal((T, hq, d)))
    k = to_f16_bits(rng.standard_normal((T, hkv, d)))
    v = to_f16_bits(rng.standard_normal((T, hkv, d)))
    geom = oracle.Geometry(pool.shape[0], hq, hkv, d, int(lengths.max()) + 1, theta)
    return geom, pool, q, k, v, pos_map.astype(np.int32), append_indptr, page_indptr, page_indices


def _ulp_diff(a, b):
    """Distance in representable fp16 steps between two arrays of finite fp16 bit patterns."""
    def ordered(x):
        x = x.astype(np.int32)
        return np.where(x & 0x8000, -(x & 0x7FFF), x)
    return np.abs(ordered(a) - ordered(b))


def test_append_placement_matches_bruteforce_layout():
    rng = np.random.default_rng(11)
    hq, hkv, d, theta = 4, 2, 8, 1e4
    lengths, new = [1, 17, 40, 33], [1, 2, 17, 1]
    geom, pool, q, k, v, pos_map, ai, pi, px = _append_case(rng, lengths, new, hq, hkv, d, theta)
    before = pool.copy()
    got = pool.copy()
    q_out = oracle.append(geom, q, k, v, pos_map, ai, pi, px, got)
    # brute force: expected image via 5-D indexing and the complex formulation of RoPE
    exp = before.copy()
    qexp = np.empty_like(q)
    for s in range(len(lengths)):
        own = px[pi[s]:pi[s + 1]]
        for t in range(ai[s], ai[s + 1]):
            p = int(pos_map[t])
            page, slot = own[p // PAGE], p % PAGE
            exp[page, 0, :, slot, :] = to_f16_bits(rope_complex(f16(k[t]), p, theta))
            exp[page, 1, :, slot, :] = v[t]
            qexp[t] = to_f16_bits(rope_complex(f16(q[t]), p, theta))
    nan_exp = (exp & 0x7C00) == 0x7C00
    assert np.array_equal(nan_exp, (got & 0x7C00) == 0x7C00), "written slot set differs"
    assert np.array_equal(got[:, 1], exp[:, 1]), "V must be a bit copy"
    assert _ulp_diff(got[:, 0][~nan_exp[:, 0]], exp[:, 0][~nan_exp[:, 0]]).max() <= 1
    assert _ulp_diff(q_out, qexp).max() <= 1
    untouched = (before == exp).all(axis=(1, 2, 4))
    assert np.array_equal(got.transpose(0, 3, 1, 2, 4)[untouched], before.transpose(0, 3, 1, 2, 4)[untouched])


def test_append_rejects_duplicate_and_out_of_range_positions():
    rng = np.random.default_rng(12)
    geom, pool, q, k, v, pos_map, ai, pi, px = _append_case(rng, [20, 20], [2, 1], 2, 2, 8)
    dup = pos_map.copy()
    dup[1] = dup[0]
    with pytest.raises(oracle.OracleError) as e:
        oracle.append(geom, q, k, v, dup, ai, pi, px, pool.copy())
    assert e.value.code == 5
    far = pos_map.copy()
    far[0] = 10 * PAGE * 100
    with pytest.raises(oracle.OracleError) as e:
        oracle.append(geom, q, k, v, far, ai, pi, px, pool.copy())
    assert e.value.code == 3


def test_append_at_position_zero_stores_k_unchanged():
    rng = np.random.default_rng(13)
    geom, pool, q, k, v, pos_map, ai, pi, px = _append_case(rng, [1], [1], 2, 2, 16)
    q_out = oracle.append(geom, q, k, v, pos_map, ai, pi, px, pool)
    assert np.array_equal(pool[px[0], 0, :, 0, :], k[0])
    assert np.array_equal(q_out, q)


# ------------------------------------------------------------------------------------------------
# attention


def _geom(pool, hq, hkv, d, theta=1e4):
    return oracle.Geometry(pool.shape[0], hq, hkv, d, 1 << 20, theta)


@pytest.mark.parametrize("hq,hkv", [(4, 4), (4, 2), (8, 2), (6, 2)])
def test_attention_matches_dense_softmax(hq, hkv):
    rng = np.random.default_rng(hq * 10 + hkv)
    d = 16
    lengths = [1, 16, 17, 40, 100]
    pool, q, pi, px, last = random_paged_case(rng, lengths, hq, hkv, d)
    out, lse = oracle.attention(_geom(pool, hq, hkv, d), pool, q, pi, px, last)
    for s, L in enumerate(lengths):
        K = f16(logical_kv(pool, pi, px, s, L, 0))
        V = f16(logical_kv(pool, pi, px, s, L, 1))
        ro, rl = dense_attention(f16(q[s]), K, V, 1 / math.sqrt(d))
        np.testing.assert_allclose(out[s], ro, atol=1e-12, rtol=1e-12)
        np.testing.assert_allclose(lse[s], rl, atol=1e-12, rtol=1e-12)


def test_attention_length_one_returns_v_exactly():
    rng = np.random.default_rng(21)
    pool, q, pi, px, last = random_paged_case(rng, [1, 1], 4, 2, 32)
    out, lse = oracle.attention(_geom(pool, 4, 2, 32), pool, q, pi, px, last)
    for s in range(2):
        V = f16(pool[px[pi[s]], 1, :, 0, :])
        assert np.array_equal(out[s], np.repeat(V, 2, axis=0))


def test_attention_zero_query_is_mean_of_v_with_lse_log_len():
    rng = np.random.default_rng(22)
    lengths = [5, 37]
    pool, q, pi, px, last = random_paged_case(rng, lengths, 2, 2, 8)
    q[:] = 0
    out, lse = oracle.attention(_geom(pool, 2, 2, 8), pool, q, pi, px, last)
    for s, L in enumerate(lengths):
        V = f16(logical_kv(pool, pi, px, s, L, 1))
        np.testing.assert_allclose(out[s], V.mean(axis=1), atol=1e-13)
        np.testing.assert_allclose(lse[s], math.log(L), atol=1e-13)


def test_attention_equal_keys_give_mean_of_v():
    rng = np.random.default_rng(23)
    lengths = [50]
    pool, q, pi, px, last = random_paged_case(rng, lengths, 2, 1, 8)
    key_row = to_f16_bits(rng.standard_normal(8))
    pages = px[pi[0]:pi[1]]
    for t in range(50):
        pool[pages[t // PAGE], 0, 0, t % PAGE, :] = key_row
    out, lse = oracle.attention(_geom(pool, 2, 1, 8), pool, q, pi, px, last)
    V = f16(logical_kv(pool, pi, px, 0, 50, 1))[0]
    np.testing.assert_allclose(out[0], np.stack([V.mean(axis=0)] * 2), atol=1e-13)


def test_attention_page_permutation_invariance_is_exact():
    rng = np.random.default_rng(24)
    lengths = [33, 70, 5]
    pool, q, pi, px, last = random_paged_case(rng, lengths, 4, 2, 16, extra_pages=6)
    g = _geom(pool, 4, 2, 16)
    out, lse = oracle.attention(g, pool, q, pi, px, last)
    perm = rng.permutation(pool.shape[0])        # new physical id of old page i is perm[i]
    pool2 = np.empty_like(pool)
    pool2[perm] = pool
    out2, lse2 = oracle.attention(g, pool2, q, pi, perm[px].astype(np.int32), last)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_empty_sequence_gives_zero_and_minus_inf():
    rng = np.random.default_rng(25)
    pool, q, pi, px, last = random_paged_case(rng, [0, 3], 2, 2, 8)
    out, lse = oracle.attention(_geom(pool, 2, 2, 8), pool, q, pi, px, last)
    assert np.all(out[0] == 0) and np.all(lse[0] == -np.inf)
    po, pl = oracle.split_attention(_geom(pool, 2, 2, 8), pool, q, pi, px, last, num_splits=3)
    o, o16, l = oracle.combine(po, pl)
    assert np.all(o[0] == 0) and np.all(l[0] == -np.inf)


@pytest.mark.parametrize("mode", ["splits", "chunk"])
def test_split_then_combine_equals_unsplit(mode):
    rng = np.random.default_rng(26)
    lengths = [1, 16, 17, 150, 333]
    hq, hkv, d = 4, 2, 16
    pool, q, pi, px, last = random_paged_case(rng, lengths, hq, hkv, d)
    g = _geom(pool, hq, hkv, d)
    ref, ref_lse = oracle.attention(g, pool, q, pi, px, last)
    nmax = int(np.diff(pi).max())
    values = [1, 2, 3, 7, nmax, nmax + 3] if mode == "splits" else [1, 2, 5, nmax]
    for val in values:
        kw = {"num_splits": val} if mode == "splits" else {"chunk_pages": val}
        po, pl = oracle.split_attention(g, pool, q, pi, px, last, **kw)
        out, out16, lse = oracle.combine(po, pl)
        np.testing.assert_allclose(out, ref, atol=1e-12)
        np.testing.assert_allclose(lse, ref_lse, atol=1e-12)
        assert np.array_equal(out16, oracle.f64_to_f16(ref)) or \
            _ulp_diff(out16, oracle.f64_to_f16(ref)).max() <= 1


def test_split_chunks_are_page_aligned_and_match_dense_pieces():
    rng = np.random.default_rng(27)
    lengths = [100]
    pool, q, pi, px, last = random_paged_case(rng, lengths, 2, 2, 8)
    po, pl = oracle.split_attention(_geom(pool, 2, 2, 8), pool, q, pi, px, last, num_splits=2)
    # 7 pages, ceil(7/2) = 4 pages per chunk: tokens [0, 64) and [64, 100)
    K = f16(logical_kv(pool, pi, px, 0, 100, 0))
    V = f16(logical_kv(pool, pi, px, 0, 100, 1))
    for j, (a, b) in enumerate([(0, 64), (64, 100)]):
        ro, rl = dense_attention(f16(q[0]), K[:, a:b], V[:, a:b], 1 / math.sqrt(8))
        np.testing.assert_allclose(po[0, :, j], ro, atol=1e-12)
        np.testing.assert_allclose(pl[0, :, j], rl, atol=1e-12)


def test_combine_two_partials_closed_form():
    rng = np.random.default_rng(28)
    o = rng.standard_normal((1, 1, 2, 4))
    l = np.array([[[0.3, -1.7]]])
    out, _, lse = oracle.combine(o, l)
    w = np.exp(l[0, 0] - np.logaddexp(l[0, 0, 0], l[0, 0, 1]))
    np.testing.assert_allclose(out[0, 0], w[0] * o[0, 0, 0] + w[1] * o[0, 0, 1], atol=1e-15)
    np.testing.assert_allclose(lse[0, 0], np.logaddexp(0.3, -1.7), atol=1e-15)
    l2 = np.array([[[0.3, -np.inf]]])
    out, _, lse = oracle.combine(o, l2)
    np.testing.assert_allclose(out[0, 0], o[0, 0, 0], atol=1e-15)


def test_scale_zero_gives_uniform_weights():
    rng = np.random.default_rng(29)
    pool, q, pi, px, last = random_paged_case(rng, [20], 2, 2, 8)
    out, lse = oracle.attention(_geom(pool, 2, 2, 8), pool, q, pi, px, last, sm_scale=0.0)
    V = f16(logical_kv(pool, pi, px, 0, 20, 1))
    np.testing.assert_allclose(out[0], V.mean(axis=1), atol=1e-13)


@pytest.mark.parametrize("warps", [1, 3, 7, 40, 200])
def test_balanced_partition_covers_each_segment_once_and_merges_to_unsplit(warps):
    """The page-balanced partition: runs of equal size (within one page) whose pieces tile every
    (sequence, KV head) segment exactly once; merging the pieces gives the unsplit result."""
    rng = np.random.default_rng(31)
    lengths = [1, 16, 17, 150, 333, 40]
    hq, hkv, d = 4, 2, 16
    pool, q, pi, px, last = random_paged_case(rng, lengths, hq, hkv, d)
    g = _geom(pool, hq, hkv, d)
    U = hkv * int(pi[-1])
    if warps > U:
        pytest.skip("more runs than units")
    ref, ref_lse = oracle.attention(g, pool, q, pi, px, last)
    S = -(-int(np.diff(pi).max()) * warps // U) + 1
    po, pl = oracle.split_attention_balanced(g, pool, q, pi, px, last, warps, S)
    out, out16, lse = oracle.combine(po, pl)
    np.testing.assert_allclose(out, ref, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, atol=1e-12)
    # run sizes differ by at most one page; pieces of a segment are contiguous and cover it
    sizes = [(w + 1) * U // warps - w * U // warps for w in range(warps)]
    assert max(sizes) - min(sizes) <= 1 and sum(sizes) == U
    n_pieces = (~np.isinf(pl)).sum(axis=2)
    for s_, L in enumerate(lengths):
        n = int(pi[s_ + 1] - pi[s_])
        for h in range(hq):
            b = hkv * int(pi[s_]) + (h // (hq // hkv)) * n
            expect = len({w for w in range(warps) for u in range(b, b + n) if w * U // warps <= u < (w + 1) * U // warps})
            assert n_pieces[s_, h] == expect
