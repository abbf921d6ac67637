"""Pins of the oracle's int8 KV cache (CPU): the row quantizer against its defining properties
(the largest magnitude maps to 127, every value is within half a step of code * scale, zero rows,
odd symmetry), the block layout against a brute force of the format, and attention over the int8
pool against a dense numpy softmax over independently dequantized values."""
import math

import numpy as np
import pytest

import oracle
from tests.dense_ref import f16, logical_kv, random_paged_case, to_f16_bits


@pytest.mark.parametrize("d", [64, 96, 128])
def test_quantizer_properties(d):
    rng = np.random.default_rng(d)
    for trial in range(200):
        x = rng.standard_normal(d) * 10.0 ** rng.uniform(-4, 2)
        bits = to_f16_bits(x)
        xv = f16(bits)
        codes, s = oracle.quantize_row(bits)
        amax = np.abs(xv).max()
        assert np.all(np.abs(codes.astype(np.int32)) <= 127)
        if amax == 0:
            assert s == 0 and np.all(codes == 0)
            continue
        assert np.float32(s) == np.float32(amax) / np.float32(127)
        i = int(np.argmax(np.abs(xv)))
        assert abs(int(codes[i])) == 127 and np.sign(codes[i]) == np.sign(xv[i])
        # within half a step, plus the fp32 rounding of x / s (at most 2^-24 * 128 steps)
        err = np.abs(xv - codes.astype(np.float64) * float(s))
        assert np.all(err <= float(s) * (0.5 + 2.0 ** -24 * 128))
        neg, sn = oracle.quantize_row(to_f16_bits(-xv))
        assert sn == s and np.array_equal(neg, -codes)


def test_zero_row_and_ties_round_to_even():
    codes, s = oracle.quantize_row(to_f16_bits(np.zeros(64)))
    assert s == 0 and np.all(codes == 0)
    # values at exactly half a step: 127 * 0.5 / 127 = 0.5 step -> 0 (even), 1.5 steps -> 2
    x = np.zeros(64)
    x[0] = 127.0
    x[1] = 0.5
    x[2] = 1.5
    x[3] = 2.5
    codes, s = oracle.quantize_row(to_f16_bits(x))
    assert s == np.float32(1.0) and list(codes[:4]) == [127, 0, 2, 2]


def _pool8_case(rng, lengths, hq, hkv, d):
    pool, q, pi, px, last = random_paged_case(rng, lengths, hq, hkv, d)
    g = oracle.Geometry(pool.shape[0], hq, hkv, d, 1 << 20, 1e4)
    blk = oracle.int8_block_bytes(d)
    # quantize every written slot of the fp16 pool with the row quantizer, block by block
    pool8 = np.full((pool.shape[0], 2, hkv, blk), 0x55, dtype=np.uint8)
    for s, L in enumerate(lengths):
        for t in range(L):
            page = px[pi[s] + t // 16]
            for kv in range(2):
                for h in range(hkv):
                    codes, sc = oracle.quantize_row(pool[page, kv, h, t % 16])
                    stored = _stored(codes)
                    if kv == 0:  # K codes slot-major [16][d]
                        pool8[page, kv, h, (t % 16) * d:(t % 16 + 1) * d] = stored
                    else:        # V codes dim-major [d][16]
                        pool8[page, kv, h, t % 16:16 * d:16] = stored
                    pool8[page, kv, h, 16 * d + 4 * (t % 16):16 * d + 4 * (t % 16) + 4] = \
                        np.array([sc], np.float32).view(np.uint8)
    return g, pool, pool8, q, pi, px, last


def _stored(codes):
    """The bytes a block stores for int8 codes: code + 128 (offset binary)."""
    return (codes.astype(np.int16) + 128).astype(np.uint8)


def _row_bytes(blk, kv, slot, d):
    """The stored bytes of one slot row in a block: K rows are contiguous, V rows a stride-16 column."""
    return blk[slot * d:(slot + 1) * d] if kv == 0 else blk[slot:16 * d:16]


def _row_codes(blk, kv, slot, d):
    """The codes of one slot row in a block, read back from their offset-binary bytes."""
    return (_row_bytes(blk, kv, slot, d).astype(np.int16) - 128).astype(np.int8)


def _dequant(pool8, d):
    """Independent read of the block format: int8 codes stored as code + 128 (K blocks [16][d], V
    blocks [d][16]), then fp32 scales [16]."""
    raw = pool8[..., :16 * d].astype(np.int16) - 128
    k = raw[:, 0].reshape(raw.shape[0], raw.shape[2], 16, d)
    v = raw[:, 1].reshape(raw.shape[0], raw.shape[2], d, 16).transpose(0, 1, 3, 2)
    codes = np.stack([k, v], axis=1).astype(np.float64)
    scales = pool8[..., 16 * d:].copy().view(np.float32).astype(np.float64)
    return codes * scales[..., None]


def test_dequantize_pool_reads_the_block_format():
    rng = np.random.default_rng(3)
    g, pool, pool8, q, pi, px, last = _pool8_case(rng, [20, 37], 4, 2, 32)
    deq = oracle.dequantize_pool(g, pool8)
    ref = _dequant(pool8, 32)
    for s, L in enumerate([20, 37]):
        for t in range(L):
            page = px[pi[s] + t // 16]
            assert np.array_equal(deq[page, :, :, t % 16], ref[page, :, :, t % 16])


def test_append_int8_writes_the_quantized_rotated_rows():
    rng = np.random.default_rng(4)
    hq, hkv, d = 4, 2, 32
    lengths = [20, 5]
    pool, _, pi, px, last = random_paged_case(rng, lengths, hq, hkv, d)
    g = oracle.Geometry(pool.shape[0], hq, hkv, d, 1 << 20, 1e4)
    pos = np.array([19, 4], np.int32)
    ai = np.array([0, 1, 2], np.int32)
    qn = to_f16_bits(rng.standard_normal((2, hq, d)))
    kn = to_f16_bits(rng.standard_normal((2, hkv, d)))
    vn = to_f16_bits(rng.standard_normal((2, hkv, d)))
    pool16 = pool.copy()
    q_ref = oracle.append(g, qn, kn, vn, pos, ai, pi, px, pool16)
    pool8 = np.full((pool.shape[0], 2, hkv, oracle.int8_block_bytes(d)), 0x55, dtype=np.uint8)
    q_out = oracle.append_int8(g, qn, kn, vn, pos, ai, pi, px, pool8)
    assert np.array_equal(q_out, q_ref)
    for t, s in enumerate([0, 1]):
        page, slot = px[pi[s] + pos[t] // 16], pos[t] % 16
        for kv in range(2):
            for h in range(hkv):
                codes, sc = oracle.quantize_row(pool16[page, kv, h, slot])
                blk = pool8[page, kv, h]
                assert np.array_equal(_row_codes(blk, kv, slot, d), codes)
                assert blk[16 * d + 4 * slot:16 * d + 4 * slot + 4].view(np.float32)[0] == sc
    # nothing else was written
    touched = np.zeros(pool8.shape[:-1] + (16,), dtype=bool)
    for t, s in enumerate([0, 1]):
        touched[px[pi[s] + pos[t] // 16], :, :, pos[t] % 16] = True
    for page in range(pool8.shape[0]):
        for kv in range(2):
            for h in range(hkv):
                for slot in range(16):
                    if not touched[page, kv, h, slot]:
                        assert np.all(_row_bytes(pool8[page, kv, h], kv, slot, d) == 0x55)


@pytest.mark.parametrize("window", [0, 20])
def test_int8_attention_matches_dense_softmax_over_dequantized_values(window):
    rng = np.random.default_rng(5 + window)
    lengths = [1, 17, 60]
    hq, hkv, d = 4, 2, 16
    g, pool, pool8, q, pi, px, last = _pool8_case(rng, lengths, hq, hkv, d)
    out, lse = oracle.attention_int8(g, pool8, q, pi, px, last, window=window)
    deq = _dequant(pool8, d)
    for s, L in enumerate(lengths):
        pages = px[pi[s]:pi[s + 1]]
        K = np.transpose(deq[pages, 0], (1, 0, 2, 3)).reshape(hkv, -1, d)[:, :L]
        V = np.transpose(deq[pages, 1], (1, 0, 2, 3)).reshape(hkv, -1, d)[:, :L]
        t0 = max(0, L - window) if window else 0
        Kr = np.repeat(K[:, t0:], hq // hkv, axis=0)
        Vr = np.repeat(V[:, t0:], hq // hkv, axis=0)
        sc = np.einsum("hd,hld->hl", f16(q[s]), Kr) / math.sqrt(d)
        m = sc.max(axis=1, keepdims=True)
        e = np.exp(sc - m)
        ro = np.einsum("hl,hld->hd", e, Vr) / e.sum(axis=1, keepdims=True)
        np.testing.assert_allclose(out[s], ro, atol=1e-12, rtol=1e-12)
        np.testing.assert_allclose(lse[s], m[:, 0] + np.log(e.sum(axis=1)), atol=1e-12)


def test_int8_split_and_combine_equal_unsplit():
    rng = np.random.default_rng(6)
    lengths = [16, 40, 90]
    g, pool, pool8, q, pi, px, last = _pool8_case(rng, lengths, 4, 2, 16)
    ref, ref_lse = oracle.attention_int8(g, pool8, q, pi, px, last)
    po, pl = oracle.split_attention_int8(g, pool8, q, pi, px, last, num_splits=3, num_out_splits=3)
    out, _, lse = oracle.combine(po, pl)
    np.testing.assert_allclose(out, ref, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, atol=1e-12)


def test_quantize_pool_matches_the_row_quantizer():
    rng = np.random.default_rng(7)
    pool, q, pi, px, last = random_paged_case(rng, [20, 5], 2, 2, 16)
    g = oracle.Geometry(pool.shape[0], 2, 2, 16, 1 << 20, 1e4)
    pool8 = oracle.quantize_pool(g, pool)
    for page in range(pool.shape[0]):
        for kv in range(2):
            for h in range(2):
                for slot in range(16):
                    codes, sc = oracle.quantize_row(pool[page, kv, h, slot])
                    blk = pool8[page, kv, h]
                    assert np.array_equal(_row_codes(blk, kv, slot, 16), codes)
                    assert blk[256 + 4 * slot:256 + 4 * slot + 4].view(np.float32)[0] == sc or (np.isnan(sc))
