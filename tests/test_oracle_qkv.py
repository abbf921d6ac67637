"""Pins of the oracle's Q4F16_1 QKV projection (CPU), against the format as the Zero TVM
Documentation prints it ("Q4F16 quantization format": element i of a uint32 in bits 4i..4i+3,
value f16(nibble - 7) * scale with one fp16 scale per 32 weights): hand-built words, the fp16
rounding of the product, and a dense numpy projection of independently dequantized weights."""
import numpy as np
import pytest

import oracle


def _f16(x):
    return np.asarray(x, dtype=np.float16).view(np.uint16)


def test_nibble_order_and_centering_from_hand_built_words():
    hidden, N = 32, 2
    w = np.zeros((N, hidden // 8), dtype=np.uint32)
    w[0, :] = 0x76543210          # elements 0..7 of every word hold nibbles 0..7
    w[1, :] = 0xFEDCBA98          # nibbles 8..15
    scales = _f16(np.ones((N, 1)))
    for k in range(8):
        x = np.zeros((1, hidden), dtype=np.float16)
        x[0, 8 + k] = 1.0         # one-hot input, in the second word
        y = oracle.qkv_project(x.view(np.uint16), w, scales).view(np.float16)
        assert y[0, 0] == k - 7 and y[0, 1] == k + 1


def test_scale_groups_of_32_inputs():
    hidden, N = 96, 1
    w = np.full((N, hidden // 8), 0x88888888, dtype=np.uint32)   # every weight is (8 - 7) * scale
    scales = _f16([[1.0, 2.0, 4.0]])
    for grp, s in enumerate([1.0, 2.0, 4.0]):
        x = np.zeros((1, hidden), dtype=np.float16)
        x[0, 32 * grp + 5] = 1.0
        y = oracle.qkv_project(x.view(np.uint16), w, scales).view(np.float16)
        assert y[0, 0] == s


def test_weight_is_the_fp16_product():
    # (nibble - 7) * scale = 3 * (1 + 2^-10) lies exactly between two fp16 values; the fp16
    # multiply rounds it to even, which one-hot input then shows unchanged
    hidden = 32
    w = np.full((1, hidden // 8), 0xAAAAAAAA, dtype=np.uint32)  # nibble 10 -> 3
    s = np.float16(1.0009765625)
    scales = _f16([[s]])
    x = np.zeros((1, hidden), dtype=np.float16)
    x[0, 0] = 1.0
    y = oracle.qkv_project(x.view(np.uint16), w, scales).view(np.float16)
    expect = np.float16(3) * s                      # numpy: exact product rounded to fp16
    assert y[0, 0] == expect and float(expect) != 3 * float(s)


def _dequantize(w, scales, hidden):
    """Independent dequantization: shifts over the packed words, fp16 products."""
    N = w.shape[0]
    nib = (w[:, :, None] >> (4 * np.arange(8, dtype=np.uint32))) & 0xF     # [N, hidden/8, 8]
    nib = nib.reshape(N, hidden).astype(np.int32) - 7
    sc = np.repeat(scales.view(np.float16), 32, axis=1)                       # [N, hidden]
    return (nib.astype(np.float16) * sc).astype(np.float64)                   # fp16 product


@pytest.mark.parametrize("T,hidden,N", [(1, 64, 24), (3, 256, 40), (2, 3072, 96)])
def test_projection_matches_dense_numpy(T, hidden, N):
    rng = np.random.default_rng(T * 1000 + hidden + N)
    w = rng.integers(0, 1 << 32, size=(N, hidden // 8), dtype=np.uint64).astype(np.uint32)
    scales = _f16(np.abs(rng.standard_normal((N, hidden // 32))) * 0.03)
    x = _f16(rng.standard_normal((T, hidden)))
    y = oracle.qkv_project(x, w, scales).view(np.float16).astype(np.float64)
    ref = x.view(np.float16).astype(np.float64) @ _dequantize(w, scales, hidden).T
    ref16 = ref.astype(np.float16).astype(np.float64)     # the projection rounded to fp16
    # fp64 sums in different orders may land on either side of an fp16 rounding boundary only
    # when the exact value is within ~1e-16 relative of it: allow that one step, nothing more
    diff = np.abs(y - ref16)
    ulp = np.spacing(np.abs(ref16).astype(np.float16)).astype(np.float64)
    assert np.all(diff <= ulp)
    assert np.mean(diff == 0) > 0.999


def test_qkv_append_splits_rows_into_q_k_v_heads():
    rng = np.random.default_rng(5)
    hq, hkv, d, hidden = 4, 2, 16, 64
    N = (hq + 2 * hkv) * d
    g = oracle.Geometry(4, hq, hkv, d, 64, 1e4)
    w = rng.integers(0, 1 << 32, size=(N, hidden // 8), dtype=np.uint64).astype(np.uint32)
    scales = _f16(np.abs(rng.standard_normal((N, hidden // 32))) * 0.05)
    x = _f16(rng.standard_normal((1, hidden)))
    pool = np.full((4, 2, hkv, 16, d), 0x7E00, dtype=np.uint16)
    pos = np.array([0], dtype=np.int32)            # position 0: RoPE is the identity
    y, q_out = oracle.qkv_append(g, x, w, scales, pos, np.array([0, 1], np.int32), np.array([0, 1], np.int32),
                                 np.array([2], np.int32), pool)
    assert np.array_equal(q_out.reshape(-1), y[0, :hq * d])
    assert np.array_equal(pool[2, 0, :, 0, :].reshape(-1), y[0, hq * d:(hq + hkv) * d])
    assert np.array_equal(pool[2, 1, :, 0, :].reshape(-1), y[0, (hq + hkv) * d:])
