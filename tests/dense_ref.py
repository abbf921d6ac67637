"""Independent numpy formulations used to pin the oracle (tests only).

None of this shares code with ``oracle/``: the page layout is expressed with
numpy's 5-D indexing instead of flat offsets, RoPE as multiplication of complex
numbers by unit phasors, and attention as one dense softmax over the gathered
logical sequence.  They are for tiny inputs.
"""
import numpy as np

PAGE = 16


def f16(bits):
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def to_f16_bits(x):
    return np.asarray(x, dtype=np.float64).astype(np.float16).view(np.uint16)


def rope_complex(x, pos, theta):
    """Rotate-half RoPE as complex multiplication: z_i = x_i + j x_{i+d/2}, z_i *= exp(j pos w_i).

    ``pos`` broadcasts against ``x.shape[:-1]``."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    half = d // 2
    w = theta ** (-np.arange(half, dtype=np.float64) * 2.0 / d)
    ang = np.asarray(pos, dtype=np.float64)[..., None] * w
    z = (x[..., :half] + 1j * x[..., half:]) * np.exp(1j * ang)
    return np.concatenate([z.real, z.imag], axis=-1)


def logical_kv(pool, page_indptr, page_indices, seq, length, kv):
    """Tokens 0..length-1 of one sequence gathered from a [P, 2, H, 16, d] pool: [H, length, d]."""
    pages = page_indices[page_indptr[seq]:page_indptr[seq + 1]]
    blocks = pool[pages, kv]                       # [n, H, 16, d]
    seqv = np.transpose(blocks, (1, 0, 2, 3))      # [H, n, 16, d]
    H, n, _, d = seqv.shape
    return seqv.reshape(H, n * PAGE, d)[:, :length]


def dense_attention(q, K, V, scale):
    """q [Hq, d], K/V [Hkv, L, d] (float64) -> out [Hq, d], lse [Hq]; KV heads repeated in groups."""
    Hq, Hkv = q.shape[0], K.shape[0]
    Kr = np.repeat(K, Hq // Hkv, axis=0)
    Vr = np.repeat(V, Hq // Hkv, axis=0)
    if Kr.shape[1] == 0:
        return np.zeros_like(q), np.full(Hq, -np.inf)
    s = scale * np.einsum("hd,hld->hl", q, Kr)
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    out = np.einsum("hl,hld->hd", e, Vr) / e.sum(axis=1, keepdims=True)
    lse = (m[:, 0] + np.log(e.sum(axis=1)))
    return out, lse


def random_paged_case(rng, lengths, hq, hkv, d, extra_pages=3, permute=True):
    """A random pool with NaN in every slot beyond each sequence's length, and its page table."""
    lengths = np.asarray(lengths)
    n = (lengths + PAGE - 1) // PAGE
    total = int(n.sum())
    P = total + extra_pages
    order = rng.permutation(P)[:total] if permute else np.arange(total)
    page_indptr = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    page_indices = order.astype(np.int32)
    last = np.where(n > 0, lengths - (n - 1) * PAGE, 1).astype(np.int32)
    vals = rng.standard_normal((P, 2, hkv, PAGE, d))
    pool = to_f16_bits(vals)
    valid = np.zeros((P, PAGE), dtype=bool)
    for s, L in enumerate(lengths):
        pages = page_indices[page_indptr[s]:page_indptr[s + 1]]
        for t in range(L):
            valid[pages[t // PAGE], t % PAGE] = True
    pool[np.broadcast_to(~valid[:, None, None, :, None], pool.shape)] = 0x7E00
    q = to_f16_bits(rng.standard_normal((lengths.size, hq, d)))
    return pool, q, page_indptr, page_indices, last
