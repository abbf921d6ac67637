"""Workload table and seeded construction of one decode step's inputs.

Shapes come from the pages' workloads: the Phi-3-mini constants of the
Zero-TVM documentation ("Phi-3 model constants": hidden 3072, 32 heads of 96,
32 layers, 16-slot pages) and the 32-query / 8-KV-head x 128 attention of the
Splash models page.  Everything here is input construction: sequence lengths,
page allocation, token positions, the raw q/k/v of the new tokens and the
cache contents written by earlier steps.  None of it computes attention.

Recipe (all draws from :mod:`pkv_inputs` with seed ``0x504B5600 + config id``):

* lengths: fixed, uniform integer in [lo, hi] (``lo + w % (hi-lo+1)``), or
  log-uniform (``floor(lo * (hi/lo)**u)``, ``u = (w >> 11) * 2**-53``);
* a sequence of length L that appends one token holds L-1 cached tokens and
  appends position L-1 (it attends to itself); a sequence that appends a chunk
  of C tokens holds L cached tokens and appends positions L .. L+C-1;
* page tables: ``identity`` gives each sequence a contiguous run of pages in
  sequence order; ``permuted`` hands out pages in the order of a seeded random
  permutation of the whole pool (argsort of 64-bit draws);
* cache contents before the step: K and V of every pool page are generated as
  two tensors [pages, kv_heads, 16, head_dim] (element index = flat index),
  then every slot that holds no cached token (unreferenced pages, slots at or
  after a sequence's cached length, including the slots the step appends to)
  is set to the fp16 NaN pattern 0x7E00;
* new tokens: q [T, Hq, d], k and v [T, Hkv, d] from their own streams;
* optional outlier keys: a seeded ``pct`` percent of key rows (one key vector
  of one head at one slot or token) are multiplied by 8 before fp16 rounding.
"""
from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass, field

import numpy as np

from . import dev_fill_range, fill_blocks, fill_range, key, words

PAGE_SIZE = 16
SEED_BASE = 0x504B5600
NAN16 = 0x7E00

# stream tags: per layer l the tag is l * 16 + one of these
TAG_K_HIST, TAG_V_HIST, TAG_Q_NEW, TAG_K_NEW, TAG_V_NEW, TAG_OUT_K_HIST, TAG_OUT_K_NEW = range(7)
# step-level tags (not per layer)
TAG_LENGTHS = 1 << 40
TAG_PERM = (1 << 40) + 1
TAG_CHUNK_SEQS = (1 << 40) + 2


@dataclass(frozen=True)
class Config:
    cid: int
    name: str
    layers: int
    batch: int
    hq: int
    hkv: int
    head_dim: int
    theta: float
    lengths: tuple            # ("fixed", n) | ("uniform", lo, hi) | ("loguniform", lo, hi)
    page_table: str           # "identity" | "permuted"
    pool_pages: int           # pages per layer pool; 0 = exactly the referenced pages
    value_scale: float = 1.0  # N(0,1) draws are multiplied by this before fp16 rounding
    outlier_pct: int = 0      # percent of key rows scaled by 8
    chunk_seqs: int = 0       # sequences that append a chunk instead of one token
    chunk_tokens: int = 0
    num_splits: int = 0       # explicit split count; 0 = the planner chooses
    window: int = 0           # sliding window of every layer (0 = full attention)
    sinks: bool = False       # per-layer attention-sink logits, one per query head

    @property
    def group(self) -> int:
        return self.hq // self.hkv


CONFIGS = {
    1: Config(1, "tiny_h4_d64_ctx100", layers=1, batch=1, hq=4, hkv=4, head_dim=64, theta=1e4,
              lengths=("fixed", 100), page_table="identity", pool_pages=7, num_splits=2),
    2: Config(2, "phi3_mini_b1_ctx4096_32layers", layers=32, batch=1, hq=32, hkv=32, head_dim=96,
              theta=1e4, lengths=("fixed", 4096), page_table="identity", pool_pages=256,
              value_scale=float(np.float32(1.0 / math.sqrt(96.0)))),
    3: Config(3, "phi3_ragged_b64_u128_4096", layers=1, batch=64, hq=32, hkv=32, head_dim=96,
              theta=1e4, lengths=("uniform", 128, 4096), page_table="permuted", pool_pages=20000),
    4: Config(4, "gqa16x8_d128_b8_ctx32768_28layers", layers=28, batch=8, hq=16, hkv=8,
              head_dim=128, theta=1e6, lengths=("fixed", 32768), page_table="identity",
              pool_pages=16384, outlier_pct=1),
    5: Config(5, "gqa32x8_d128_b128_loguniform16_65536_chunk512", layers=1, batch=128, hq=32,
              hkv=8, head_dim=128, theta=1e6, lengths=("loguniform", 16, 65536),
              page_table="permuted", pool_pages=600000, chunk_seqs=16, chunk_tokens=512),
    # the 32/8 x 128 attention with a 2048-token window of the Splash page's drafts, with
    # attention sinks on every layer (its families' attn_sinks)
    6: Config(6, "gqa32x8_d128_b32_ctx8192_window2048_sinks_8layers", layers=8, batch=32, hq=32, hkv=8,
              head_dim=128, theta=1e6, lengths=("fixed", 8192), page_table="identity", pool_pages=16384,
              window=2048, sinks=True),
}


@dataclass
class Step:
    """One decode step: host-side int32 metadata shared by both sides."""
    cfg: Config
    seed: int
    seq_len: np.ndarray        # [B] tokens after the append
    new_tokens: np.ndarray     # [B] tokens appended this step
    page_indptr: np.ndarray    # [B+1] int32
    page_indices: np.ndarray   # [nnz] int32
    last_page_len: np.ndarray  # [B] int32, in [1, 16]
    append_indptr: np.ndarray  # [B+1] int32
    pos_map: np.ndarray        # [T] int32
    num_pages: int
    page_origin: np.ndarray = field(default=None)  # for sub-steps: original page id of each page

    @property
    def batch(self) -> int:
        return int(self.seq_len.size)

    @property
    def hist_len(self) -> np.ndarray:
        return self.seq_len - self.new_tokens

    @property
    def num_tokens(self) -> int:
        return int(self.append_indptr[-1])

    @property
    def max_position(self) -> int:
        return int(self.seq_len.max()) if self.seq_len.size else 1

    @property
    def max_pages_per_seq(self) -> int:
        n = np.diff(self.page_indptr)
        return int(n.max()) if n.size else 0

    def kv_bytes(self) -> int:
        """Algorithmic KV bytes one decode pass reads per layer (each attended token once per KV
        head; under a sliding window only the window's tokens)."""
        seen = np.minimum(self.seq_len, self.cfg.window) if self.cfg.window > 0 else self.seq_len
        return int(seen.sum()) * self.cfg.hkv * self.cfg.head_dim * 2 * 2


def _lengths(cfg: Config, seed: int) -> np.ndarray:
    kind = cfg.lengths[0]
    B = cfg.batch
    if kind == "fixed":
        return np.full(B, cfg.lengths[1], dtype=np.int64)
    w = words(key(seed, TAG_LENGTHS), B)
    lo, hi = cfg.lengths[1], cfg.lengths[2]
    if kind == "uniform":
        return (lo + (w % np.uint64(hi - lo + 1))).astype(np.int64)
    if kind == "loguniform":
        u = (w >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
        L = np.floor(lo * np.exp(u * math.log(hi / lo))).astype(np.int64)
        return np.clip(L, lo, hi)
    raise ValueError(kind)


def _permutation(n: int, k: int) -> np.ndarray:
    return np.argsort(words(k, n), kind="stable").astype(np.int64)


def make_step(cfg: Config, seed: int | None = None) -> Step:
    seed = SEED_BASE + cfg.cid if seed is None else seed
    B = cfg.batch
    L = _lengths(cfg, seed)
    new = np.ones(B, dtype=np.int64)
    seq_len = L.copy()
    if cfg.chunk_seqs:
        chosen = _permutation(B, key(seed, TAG_CHUNK_SEQS))[: cfg.chunk_seqs]
        new[chosen] = cfg.chunk_tokens
        seq_len[chosen] = L[chosen] + cfg.chunk_tokens
    n_pages = (seq_len + PAGE_SIZE - 1) // PAGE_SIZE
    total = int(n_pages.sum())
    pool = cfg.pool_pages or total
    if total > pool:
        raise ValueError(f"{cfg.name}: {total} pages referenced but the pool holds {pool}")
    if cfg.page_table == "identity":
        order = np.arange(total, dtype=np.int64)
    elif cfg.page_table == "permuted":
        order = _permutation(pool, key(seed, TAG_PERM))[:total]
    else:
        raise ValueError(cfg.page_table)
    page_indptr = np.zeros(B + 1, dtype=np.int64)
    page_indptr[1:] = np.cumsum(n_pages)
    append_indptr = np.zeros(B + 1, dtype=np.int64)
    append_indptr[1:] = np.cumsum(new)
    pos_map = np.concatenate([np.arange(seq_len[s] - new[s], seq_len[s]) for s in range(B)]) \
        if B else np.zeros(0, dtype=np.int64)
    last = seq_len - (n_pages - 1) * PAGE_SIZE
    return Step(cfg=cfg, seed=seed, seq_len=seq_len, new_tokens=new,
                page_indptr=page_indptr.astype(np.int32), page_indices=order.astype(np.int32),
                last_page_len=last.astype(np.int32), append_indptr=append_indptr.astype(np.int32),
                pos_map=pos_map.astype(np.int32), num_pages=pool)


def scaled(cfg: Config, **changes) -> Config:
    """A copy of a configuration with some fields changed (smaller parity cases)."""
    return dataclasses.replace(cfg, **changes)


def substep(step: Step, seqs) -> Step:
    """The step restricted to some sequences, with their pages renumbered 0..n-1.

    ``page_origin[i]`` is the original page id of page i, so the cache
    contents of the sub-step are regenerated with :func:`host_pool_pages`."""
    seqs = np.asarray(seqs, dtype=np.int64)
    pi, ai = step.page_indptr, step.append_indptr
    pages = [step.page_indices[pi[s]:pi[s + 1]].astype(np.int64) for s in seqs]
    counts = np.array([p.size for p in pages], dtype=np.int64)
    origin = np.concatenate(pages) if pages else np.zeros(0, dtype=np.int64)
    page_indptr = np.zeros(seqs.size + 1, dtype=np.int64)
    page_indptr[1:] = np.cumsum(counts)
    new = step.new_tokens[seqs]
    append_indptr = np.zeros(seqs.size + 1, dtype=np.int64)
    append_indptr[1:] = np.cumsum(new)
    pos_map = np.concatenate([step.pos_map[ai[s]:ai[s + 1]] for s in seqs]).astype(np.int32)
    return Step(cfg=step.cfg, seed=step.seed, seq_len=step.seq_len[seqs].copy(), new_tokens=new.copy(),
                page_indptr=page_indptr.astype(np.int32),
                page_indices=np.arange(origin.size, dtype=np.int32),
                last_page_len=step.last_page_len[seqs].copy(), append_indptr=append_indptr.astype(np.int32),
                pos_map=pos_map, num_pages=int(origin.size), page_origin=origin)


def token_rows(step: Step, seqs) -> np.ndarray:
    """Indices of the appended tokens of the given sequences, in order."""
    ai = step.append_indptr
    return np.concatenate([np.arange(ai[s], ai[s + 1]) for s in np.asarray(seqs)]).astype(np.int64)


# ----------------------------------------------------------------------------------------------
# new tokens


def new_qkv(step: Step, layer: int, rows=None):
    """Raw (pre-RoPE) q [T,Hq,d], k, v [T,Hkv,d] of the appended tokens, fp16 bits (uint16).

    ``rows`` restricts the result to some token indices of the full step."""
    cfg, s = step.cfg, step.seed
    d, hq, hkv = cfg.head_dim, cfg.hq, cfg.hkv
    T = step.num_tokens
    rows = np.arange(T, dtype=np.int64) if rows is None else np.asarray(rows, dtype=np.int64)
    base = layer * 16
    okey = key(s, base + TAG_OUT_K_NEW)
    q = fill_blocks(rows, hq * d, key(s, base + TAG_Q_NEW), cfg.value_scale).reshape(-1, hq, d)
    k = fill_blocks(rows, hkv * d, key(s, base + TAG_K_NEW), cfg.value_scale, okey, d,
                    cfg.outlier_pct).reshape(-1, hkv, d)
    v = fill_blocks(rows, hkv * d, key(s, base + TAG_V_NEW), cfg.value_scale).reshape(-1, hkv, d)
    return q, k, v


TAG_SINKS = 7  # per layer, beside the new-token tags
TAG_QKV_W, TAG_QKV_SCALE, TAG_HIDDEN = 8, 9, 10


def qkv_hidden(cfg: Config) -> int:
    """Hidden width feeding the QKV projection: Hq * head_dim (the Phi-3 shape: 3072)."""
    return cfg.hq * cfg.head_dim


def qkv_weights(step: Step, layer: int):
    """Q4F16_1 weights of the layer's QKV projection: packed uint32 [N, hidden/8] (uniform random
    nibbles) and fp16 scale bits [N, hidden/32] (seeded N(0,1) x 0.003)."""
    cfg = step.cfg
    hidden = qkv_hidden(cfg)
    n = (cfg.hq + 2 * cfg.hkv) * cfg.head_dim
    w = (words(key(step.seed, layer * 16 + TAG_QKV_W), n * hidden // 8) & 0xFFFFFFFF).astype(np.uint32)
    sc = fill_range(n * (hidden // 32), key(step.seed, layer * 16 + TAG_QKV_SCALE), scale=0.003)
    return w.reshape(n, hidden // 8), sc.reshape(n, hidden // 32)


def hidden_states(step: Step, layer: int, rows=None):
    """The new tokens' inputs of the QKV projection, fp16 bits [T, hidden] (seeded N(0,1))."""
    hidden = qkv_hidden(step.cfg)
    rows = np.arange(step.num_tokens, dtype=np.int64) if rows is None else np.asarray(rows, dtype=np.int64)
    return fill_blocks(rows, hidden, key(step.seed, layer * 16 + TAG_HIDDEN))


def sink_logits(step: Step, layer: int) -> np.ndarray:
    """The layer's attention-sink logits, float32 [Hq]: seeded N(0,1) draws (fp16-representable)."""
    bits = fill_range(step.cfg.hq, key(step.seed, layer * 16 + TAG_SINKS))
    return bits.view(np.float16).astype(np.float32)


# ----------------------------------------------------------------------------------------------
# cache contents before the step


def cached_slot_mask(step: Step, page_ids=None) -> np.ndarray:
    """bool [n, 16]: which slots of the listed pages (default: all pool pages) hold a cached token."""
    P = step.num_pages
    valid = np.zeros((P, PAGE_SIZE), dtype=bool)
    pi, hist = step.page_indptr, step.hist_len
    for s in range(step.batch):
        pages = step.page_indices[pi[s]:pi[s + 1]]
        full, rem = int(hist[s]) // PAGE_SIZE, int(hist[s]) % PAGE_SIZE
        valid[pages[:full]] = True
        if rem:
            valid[pages[full], :rem] = True
    return valid if page_ids is None else valid[np.asarray(page_ids)]


def _hist_keys(step: Step, layer: int):
    s, base = step.seed, layer * 16
    return key(s, base + TAG_K_HIST), key(s, base + TAG_V_HIST), key(s, base + TAG_OUT_K_HIST)


def host_pool_pages(step: Step, layer: int, page_ids) -> np.ndarray:
    """Cache contents of the listed pages before the step: uint16 [n, 2, Hkv, 16, d].

    Page ids refer to ``step`` (for a sub-step, its renumbered pages)."""
    cfg = step.cfg
    page_ids = np.asarray(page_ids, dtype=np.int64)
    origin = page_ids if step.page_origin is None else step.page_origin[page_ids]
    hkv, d = cfg.hkv, cfg.head_dim
    kk, vk, ok = _hist_keys(step, layer)
    blk = hkv * PAGE_SIZE * d
    K = fill_blocks(origin, blk, kk, cfg.value_scale, ok, d, cfg.outlier_pct)
    V = fill_blocks(origin, blk, vk, cfg.value_scale)
    out = np.empty((page_ids.size, 2, hkv, PAGE_SIZE, d), dtype=np.uint16)
    out[:, 0] = K.reshape(-1, hkv, PAGE_SIZE, d)
    out[:, 1] = V.reshape(-1, hkv, PAGE_SIZE, d)
    valid = cached_slot_mask(step, page_ids)
    out[np.broadcast_to(~valid[:, None, None, :, None], out.shape)] = NAN16
    return out


def host_pool(step: Step, layer: int) -> np.ndarray:
    """Cache contents of the whole pool before the step (small pools only)."""
    return host_pool_pages(step, layer, np.arange(step.num_pages))


def device_pool(step: Step, layer: int, out=None, stream: int = 0):
    """The same cache contents as :func:`host_pool`, generated directly in device memory.

    Returns a torch.float16 tensor [pages, 2, Hkv, 16, d] (``out`` if given)."""
    import torch

    assert step.page_origin is None, "device pools are built for full steps only"
    cfg = step.cfg
    P, hkv, d = step.num_pages, cfg.hkv, cfg.head_dim
    kk, vk, ok = _hist_keys(step, layer)
    if out is None:
        out = torch.empty((P, 2, hkv, PAGE_SIZE, d), dtype=torch.float16, device="cuda")
    n = P * hkv * PAGE_SIZE * d
    tmp = torch.empty(n, dtype=torch.float16, device=out.device)
    dev_fill_range(tmp.data_ptr(), n, kk, 0, cfg.value_scale, ok, d, cfg.outlier_pct, stream)
    out[:, 0].copy_(tmp.view(P, hkv, PAGE_SIZE, d))
    dev_fill_range(tmp.data_ptr(), n, vk, 0, cfg.value_scale, 0, 0, 0, stream)
    out[:, 1].copy_(tmp.view(P, hkv, PAGE_SIZE, d))
    del tmp
    valid = torch.from_numpy(cached_slot_mask(step)).to(out.device)
    out.view(torch.int16).masked_fill_(~valid[:, None, None, :, None], NAN16)
    return out
