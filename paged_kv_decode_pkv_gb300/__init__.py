"""GB300 paged-KV decode attention: Python binding of libpkv.so.

Argument marshalling only.  Every step of the path (RoPE + KV append, split-K decode attention,
log-sum-exp combine) runs in the library's CUDA kernels; PyTorch provides device memory and the
stream.  There is no fallback: importing works without a GPU, but every compute call needs the
built library and a CUDA device, and raises otherwise.

Names follow include/pkv.h: ``Cache`` wraps pkv_create_cache / pkv_destroy, and its methods
``append_rope``, ``decode_attention``, ``combine``, ``plan_decode`` and ``check_status`` wrap the
entry points of the same names.
"""
from __future__ import annotations

import ctypes
import os

from . import _build

LIB_PATH = _build.LIB
PAGE_SIZE = 16

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_OUT_OF_RANGE, ERR_CUDA, ERR_TIMEOUT = range(6)
FLAG_BAD_PAGE, FLAG_BAD_POSITION, FLAG_BAD_SEQUENCE, FLAG_TIMEOUT = 0x1, 0x2, 0x4, 0x8
OPT_PDL = 0x1
OPT_EARLY_PAGES = 0x2  # PKV_OPT_EARLY_PAGES
OPT_INT8_KV = 0x4  # PKV_OPT_INT8_KV


class PkvError(RuntimeError):
    def __init__(self, code: int, what: str, detail: str = ""):
        super().__init__(f"{what}: {status_string(code)} ({code})" + (f" - {detail}" if detail else ""))
        self.code = code


class _Desc(ctypes.Structure):
    _fields_ = [("num_layers", ctypes.c_int), ("num_pages", ctypes.c_int), ("page_size", ctypes.c_int),
                ("num_qo_heads", ctypes.c_int), ("num_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int),
                ("max_position", ctypes.c_int), ("rope_theta", ctypes.c_double),
                ("layer_pools", ctypes.POINTER(ctypes.c_void_p)), ("rope_table", ctypes.c_void_p),
                ("status_word", ctypes.c_void_p), ("options", ctypes.c_int),
                ("layer_window", ctypes.POINTER(ctypes.c_int32)), ("layer_sinks", ctypes.POINTER(ctypes.c_void_p))]


_lib = None


def lib():
    """The loaded libpkv.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                               "(the CUDA path has no fallback)")
        L = ctypes.CDLL(LIB_PATH)
        P, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        L.pkv_pool_bytes.restype = sz
        L.pkv_pool_bytes.argtypes = [i, i, i]
        L.pkv_rope_table_bytes.restype = sz
        L.pkv_rope_table_bytes.argtypes = [i, i]
        L.pkv_partial_bytes.restype = sz
        L.pkv_partial_bytes.argtypes = [i, i, i, i]
        L.pkv_status_string.restype = ctypes.c_char_p
        L.pkv_status_string.argtypes = [i]
        L.pkv_last_error.restype = ctypes.c_char_p
        L.pkv_last_error.argtypes = []
        L.pkv_create_cache.restype = i
        L.pkv_create_cache.argtypes = [ctypes.POINTER(_Desc), ctypes.POINTER(P)]
        L.pkv_destroy.restype = None
        L.pkv_destroy.argtypes = [P]
        L.pkv_device_info.restype = i
        L.pkv_device_info.argtypes = [P, i, ctypes.POINTER(i), ctypes.POINTER(i)]
        L.pkv_append_rope.restype = i
        L.pkv_append_rope.argtypes = [P, i, P, P, P, P, P, i, i, P, P, P, P]
        L.pkv_plan_decode.restype = i
        L.pkv_plan_decode.argtypes = [P, i, i, i, i, i, i, ctypes.POINTER(i), ctypes.POINTER(i)]
        L.pkv_decode_attention.restype = i
        L.pkv_decode_attention.argtypes = [P, i, P, P, P, P, P, i, i, i, i, i, i, f, P, P,
                                           ctypes.POINTER(i), P]
        L.pkv_decode_attention_merged.restype = i
        L.pkv_decode_attention_merged.argtypes = [P, i, P, P, P, P, P, i, i, i, i, i, i, f, P, P, P, P, P,
                                                  ctypes.POINTER(i), P]
        L.pkv_append_decode_attention.restype = i
        L.pkv_append_decode_attention.argtypes = [P, i, P, P, P, P, P, i, P, P, P, i, i, i, i, i, i, f, P, P, P, P,
                                                  P, P, ctypes.POINTER(i), P]
        L.pkv_decode_attention_noalloc.restype = i
        L.pkv_decode_attention_noalloc.argtypes = [P, i, P, P, P, P, P, i, i, i, i, i, f, P, P,
                                                   ctypes.POINTER(i), P]
        L.pkv_prefill_attention.restype = i
        L.pkv_prefill_attention.argtypes = [P, i, P, P, P, i, P, P, P, i, ctypes.c_float, P, P, P]
        L.pkv_qkv_project.restype = i
        L.pkv_qkv_project.argtypes = [P, P, P, P, i, i, P, P]
        L.pkv_qkv_append_rope.restype = i
        L.pkv_qkv_append_rope.argtypes = [P, i, P, P, P, i, P, P, i, i, P, P, P, P]
        L.pkv_combine.restype = i
        L.pkv_combine.argtypes = [P, P, P, P, i, i, i, i, P, P, P]
        L.pkv_check_status.restype = i
        L.pkv_check_status.argtypes = [P, P, ctypes.POINTER(i)]
        L.pkv_set_wait_limit.restype = i
        L.pkv_set_wait_limit.argtypes = [P, ctypes.c_ulonglong]
        L.pkv_set_stage_stall.restype = i
        L.pkv_set_stage_stall.argtypes = [P, i]
        _lib = L
    return _lib


def status_string(code: int) -> str:
    return lib().pkv_status_string(code).decode()


def _check(code: int, what: str) -> None:
    if code != OK:
        raise PkvError(code, what, lib().pkv_last_error().decode())


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    import torch

    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def pool_bytes(num_pages: int, num_kv_heads: int, head_dim: int) -> int:
    return lib().pkv_pool_bytes(num_pages, num_kv_heads, head_dim)


def rope_table_bytes(max_position: int, head_dim: int) -> int:
    return lib().pkv_rope_table_bytes(max_position, head_dim)


def partial_bytes(batch: int, num_qo_heads: int, splits: int, head_dim: int) -> int:
    return lib().pkv_partial_bytes(batch, num_qo_heads, splits, head_dim)


class Cache:
    """A paged KV cache over caller-owned device memory (torch tensors).

    ``pools`` is a list of fp16 tensors [num_pages, 2, num_kv_heads, 16, head_dim] (allocated
    here when omitted).  The RoPE table and the status word are allocated here as tensors.
    ``windows``: per layer sliding window (0 = full attention), or None; ``sinks``: per layer
    None or an fp32 tensor [num_qo_heads] of attention-sink logits (kept alive here), or None."""

    def __init__(self, num_layers, num_pages, num_qo_heads, num_kv_heads, head_dim, max_position,
                 rope_theta, pools=None, options: int = 0, device=None, windows=None, sinks=None):
        import torch

        device = torch.device("cuda") if device is None else torch.device(device)
        self.num_layers, self.num_pages = int(num_layers), int(num_pages)
        self.num_qo_heads, self.num_kv_heads = int(num_qo_heads), int(num_kv_heads)
        self.head_dim, self.max_position = int(head_dim), int(max_position)
        self.rope_theta = float(rope_theta)
        self.int8 = bool(int(options) & OPT_INT8_KV)
        if self.int8:  # uint8 blocks: codes [16][d] then fp32 scales [16]
            shape, dtype = (self.num_pages, 2, self.num_kv_heads, 16 * self.head_dim + 64), torch.uint8
        else:
            shape, dtype = (self.num_pages, 2, self.num_kv_heads, PAGE_SIZE, self.head_dim), torch.float16
        if pools is None:
            pools = [torch.empty(shape, dtype=dtype, device=device) for _ in range(self.num_layers)]
        if len(pools) != self.num_layers:
            raise ValueError("one pool per layer is required")
        for t in pools:
            if t.dtype != dtype or tuple(t.shape) != shape or not t.is_contiguous():
                raise ValueError(f"pools must be contiguous {dtype} tensors of shape {shape}")
        self.pools = list(pools)
        nbytes = rope_table_bytes(self.max_position, self.head_dim)
        self.rope_table = torch.empty(max(nbytes // 4, 4), dtype=torch.float32, device=device)
        self.status_word = torch.zeros(1, dtype=torch.int32, device=device)
        self._pool_ptrs = (ctypes.c_void_p * self.num_layers)(*[t.data_ptr() for t in self.pools])
        win_ptr = ctypes.POINTER(ctypes.c_int32)()
        sink_ptr = ctypes.POINTER(ctypes.c_void_p)()
        self.windows = [0] * self.num_layers if windows is None else [int(w) for w in windows]
        self.sinks = [None] * self.num_layers if sinks is None else list(sinks)
        if len(self.windows) != self.num_layers or len(self.sinks) != self.num_layers:
            raise ValueError("windows and sinks take one entry per layer")
        for t in self.sinks:
            if t is not None and (t.dtype != torch.float32 or tuple(t.shape) != (self.num_qo_heads,)
                                  or not t.is_contiguous() or t.device.type != "cuda"):
                raise ValueError("sinks must be contiguous float32 CUDA tensors of shape [num_qo_heads]")
        if windows is not None:
            self._windows = (ctypes.c_int32 * self.num_layers)(*self.windows)
            win_ptr = ctypes.cast(self._windows, ctypes.POINTER(ctypes.c_int32))
        if sinks is not None:
            self._sink_ptrs = (ctypes.c_void_p * self.num_layers)(
                *[None if t is None else t.data_ptr() for t in self.sinks])
            sink_ptr = ctypes.cast(self._sink_ptrs, ctypes.POINTER(ctypes.c_void_p))
        d = _Desc(self.num_layers, self.num_pages, PAGE_SIZE, self.num_qo_heads, self.num_kv_heads,
                  self.head_dim, self.max_position, self.rope_theta,
                  ctypes.cast(self._pool_ptrs, ctypes.POINTER(ctypes.c_void_p)),
                  self.rope_table.data_ptr(), self.status_word.data_ptr(), int(options), win_ptr, sink_ptr)
        handle = ctypes.c_void_p()
        with torch.cuda.device(device):
            _check(lib().pkv_create_cache(ctypes.byref(d), ctypes.byref(handle)), "pkv_create_cache")
        self.handle = handle
        self.device = device

    def close(self):
        if getattr(self, "handle", None):
            lib().pkv_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- entry points ---------------------------------------------------------------------------

    def device_info(self, batch=1):
        """pkv_device_info: (SMs, decode warps per SM for a batch of ``batch`` sequences)."""
        n, w = ctypes.c_int(), ctypes.c_int()
        _check(lib().pkv_device_info(self.handle, int(batch), ctypes.byref(n), ctypes.byref(w)), "pkv_device_info")
        return n.value, w.value

    def append_rope(self, layer, q, k, v, pos_map, append_indptr, page_indptr, page_indices, q_out=None,
                    stream=None):
        """pkv_append_rope; returns q_out (fp16 [T, Hq, d])."""
        import torch

        if q_out is None:
            q_out = torch.empty_like(q)
        T, B = int(pos_map.numel()), int(append_indptr.numel()) - 1
        _check(lib().pkv_append_rope(self.handle, layer, _ptr(q), _ptr(k), _ptr(v), _ptr(pos_map),
                                     _ptr(append_indptr), T, B, _ptr(page_indptr), _ptr(page_indices),
                                     _ptr(q_out), _stream(stream)), "pkv_append_rope")
        return q_out

    def plan_decode(self, batch, max_pages_per_seq, total_pages=0, num_splits=0, chunk_pages=0,
                    max_splits=1 << 16):
        """pkv_plan_decode; returns (splits, chunk_pages)."""
        s, c = ctypes.c_int(), ctypes.c_int()
        _check(lib().pkv_plan_decode(self.handle, batch, max_pages_per_seq, total_pages, num_splits,
                                     chunk_pages, max_splits, ctypes.byref(s), ctypes.byref(c)),
               "pkv_plan_decode")
        return s.value, c.value

    def decode_attention(self, layer, q_rope, page_indptr, page_indices, last_page_len, max_pages_per_seq,
                         q_indptr=None, total_pages=0, num_splits=0, chunk_pages=0, sm_scale=0.0,
                         partial_o=None, partial_lse=None, stream=None):
        """pkv_decode_attention; returns (partial_o [B,Hq,S,d], partial_lse [B,Hq,S], S)."""
        import torch

        B = int(page_indptr.numel()) - 1
        if partial_o is None or partial_lse is None:
            S, _ = self.plan_decode(B, max_pages_per_seq, total_pages, num_splits, chunk_pages)
            partial_o = torch.empty((B, self.num_qo_heads, S, self.head_dim), dtype=torch.float32,
                                    device=q_rope.device)
            partial_lse = torch.empty((B, self.num_qo_heads, S), dtype=torch.float32, device=q_rope.device)
        cap = int(partial_lse.numel()) // max(1, B * self.num_qo_heads)
        used = ctypes.c_int()
        _check(lib().pkv_decode_attention(self.handle, layer, _ptr(q_rope), _ptr(q_indptr), _ptr(page_indptr),
                                          _ptr(page_indices), _ptr(last_page_len), B, max_pages_per_seq,
                                          total_pages, num_splits, chunk_pages, max(cap, 1), float(sm_scale),
                                          _ptr(partial_o), _ptr(partial_lse), ctypes.byref(used),
                                          _stream(stream)), "pkv_decode_attention")
        S = used.value
        if partial_lse.dim() != 3 or partial_lse.shape[2] != S:
            partial_o = partial_o.view(-1)[: B * self.num_qo_heads * S * self.head_dim].view(
                B, self.num_qo_heads, S, self.head_dim)
            partial_lse = partial_lse.view(-1)[: B * self.num_qo_heads * S].view(B, self.num_qo_heads, S)
        return partial_o, partial_lse, S

    def decode_attention_merged(self, layer, q_rope, page_indptr, page_indices, last_page_len,
                                max_pages_per_seq, chunk_counters, q_indptr=None, total_pages=0, num_splits=0,
                                chunk_pages=0, sm_scale=0.0, partial_o=None, partial_lse=None, out=None,
                                lse=None, stream=None):
        """pkv_decode_attention_merged; returns (out fp16 [B,Hq,d], lse fp32 [B,Hq]).

        ``chunk_counters`` is an int32 device tensor of at least B * Hkv zeros (left zero)."""
        import torch

        B = int(page_indptr.numel()) - 1
        dev = q_rope.device
        if partial_o is None or partial_lse is None:
            S, _ = self.plan_decode(B, max_pages_per_seq, total_pages, num_splits, chunk_pages)
            partial_o = torch.empty((B, self.num_qo_heads, S, self.head_dim), dtype=torch.float32, device=dev)
            partial_lse = torch.empty((B, self.num_qo_heads, S), dtype=torch.float32, device=dev)
        if out is None:
            out = torch.empty((B, self.num_qo_heads, self.head_dim), dtype=torch.float16, device=dev)
        if lse is None:
            lse = torch.empty((B, self.num_qo_heads), dtype=torch.float32, device=dev)
        if chunk_counters.dtype != torch.int32 or chunk_counters.numel() < B * self.num_kv_heads:
            raise ValueError("chunk_counters must be an int32 tensor of at least batch * num_kv_heads elements")
        cap = int(partial_lse.numel()) // max(1, B * self.num_qo_heads)
        used = ctypes.c_int()
        _check(lib().pkv_decode_attention_merged(
            self.handle, layer, _ptr(q_rope), _ptr(q_indptr), _ptr(page_indptr), _ptr(page_indices),
            _ptr(last_page_len), B, max_pages_per_seq, total_pages, num_splits, chunk_pages, max(cap, 1),
            float(sm_scale), _ptr(partial_o), _ptr(partial_lse), _ptr(chunk_counters), _ptr(out), _ptr(lse),
            ctypes.byref(used), _stream(stream)), "pkv_decode_attention_merged")
        return out, lse

    def append_decode_attention(self, layer, q, k, v, pos_map, append_indptr, page_indptr, page_indices,
                                last_page_len, max_pages_per_seq, chunk_counters, total_pages=0, num_splits=0,
                                chunk_pages=0, sm_scale=0.0, q_out=None, partial_o=None, partial_lse=None,
                                out=None, lse=None, stream=None):
        """pkv_append_decode_attention (append + merged decode in one launch); returns (q_out, out, lse)."""
        import torch

        B = int(page_indptr.numel()) - 1
        dev = q.device
        if partial_o is None or partial_lse is None:
            S, _ = self.plan_decode(B, max_pages_per_seq, total_pages, num_splits, chunk_pages)
            partial_o = torch.empty((B, self.num_qo_heads, S, self.head_dim), dtype=torch.float32, device=dev)
            partial_lse = torch.empty((B, self.num_qo_heads, S), dtype=torch.float32, device=dev)
        if q_out is None:
            q_out = torch.empty_like(q)
        if out is None:
            out = torch.empty((B, self.num_qo_heads, self.head_dim), dtype=torch.float16, device=dev)
        if lse is None:
            lse = torch.empty((B, self.num_qo_heads), dtype=torch.float32, device=dev)
        if chunk_counters.dtype != torch.int32 or chunk_counters.numel() < B * self.num_kv_heads:
            raise ValueError("chunk_counters must be an int32 tensor of at least batch * num_kv_heads elements")
        cap = int(partial_lse.numel()) // max(1, B * self.num_qo_heads)
        used = ctypes.c_int()
        _check(lib().pkv_append_decode_attention(
            self.handle, layer, _ptr(q), _ptr(k), _ptr(v), _ptr(pos_map), _ptr(append_indptr), int(pos_map.numel()),
            _ptr(page_indptr), _ptr(page_indices), _ptr(last_page_len), B, max_pages_per_seq, total_pages,
            num_splits, chunk_pages, max(cap, 1), float(sm_scale), _ptr(q_out), _ptr(partial_o), _ptr(partial_lse),
            _ptr(chunk_counters), _ptr(out), _ptr(lse), ctypes.byref(used), _stream(stream)),
            "pkv_append_decode_attention")
        return q_out, out, lse

    def decode_attention_noalloc(self, layer, q_rope, page_indptr, page_indices, last_page_len,
                                 max_pages_per_seq, out, lse=None, q_indptr=None, total_pages=0, num_splits=0,
                                 chunk_pages=0, sm_scale=0.0, stream=None):
        """pkv_decode_attention_noalloc: the merged decode with the library's own fixed scratch.

        For callers that cannot allocate device memory on this path: ``out`` (fp16 [B,Hq,d]) and
        ``lse`` (fp32 [B,Hq] or None) are caller tensors, and nothing is allocated here or in the
        library.  Calls share one scratch array: do not let them overlap on the GPU."""
        B = int(page_indptr.numel()) - 1
        used = ctypes.c_int()
        _check(lib().pkv_decode_attention_noalloc(
            self.handle, layer, _ptr(q_rope), _ptr(q_indptr), _ptr(page_indptr), _ptr(page_indices),
            _ptr(last_page_len), B, max_pages_per_seq, total_pages, num_splits, chunk_pages, float(sm_scale),
            _ptr(out), _ptr(lse), ctypes.byref(used), _stream(stream)), "pkv_decode_attention_noalloc")
        return out, lse

    def combine(self, partial_o, partial_lse, out=None, lse=None, stream=None, sinks=None):
        """pkv_combine; returns (out fp16 [B,Hq,d], lse fp32 [B,Hq]); sinks: fp32 [Hq] or None."""
        import torch

        B, Hq, S, d = (int(x) for x in partial_o.shape)
        if out is None:
            out = torch.empty((B, Hq, d), dtype=torch.float16, device=partial_o.device)
        if lse is None:
            lse = torch.empty((B, Hq), dtype=torch.float32, device=partial_o.device)
        _check(lib().pkv_combine(self.handle, _ptr(partial_o), _ptr(partial_lse), _ptr(sinks), B, Hq, S, d,
                                 _ptr(out), _ptr(lse), _stream(stream)), "pkv_combine")
        return out, lse

    def prefill_attention(self, layer, q_rope, append_indptr, pos_map, page_indptr, page_indices, last_page_len,
                          sm_scale=0.0, out=None, lse=None, stream=None):
        """pkv_prefill_attention: every appended token attends causally; returns (out, lse)."""
        import torch

        T = int(q_rope.shape[0])
        B = int(append_indptr.numel()) - 1
        if out is None:
            out = torch.empty((T, self.num_qo_heads, self.head_dim), dtype=torch.float16, device=q_rope.device)
        if lse is None:
            lse = torch.empty((T, self.num_qo_heads), dtype=torch.float32, device=q_rope.device)
        _check(lib().pkv_prefill_attention(self.handle, layer, _ptr(q_rope), _ptr(append_indptr), _ptr(pos_map), T,
                                           _ptr(page_indptr), _ptr(page_indices), _ptr(last_page_len), B,
                                           float(sm_scale), _ptr(out), _ptr(lse), _stream(stream)),
               "pkv_prefill_attention")
        return out, lse

    def qkv_project(self, x, w, scales, y=None, stream=None):
        """pkv_qkv_project: x fp16 [T, hidden], w int32/uint32 [N, hidden/8], scales fp16
        [N, hidden/32] -> y fp16 [T, N]."""
        import torch

        T, hidden = (int(v) for v in x.shape)
        if y is None:
            y = torch.empty((T, int(w.shape[0])), dtype=torch.float16, device=x.device)
        _check(lib().pkv_qkv_project(self.handle, _ptr(x), _ptr(w), _ptr(scales), hidden, T, _ptr(y),
                                     _stream(stream)), "pkv_qkv_project")
        return y

    def qkv_append_rope(self, layer, x, w, scales, pos_map, append_indptr, page_indptr, page_indices,
                        q_out=None, stream=None):
        """pkv_qkv_append_rope: the Q4F16_1 projection of x, then RoPE and the append; returns q_out."""
        import torch

        T, hidden = (int(v) for v in x.shape)
        B = int(append_indptr.numel()) - 1
        if q_out is None:
            q_out = torch.empty((T, self.num_qo_heads, self.head_dim), dtype=torch.float16, device=x.device)
        _check(lib().pkv_qkv_append_rope(self.handle, layer, _ptr(x), _ptr(w), _ptr(scales), hidden, _ptr(pos_map),
                                         _ptr(append_indptr), T, B, _ptr(page_indptr), _ptr(page_indices),
                                         _ptr(q_out), _stream(stream)), "pkv_qkv_append_rope")
        return q_out

    def set_wait_limit(self, limit_ns: int = 0):
        """pkv_set_wait_limit: limit of the kernels' waits for staged copies (0 = the 2 s default)."""
        _check(lib().pkv_set_wait_limit(self.handle, int(limit_ns)), "pkv_set_wait_limit")

    def set_stage_stall(self, on: bool = True):
        """pkv_set_stage_stall (test setting): the decode kernel's stage barriers wait for an
        arrival that nothing makes, so that every stage wait runs out at the wait limit."""
        _check(lib().pkv_set_stage_stall(self.handle, 1 if on else 0), "pkv_set_stage_stall")

    def check_status(self, stream=None):
        """pkv_check_status; returns (status code, flag bits) without raising."""
        flags = ctypes.c_int()
        code = lib().pkv_check_status(self.handle, _stream(stream), ctypes.byref(flags))
        return code, flags.value


def combine(partial_o, partial_lse, out=None, lse=None, stream=None, sinks=None):
    """pkv_combine without a cache (plain launches); sinks: fp32 [Hq] or None."""
    import torch

    B, Hq, S, d = (int(x) for x in partial_o.shape)
    if out is None:
        out = torch.empty((B, Hq, d), dtype=torch.float16, device=partial_o.device)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=partial_o.device)
    _check(lib().pkv_combine(None, _ptr(partial_o), _ptr(partial_lse), _ptr(sinks), B, Hq, S, d, _ptr(out),
                             _ptr(lse), _stream(stream)), "pkv_combine")
    return out, lse
