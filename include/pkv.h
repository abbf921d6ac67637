/*
 * pkv.h - C ABI of the GB300 paged-KV decode attention library (libpkv.so).
 *
 * The library implements, for one transformer layer at a time, the decode-step
 * attention path over a paged KV cache:
 *
 *   1. pkv_append_rope       rotate the new tokens' q and k with RoPE and write
 *                            k and v into 16-slot pages of the cache;
 *   2. pkv_decode_attention  split-K partial attention of every query head over
 *                            its sequence's pages;
 *   3. pkv_combine           log-sum-exp merge of the partials.
 *
 * Sources: Zero TVM Documentation ("KV cache", "Decode loop", "How it works",
 * "Port to Phi-4-mini or Qwen3"); the MLC model artifact manifest page (the
 * create_kv_cache role "takes only its size arguments"; decode_tokens takes a
 * [batch_size, 1] batch); everything-webgpu AI.md (fail fast, typed errors).
 *
 * Conventions that hold for every entry point:
 *  - Ownership: the caller allocates and frees every device buffer (pools, the
 *    RoPE table, the status word, q/k/v, page tables, partials, outputs).  A
 *    pkv_cache handle owns its host memory and one 8-byte device counter (the
 *    prefill kernel's work counter); pkv_destroy frees both and nothing else.
 *  - Device: a cache is bound to the CUDA device that was current when it was
 *    created; call the other entry points with that device current.
 *  - Asynchrony: calls enqueue kernels on the given stream and return; results
 *    are stream-ordered.  Only pkv_create_cache and pkv_check_status block.
 *  - Errors found on the host (null pointers, bad sizes, unsupported shapes)
 *    return a status before anything is enqueued and nothing is written.
 *    Errors that only the device can see (an index out of range in a page table
 *    or position map) make the kernel skip the offending read or write and set
 *    bits in the cache's status word; pkv_check_status reports them.  No
 *    kernel traps, asserts or aborts.
 *  - int32 index arrays are device arrays of the stated length.
 *  - fp16 means IEEE binary16; results are rounded to nearest even.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Slots per KV page (Zero TVM Documentation, "KV cache": fixed pages of 16 slots). */
#define PKV_PAGE_SIZE 16

typedef struct CUstream_st* pkv_stream_t; /* a cudaStream_t; NULL is the legacy default stream */

typedef enum {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARG = 1,  /* null pointer, negative size, inconsistent sizes */
  PKV_ERR_UNSUPPORTED = 2,  /* shape outside what the kernels are built for */
  PKV_ERR_OUT_OF_RANGE = 3, /* device saw an index out of range (see pkv_check_status) */
  PKV_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
  PKV_ERR_TIMEOUT = 5       /* a device-side wait gave up (reported by pkv_check_status) */
} pkv_status;

/* Bits of the device status word (pkv_check_status returns them in *flags). */
#define PKV_FLAG_BAD_PAGE 0x1     /* a page-table entry outside [0, num_pages) */
#define PKV_FLAG_BAD_POSITION 0x2 /* a position < 0, >= max_position, or past the sequence's pages */
#define PKV_FLAG_BAD_SEQUENCE 0x4 /* last_page_len outside [1, 16], more pages than declared, bad token or query range */
#define PKV_FLAG_TIMEOUT 0x8      /* a bounded wait on a shared-memory barrier expired */

/* Cache option bits (pkv_cache_desc.options). */
#define PKV_OPT_PDL 0x1 /* launch with programmatic dependent launch: each kernel may start while
                           the previous kernel in the stream finishes.  Kernels wait for it (the
                           launch wait) before reading q, k, v, x, the pool, the partials and the
                           counters, but read their int32 index arrays (page_indptr, page_indices,
                           last_page_len, append_indptr, q_indptr, pos_map) and, for the QKV entry
                           points, the weights and scales before it.  Those arrays must be complete
                           when the kernel starts: written by the host, by a copy, or by a kernel
                           that does not let its dependents start early (a kernel launched without
                           programmatic dependent launch signals the next one only when it has
                           finished).  Do not produce them in a kernel that starts its dependents
                           early, such as this library's own kernels under this option. */
#define PKV_OPT_INT8_KV 0x4 /* int8 KV pages (Zero TVM Documentation, "The memory-bandwidth ceiling":
                               int8 KV behind a flag; the format is this library's reading): each
                               layer's pool is uint8 blocks
                               [num_pages][2][Hkv][16 * head_dim + 64] holding the 16 slots' int8
                               codes, each stored as the byte code + 128, then their fp32 scales
                               [16]: K codes slot-major
                               [16][head_dim], V codes dim-major [head_dim][16].  The append
                               quantizes each new K row (after RoPE and its fp16 rounding) and V row:
                               s = max|x| / 127 (fp32), code = clamp(rint(x / s), -127, 127) (fp32);
                               attention runs on the exact codes (tensor cores when Hq / Hkv >= 2,
                               CUDA cores for one query head per KV head, as for fp16 pages) and
                               applies the scales in fp32 to the scores (K) and the
                               probabilities (V).  pkv_append_decode_attention runs as two
                               launches; pkv_prefill_attention and pkv_qkv_append_rope return
                               PKV_ERR_UNSUPPORTED. */
#define PKV_OPT_EARLY_PAGES 0x2 /* with PKV_OPT_PDL, the one-launch step (pkv_append_decode_attention
                                   with one token per sequence) starts copying the layer's cached
                                   pages before the launch wait, so the copies overlap the end of the
                                   previous kernels; the new tokens' q, k, v are read after it.  The
                                   last two pages of every sequence, which hold the 16 positions
                                   before its new token (written by the preceding decode steps of
                                   the layer, which may still be running), are always copied after
                                   the wait.  A layer whose pool was written by another call since
                                   its last one-launch step (pkv_append_rope, pkv_qkv_append_rope, a
                                   chunked pkv_append_decode_attention) runs its next one-launch step
                                   without early copies; the choice is made when the call is made
                                   (also while a stream is being captured).  The caller's own writes
                                   to a pool must come from kernels that do not start their
                                   dependents early (see PKV_OPT_PDL).  The whole ring goes early
                                   when Hq / Hkv >= 2 (tensor-core path), two stages per warp
                                   otherwise (the depths that measured fastest). */

typedef struct pkv_cache pkv_cache; /* opaque, host-only */

/*
 * Geometry and caller-owned device storage of a paged KV cache.
 *
 * Pool layout, one pool per layer (a reading of Zero TVM Documentation, "KV
 * cache": one buffer of pages per layer; the page-internal order is ours):
 *     fp16 pool[num_pages][2][num_kv_heads][16][head_dim]
 * index 0 of the second dimension holds K (rotated), index 1 holds V, so the
 * K (or V) of one page and one KV head is a contiguous 16*head_dim*2-byte run.
 */
typedef struct {
  int num_layers;        /* >= 1 */
  int num_pages;         /* pages in each layer's pool, >= 1 */
  int page_size;         /* must be PKV_PAGE_SIZE */
  int num_qo_heads;      /* Hq >= 1 */
  int num_kv_heads;      /* Hkv >= 1, Hq % Hkv == 0, Hq / Hkv <= 8 */
  int head_dim;          /* 64, 96 or 128 */
  int max_position;      /* appended positions must lie in [0, max_position) */
  double rope_theta;     /* RoPE base (e.g. 1e4, 1e6) */
  void* const* layer_pools; /* host array [num_layers] of device pointers, each 256-byte aligned,
                               pkv_pool_bytes(num_pages, num_kv_heads, head_dim) bytes */
  float* rope_table;     /* device buffer of pkv_rope_table_bytes(max_position, head_dim) bytes,
                            filled by pkv_create_cache; must outlive the cache */
  int* status_word;      /* device int32, zeroed by pkv_create_cache; must outlive the cache */
  int options;           /* PKV_OPT_* bits */
  /* Per-layer attention variants (Splash models page: a family's sliding_window, its
   * layer_types, and each layer's attn_sinks, F32).  Both may be NULL (every layer full
   * attention, no sinks); both are read by pkv_create_cache, which copies them.
   *   layer_window  host int32 [num_layers]: 0 = full attention; W > 0 = the query at position
   *                 len-1 attends to positions [max(0, len-W), len), the W most recent tokens
   *                 including itself.  Such a layer is split into chunks of its visible pages.
   *   layer_sinks   host array [num_layers] of device pointers (each NULL or fp32 [num_qo_heads],
   *                 caller-owned, alive while the cache is used): one logit per query head, in
   *                 the units of the scaled scores (natural log), that joins the softmax's
   *                 denominator and carries no value:
   *                   out = sum_t e^s_t V_t / (sum_t e^s_t + e^sink),
   *                   lse = ln(sum_t e^s_t + e^sink).
   *                 The partials of pkv_decode_attention do not include it; pass the layer's
   *                 sinks to pkv_combine.  The merged entry points apply it. */
  const int32_t* layer_window;
  const float* const* layer_sinks;
} pkv_cache_desc;

/* Bytes of one layer's pool. */
size_t pkv_pool_bytes(int num_pages, int num_kv_heads, int head_dim);

/* Bytes of one layer's int8 pool (PKV_OPT_INT8_KV): num_pages * 2 * Hkv * (16 * head_dim + 64). */
size_t pkv_pool_bytes_int8(int num_pages, int num_kv_heads, int head_dim);

/* Bytes of the RoPE table: max_position * (head_dim / 2) (cos, sin) pairs of fp32, computed on
 * the host in fp64 as cos/sin(p * theta^(-2i/head_dim)) and rounded once to fp32. */
size_t pkv_rope_table_bytes(int max_position, int head_dim);

/*
 * Create a cache handle over caller-owned storage (the create_kv_cache role of the MLC model
 * artifact manifest page: the constructor takes sizes only; here also the storage).
 * Blocks: fills desc->rope_table and zeroes desc->status_word with synchronous copies,
 * allocates and zeroes the handle's 8-byte device work counter, and builds the TMA descriptors
 * of each layer pool.  The pools' contents are not touched.
 * Returns PKV_ERR_INVALID_ARG / PKV_ERR_UNSUPPORTED for bad descriptors, PKV_ERR_CUDA if a
 * CUDA call fails; *out is set only on PKV_OK.
 */
pkv_status pkv_create_cache(const pkv_cache_desc* desc, pkv_cache** out);

/* Free the handle and its device work counter (on the cache's device).  NULL is ignored. */
void pkv_destroy(pkv_cache* cache);

/*
 * RoPE + KV append for one layer (Zero TVM Documentation, "Decode loop": the QKV dispatch
 * rotates q and k at posMap and scatters k and v into page slots; "KV cache": K is rotated
 * before the cache write).
 *
 *   q       fp16 [num_tokens][Hq][head_dim]   raw queries of the new tokens
 *   k, v    fp16 [num_tokens][Hkv][head_dim]  raw keys and values of the new tokens
 *   pos_map int32 [num_tokens]                position of each new token in its sequence
 *   append_indptr int32 [batch+1]             tokens of sequence s are append_indptr[s] ..
 *                                             append_indptr[s+1]-1 (non-decreasing, [0] = 0,
 *                                             [batch] = num_tokens)
 *   page_indptr   int32 [batch+1]             pages of sequence s are page_indices[page_indptr[s]
 *   page_indices  int32 [page_indptr[batch]]  .. page_indptr[s+1]-1], logical page order
 *   q_out   fp16 [num_tokens][Hq][head_dim]   rotated queries (may not alias q)
 *
 * Token t of sequence s at position p = pos_map[t] goes to page
 * page_indices[page_indptr[s] + p / 16], slot p % 16:
 *   pool[page][0][g][slot][:] = RoPE(k[t][g][:], p)   for every KV head g
 *   pool[page][1][g][slot][:] = v[t][g][:]            (bit copy)
 *   q_out[t][h][:]            = RoPE(q[t][h][:], p)   for every query head h
 * RoPE is the rotate-half form: element i pairs with i + head_dim/2.  Rotations are computed
 * in fp32 from the fp64-derived table; results are rounded to fp16.
 * Positions must be distinct within a sequence (duplicates: the last write wins, unspecified).
 * Device-detected: positions out of range (PKV_FLAG_BAD_POSITION), page ids out of range
 * (PKV_FLAG_BAD_PAGE), token ranges outside [0, num_tokens) (PKV_FLAG_BAD_SEQUENCE);
 * the affected token is skipped.  num_tokens == 0 or batch == 0 is a no-op.
 */
pkv_status pkv_append_rope(pkv_cache* cache, int layer, const void* q, const void* k, const void* v,
                           const int32_t* pos_map, const int32_t* append_indptr, int num_tokens,
                           int batch, const int32_t* page_indptr, const int32_t* page_indices,
                           void* q_out, pkv_stream_t stream);

/*
 * Chunked-prefill attention (the step after a multi-token append: every appended token attends
 * causally to its sequence; Zero TVM Documentation, "Decode loop": a token attends to itself and
 * to the earlier positions of its sequence).  Token t of sequence s (append_indptr), at position
 * p = pos_map[t] < len_s, attends to the positions [max(0, p + 1 - W), p] of s (W = the layer's
 * window, 0 = all) in the cache after the append; the layer's sinks join the denominator:
 *   out[t][h][:] = fp16( sum_u e^{s_u} V_u / (sum_u e^{s_u} + e^{sink_h}) ),
 *   lse_out[t][h] = ln(sum_u e^{s_u} + e^{sink_h}),   s_u = sm_scale * q_t,h . K_u.
 *   q_rope   fp16 [num_tokens][Hq][head_dim] (e.g. q_out of pkv_append_rope), 16-byte aligned
 *   out      fp16 [num_tokens][Hq][head_dim], 16-byte aligned;  lse_out fp32 [num_tokens][Hq] or NULL
 * Tiles of (sequence, KV head, 128 / G tokens x G heads) run tcgen05.mma over 128-key blocks of
 * the pages the tile attends to, taken longest first by the CTAs through the cache's device work
 * counter: prefill calls on one cache must not overlap on the GPU (call them on one stream, or
 * order their streams).  Device-detected errors: page ids out of range, positions outside
 * [0, len_s), bad last_page_len (the token's rows are left unwritten).  With one token per
 * sequence at its last position this equals the merged decode up to rounding.
 */
pkv_status pkv_prefill_attention(const pkv_cache* cache, int layer, const void* q_rope,
                                 const int32_t* append_indptr, const int32_t* pos_map, int num_tokens,
                                 const int32_t* page_indptr, const int32_t* page_indices,
                                 const int32_t* last_page_len, int batch, float sm_scale, void* out,
                                 float* lse_out, pkv_stream_t stream);

/*
 * QKV projection with Q4F16_1 weights, fused with RoPE and the KV append (Zero TVM Documentation,
 * "Decode loop": the QKV matmul, RoPE and the KV append in one dispatch; "Q4F16 quantization
 * format": eight int4 values per uint32, element i in bits 4i..4i+3, one fp16 scale per 32
 * weights, weight value f16(nibble - 7) * scale evaluated in fp16).
 *   x        fp16 [num_tokens][hidden] (16-byte aligned), hidden a multiple of 32, <= 4096
 *   w        uint32 [N][hidden / 8] (16-byte aligned), N = (Hq + 2 Hkv) * head_dim output rows
 *            ordered [q heads | k heads | v heads]; input k of row n is nibble k % 8 of
 *            w[n][k / 8]
 *   scales   fp16 [N][hidden / 32]
 * For every token and output row n: y = fp16(sum_k x_k * f16((nibble - 7) * scale)), the
 * products rounded to fp16 as the format states and summed in fp32.  The q, k and v rows of y
 * then go through pkv_append_rope (same arguments and errors), bit for bit as if y had been
 * written and pkv_append_rope called on it.  The weights are read before the programmatic
 * dependent launch wait (they are not produced by the preceding kernel).
 */
pkv_status pkv_qkv_append_rope(pkv_cache* cache, int layer, const void* x, const uint32_t* w, const void* scales,
                               int hidden, const int32_t* pos_map, const int32_t* append_indptr, int num_tokens,
                               int batch, const int32_t* page_indptr, const int32_t* page_indices, void* q_out,
                               pkv_stream_t stream);

/*
 * The projection of pkv_qkv_append_rope alone: y fp16 [num_tokens][N] (16-byte aligned), the
 * same bits the fused call rotates and appends.  Arguments as there.
 */
pkv_status pkv_qkv_project(const pkv_cache* cache, const void* x, const uint32_t* w, const void* scales,
                           int hidden, int num_tokens, void* y, pkv_stream_t stream);

/*
 * Split plan (host only, no device access).  Returns in *splits the number of partial slots per
 * (sequence, query head) that pkv_decode_attention will produce for these arguments, and in
 * *chunk_pages the uniform chunk size in pages (0 when num_splits > 0 selects per-sequence
 * chunks of ceil(n_s / num_splits) pages).
 *   num_splits > 0            per-sequence chunks: c_s = ceil(n_s / num_splits), splits = num_splits
 *   chunk_pages > 0           uniform chunks of chunk_pages pages, splits = ceil(max_pages / c)
 *   both 0, total_pages > 0   the balanced partition (*chunk_pages_out = -1): the page units of all
 *                             (sequence, KV head) pairs, in sequence, head, page order, are cut
 *                             into W = min(SMs x resident decode warps, U) equal runs, run w being
 *                             units [floor(w*U/W), floor((w+1)*U/W)) with U = Hkv * total_pages;
 *                             chunk j of a (sequence, KV head) is its piece in the j-th run that
 *                             meets it; splits = ceil(max_pages * W / U) + 1.  total_pages must
 *                             equal page_indptr[batch].
 *   both 0, total_pages == 0  a uniform chunk size from the batch, the KV heads, max_pages_per_seq
 *                             and the SM count, so that the work items fill the resident warps.
 *   The split count never exceeds max_splits (the balanced partition is not used when it would).
 * A layer with a sliding window (pkv_cache_desc.layer_window) walks each sequence's visible pages
 * (at most V = ceil(W/16) + 1): num_splits and chunk_pages apply to them; with neither, the
 * balanced partition of the visible page units (the kernel counts them; splits = V + 1), or, if
 * that exceeds max_splits, chunks of about four work items per resident warp.  *splits is the
 * most any layer of the cache produces (the capacity partial buffers need); *chunk_pages_out
 * describes the layers without a window.
 * (Zero TVM Documentation, "How it works": split-K over KV chunks with a fixed ?splitk=N; the
 * choice from length and SM count is this library's.)
 */
pkv_status pkv_plan_decode(const pkv_cache* cache, int batch, int max_pages_per_seq, int total_pages,
                           int num_splits, int chunk_pages, int max_splits, int* splits,
                           int* chunk_pages_out);

/* Bytes of partial_o for (batch, Hq, splits, head_dim): batch*Hq*splits*head_dim*4.
 * partial_lse takes batch*Hq*splits*4 bytes. */
size_t pkv_partial_bytes(int batch, int num_qo_heads, int splits, int head_dim);

/*
 * Split-K partial attention for one layer (Zero TVM Documentation, "How it works": attention
 * split over KV chunks; "Port to Phi-4-mini or Qwen3": KV heads repeated for grouped queries).
 *
 *   q_rope  fp16 [rows][Hq][head_dim]  rotated queries (e.g. q_out of pkv_append_rope)
 *   q_indptr int32 [batch+1] or NULL   NULL: sequence s uses row s; otherwise row
 *                                      q_indptr[s+1]-1 (the last appended token of s)
 *   page_indptr, page_indices          as for pkv_append_rope (after the append)
 *   last_page_len int32 [batch]        valid slots of each sequence's last page, in [1, 16];
 *                                      sequence length = 16 * (n_s - 1) + last_page_len[s]
 *                                      (n_s = 0 means an empty sequence)
 *   max_pages_per_seq                  an upper bound of every n_s
 *   total_pages                        page_indptr[batch] if known on the host (then exact), else 0
 *   num_splits, chunk_pages, max_splits  split selection, see pkv_plan_decode
 *   sm_scale                           score scale; 0 selects 1/sqrt(head_dim)
 *   partial_o   fp32 [batch][Hq][S][head_dim]  S = *splits_used (capacity max_splits);
 *                                      16-byte aligned, like q_rope and out
 *   partial_lse fp32 [batch][Hq][S]            natural-log LSE of each chunk
 *   splits_used (host, nullable)       receives S
 *
 * Query head h reads KV head h / (Hq / Hkv).  Chunk j of sequence s covers its pages
 * [j*c, min((j+1)*c, n_s)) (or its j-th piece of the balanced partition); for each (s, h, j)
 * with at least one token:
 *   partial_lse = ln sum_t exp(sm_scale * q.K_t),  partial_o = sum_t softmax_t * V_t
 * in fp32 from fp16 data.  Chunks with no token get partial_lse = -inf and partial_o is not
 * written.  Device-detected: page ids out of range (the page is masked out), n_s above
 * max_pages_per_seq, bad last_page_len or q_indptr rows (the sequence is reported empty).
 */
pkv_status pkv_decode_attention(const pkv_cache* cache, int layer, const void* q_rope,
                                const int32_t* q_indptr, const int32_t* page_indptr,
                                const int32_t* page_indices, const int32_t* last_page_len, int batch,
                                int max_pages_per_seq, int total_pages, int num_splits,
                                int chunk_pages, int max_splits, float sm_scale, float* partial_o,
                                float* partial_lse, int* splits_used, pkv_stream_t stream);

/*
 * Split-K decode attention and the log-sum-exp combine in one launch: the same chunks as
 * pkv_decode_attention, but the last chunk of each (sequence, KV head) to finish merges the
 * chunks' partials exactly as pkv_combine does and writes the result, so no separate combine
 * kernel runs.  A sequence with a single chunk writes its result directly (the same bits as the
 * merge of one split).  Arguments as pkv_decode_attention, plus:
 *   partial_o, partial_lse  workspace of the same shapes (contents undefined on return)
 *   chunk_counters  int32 [batch * Hkv] device workspace; all zero before the first call and left
 *                   all zero by every call that completes (re-zero it after PKV_ERR_TIMEOUT)
 *   out             fp16 [batch][Hq][head_dim] result;  lse_out  fp32 [batch][Hq] or NULL
 * Calls that share chunk_counters must not overlap on the device.
 */
pkv_status pkv_decode_attention_merged(const pkv_cache* cache, int layer, const void* q_rope,
                                       const int32_t* q_indptr, const int32_t* page_indptr,
                                       const int32_t* page_indices, const int32_t* last_page_len,
                                       int batch, int max_pages_per_seq, int total_pages, int num_splits,
                                       int chunk_pages, int max_splits, float sm_scale, float* partial_o,
                                       float* partial_lse, int32_t* chunk_counters, void* out,
                                       float* lse_out, int* splits_used, pkv_stream_t stream);

/*
 * One layer's whole decode step: the append of pkv_append_rope, then pkv_decode_attention_merged
 * over the updated cache, with the same results bit for bit.  Arguments as pkv_append_rope (q, k,
 * v are the raw new tokens; q_out receives the rotated q) and pkv_decode_attention_merged (the
 * query of sequence s is its last new token, row append_indptr[s+1]-1; every sequence with pages
 * must append at least one token).
 * When num_tokens == batch (one new token per sequence, the decode step) everything runs in one
 * launch: the stage that starts a work item also brings the token's raw k and v, the consumer
 * rotates k (the append kernel's arithmetic) and, on the page that holds the token, writes the
 * rotated K and V rows into the staged copy and into the cache; every item rotates its query
 * itself and the first item of each (sequence, KV head) writes that group's q_out rows and reports
 * positions out of range.  A sequence whose append_indptr range is not exactly one token is then
 * reported as PKV_FLAG_BAD_SEQUENCE.  Otherwise (a chunked append) the call issues the two
 * launches of pkv_append_rope and pkv_decode_attention_merged.
 * (Zero TVM Documentation, "Decode loop": QKV + RoPE + KV-append fused into one dispatch; here
 * the append is fused with the attention that follows it instead.)
 */
pkv_status pkv_append_decode_attention(pkv_cache* cache, int layer, const void* q, const void* k,
                                       const void* v, const int32_t* pos_map, const int32_t* append_indptr,
                                       int num_tokens, const int32_t* page_indptr,
                                       const int32_t* page_indices, const int32_t* last_page_len, int batch,
                                       int max_pages_per_seq, int total_pages, int num_splits,
                                       int chunk_pages, int max_splits, float sm_scale, void* q_out,
                                       float* partial_o, float* partial_lse, int32_t* chunk_counters,
                                       void* out, float* lse_out, int* splits_used, pkv_stream_t stream);

/*
 * pkv_decode_attention_merged without caller workspace, for callers that cannot allocate device
 * memory on this path: a framework that reserved the whole device for its own allocator up
 * front, or a serving loop that must not risk an allocation failure or the implicit device
 * synchronisation an allocation can cause in the middle of a step.  (This entry point has no
 * counterpart in the source pages; it is a property of this library's memory handling.)
 *
 * The caller passes inputs and outputs only (arguments as pkv_decode_attention_merged).  The
 * chunk counters and partials live in one file-scope device array of 32 MiB that every GPU that
 * loads the library holds until the process exits; nothing is allocated or freed by the call.
 * A request whose partials (batch * Hq * splits * (head_dim + 1) * 4 bytes) and counters
 * (batch * Hkv * 4 bytes) exceed 32 MiB returns PKV_ERR_UNSUPPORTED (see pkv_last_error).
 * The first call on a device, with that device current, looks up the array's device address
 * once; make that first call before any stream capture.  Call it with the cache's device current
 * (otherwise PKV_ERR_INVALID_ARG).  A device reset gives the device a new context, and the next
 * call looks the address up again.  Each call clears the counters on its stream before launching.
 * All calls share the one array: calls that overlap on the GPU race.
 */
pkv_status pkv_decode_attention_noalloc(const pkv_cache* cache, int layer, const void* q_rope,
                                        const int32_t* q_indptr, const int32_t* page_indptr,
                                        const int32_t* page_indices, const int32_t* last_page_len,
                                        int batch, int max_pages_per_seq, int total_pages, int num_splits,
                                        int chunk_pages, float sm_scale, void* out, float* lse_out,
                                        int* splits_used, pkv_stream_t stream);

/*
 * Log-sum-exp combine (Zero TVM Documentation, "How it works": one combine dispatch per layer
 * after split-K attention).  For each (s, h): M = max_j lse_j, w_j = exp(lse_j - M),
 *   out[s][h][:] = fp16( sum_j w_j o_j / sum_j w_j ),   lse_out[s][h] = M + ln sum_j w_j.
 * Splits with lse_j = -inf are skipped (their o_j is not read); if every split is -inf,
 * out = 0 and lse_out = -inf.  out: fp16 [batch][Hq][head_dim]; lse_out: fp32 [batch][Hq]
 * or NULL.  num_splits >= 1; head_dim in {64, 96, 128}.  sinks: NULL, or the layer's device
 * fp32 [Hq] attention sinks (see pkv_cache_desc), which join M and the denominator:
 * M = max(max_j lse_j, sink_h), out = sum_j w_j o_j / (sum_j w_j + exp(sink_h - M)).
 * The cache supplies the launch options (PKV_OPT_PDL); it may be NULL for plain launches.
 */
pkv_status pkv_combine(const pkv_cache* cache, const float* partial_o, const float* partial_lse,
                       const float* sinks, int batch, int num_qo_heads, int num_splits, int head_dim,
                       void* out, float* lse_out, pkv_stream_t stream);

/*
 * Synchronise `stream`, read and clear the cache's status word.  Returns PKV_OK when no bit was
 * set, PKV_ERR_TIMEOUT when PKV_FLAG_TIMEOUT was set, PKV_ERR_OUT_OF_RANGE for any other bit,
 * PKV_ERR_CUDA if a CUDA call failed.  flags (nullable) receives the raw bits.
 */
pkv_status pkv_check_status(pkv_cache* cache, pkv_stream_t stream, int* flags);

/*
 * Limit of the kernels' waits for their staged copies, in nanoseconds (default 2 s; 0 restores
 * it).  A decode or prefill warp whose wait runs out sets PKV_FLAG_TIMEOUT, waits up to 125 ms (a
 * fixed limit) for its own copies still in flight, and returns without writing its results;
 * pkv_check_status then reports PKV_ERR_TIMEOUT.  After a timeout, outputs are undefined and
 * chunk_counters must be re-zeroed.  The decode kernels count the limit on the GPU's global timer
 * and poll with suspending waits; the prefill kernel does the same from 1 ms up, and counts limits
 * below 1 ms (a test setting) in SM clock cycles (about half a nanosecond each), polling without
 * suspending, so that a limit shorter than a copy's latency (say 1) makes its waits run out on a
 * healthy GPU.  The decode kernels' failure path is tested with pkv_set_stage_stall.
 * Applies to the launches that follow the call.  Host only; returns PKV_ERR_INVALID_ARG for NULL.
 * (Everything WebGPU AI.md, "Fail Fast": failures surface as typed errors, not hangs.)
 */
pkv_status pkv_set_wait_limit(pkv_cache* cache, unsigned long long limit_ns);

/*
 * Test setting of the decode kernels (pkv_decode_attention, pkv_decode_attention_merged,
 * pkv_append_decode_attention and the no-alloc entry point): with `on` nonzero, each stage
 * barrier of the decode kernel is initialised for two arrivals where the producer makes one, so
 * that no stage's phase completes and every stage wait runs out at the wait limit (a wait for
 * something nothing provides), on every lane of every warp alike.  The copies themselves land as
 * usual.  With `on` zero (the default) one arrival completes a stage.  Applies to the launches that
 * follow the call.  Host only; returns PKV_ERR_INVALID_ARG for NULL.
 */
pkv_status pkv_set_stage_stall(pkv_cache* cache, int on);

/* Static description of a status code. */
const char* pkv_status_string(pkv_status status);

/* Description of the last failure on the calling thread (the CUDA call and its error string, or
 * the rejected argument); empty before any failure.  Valid until the thread's next failing call. */
const char* pkv_last_error(void);

/* Number of streaming multiprocessors of the cache's device and the resident warps the decode
 * kernel uses per SM for a batch of `batch` sequences (the page-balanced partition cuts the work
 * into num_sms * decode_warps_per_sm runs; the CUDA-core path runs more warps for large batches).
 * PKV_ERR_INVALID_ARG for a null cache or batch < 1. */
pkv_status pkv_device_info(const pkv_cache* cache, int batch, int* num_sms, int* decode_warps_per_sm);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
