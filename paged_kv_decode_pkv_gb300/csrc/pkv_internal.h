// Internal interface between the host library (pkv_host.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace pkv {

constexpr int kPageSize = 16;
constexpr int kMaxGroup = 8;        // Hq / Hkv handled by the kernels
constexpr int kMaxDecodeBatch = 4096;  // sequences per decode call (per-CTA shared-memory prefix)
constexpr int kMaxDecodeWarps = 8;     // warps per decode CTA, at most
// The CUDA-core decode (one query head per KV head), from this many sequences on: 12 warps per SM
// (two CTAs of six), the most of any decode layout
constexpr int kWideBatch = 8;
constexpr int kWideWarps = 12;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // bounded device waits: 2 s (default)
// A warp that gave up waits this long for its own copies still in flight before it returns, so
// that no copy lands in the shared memory of a finished block.  Not affected by the settable limit.
constexpr unsigned long long kDrainLimitNs = kWaitLimitNs / 16;

// Device status word bits (mirrors PKV_FLAG_* of include/pkv.h).
constexpr int kFlagBadPage = 0x1;
constexpr int kFlagBadPosition = 0x2;
constexpr int kFlagBadSequence = 0x4;
constexpr int kFlagTimeout = 0x8;

struct AppendParams {
  const __half* q;
  const __half* k;
  const __half* v;
  const int* pos_map;
  const int* append_indptr;
  const int* page_indptr;
  const int* page_indices;
  __half* q_out;
  __half* pool;
  const float2* rope;  // [max_position][head_dim / 2] (cos, sin)
  int* status;
  int num_tokens, batch, hq, hkv, head_dim, max_position, num_pages;
  unsigned char* pool8;  // int8 cache (PKV_OPT_INT8_KV): blocks [num_pages][2][hkv][16 * d + 64]
};

// QKV projection (Q4F16_1) fused with RoPE and the KV append.
struct QkvParams {
  const __half* x;           // [num_tokens][hidden]
  const uint32_t* w;         // [N][hidden / 8], N = (hq + 2 hkv) * head_dim
  const __half* scales;      // [N][hidden / 32]
  __half* y_out;             // nullable: write the projection [num_tokens][N] instead of appending
  const int* pos_map;
  const int* append_indptr;
  const int* page_indptr;
  const int* page_indices;
  __half* q_out;
  __half* pool;              // null with y_out
  const float2* rope;
  int* status;
  int num_tokens, batch, hidden, hq, hkv, head_dim, max_position, num_pages;
};
constexpr int kQkvMaxHidden = 4096;          // four input parts of 1024 (x two row halves = 8 warps)
constexpr int kQkvMaxSmem = 2 * kQkvMaxHidden * 2 + 4 * 2 * 16 * 4;

// Chunked-prefill attention: every appended token attends causally over its sequence's pages.
struct PrefillParams {
  const __half* q;  // [num_tokens][hq][head_dim], rotated
  const int* append_indptr;
  const int* pos_map;
  const int* page_indptr;
  const int* page_indices;
  const int* last_page_len;
  __half* out;      // [num_tokens][hq][head_dim]
  float* lse;       // [num_tokens][hq], nullable
  int* status;
  const float* sinks;  // nullable, per query head
  int batch, num_tokens, hq, hkv, group, num_pages;
  int window;       // 0 = full attention
  int nstage;       // K stages
  float scale_log2;
  unsigned long long wait_ns;  // limit of a wait for a staged copy (kWaitLimitNs unless set)
  int* work;  // device [2]: next work item, CTAs finished (the last CTA resets both to 0)
};
struct PrefillConfig {
  int nstage;
  size_t smem_bytes;
};
PrefillConfig prefill_config(int head_dim, int batch);
cudaError_t prefill_prepare();
cudaError_t launch_prefill(const PrefillParams& p, const CUtensorMap& map, const PrefillConfig& cfg, int head_dim,
                           int grid, cudaStream_t stream, bool pdl);

struct DecodeParams {
  const __half* q;
  const int* q_indptr;  // nullable
  const int* page_indptr;
  const int* page_indices;
  const int* last_page_len;
  float* partial_o;
  float* partial_lse;
  int* status;
  int batch, hq, hkv, group, num_pages;
  int splits;       // S: partial slots per (sequence, head)
  int chunk_pages;  // > 0: uniform chunks of this many pages; 0: ceil(n_s / splits) per sequence
  int max_pages;    // declared bound of n_s
  float scale_log2; // sm_scale * log2(e)
  int nstage;       // ring depth per warp
  int warps;        // consumer warps per CTA
  // Merged mode: the last chunk of each (sequence, KV head) to finish merges the partials and
  // writes out / lse_out; counters[s * hkv + g] counts finished chunks and is reset to zero.
  int merged;
  int* counters;
  __half* out;
  float* lse_out;   // nullable
  // Balanced mode: the page units of all (sequence, KV head) segments, in sequence, head, page
  // order, are cut into part_warps equal runs (run w = units [w*U/W, (w+1)*U/W)); warp w of the
  // grid processes run w.  units = U = hkv * page_indptr[batch] as declared by the host.
  int balanced;
  long long units;
  int part_warps;
  // Fused mode: the step's append runs inside the decode.  q is then the raw (unrotated) query,
  // q_indptr the append_indptr (the query of a sequence is its last new token), and the kernel
  // writes the rotated K and V of the new tokens into the pool and the rotated q into q_out.
  int fused;
  const __half* k_new;
  const __half* v_new;
  const int* pos_map;
  __half* q_out;
  __half* pool;
  const float2* rope;
  int max_position;
  // Layer variants: a sliding window of `window` positions (0 = full attention; chunk mode only,
  // the chunks then cover each sequence's visible pages) and per query head sink logits (natural
  // log, units of the scaled scores; nullable) that join the merge's denominator.
  int window;
  const float* sinks;
  int early;  // one-launch mode: stages per warp copied before the launch wait (PKV_OPT_EARLY_PAGES)
  const unsigned char* pool8;  // int8 cache: blocks [num_pages][2][hkv][16 * d + 64]
  unsigned long long wait_ns;  // limit of a wait for a staged copy (kWaitLimitNs unless set)
  int stall;  // test setting (pkv_set_stage_stall): stage barriers wait for a second arrival
};

struct CombineParams {
  const float* partial_o;
  const float* partial_lse;
  __half* out;
  float* lse;
  const float* sinks;  // nullable: per query head sink logits
  int batch, hq, splits, head_dim;
};

// Decode launch geometry for a (group, head_dim) pair and a batch size.
struct DecodeConfig {
  bool mma;             // tensor-core path (group >= 2)
  bool fused;           // append folded into the decode
  bool q8;              // int8 cache
  int warps;            // warps per CTA
  int ctas_per_sm;      // resident CTAs per SM (the grid of a full launch is SMs x this)
  int nstage;           // per-warp ring depth
  bool wide;            // CUDA-core layout of 12 warps per SM (its kernel holds at most 168 registers)
  size_t smem_bytes;    // dynamic shared memory
  int box_inner;        // TMA box extent along head_dim (elements)
  int swizzle_bytes;    // 0 (none), 64 or 128
};

DecodeConfig decode_config(int group, int head_dim, int batch, bool fused = false, bool windowed = false,
                           bool q8 = false);
cudaError_t decode_prepare(const DecodeConfig& cfg, int head_dim);  // function attributes
cudaError_t launch_decode(const DecodeParams& p, const CUtensorMap& map, const DecodeConfig& cfg, int head_dim,
                          int grid, cudaStream_t stream, bool pdl);
cudaError_t launch_append(const AppendParams& p, cudaStream_t stream, bool pdl);
cudaError_t launch_append_q8(const AppendParams& p, cudaStream_t stream, bool pdl);
__host__ __device__ constexpr int int8_block_bytes(int head_dim) { return 16 * head_dim + 64; }
cudaError_t append_prepare();   // function attributes (shared-memory carveout)
cudaError_t combine_prepare();
cudaError_t qkv_prepare();
cudaError_t launch_qkv(const QkvParams& p, cudaStream_t stream, bool pdl);
cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream, bool pdl);

}  // namespace pkv

struct pkv_cache;

namespace pkv {

// Host-side helpers for entry points defined outside pkv_host.cu.
void cache_geometry(const pkv_cache* cache, int* num_qo_heads, int* num_kv_heads, int* head_dim);
int cache_device(const pkv_cache* cache);  // the device that was current when the cache was created
void set_last_error(const char* what);

}  // namespace pkv
