// Host side of libpkv.so: argument validation, the split planner, the RoPE table, TMA
// descriptors and kernel launches.  Every entry point of include/pkv.h is defined here.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "../../include/pkv.h"
#include "pkv_internal.h"

struct pkv_cache {
  pkv_cache_desc desc;
  std::vector<void*> pools;
  std::vector<int> windows;         // per layer, 0 = full attention
  std::vector<const float*> sinks;  // per layer, device fp32 [Hq] or null
  std::vector<CUtensorMap> maps;     // one per layer pool: boxes of one page's K and V (decode)
  std::vector<CUtensorMap> maps_pf;  // one per layer pool: one page's K or V of one KV head (prefill)
  int device = 0;
  int num_sms = 0;
  int group = 1;
  bool pdl = false;
  bool int8 = false;  // PKV_OPT_INT8_KV: int8 blocks with per-slot scales
  unsigned long long wait_ns = pkv::kWaitLimitNs;  // limit of the kernels' waits for staged copies
  bool stall = false;  // test setting (pkv_set_stage_stall): decode stages never complete
  // Per layer: the pool was written by a call other than the one-launch step (an append or a QKV
  // append) since the last one-launch step of that layer.  The next one-launch step of the layer
  // then copies no page before its launch wait, since the writing kernel may still be running.
  std::vector<char> pool_dirty;
  int* prefill_work = nullptr;  // device int[2], owned: the prefill kernel's work counter
};

namespace {

using pkv::DecodeConfig;

constexpr int kEarlyStagesOneHead = 2;  // early stages per warp on the CUDA-core path
constexpr int kEarlyStagesGroup = 8;    // and on the tensor-core path (the whole ring)

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

thread_local std::string g_last_error;

void set_error(const char* what, const char* detail) {
  g_last_error = what;
  if (detail != nullptr) {
    g_last_error += ": ";
    g_last_error += detail;
  }
}

pkv_status fail(pkv_status s, const char* what, const char* detail = nullptr) {
  set_error(what, detail);
  return s;
}

pkv_status cuda_fail(const char* what, cudaError_t e) {
  set_error(what, cudaGetErrorString(e));
  return PKV_ERR_CUDA;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool head_dim_ok(int d) { return d == 64 || d == 96 || d == 128; }

pkv_status launch_status(const char* what, cudaError_t e) { return e == cudaSuccess ? PKV_OK : cuda_fail(what, e); }

// Split selection shared by pkv_plan_decode and pkv_decode_attention.
pkv_status plan(const pkv_cache* c, int batch, int max_pages, int total_pages, int num_splits, int chunk_pages,
                int max_splits, int* splits, int* chunk) {
  if (batch < 0 || max_pages < 0 || total_pages < 0 || num_splits < 0 || chunk_pages < 0 || max_splits < 1)
    return PKV_ERR_INVALID_ARG;
  if (num_splits > 0 && chunk_pages > 0) return PKV_ERR_INVALID_ARG;
  if (num_splits > 0) {
    if (num_splits > max_splits) return PKV_ERR_INVALID_ARG;
    *splits = num_splits;
    *chunk = 0;
    return PKV_OK;
  }
  if (chunk_pages > 0) {
    const int s = max_pages > 0 ? (max_pages + chunk_pages - 1) / chunk_pages : 1;
    if (s > max_splits) return PKV_ERR_INVALID_ARG;
    *splits = s;
    *chunk = chunk_pages;
    return PKV_OK;
  }
  const DecodeConfig cfg = pkv::decode_config(c->group, c->desc.head_dim, batch > 0 ? batch : 1);
  const long long warps = (long long)c->num_sms * cfg.ctas_per_sm * cfg.warps;
  // Automatic with the exact page total: the balanced partition, every warp of the grid taking an
  // equal run of (sequence, KV head, page) units; a segment of n pages meets at most
  // ceil(n * W / U) + 1 runs.
  // The bound takes the most warps any decode launch runs (the one-launch layout may run more warps
  // per CTA than the plain one; the CUDA-core layout runs 12 per SM for large batches), so one plan
  // serves every entry point.
  if (total_pages > 0) {
    const long long U = (long long)total_pages * c->desc.num_kv_heads;
    const int sm_warps = std::max(pkv::kMaxDecodeWarps, pkv::kWideWarps);
    const long long W = std::min((long long)c->num_sms * sm_warps, U);
    const long long s_bal = ((long long)max_pages * W + U - 1) / U + 1;
    if (U < 0x7fffffffLL && s_bal <= max_splits) {
      *splits = (int)s_bal;
      *chunk = -1;
      return PKV_OK;
    }
  }
  // Automatic without it: chunk size so that the items fill the resident warps once (uniform
  // lengths) or about four times (ragged lengths, where small items balance the long ones).
  const long long uniform_pages = (long long)batch * max_pages;
  const long long pages = total_pages > 0 ? total_pages : uniform_pages;
  const bool ragged = total_pages > 0 && 10 * (long long)total_pages < 9 * uniform_pages;
  const long long units = pages * c->desc.num_kv_heads;
  const long long heads = (long long)batch * c->desc.num_kv_heads;
  const long long per_head = heads > 0 ? warps / heads : 0;  // items each (sequence, KV head) may have
  long long cp;
  if (!ragged && per_head >= 1) {
    // uniform lengths: at most one item per warp, as small as that allows
    cp = std::max((units + warps - 1) / warps, ((long long)max_pages + per_head - 1) / per_head);
  } else {
    // ragged lengths or more (sequence, head) pairs than warps: about four items per warp, so that
    // small items even out the long ones under the static round-robin assignment
    cp = (units + 4 * warps - 1) / (4 * warps);
  }
  if (cp < 1) cp = 1;
  if (max_pages > 0 && cp > max_pages) cp = max_pages;
  int s = max_pages > 0 ? (int)((max_pages + cp - 1) / cp) : 1;
  if (s > max_splits) {
    cp = (max_pages + max_splits - 1) / max_splits;
    s = (int)((max_pages + cp - 1) / cp);
  }
  *splits = s;
  *chunk = (int)cp;
  return PKV_OK;
}

// Plan of a layer with a sliding window of `window` positions: each sequence walks its visible
// pages (at most ceil(window / 16) + 1 of them).  Explicit split counts and chunk sizes apply to
// them; otherwise the page-balanced partition of the visible pages (the kernel counts them), or,
// when its split bound exceeds max_splits, chunks of about four work items per resident warp.
pkv_status plan_windowed(const pkv_cache* c, int window, int batch, int max_pages, int num_splits, int chunk_pages,
                         int max_splits, int* splits, int* chunk) {
  if (batch < 0 || max_pages < 0 || num_splits < 0 || chunk_pages < 0 || max_splits < 1) return PKV_ERR_INVALID_ARG;
  if (num_splits > 0 && chunk_pages > 0) return PKV_ERR_INVALID_ARG;
  const int max_vis = std::max(1, std::min(max_pages, (window + PKV_PAGE_SIZE - 1) / PKV_PAGE_SIZE + 1));
  if (num_splits > 0) {
    if (num_splits > max_splits) return PKV_ERR_INVALID_ARG;
    *splits = num_splits;
    *chunk = 0;
    return PKV_OK;
  }
  if (chunk_pages <= 0 && max_vis + 1 <= max_splits) {
    // the page-balanced partition over the visible pages, whose total the kernel counts itself; a
    // segment of n' visible pages meets at most n' + 1 runs
    *splits = max_vis + 1;
    *chunk = -1;
    return PKV_OK;
  }
  long long cp = chunk_pages;
  if (cp <= 0) {
    const DecodeConfig cfg = pkv::decode_config(c->group, c->desc.head_dim, batch > 0 ? batch : 1);
    const long long warps = (long long)c->num_sms * cfg.ctas_per_sm * cfg.warps;
    const long long units = (long long)std::max(batch, 1) * c->desc.num_kv_heads * max_vis;
    cp = std::max(1LL, (units + 4 * warps - 1) / (4 * warps));
    if ((max_vis + cp - 1) / cp > max_splits) cp = (max_vis + max_splits - 1) / max_splits;
  }
  const long long s = (max_vis + cp - 1) / cp;
  if (s > max_splits) return PKV_ERR_INVALID_ARG;
  *splits = (int)s;
  *chunk = (int)cp;
  return PKV_OK;
}

// The plan of one layer (sliding window or not).
pkv_status plan_layer(const pkv_cache* c, int layer, int batch, int max_pages, int total_pages, int num_splits,
                      int chunk_pages, int max_splits, int* splits, int* chunk) {
  const int window = c->windows[layer];
  if (window > 0) return plan_windowed(c, window, batch, max_pages, num_splits, chunk_pages, max_splits, splits, chunk);
  return plan(c, batch, max_pages, total_pages, num_splits, chunk_pages, max_splits, splits, chunk);
}

}  // namespace

namespace pkv {

void cache_geometry(const pkv_cache* c, int* hq, int* hkv, int* d) {
  *hq = c->desc.num_qo_heads;
  *hkv = c->desc.num_kv_heads;
  *d = c->desc.head_dim;
}

int cache_device(const pkv_cache* c) { return c->device; }

void set_last_error(const char* what) { ::set_error(what, nullptr); }

}  // namespace pkv

extern "C" {

size_t pkv_pool_bytes(int num_pages, int num_kv_heads, int head_dim) {
  if (num_pages <= 0 || num_kv_heads <= 0 || head_dim <= 0) return 0;
  return (size_t)num_pages * 2 * num_kv_heads * PKV_PAGE_SIZE * head_dim * 2;
}

size_t pkv_pool_bytes_int8(int num_pages, int num_kv_heads, int head_dim) {
  if (num_pages <= 0 || num_kv_heads <= 0 || head_dim <= 0) return 0;
  return (size_t)num_pages * 2 * num_kv_heads * pkv::int8_block_bytes(head_dim);
}

size_t pkv_rope_table_bytes(int max_position, int head_dim) {
  if (max_position <= 0 || head_dim <= 0 || head_dim % 2) return 0;
  return (size_t)max_position * (head_dim / 2) * 2 * sizeof(float);
}

size_t pkv_partial_bytes(int batch, int num_qo_heads, int splits, int head_dim) {
  if (batch < 0 || num_qo_heads <= 0 || splits <= 0 || head_dim <= 0) return 0;
  return (size_t)batch * num_qo_heads * splits * head_dim * sizeof(float);
}

const char* pkv_last_error(void) { return g_last_error.c_str(); }

const char* pkv_status_string(pkv_status s) {
  switch (s) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID_ARG: return "invalid argument";
    case PKV_ERR_UNSUPPORTED: return "unsupported shape";
    case PKV_ERR_OUT_OF_RANGE: return "index out of range (device)";
    case PKV_ERR_CUDA: return "CUDA error";
    case PKV_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

pkv_status pkv_create_cache(const pkv_cache_desc* d, pkv_cache** out) {
  if (d == nullptr || out == nullptr) return PKV_ERR_INVALID_ARG;
  if (d->num_layers < 1 || d->num_pages < 1 || d->num_qo_heads < 1 || d->num_kv_heads < 1 ||
      d->max_position < 1 || !(d->rope_theta > 0.0) || d->layer_pools == nullptr || d->rope_table == nullptr ||
      d->status_word == nullptr)
    return PKV_ERR_INVALID_ARG;
  if (d->page_size != PKV_PAGE_SIZE || !head_dim_ok(d->head_dim)) return PKV_ERR_UNSUPPORTED;
  if (d->num_qo_heads % d->num_kv_heads) return PKV_ERR_INVALID_ARG;
  const int group = d->num_qo_heads / d->num_kv_heads;
  if (group > pkv::kMaxGroup) return PKV_ERR_UNSUPPORTED;
  if ((long long)d->num_pages * 2 > 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;
  if (!aligned(d->rope_table, 16)) return PKV_ERR_INVALID_ARG;
  for (int l = 0; l < d->num_layers; ++l)
    if (d->layer_pools[l] == nullptr || !aligned(d->layer_pools[l], 256)) return PKV_ERR_INVALID_ARG;
  if (d->options & ~(PKV_OPT_PDL | PKV_OPT_EARLY_PAGES | PKV_OPT_INT8_KV)) return PKV_ERR_INVALID_ARG;
  for (int l = 0; l < d->num_layers; ++l) {
    if (d->layer_window != nullptr && d->layer_window[l] < 0) return PKV_ERR_INVALID_ARG;
    if (d->layer_sinks != nullptr && d->layer_sinks[l] != nullptr && !aligned(d->layer_sinks[l], 4))
      return PKV_ERR_INVALID_ARG;
  }

  EncodeTiledFn encode = encode_tiled_fn();
  if (encode == nullptr) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");

  pkv_cache* c = new (std::nothrow) pkv_cache();
  if (c == nullptr) return fail(PKV_ERR_CUDA, "out of host memory");
  c->desc = *d;
  c->pools.assign(d->layer_pools, d->layer_pools + d->num_layers);
  c->desc.layer_pools = nullptr;
  c->windows.assign(d->num_layers, 0);
  c->sinks.assign(d->num_layers, nullptr);
  c->pool_dirty.assign(d->num_layers, 0);
  for (int l = 0; l < d->num_layers; ++l) {
    if (d->layer_window != nullptr) c->windows[l] = d->layer_window[l];
    if (d->layer_sinks != nullptr) c->sinks[l] = d->layer_sinks[l];
  }
  c->desc.layer_window = nullptr;
  c->desc.layer_sinks = nullptr;
  c->group = group;
  c->pdl = (d->options & PKV_OPT_PDL) != 0;
  c->int8 = (d->options & PKV_OPT_INT8_KV) != 0;
  cudaError_t e = cudaGetDevice(&c->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device);
  if (e != cudaSuccess) {
    delete c;
    return cuda_fail("querying the device", e);
  }

  // RoPE table: cos/sin(p * theta^(-2i/d)) in fp64, rounded once to fp32, interleaved (cos, sin).
  const int D = d->head_dim, half = D / 2;
  std::vector<double> inv_freq(half);
  for (int i = 0; i < half; ++i) inv_freq[i] = std::pow(d->rope_theta, -2.0 * i / D);
  std::vector<float> table((size_t)d->max_position * half * 2);
  for (int p = 0; p < d->max_position; ++p) {
    for (int i = 0; i < half; ++i) {
      const double phi = (double)p * inv_freq[i];
      table[((size_t)p * half + i) * 2] = (float)std::cos(phi);
      table[((size_t)p * half + i) * 2 + 1] = (float)std::sin(phi);
    }
  }
  e = cudaMemcpy(d->rope_table, table.data(), table.size() * sizeof(float), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemset(d->status_word, 0, sizeof(int));
  if (e == cudaSuccess) e = cudaMalloc(&c->prefill_work, 2 * sizeof(int));
  if (e == cudaSuccess) e = cudaMemset(c->prefill_work, 0, 2 * sizeof(int));
  if (e != cudaSuccess) {
    pkv_destroy(c);
    return cuda_fail("writing the RoPE table / status word", e);
  }

  // One 4-D tensor map per pool: dims (head_dim, slot, kv_head, page*2 + kv).
  const DecodeConfig cfg = pkv::decode_config(group, D, 1);
  e = pkv::decode_prepare(cfg, D);
  if (e == cudaSuccess) e = pkv::decode_prepare(pkv::decode_config(group, D, 1, true), D);
  if (e == cudaSuccess && c->int8) e = pkv::decode_prepare(pkv::decode_config(group, D, 1, false, false, true), D);
  if (e == cudaSuccess) e = pkv::qkv_prepare();
  if (e == cudaSuccess) e = pkv::prefill_prepare();
  if (e == cudaSuccess) e = pkv::append_prepare();
  if (e == cudaSuccess) e = pkv::combine_prepare();
  if (e != cudaSuccess) {
    pkv_destroy(c);
    return cuda_fail("setting kernel attributes", e);
  }
  c->maps.resize(d->num_layers);
  c->maps_pf.resize(d->num_layers);
  if (c->int8) {  // int8 pages use plain copies
    memset(c->maps.data(), 0, sizeof(CUtensorMap) * c->maps.size());
    memset(c->maps_pf.data(), 0, sizeof(CUtensorMap) * c->maps_pf.size());
  }
  for (int l = 0; l < d->num_layers && !c->int8; ++l) {
    const cuuint64_t gdim[4] = {(cuuint64_t)D, (cuuint64_t)PKV_PAGE_SIZE, (cuuint64_t)d->num_kv_heads,
                                (cuuint64_t)d->num_pages * 2};
    const cuuint64_t gstride[3] = {(cuuint64_t)D * 2, (cuuint64_t)PKV_PAGE_SIZE * D * 2,
                                   (cuuint64_t)d->num_kv_heads * PKV_PAGE_SIZE * D * 2};
    const cuuint32_t box[4] = {(cuuint32_t)cfg.box_inner, (cuuint32_t)PKV_PAGE_SIZE, 1, 2};
    const cuuint32_t estride[4] = {1, 1, 1, 1};
    const CUtensorMapSwizzle swz = cfg.swizzle_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                                   : cfg.swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                             : CU_TENSOR_MAP_SWIZZLE_NONE;
    CUresult r = encode(&c->maps[l], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, c->pools[l], gdim, gstride, box, estride,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    // The prefill kernel copies a page's K (or V) of one KV head in one box, landing as
    // [half page][swizzle atom][8 slots][one swizzle row]: the dimensions, innermost first, are the
    // elements of an atom, the slot within a half page, the atom, the half page, and (page, K or V,
    // KV head) together.
    const int E = cfg.box_inner, NA = D / E;
    const cuuint64_t gdim5[5] = {(cuuint64_t)E, 8, (cuuint64_t)NA, 2,
                                 (cuuint64_t)d->num_pages * 2 * (cuuint64_t)d->num_kv_heads};
    const cuuint64_t gstride5[4] = {(cuuint64_t)D * 2, (cuuint64_t)E * 2, (cuuint64_t)8 * D * 2,
                                    (cuuint64_t)PKV_PAGE_SIZE * D * 2};
    const cuuint32_t box5[5] = {(cuuint32_t)E, 8, (cuuint32_t)NA, 2, 1};
    const cuuint32_t estride5[5] = {1, 1, 1, 1, 1};
    if (r == CUDA_SUCCESS)
      r = encode(&c->maps_pf[l], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 5, c->pools[l], gdim5, gstride5, box5, estride5,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
      pkv_destroy(c);
      char msg[64];
      snprintf(msg, sizeof(msg), "CUresult %d for layer %d", (int)r, l);
      return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled", msg);
    }
  }
  *out = c;
  return PKV_OK;
}

void pkv_destroy(pkv_cache* c) {
  if (c == nullptr) return;
  if (c->prefill_work != nullptr) {
    int cur = 0;
    const bool restore = cudaGetDevice(&cur) == cudaSuccess && cur != c->device;
    if (restore) cudaSetDevice(c->device);
    cudaFree(c->prefill_work);
    if (restore) cudaSetDevice(cur);
  }
  delete c;
}

pkv_status pkv_device_info(const pkv_cache* c, int batch, int* num_sms, int* decode_warps_per_sm) {
  if (c == nullptr || batch < 1) return PKV_ERR_INVALID_ARG;
  if (num_sms) *num_sms = c->num_sms;
  if (decode_warps_per_sm) {
    const DecodeConfig cfg = pkv::decode_config(c->group, c->desc.head_dim, batch, false, false, c->int8);
    *decode_warps_per_sm = cfg.warps * cfg.ctas_per_sm;
  }
  return PKV_OK;
}

pkv_status pkv_append_rope(pkv_cache* c, int layer, const void* q, const void* k, const void* v,
                           const int32_t* pos_map, const int32_t* append_indptr, int num_tokens, int batch,
                           const int32_t* page_indptr, const int32_t* page_indices, void* q_out,
                           pkv_stream_t stream) {
  if (c == nullptr || layer < 0 || layer >= c->desc.num_layers || num_tokens < 0 || batch < 0)
    return PKV_ERR_INVALID_ARG;
  if (num_tokens == 0 || batch == 0) return PKV_OK;
  if (q == nullptr || k == nullptr || v == nullptr || pos_map == nullptr || append_indptr == nullptr ||
      page_indptr == nullptr || page_indices == nullptr || q_out == nullptr)
    return PKV_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(q_out, 16) || q_out == q)
    return PKV_ERR_INVALID_ARG;
  pkv::AppendParams p;
  p.q = static_cast<const __half*>(q);
  p.k = static_cast<const __half*>(k);
  p.v = static_cast<const __half*>(v);
  p.pos_map = pos_map;
  p.append_indptr = append_indptr;
  p.page_indptr = page_indptr;
  p.page_indices = page_indices;
  p.q_out = static_cast<__half*>(q_out);
  p.pool = static_cast<__half*>(c->pools[layer]);
  p.rope = reinterpret_cast<const float2*>(c->desc.rope_table);
  p.status = c->desc.status_word;
  p.num_tokens = num_tokens;
  p.batch = batch;
  p.hq = c->desc.num_qo_heads;
  p.hkv = c->desc.num_kv_heads;
  p.head_dim = c->desc.head_dim;
  p.max_position = c->desc.max_position;
  p.num_pages = c->desc.num_pages;
  if (c->int8) {
    p.pool = nullptr;
    p.pool8 = static_cast<unsigned char*>(c->pools[layer]);
    const pkv_status st = launch_status("append_rope launch", pkv::launch_append_q8(p, stream, c->pdl));
    if (st == PKV_OK) c->pool_dirty[layer] = 1;
    return st;
  }
  p.pool8 = nullptr;
  const pkv_status st = launch_status("append_rope launch", pkv::launch_append(p, stream, c->pdl));
  if (st == PKV_OK) c->pool_dirty[layer] = 1;
  return st;
}

namespace {

// Shared checks and parameters of the QKV entry points.
pkv_status qkv_params(const pkv_cache* c, const void* x, const uint32_t* w, const void* scales, int hidden,
                      int num_tokens, pkv::QkvParams* p) {
  if (c == nullptr || num_tokens < 0) return fail(PKV_ERR_INVALID_ARG, "null cache or negative num_tokens");
  if (hidden <= 0 || hidden % 32 || hidden > pkv::kQkvMaxHidden)
    return fail(PKV_ERR_UNSUPPORTED, "hidden must be a positive multiple of 32, at most 4096");
  if (num_tokens > 0 && (x == nullptr || w == nullptr || scales == nullptr))
    return fail(PKV_ERR_INVALID_ARG, "null pointer");
  if (!aligned(x, 16) || !aligned(w, 16) || !aligned(scales, 2)) return fail(PKV_ERR_INVALID_ARG, "misaligned pointer");
  *p = pkv::QkvParams{};
  p->x = static_cast<const __half*>(x);
  p->w = w;
  p->scales = static_cast<const __half*>(scales);
  p->num_tokens = num_tokens;
  p->hidden = hidden;
  p->hq = c->desc.num_qo_heads;
  p->hkv = c->desc.num_kv_heads;
  p->head_dim = c->desc.head_dim;
  p->max_position = c->desc.max_position;
  p->num_pages = c->desc.num_pages;
  p->rope = reinterpret_cast<const float2*>(c->desc.rope_table);
  p->status = c->desc.status_word;
  return PKV_OK;
}

}  // namespace

pkv_status pkv_qkv_append_rope(pkv_cache* c, int layer, const void* x, const uint32_t* w, const void* scales,
                               int hidden, const int32_t* pos_map, const int32_t* append_indptr, int num_tokens,
                               int batch, const int32_t* page_indptr, const int32_t* page_indices, void* q_out,
                               pkv_stream_t stream) {
  pkv::QkvParams p;
  const pkv_status st = qkv_params(c, x, w, scales, hidden, num_tokens, &p);
  if (st != PKV_OK) return st;
  if (layer < 0 || layer >= c->desc.num_layers || batch < 0) return fail(PKV_ERR_INVALID_ARG, "layer or batch");
  if (c->int8) return fail(PKV_ERR_UNSUPPORTED, "int8 cache: use pkv_qkv_project and pkv_append_rope");
  if (num_tokens == 0 || batch == 0) return PKV_OK;
  if (pos_map == nullptr || append_indptr == nullptr || page_indptr == nullptr || page_indices == nullptr ||
      q_out == nullptr)
    return fail(PKV_ERR_INVALID_ARG, "null pointer");
  if (!aligned(q_out, 16)) return fail(PKV_ERR_INVALID_ARG, "misaligned q_out");
  p.pos_map = pos_map;
  p.append_indptr = append_indptr;
  p.page_indptr = page_indptr;
  p.page_indices = page_indices;
  p.batch = batch;
  p.q_out = static_cast<__half*>(q_out);
  p.pool = static_cast<__half*>(c->pools[layer]);
  const pkv_status ls = launch_status("qkv launch", pkv::launch_qkv(p, stream, c->pdl));
  if (ls == PKV_OK) c->pool_dirty[layer] = 1;
  return ls;
}

pkv_status pkv_qkv_project(const pkv_cache* c, const void* x, const uint32_t* w, const void* scales, int hidden,
                           int num_tokens, void* y, pkv_stream_t stream) {
  pkv::QkvParams p;
  const pkv_status st = qkv_params(c, x, w, scales, hidden, num_tokens, &p);
  if (st != PKV_OK) return st;
  if (num_tokens == 0) return PKV_OK;
  if (y == nullptr || !aligned(y, 16)) return fail(PKV_ERR_INVALID_ARG, "null or misaligned y");
  p.y_out = static_cast<__half*>(y);
  return launch_status("qkv launch", pkv::launch_qkv(p, stream, c->pdl));
}

pkv_status pkv_prefill_attention(const pkv_cache* c, int layer, const void* q_rope, const int32_t* append_indptr,
                                 const int32_t* pos_map, int num_tokens, const int32_t* page_indptr,
                                 const int32_t* page_indices, const int32_t* last_page_len, int batch,
                                 float sm_scale, void* out, float* lse_out, pkv_stream_t stream) {
  if (c == nullptr || layer < 0 || layer >= c->desc.num_layers || num_tokens < 0 || batch < 0)
    return fail(PKV_ERR_INVALID_ARG, "cache, layer or sizes");
  if (c->int8) return fail(PKV_ERR_UNSUPPORTED, "int8 cache: prefill attention reads fp16 pages");
  if (num_tokens == 0 || batch == 0) return PKV_OK;
  if (batch > pkv::kMaxDecodeBatch) return fail(PKV_ERR_UNSUPPORTED, "batch above 4096 sequences");
  if (q_rope == nullptr || append_indptr == nullptr || pos_map == nullptr || page_indptr == nullptr ||
      page_indices == nullptr || last_page_len == nullptr || out == nullptr)
    return fail(PKV_ERR_INVALID_ARG, "null pointer");
  if (!aligned(q_rope, 16) || !aligned(out, 16)) return fail(PKV_ERR_INVALID_ARG, "misaligned pointer");
  if (!(sm_scale >= 0.f) || std::isinf(sm_scale)) return fail(PKV_ERR_INVALID_ARG, "sm_scale");
  const int D = c->desc.head_dim;
  const pkv::PrefillConfig cfg = pkv::prefill_config(D, batch);
  if (cfg.nstage < 2) return fail(PKV_ERR_UNSUPPORTED, "shared memory too small for this batch");
  pkv::PrefillParams p{};
  p.q = static_cast<const __half*>(q_rope);
  p.append_indptr = append_indptr;
  p.pos_map = pos_map;
  p.page_indptr = page_indptr;
  p.page_indices = page_indices;
  p.last_page_len = last_page_len;
  p.out = static_cast<__half*>(out);
  p.lse = lse_out;
  p.status = c->desc.status_word;
  p.sinks = c->sinks[layer];
  p.batch = batch;
  p.num_tokens = num_tokens;
  p.hq = c->desc.num_qo_heads;
  p.hkv = c->desc.num_kv_heads;
  p.group = c->group;
  p.num_pages = c->desc.num_pages;
  p.window = c->windows[layer];
  p.nstage = cfg.nstage;
  const float scale = sm_scale > 0.f ? sm_scale : (float)(1.0 / std::sqrt((double)D));
  p.scale_log2 = (float)((double)scale * 1.4426950408889634);
  p.work = c->prefill_work;
  p.wait_ns = c->wait_ns;
  const int grid = c->num_sms;
  return launch_status("prefill launch", pkv::launch_prefill(p, c->maps_pf[layer], cfg, D, grid, stream, c->pdl));
}

pkv_status pkv_plan_decode(const pkv_cache* c, int batch, int max_pages, int total_pages, int num_splits,
                           int chunk_pages, int max_splits, int* splits, int* chunk_out) {
  if (c == nullptr || splits == nullptr || chunk_out == nullptr) return PKV_ERR_INVALID_ARG;
  const pkv_status st = plan(c, batch, max_pages, total_pages, num_splits, chunk_pages, max_splits, splits, chunk_out);
  if (st != PKV_OK) return st;
  // the split count is the most any layer produces (windowed layers plan their own chunks)
  for (int l = 0; l < c->desc.num_layers; ++l) {
    if (c->windows[l] <= 0) continue;
    int s = 0, ch = 0;
    const pkv_status sw = plan_windowed(c, c->windows[l], batch, max_pages, num_splits, chunk_pages, max_splits, &s, &ch);
    if (sw != PKV_OK) return sw;
    *splits = std::max(*splits, s);
  }
  return PKV_OK;
}

}  // extern "C"

namespace {

// The append inputs of the fused entry point.
struct FusedArgs {
  const void* k;
  const void* v;
  const int32_t* pos_map;
  void* q_out;
  bool early_ok;  // no other call wrote the layer's pool since its last one-launch step
};

// Shared body of pkv_decode_attention, pkv_decode_attention_merged and pkv_append_decode_attention.
pkv_status decode_common(const pkv_cache* c, int layer, const void* q_rope, const int32_t* q_indptr,
                         const int32_t* page_indptr, const int32_t* page_indices, const int32_t* last_page_len,
                         int batch, int max_pages, int total_pages, int num_splits, int chunk_pages, int max_splits,
                         float sm_scale, float* partial_o, float* partial_lse, int32_t* counters, void* out,
                         float* lse_out, bool merged, int* splits_used, cudaStream_t stream,
                         const FusedArgs* fused = nullptr) {
  if (c == nullptr || layer < 0 || layer >= c->desc.num_layers) return fail(PKV_ERR_INVALID_ARG, "cache or layer");
  int S = 0, chunk = 0;
  const pkv_status ps =
      plan_layer(c, layer, batch, max_pages, total_pages, num_splits, chunk_pages, max_splits, &S, &chunk);
  if (ps != PKV_OK) return fail(ps, "split plan arguments");
  const int window = c->windows[layer];
  if (splits_used) *splits_used = S;
  if (batch == 0) return PKV_OK;
  if (batch > pkv::kMaxDecodeBatch) return fail(PKV_ERR_UNSUPPORTED, "batch above 4096 sequences");
  if (q_rope == nullptr || page_indptr == nullptr || page_indices == nullptr || last_page_len == nullptr ||
      partial_o == nullptr || partial_lse == nullptr)
    return fail(PKV_ERR_INVALID_ARG, "null pointer");
  if (merged && (counters == nullptr || out == nullptr)) return fail(PKV_ERR_INVALID_ARG, "null pointer");
  if (!aligned(q_rope, 16) || !aligned(partial_o, 16) || !aligned(partial_lse, 4) ||
      (merged && (!aligned(out, 16) || !aligned(counters, 4))))
    return fail(PKV_ERR_INVALID_ARG, "misaligned pointer");
  if (!(sm_scale >= 0.f) || std::isinf(sm_scale)) return fail(PKV_ERR_INVALID_ARG, "sm_scale");
  const long long items = (long long)batch * c->desc.num_kv_heads * S;
  if (items > 0x3fffffffLL) return fail(PKV_ERR_UNSUPPORTED, "too many work items");

  if (fused != nullptr &&
      (fused->k == nullptr || fused->v == nullptr || fused->pos_map == nullptr || fused->q_out == nullptr ||
       q_indptr == nullptr))
    return fail(PKV_ERR_INVALID_ARG, "null pointer");
  if (fused != nullptr && (!aligned(fused->k, 16) || !aligned(fused->v, 16) || !aligned(fused->q_out, 16) ||
                           fused->q_out == q_rope))
    return fail(PKV_ERR_INVALID_ARG, "misaligned or aliased q/k/v/q_out");
  const int D = c->desc.head_dim;
  if (c->int8 && fused != nullptr) return fail(PKV_ERR_UNSUPPORTED, "int8 cache: one-launch layout");
  const DecodeConfig cfg = pkv::decode_config(c->group, D, batch, fused != nullptr, window > 0, c->int8);
  if (cfg.nstage < 2) return fail(PKV_ERR_UNSUPPORTED, "shared memory too small for this batch");
  pkv::DecodeParams p;
  p.q = static_cast<const __half*>(q_rope);
  p.q_indptr = q_indptr;
  p.page_indptr = page_indptr;
  p.page_indices = page_indices;
  p.last_page_len = last_page_len;
  p.partial_o = partial_o;
  p.partial_lse = partial_lse;
  p.status = c->desc.status_word;
  p.batch = batch;
  p.hq = c->desc.num_qo_heads;
  p.hkv = c->desc.num_kv_heads;
  p.group = c->group;
  p.num_pages = c->desc.num_pages;
  p.splits = S;
  p.chunk_pages = chunk;
  p.max_pages = max_pages;
  const float scale = sm_scale > 0.f ? sm_scale : (float)(1.0 / std::sqrt((double)D));
  p.scale_log2 = (float)((double)scale * 1.4426950408889634);
  p.nstage = cfg.nstage;
  p.warps = cfg.warps;
  p.merged = merged ? 1 : 0;
  p.counters = counters;
  p.out = static_cast<__half*>(out);
  p.lse_out = lse_out;
  p.balanced = chunk < 0 ? 1 : 0;
  p.units = (long long)total_pages * c->desc.num_kv_heads;
  const long long full_grid = (long long)c->num_sms * cfg.ctas_per_sm;
  long long grid = (items + cfg.warps - 1) / cfg.warps;
  if (grid > full_grid || p.balanced) grid = full_grid;
  if (grid < 1) grid = 1;
  p.part_warps = (int)std::min(grid * cfg.warps, std::max(p.units, 1LL));
  if (p.balanced) p.chunk_pages = 0;
  p.fused = fused != nullptr ? 1 : 0;
  p.k_new = fused ? static_cast<const __half*>(fused->k) : nullptr;
  p.v_new = fused ? static_cast<const __half*>(fused->v) : nullptr;
  p.pos_map = fused ? fused->pos_map : nullptr;
  p.q_out = fused ? static_cast<__half*>(fused->q_out) : nullptr;
  p.pool = static_cast<__half*>(c->pools[layer]);
  p.rope = reinterpret_cast<const float2*>(c->desc.rope_table);
  p.max_position = c->desc.max_position;
  p.window = window;
  p.sinks = c->sinks[layer];
  // Early page copies, measured: tensor-core path, the whole ring (GQA long context 6 400 -> 6 580
  // GB/s; 1 to 3 stages were slower); CUDA-core path, two stages per warp (single stream 3 230 ->
  // 3 510 GB/s; one stage 3 390, three 3 435, the whole ring 3 125, where the early copies slow the
  // previous launch's merge tail).
  p.early = 0;
  if (fused != nullptr && fused->early_ok && (c->desc.options & PKV_OPT_EARLY_PAGES))
    p.early = c->group >= 2 ? kEarlyStagesGroup : kEarlyStagesOneHead;
  p.wait_ns = c->wait_ns;
  p.stall = c->stall ? 1 : 0;
  p.pool8 = c->int8 ? static_cast<const unsigned char*>(c->pools[layer]) : nullptr;
  if (c->int8) p.pool = nullptr;
  return launch_status("decode launch", pkv::launch_decode(p, c->maps[layer], cfg, D, (int)grid, stream, c->pdl));
}

}  // namespace

extern "C" {

pkv_status pkv_decode_attention(const pkv_cache* c, int layer, const void* q_rope, const int32_t* q_indptr,
                                const int32_t* page_indptr, const int32_t* page_indices,
                                const int32_t* last_page_len, int batch, int max_pages, int total_pages,
                                int num_splits, int chunk_pages, int max_splits, float sm_scale, float* partial_o,
                                float* partial_lse, int* splits_used, pkv_stream_t stream) {
  return decode_common(c, layer, q_rope, q_indptr, page_indptr, page_indices, last_page_len, batch, max_pages,
                       total_pages, num_splits, chunk_pages, max_splits, sm_scale, partial_o, partial_lse, nullptr,
                       nullptr, nullptr, false, splits_used, stream);
}

pkv_status pkv_append_decode_attention(pkv_cache* c, int layer, const void* q, const void* k, const void* v,
                                       const int32_t* pos_map, const int32_t* append_indptr, int num_tokens,
                                       const int32_t* page_indptr, const int32_t* page_indices,
                                       const int32_t* last_page_len, int batch, int max_pages, int total_pages,
                                       int num_splits, int chunk_pages, int max_splits, float sm_scale, void* q_out,
                                       float* partial_o, float* partial_lse, int32_t* chunk_counters, void* out,
                                       float* lse_out, int* splits_used, pkv_stream_t stream) {
  if (c == nullptr || layer < 0 || layer >= c->desc.num_layers) return fail(PKV_ERR_INVALID_ARG, "cache or layer");
  if (num_tokens < 0) return fail(PKV_ERR_INVALID_ARG, "negative num_tokens");
  if (num_tokens != batch || c->int8) {
    // several new tokens per sequence (a chunked append), or an int8 cache: the append launch, then
    // the merged decode
    const pkv_status st = pkv_append_rope(c, layer, q, k, v, pos_map, append_indptr, num_tokens, batch,
                                          page_indptr, page_indices, q_out, stream);
    if (st != PKV_OK) return st;
    return decode_common(c, layer, q_out, append_indptr, page_indptr, page_indices, last_page_len, batch,
                         max_pages, total_pages, num_splits, chunk_pages, max_splits, sm_scale, partial_o,
                         partial_lse, chunk_counters, out, lse_out, true, splits_used, stream);
  }
  const FusedArgs fa{k, v, pos_map, q_out, c->pool_dirty[layer] == 0};
  const pkv_status st = decode_common(c, layer, q, append_indptr, page_indptr, page_indices, last_page_len, batch,
                                      max_pages, total_pages, num_splits, chunk_pages, max_splits, sm_scale, partial_o,
                                      partial_lse, chunk_counters, out, lse_out, true, splits_used, stream, &fa);
  if (st == PKV_OK) c->pool_dirty[layer] = 0;
  return st;
}

pkv_status pkv_decode_attention_merged(const pkv_cache* c, int layer, const void* q_rope, const int32_t* q_indptr,
                                       const int32_t* page_indptr, const int32_t* page_indices,
                                       const int32_t* last_page_len, int batch, int max_pages, int total_pages,
                                       int num_splits, int chunk_pages, int max_splits, float sm_scale,
                                       float* partial_o, float* partial_lse, int32_t* chunk_counters, void* out,
                                       float* lse_out, int* splits_used, pkv_stream_t stream) {
  return decode_common(c, layer, q_rope, q_indptr, page_indptr, page_indices, last_page_len, batch, max_pages,
                       total_pages, num_splits, chunk_pages, max_splits, sm_scale, partial_o, partial_lse,
                       chunk_counters, out, lse_out, true, splits_used, stream);
}

pkv_status pkv_combine(const pkv_cache* c, const float* partial_o, const float* partial_lse, const float* sinks,
                       int batch, int num_qo_heads, int num_splits, int head_dim, void* out, float* lse_out,
                       pkv_stream_t stream) {
  if (batch < 0 || num_qo_heads < 1 || num_splits < 1) return PKV_ERR_INVALID_ARG;
  if (!head_dim_ok(head_dim)) return PKV_ERR_UNSUPPORTED;
  if (batch == 0) return PKV_OK;
  if (partial_o == nullptr || partial_lse == nullptr || out == nullptr) return PKV_ERR_INVALID_ARG;
  if (!aligned(partial_o, 16) || !aligned(out, 16)) return PKV_ERR_INVALID_ARG;
  pkv::CombineParams p;
  p.partial_o = partial_o;
  p.partial_lse = partial_lse;
  p.out = static_cast<__half*>(out);
  p.lse = lse_out;
  p.sinks = sinks;
  p.batch = batch;
  p.hq = num_qo_heads;
  p.splits = num_splits;
  p.head_dim = head_dim;
  return launch_status("combine launch", pkv::launch_combine(p, stream, c != nullptr && c->pdl));
}

pkv_status pkv_set_wait_limit(pkv_cache* c, unsigned long long limit_ns) {
  if (c == nullptr) return fail(PKV_ERR_INVALID_ARG, "null cache");
  c->wait_ns = limit_ns == 0 ? pkv::kWaitLimitNs : limit_ns;
  return PKV_OK;
}

pkv_status pkv_set_stage_stall(pkv_cache* c, int on) {
  if (c == nullptr) return fail(PKV_ERR_INVALID_ARG, "null cache");
  c->stall = on != 0;
  return PKV_OK;
}

pkv_status pkv_check_status(pkv_cache* c, pkv_stream_t stream, int* flags) {
  if (c == nullptr) return PKV_ERR_INVALID_ARG;
  int v = 0;
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail("synchronising the stream", e);
  e = cudaMemcpy(&v, c->desc.status_word, sizeof(int), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && v != 0) e = cudaMemset(c->desc.status_word, 0, sizeof(int));
  if (e != cudaSuccess) return cuda_fail("reading the status word", e);
  if (flags) *flags = v;
  if (v == 0) return PKV_OK;
  return (v & PKV_FLAG_TIMEOUT) ? PKV_ERR_TIMEOUT : PKV_ERR_OUT_OF_RANGE;
}

}  // extern "C"
