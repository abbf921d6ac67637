// Allocation-free variant of the merged decode (pkv_decode_attention_noalloc).
//
// Some callers cannot allocate device memory on the path that runs attention: a framework that
// reserved the whole device for its own allocator up front, or a serving loop that must not risk an
// allocation failure or the implicit device synchronisation an allocation can cause mid-step.
// For them this entry point takes only inputs and outputs and keeps the merged decode's scratch
// (chunk counters, partial outputs and their LSEs) in one file-scope device array of
// kNoAllocScratchBytes, which every GPU that loads the library holds until the process exits.
//
// The array's device address is looked up once per device, on the first call made with that
// device current (cudaGetSymbolAddress; its return code is checked), and passed to the kernel as
// ordinary pointers.  That first call on a device should come before any stream capture.  The
// address belongs to the device's context: after a device reset (cudaDeviceReset) the next call
// finds a new context and looks the address up again (a cache created before the reset is itself
// no longer usable: its pools and tables were freed with the old context).  Every call shares the
// one array and it keeps the last call's contents: each call clears the chunk counters on its
// stream before the kernel runs, and calls that overlap on the GPU race on the array.
#include <mutex>

#include "../../include/pkv.h"
#include "pkv_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB per device
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_address[kMaxDevices] = {};
unsigned long long g_scratch_context[kMaxDevices] = {};  // context id the address belongs to

size_t round_up(size_t x) { return (x + 255) & ~size_t(255); }

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Unique id of the current context (0 if the driver cannot tell): a device reset creates a new one.
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static bool looked_up = false;
  if (!looked_up) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
    looked_up = true;
  }
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current == nullptr || get_id == nullptr || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
      get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of the scratch array on the current device, looked up on first use (and again
// when the device's context changed).
pkv_status scratch_address(int dev, void** out) {
  if (dev < 0 || dev >= kMaxDevices) {
    pkv::set_last_error("pkv_decode_attention_noalloc: device ordinal above 63");
    return PKV_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  // the runtime makes the device's primary context current on its first call; the symbol lookup
  // below is such a call, so the context id is taken after it
  if (g_scratch_address[dev] != nullptr && g_scratch_context[dev] != 0 &&
      g_scratch_context[dev] == current_context_id()) {
    *out = g_scratch_address[dev];
    return PKV_OK;
  }
  void* ptr = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
  if (e != cudaSuccess || ptr == nullptr) {
    pkv::set_last_error("pkv_decode_attention_noalloc: cudaGetSymbolAddress of the scratch array failed");
    return PKV_ERR_CUDA;
  }
  g_scratch_address[dev] = ptr;
  g_scratch_context[dev] = current_context_id();
  *out = ptr;
  return PKV_OK;
}

}  // namespace

extern "C" pkv_status pkv_decode_attention_noalloc(const pkv_cache* cache, int layer, const void* q_rope,
                                                   const int32_t* q_indptr, const int32_t* page_indptr,
                                                   const int32_t* page_indices, const int32_t* last_page_len,
                                                   int batch, int max_pages_per_seq, int total_pages,
                                                   int num_splits, int chunk_pages, float sm_scale, void* out,
                                                   float* lse_out, int* splits_used, pkv_stream_t stream) {
  if (cache == nullptr || batch < 0) {
    pkv::set_last_error("pkv_decode_attention_noalloc: null cache or negative batch");
    return PKV_ERR_INVALID_ARG;
  }
  int hq = 0, hkv = 0, d = 0;
  pkv::cache_geometry(cache, &hq, &hkv, &d);
  int S = 0, chunk = 0;
  const pkv_status ps = pkv_plan_decode(cache, batch, max_pages_per_seq, total_pages, num_splits, chunk_pages,
                                        1 << 16, &S, &chunk);
  if (ps != PKV_OK) return ps;
  const size_t counter_bytes = round_up((size_t)batch * hkv * sizeof(int32_t));
  const size_t lse_bytes = round_up((size_t)batch * hq * S * sizeof(float));
  const size_t o_bytes = (size_t)batch * hq * S * d * sizeof(float);
  if (counter_bytes + lse_bytes + o_bytes > kNoAllocScratchBytes) {
    pkv::set_last_error(
        "pkv_decode_attention_noalloc: batch * num_qo_heads * splits * (head_dim + 1) * 4 bytes plus "
        "the chunk counters exceed the 32 MiB scratch array; use pkv_decode_attention_merged with "
        "caller-allocated workspace");
    return PKV_ERR_UNSUPPORTED;
  }
  if (batch == 0) {
    if (splits_used) *splits_used = S;
    return PKV_OK;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    pkv::set_last_error("pkv_decode_attention_noalloc: cudaGetDevice failed");
    return PKV_ERR_CUDA;
  }
  if (dev != pkv::cache_device(cache)) {
    pkv::set_last_error("pkv_decode_attention_noalloc: the current device is not the cache's device");
    return PKV_ERR_INVALID_ARG;
  }
  void* base = nullptr;
  const pkv_status as = scratch_address(dev, &base);
  if (as != PKV_OK) return as;
  unsigned char* scratch = static_cast<unsigned char*>(base);
  int32_t* counters = reinterpret_cast<int32_t*>(scratch);
  float* partial_lse = reinterpret_cast<float*>(scratch + counter_bytes);
  float* partial_o = reinterpret_cast<float*>(scratch + counter_bytes + lse_bytes);
  // the counters must start at zero; clear them on the caller's stream (no allocation)
  if (cudaMemsetAsync(counters, 0, counter_bytes, stream) != cudaSuccess) {
    pkv::set_last_error("pkv_decode_attention_noalloc: clearing the chunk counters failed");
    return PKV_ERR_CUDA;
  }
  return pkv_decode_attention_merged(cache, layer, q_rope, q_indptr, page_indptr, page_indices, last_page_len,
                                     batch, max_pages_per_seq, total_pages, num_splits, chunk_pages, S, sm_scale,
                                     partial_o, partial_lse, counters, out, lse_out, splits_used, stream);
}
