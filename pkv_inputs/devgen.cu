// Seeded synthetic inputs, device side: the twin of hostgen.c.
//
// Shared input generation only (no attention arithmetic).  Every definition
// below matches hostgen.c bit for bit: SplitMix64 words, the Irwin-Hall
// normal, the optional x8 outlier rows, one fp32 multiply by `scale`, then
// round-to-nearest-even to fp16.  It exists so that multi-GB KV pools can be
// filled in HBM directly; a GPU test checks it against the host twin.
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace {

constexpr uint64_t kGamma = 0x9e3779b97f4a7c15ULL;

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ULL;
  z = (z ^ (z >> 27)) * 0x94d049bb133111ebULL;
  return z ^ (z >> 31);
}

__device__ __forceinline__ uint64_t word(uint64_t key, uint64_t i) { return mix64(key + (i + 1) * kGamma); }

__device__ __forceinline__ uint16_t value_bits(uint64_t key, uint64_t i, float scale, uint64_t okey,
                                               uint64_t row_len, int pct) {
  int32_t sum = 0;
#pragma unroll
  for (int w = 0; w < 3; ++w) {
    uint64_t u = word(key, 3 * i + (uint64_t)w);
    sum += (int32_t)(u & 0xffff) + (int32_t)((u >> 16) & 0xffff) + (int32_t)((u >> 32) & 0xffff) +
           (int32_t)(u >> 48);
  }
  float f = __fmul_rn((float)(sum - 393210), 1.0f / 65536.0f);
  if (pct > 0 && (word(okey, i / row_len) % 100u) < (uint64_t)pct) f = __fmul_rn(f, 8.0f);
  __half h = __float2half_rn(__fmul_rn(f, scale));
  return __half_as_ushort(h);
}

__global__ void fill_range_kernel(uint16_t* __restrict__ dst, int64_t n, uint64_t key, int64_t first,
                                  float scale, uint64_t okey, int64_t row_len, int pct) {
  int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < n; j += stride)
    dst[j] = value_bits(key, (uint64_t)(first + j), scale, okey, (uint64_t)row_len, pct);
}

}  // namespace

extern "C" {

// dst[j] = value(first + j) for j in [0, n); enqueued on `stream`.
// Returns the cudaError_t of the launch (0 on success).
int pkvgen_dev_fill_range(uint16_t* dst, int64_t n, uint64_t key, int64_t first, float scale,
                          uint64_t okey, int64_t row_len, int pct, cudaStream_t stream) {
  if (n <= 0) return 0;
  if (dst == nullptr || (pct > 0 && row_len <= 0)) return (int)cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t blocks = (n + 255) / 256;
  int64_t cap = (int64_t)(sms > 0 ? sms : 1) * 16;
  if (blocks > cap) blocks = cap;
  fill_range_kernel<<<(unsigned)blocks, 256, 0, stream>>>(dst, n, key, first, scale, okey,
                                                           row_len > 0 ? row_len : 1, pct);
  return (int)cudaGetLastError();
}

}  // extern "C"
