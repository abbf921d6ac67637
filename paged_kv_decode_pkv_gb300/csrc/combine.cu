// Log-sum-exp combine of split-K partials (Zero TVM Documentation, "How it works": one combine
// dispatch per layer after split-K attention).
//
// One warp per (sequence, query head).  The warp reads the split LSEs 32 at a time, takes their
// maximum M, weights w_j = exp(lse_j - M) (splits at -inf are skipped and their partial_o is not
// read), and accumulates sum_j w_j o_j with lanes over head_dim, so each read of a partial row is
// one coalesced 128-byte transaction per 32 floats.
#include "pkv_internal.h"
#include "ptx.cuh"

namespace pkv {
namespace {

constexpr int kWarpsPerCta = 4;
constexpr int kBatch = 8;  // partial rows in flight per warp

template <int D>
__global__ void __launch_bounds__(kWarpsPerCta * 32) combine_kernel(CombineParams p) {
  pdl_launch_dependents();
  constexpr int kPerLane = D / 32;
  const int lane = threadIdx.x & 31;
  const long long sh = (long long)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  if (sh >= (long long)p.batch * p.hq) return;
  pdl_wait();  // the partials come from the preceding kernel

  const int S = p.splits;
  const float* lse = p.partial_lse + sh * S;
  const float* po = p.partial_o + sh * S * D;

  float M = -INFINITY;
  for (int j = lane; j < S; j += 32) M = fmaxf(M, lse[j]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));

  float acc[kPerLane];
#pragma unroll
  for (int e = 0; e < kPerLane; ++e) acc[e] = 0.f;
  float W = 0.f;
  if (M != -INFINITY) {
    for (int jb = 0; jb < S; jb += 32) {
      const int j = jb + lane;
      const float lj = j < S ? lse[j] : -INFINITY;
      const float wl = (lj == -INFINITY) ? 0.f : expf(lj - M);
      W += wl;
      const int n = min(32, S - jb);
      // Rows are read kBatch at a time with independent (predicated) loads so that their
      // latencies overlap instead of forming one dependent chain per split.
      for (int k0 = 0; k0 < n; k0 += kBatch) {
        float w[kBatch];
        float v[kBatch][kPerLane];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          w[u] = __shfl_sync(0xffffffffu, wl, (k0 + u) & 31);
          if (k0 + u >= n) w[u] = 0.f;
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const float* row = po + (long long)(jb + k0 + u) * D;
#pragma unroll
          for (int e = 0; e < kPerLane; ++e) v[u][e] = (w[u] != 0.f) ? row[lane + 32 * e] : 0.f;
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u)
#pragma unroll
          for (int e = 0; e < kPerLane; ++e) acc[e] = fmaf(w[u], v[u][e], acc[e]);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) W += __shfl_xor_sync(0xffffffffu, W, o);
  }
  __half* out = p.out + sh * D;
  const float inv = (W > 0.f) ? 1.f / W : 0.f;
#pragma unroll
  for (int e = 0; e < kPerLane; ++e) out[lane + 32 * e] = __float2half_rn(acc[e] * inv);
  if (p.lse != nullptr && lane == 0) p.lse[sh] = (W > 0.f) ? M + logf(W) : -INFINITY;
}

}  // namespace

cudaError_t combine_prepare() {
  const void* k[] = {(const void*)&combine_kernel<64>, (const void*)&combine_kernel<96>,
                     (const void*)&combine_kernel<128>};
  for (const void* f : k) {
    const cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout,
                                               cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream, bool pdl) {
  const long long pairs = (long long)p.batch * p.hq;
  if (pairs <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((pairs + kWarpsPerCta - 1) / kWarpsPerCta));
  cfg.blockDim = dim3(kWarpsPerCta * 32);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  switch (p.head_dim) {
    case 64: return cudaLaunchKernelEx(&cfg, combine_kernel<64>, p);
    case 96: return cudaLaunchKernelEx(&cfg, combine_kernel<96>, p);
    case 128: return cudaLaunchKernelEx(&cfg, combine_kernel<128>, p);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pkv
