// Log-sum-exp combine of split-K partials (Zero TVM Documentation, "How it works": one combine
// dispatch per layer after split-K attention).  One warp per (sequence, query head) runs the
// shared merge of merge.cuh.
#include "merge.cuh"
#include "pkv_internal.h"
#include "ptx.cuh"

namespace pkv {
namespace {

constexpr int kWarpsPerCta = 4;

template <int D>
__global__ void __launch_bounds__(kWarpsPerCta * 32) combine_kernel(CombineParams p) {
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const long long sh = (long long)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  if (sh >= (long long)p.batch * p.hq) return;
  pdl_wait();  // the partials come from the preceding kernel
  const int S = p.splits;
  merge_rows<D>(p.partial_lse + sh * S, p.partial_o + sh * S * D, S, lane, p.out + sh * D,
                p.lse != nullptr ? p.lse + sh : nullptr, p.sinks != nullptr ? p.sinks[sh % p.hq] : -INFINITY);
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
