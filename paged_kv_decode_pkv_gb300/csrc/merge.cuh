// Log-sum-exp merge of split-K partials for one (sequence, query head), executed by one warp
// (Zero TVM Documentation, "How it works": the combine step after split-K attention).
//
// M = max_j lse_j, w_j = exp(lse_j - M), out = sum_j w_j o_j / sum_j w_j, lse = M + ln sum_j w_j.
// Splits with lse_j = -inf are skipped and their o_j is not read.  Lanes own head_dim/32
// dimensions; partial rows are read kMergeBatch at a time with independent predicated loads so
// their latencies overlap.  Used by the combine kernel and by the merged decode kernel, so both
// produce bit-identical results.
#pragma once

#include "pkv_internal.h"

namespace pkv {

constexpr int kMergeBatch = 16;

// lse: [S] natural-log LSE of the splits; po: [S][D] normalised partial outputs.
template <int D>
__device__ __forceinline__ void merge_row(const float* lse, const float* po, int S, int lane, __half* out,
                                          float* lse_out) {
  constexpr int kPerLane = D / 32;
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
      for (int k0 = 0; k0 < n; k0 += kMergeBatch) {
        float w[kMergeBatch];
        float v[kMergeBatch][kPerLane];
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u) {
          w[u] = __shfl_sync(0xffffffffu, wl, (k0 + u) & 31);
          if (k0 + u >= n) w[u] = 0.f;
        }
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u) {
          const float* row = po + (long long)(jb + k0 + u) * D;
#pragma unroll
          for (int e = 0; e < kPerLane; ++e) v[u][e] = (w[u] != 0.f) ? row[lane + 32 * e] : 0.f;
        }
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u)
#pragma unroll
          for (int e = 0; e < kPerLane; ++e) acc[e] = fmaf(w[u], v[u][e], acc[e]);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) W += __shfl_xor_sync(0xffffffffu, W, o);
  }
  const float inv = (W > 0.f) ? 1.f / W : 0.f;
#pragma unroll
  for (int e = 0; e < kPerLane; ++e) out[lane + 32 * e] = __float2half_rn(acc[e] * inv);
  if (lse_out != nullptr && lane == 0) *lse_out = (W > 0.f) ? M + logf(W) : -INFINITY;
}

}  // namespace pkv

namespace pkv {

// Out-of-line merge of the G query heads of one (sequence, KV head) group, called by the chunk
// that finishes last; kept out of line so its registers do not weigh on the streaming loop.
template <int D>
__device__ __noinline__ void merge_group(const float* partial_lse, const float* partial_o, long long head_row0,
                                         int group, int splits, int nch, int lane, __half* out, float* lse_out) {
  for (int hh = 0; hh < group; ++hh) {
    const long long row = head_row0 + hh;
    merge_row<D>(partial_lse + row * splits, partial_o + row * splits * D, nch, lane, out + row * D,
                 lse_out != nullptr ? lse_out + row : nullptr);
  }
}


// The same merge with the partial rows already in shared memory (rows [S][D] at po_s) and the
// split LSEs in registers: lane l holds lse of splits l and l + 32 (lse_a, lse_b; -inf past S).
// Bit-identical to merge_row: the same operations in the same order.
template <int D>
__device__ __forceinline__ void merge_row_smem(float lse_a, float lse_b, const float* po_s, int S, int lane,
                                               __half* out, float* lse_out) {
  constexpr int kPerLane = D / 32;
  float M = fmaxf(lse_a, lse_b);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float acc[kPerLane];
#pragma unroll
  for (int e = 0; e < kPerLane; ++e) acc[e] = 0.f;
  float W = 0.f;
  if (M != -INFINITY) {
    for (int jb = 0; jb < S; jb += 32) {
      const float lj = jb == 0 ? lse_a : lse_b;
      const float wl = (lj == -INFINITY) ? 0.f : expf(lj - M);
      W += wl;
      const int n = min(32, S - jb);
      for (int k0 = 0; k0 < n; k0 += kMergeBatch) {
        float w[kMergeBatch];
        float v[kMergeBatch][kPerLane];
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u) {
          w[u] = __shfl_sync(0xffffffffu, wl, (k0 + u) & 31);
          if (k0 + u >= n) w[u] = 0.f;
        }
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u) {
          const float* row = po_s + (jb + k0 + u) * D;
#pragma unroll
          for (int e = 0; e < kPerLane; ++e) v[u][e] = (w[u] != 0.f) ? row[lane + 32 * e] : 0.f;
        }
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u)
#pragma unroll
          for (int e = 0; e < kPerLane; ++e) acc[e] = fmaf(w[u], v[u][e], acc[e]);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) W += __shfl_xor_sync(0xffffffffu, W, o);
  }
  const float inv = (W > 0.f) ? 1.f / W : 0.f;
#pragma unroll
  for (int e = 0; e < kPerLane; ++e) out[lane + 32 * e] = __float2half_rn(acc[e] * inv);
  if (lse_out != nullptr && lane == 0) *lse_out = (W > 0.f) ? M + logf(W) : -INFINITY;
}

}  // namespace pkv
