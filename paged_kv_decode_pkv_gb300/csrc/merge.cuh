// Log-sum-exp merge of split-K partials for one (sequence, query head), executed by one warp
// (Zero TVM Documentation, "How it works": the combine step after split-K attention).
//
// M = max_j lse_j, w_j = exp(lse_j - M), W = sum_j w_j, out = sum_j w_j o_j / W, lse = M + ln W.
// Splits with lse_j = -inf have w_j = 0 and their o_j is not read.  Pass 1: lane l takes splits
// l, l + 32, ... for M and W, reduced in a fixed butterfly order.  Pass 2: the warp is four groups
// of eight lanes; group g accumulates splits g, g + 4, g + 8, ... in order, each lane owning
// head_dim/8 consecutive dimensions as float4 vectors (with up to 64 splits the weights of pass 1
// arrive by shuffle, beyond that every lane recomputes its w_j, the same value); the four group
// sums are then added in a fixed order, (g0 + g1) + (g2 + g3).  A sink logit (a layer's attention
// sink, -inf for none) joins the maximum and adds its weight to the denominator, carrying no value.  Used by the combine kernel (rows and
// LSEs in global memory) and by the merged decode (in shared memory), so both give the same bits.
#pragma once

#include "pkv_internal.h"

namespace pkv {

// lse: [S] natural-log LSEs of the splits; rows: [S][D] normalised partial outputs (16-byte
// aligned); out: the fp16 result row (8-byte aligned); lse_out: the merged LSE or nullptr.  Both
// may point to global or shared memory.  Kept out of line: it runs once per merged row, and
// inlined copies would crowd the streaming loop's instruction cache.
template <int D>
__device__ __noinline__ void merge_rows(const float* lse, const float* rows, int S, int lane, __half* out,
                                        float* lse_out, float sink) {
  constexpr unsigned kAll = 0xffffffffu;
  constexpr int kVec = D / 32;  // float4 vectors per lane
  // pass 1: lane l holds the LSEs of splits l and l + 32 (the rest, if any, in a loop)
  const float la = lane < S ? lse[lane] : -INFINITY;
  const float lb = lane + 32 < S ? lse[lane + 32] : -INFINITY;
  float M = fmaxf(la, lb);
  for (int j = lane + 64; j < S; j += 32) M = fmaxf(M, lse[j]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kAll, M, o));
  M = fmaxf(M, sink);
  float4 acc[kVec];
#pragma unroll
  for (int v = 0; v < kVec; ++v) acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
  const bool any = M != -INFINITY;
  const float wa = (any && la != -INFINITY) ? expf(la - M) : 0.f;
  const float wb = (any && lb != -INFINITY) ? expf(lb - M) : 0.f;
  float W = wa + wb;
  for (int j = lane + 64; j < S; j += 32) {
    const float l = lse[j];
    W += (l == -INFINITY) ? 0.f : expf(l - M);
  }
  // pass 2: group g = lane / 8 takes splits g, g + 4, ...; lane l % 8 owns D/8 dimensions
  const int grp = lane >> 3;
  const float4* base = reinterpret_cast<const float4*>(rows) + (lane & 7) * kVec;
  auto accumulate = [&](float w, const float4* r) {
    float4 x[kVec];
#pragma unroll
    for (int v = 0; v < kVec; ++v) x[v] = r[v];
#pragma unroll
    for (int v = 0; v < kVec; ++v) {
      acc[v].x = fmaf(w, x[v].x, acc[v].x);
      acc[v].y = fmaf(w, x[v].y, acc[v].y);
      acc[v].z = fmaf(w, x[v].z, acc[v].z);
      acc[v].w = fmaf(w, x[v].w, acc[v].w);
    }
  };
  if (S <= 64) {
    // The weights come from pass 1 by shuffle.  No branch: a row past S is read as row 0 and a
    // row of weight 0 (-inf, may hold anything) is replaced by zeros, adding exactly nothing.
    const int iters = (S + 3) >> 2;
#pragma unroll 4
    for (int it = 0; it < iters; ++it) {
      const int j = 4 * it + grp;
      const float wA = __shfl_sync(kAll, wa, j & 31);
      const float wB = __shfl_sync(kAll, wb, j & 31);
      const float w = j < 32 ? wA : wB;
      const float4* r = base + (long long)(j < S ? j : 0) * (D / 4);
      float4 x[kVec];
#pragma unroll
      for (int v = 0; v < kVec; ++v) x[v] = r[v];
      const bool use = w != 0.f;
#pragma unroll
      for (int v = 0; v < kVec; ++v) {
        acc[v].x = fmaf(w, use ? x[v].x : 0.f, acc[v].x);
        acc[v].y = fmaf(w, use ? x[v].y : 0.f, acc[v].y);
        acc[v].z = fmaf(w, use ? x[v].z : 0.f, acc[v].z);
        acc[v].w = fmaf(w, use ? x[v].w : 0.f, acc[v].w);
      }
    }
  } else if (any) {
    for (int j = grp; j < S; j += 4) {
      const float l = lse[j];
      if (l != -INFINITY) accumulate(expf(l - M), base + (long long)j * (D / 4));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) W += __shfl_xor_sync(kAll, W, o);
  if (sink != -INFINITY) W += expf(sink - M);
#pragma unroll
  for (int o = 8; o <= 16; o <<= 1) {
#pragma unroll
    for (int v = 0; v < kVec; ++v) {
      acc[v].x += __shfl_xor_sync(kAll, acc[v].x, o);
      acc[v].y += __shfl_xor_sync(kAll, acc[v].y, o);
      acc[v].z += __shfl_xor_sync(kAll, acc[v].z, o);
      acc[v].w += __shfl_xor_sync(kAll, acc[v].w, o);
    }
  }
  if (lane < 8) {
    const float inv = (W > 0.f) ? 1.f / W : 0.f;
    __half2* dst = reinterpret_cast<__half2*>(out + lane * (D / 8));
#pragma unroll
    for (int v = 0; v < kVec; ++v) {
      __half2 h[2] = {__floats2half2_rn(acc[v].x * inv, acc[v].y * inv),
                      __floats2half2_rn(acc[v].z * inv, acc[v].w * inv)};
      *reinterpret_cast<uint2*>(dst + 2 * v) = *reinterpret_cast<const uint2*>(h);
    }
  }
  if (lse_out != nullptr && lane == 0) *lse_out = (W > 0.f) ? M + logf(W) : -INFINITY;
}

// Out-of-line merge of the G query heads of one (sequence, KV head) group from global memory,
// called by the chunk that finishes last when the partial rows do not fit its stage ring; kept out
// of line so its registers do not weigh on the streaming loop.
template <int D>
__device__ __noinline__ void merge_group(const float* partial_lse, const float* partial_o, long long head_row0,
                                         int group, int splits, int nch, int lane, __half* out, float* lse_out,
                                         const float* sinks, int head0) {
  for (int hh = 0; hh < group; ++hh) {
    const long long row = head_row0 + hh;
    merge_rows<D>(partial_lse + row * splits, partial_o + row * splits * D, nch, lane, out + row * D,
                  lse_out != nullptr ? lse_out + row : nullptr, sinks != nullptr ? sinks[head0 + hh] : -INFINITY);
  }
}

}  // namespace pkv
