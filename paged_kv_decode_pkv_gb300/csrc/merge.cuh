// Log-sum-exp merge of split-K partials for one (sequence, query head), executed by one warp
// (Zero TVM Documentation, "How it works": the combine step after split-K attention).
//
// M = max_j lse_j, w_j = exp(lse_j - M), W = sum_j w_j, out = sum_j w_j o_j / W, lse = M + ln W.
// Splits with lse_j = -inf have w_j = 0 and their o_j is not used.  Pass 1: lane l takes splits
// l, l + 32, ... for M and W, reduced in a fixed butterfly order.  Pass 2 takes one of two forms,
// chosen by the number of splits S:
//  * more than kColumnSplits: the warp is four groups of eight lanes; group g accumulates splits
//    g, g + 4, ... in order, each lane owning head_dim/8 consecutive dimensions as float4 vectors;
//    the four group sums are then added in a fixed order, (g0 + g1) + (g2 + g3).
//  * up to kColumnSplits: lane l owns the four dimensions 4l .. 4l + 3 (lanes past head_dim/4
//    idle) and keeps the four group sums itself (split j into sum j mod 4, in order), added in the
//    same order; no lane exchanges partial sums.
// The two forms do the same arithmetic (a split of weight 0 adds exactly nothing, whichever form
// visits it), so the result does not depend on the form, nor on trailing splits of weight 0.
// With up to 64 splits the weights of pass 1 arrive by shuffle, beyond that every lane recomputes
// w_j (the same value).  A sink logit (a layer's attention sink, -inf for none) joins the maximum
// and adds its weight to the denominator, carrying no value.  Used by the combine kernel (rows and
// LSEs in global memory) and by the merged decode (in shared memory), so both give the same bits.
#pragma once

#include "pkv_internal.h"

namespace pkv {

// Splits up to which pass 2 gives each lane a column of dimensions (no closing exchange of the
// group sums: the short chain a GQA group's few splits want); more splits are shared among four
// lane groups, which keeps the loop short.
constexpr int kColumnSplits = 16;

__device__ __forceinline__ void fma4(float w, const float4& x, float4& a) {
  a.x = fmaf(w, x.x, a.x);
  a.y = fmaf(w, x.y, a.y);
  a.z = fmaf(w, x.z, a.z);
  a.w = fmaf(w, x.w, a.w);
}

// lse: [S] natural-log LSEs of the splits; rows: [S][D] normalised partial outputs (16-byte
// aligned); out: the fp16 result row (8-byte aligned); lse_out: the merged LSE or nullptr.  Both
// may point to global or shared memory.  Kept out of line: it runs once per merged row, and
// inlined copies would crowd the streaming loop's instruction cache.
template <int D>
__device__ __noinline__ void merge_rows(const float* lse, const float* rows, int S, int lane, __half* out,
                                        float* lse_out, float sink) {
  constexpr unsigned kAll = 0xffffffffu;
  constexpr int NV = D / 4;    // float4 vectors of a row
  constexpr int kVec = D / 32;  // float4 vectors per lane in the group form
  static_assert(NV <= 32, "one float4 column per lane");
  // pass 1: lane l holds the LSEs of splits l and l + 32 (the rest, if any, in a loop)
  const float la = lane < S ? lse[lane] : -INFINITY;
  const float lb = lane + 32 < S ? lse[lane + 32] : -INFINITY;
  float M = fmaxf(la, lb);
  for (int j = lane + 64; j < S; j += 32) M = fmaxf(M, lse[j]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kAll, M, o));
  M = fmaxf(M, sink);
  const bool any = M != -INFINITY;
  const float wa = (any && la != -INFINITY) ? expf(la - M) : 0.f;
  const float wb = (any && lb != -INFINITY) ? expf(lb - M) : 0.f;
  float W = wa + wb;
  for (int j = lane + 64; j < S; j += 32) {
    const float l = lse[j];
    W += (l == -INFINITY) ? 0.f : expf(l - M);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) W += __shfl_xor_sync(kAll, W, o);
  if (sink != -INFINITY) W += expf(sink - M);
  const float inv = (W > 0.f) ? 1.f / W : 0.f;
  const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
  if (S <= kColumnSplits) {
    // Column form.  Split j's weight is lane j's wa (j < 16); a split at or past S has weight 0
    // and is read as split j, and a row of weight 0 (-inf, may hold anything) is replaced by
    // zeros, adding exactly nothing: no branch.
    const bool own = lane < NV;
    const float4* col = reinterpret_cast<const float4*>(rows) + (own ? lane : 0);
    float4 a[4] = {zero, zero, zero, zero};
    for (int j = 0; j < S; j += 4) {
#pragma unroll
      for (int h = 0; h < 4; h += 2) {
        const float w0 = __shfl_sync(kAll, wa, j + h), w1 = __shfl_sync(kAll, wa, j + h + 1);
        const float4 x0 = col[(j + h < S ? j + h : j) * NV];
        const float4 x1 = col[(j + h + 1 < S ? j + h + 1 : j) * NV];
        fma4(w0, w0 != 0.f ? x0 : zero, a[h]);
        fma4(w1, w1 != 0.f ? x1 : zero, a[h + 1]);
      }
    }
    if (own) {
      const float4 s01 = make_float4(a[0].x + a[1].x, a[0].y + a[1].y, a[0].z + a[1].z, a[0].w + a[1].w);
      const float4 s23 = make_float4(a[2].x + a[3].x, a[2].y + a[3].y, a[2].z + a[3].z, a[2].w + a[3].w);
      __half2 h[2] = {__floats2half2_rn((s01.x + s23.x) * inv, (s01.y + s23.y) * inv),
                      __floats2half2_rn((s01.z + s23.z) * inv, (s01.w + s23.w) * inv)};
      *reinterpret_cast<uint2*>(out + 4 * lane) = *reinterpret_cast<const uint2*>(h);
    }
  } else {
    // Group form: group g = lane / 8 takes splits g, g + 4, ...; lane l % 8 owns D/8 dimensions.
    const int grp = lane >> 3;
    const float4* base = reinterpret_cast<const float4*>(rows) + (lane & 7) * kVec;
    float4 acc[kVec];
#pragma unroll
    for (int v = 0; v < kVec; ++v) acc[v] = zero;
    if (S <= 64) {
      // weights by shuffle; a row past S is read as row 0, a row of weight 0 as zeros
      const int iters = (S + 3) >> 2;
#pragma unroll 4
      for (int it = 0; it < iters; ++it) {
        const int j = 4 * it + grp;
        const float wA = __shfl_sync(kAll, wa, j & 31);
        const float wB = __shfl_sync(kAll, wb, j & 31);
        const float w = j < 32 ? wA : wB;
        const float4* r = base + (long long)(j < S ? j : 0) * NV;
        float4 x[kVec];
#pragma unroll
        for (int v = 0; v < kVec; ++v) x[v] = r[v];
#pragma unroll
        for (int v = 0; v < kVec; ++v) fma4(w, w != 0.f ? x[v] : zero, acc[v]);
      }
    } else if (any) {
      for (int j = grp; j < S; j += 4) {
        const float l = lse[j];
        if (l != -INFINITY) {
          const float w = expf(l - M);
          const float4* r = base + (long long)j * NV;
#pragma unroll
          for (int v = 0; v < kVec; ++v) fma4(w, r[v], acc[v]);
        }
      }
    }
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
      __half2* dst = reinterpret_cast<__half2*>(out + lane * (D / 8));
#pragma unroll
      for (int v = 0; v < kVec; ++v) {
        __half2 h[2] = {__floats2half2_rn(acc[v].x * inv, acc[v].y * inv),
                        __floats2half2_rn(acc[v].z * inv, acc[v].w * inv)};
        *reinterpret_cast<uint2*>(dst + 2 * v) = *reinterpret_cast<const uint2*>(h);
      }
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
