// Rotate-half RoPE of eight element pairs (Zero TVM Documentation, "KV cache": K is rotated before
// the cache write; the rotation pairs element i with element i + head_dim/2 at angle
// position * theta_i).  Shared by the append kernel and the one-launch decode so that both write
// the same bits.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace pkv {

// One rotation pair: a = x_i, b = x_{i+d/2}, (c, s) = (cos, sin) of element i at the position.
__device__ __forceinline__ void rope_pair(float a, float b, float2 cs, float& out_a, float& out_b) {
  out_a = __fmaf_rn(a, cs.x, -__fmul_rn(b, cs.y));
  out_b = __fmaf_rn(b, cs.x, __fmul_rn(a, cs.y));
}

// lo: elements i..i+7 of a head row, hi: elements i+d/2..i+d/2+7, cs: the (cos, sin) pairs of
// elements i..i+7 at the token's position.  Evaluated in fp32 with fused multiply-adds and
// rounded once to fp16:
//   x'_i = x_i cos - x_{i+d/2} sin ,   x'_{i+d/2} = x_{i+d/2} cos + x_i sin.
__device__ __forceinline__ void rope8(const uint4& lo, const uint4& hi, const float2* cs, uint4& out_lo,
                                      uint4& out_hi) {
  const __half2* a = reinterpret_cast<const __half2*>(&lo);
  const __half2* b = reinterpret_cast<const __half2*>(&hi);
  __half2* ya = reinterpret_cast<__half2*>(&out_lo);
  __half2* yb = reinterpret_cast<__half2*>(&out_hi);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 xa = __half22float2(a[e]);
    const float2 xb = __half22float2(b[e]);
    const float2 c0 = cs[2 * e], c1 = cs[2 * e + 1];  // (cos, sin) of elements 2e and 2e+1
    float lo0, lo1, hi0, hi1;
    rope_pair(xa.x, xb.x, c0, lo0, hi0);
    rope_pair(xa.y, xb.y, c1, lo1, hi1);
    ya[e] = __floats2half2_rn(lo0, lo1);
    yb[e] = __floats2half2_rn(hi0, hi1);
  }
}

}  // namespace pkv
