// RoPE + KV append: rotate the new tokens' q and k at their positions and scatter k and v into
// their page slots (Zero TVM Documentation, "Decode loop": the QKV dispatch applies RoPE and
// writes the KV cache; "KV cache": K is rotated before the cache write).
//
// One CTA handles kTokensPerCta consecutive tokens.  Every thread moves 16-byte vectors: a RoPE
// unit is 8 consecutive elements i..i+7 of one head together with their rotation partners
// i+d/2..i+d/2+7 (rotate-half form), a V unit is 8 consecutive elements.  The cos/sin values come
// from the fp64-derived fp32 table built at cache creation; the rotation is evaluated in fp32
// with fused multiply-adds and rounded once to fp16.  V is a bit copy.
#include "pkv_internal.h"
#include "ptx.cuh"
#include "rope.cuh"

namespace pkv {
namespace {

constexpr int kThreads = 256;
constexpr int kTokensPerCta = 4;
constexpr int kIndptrSmemCap = 8192;  // sequences whose append_indptr fits the shared copy

struct TokenSlot {
  long long k_off;  // element offset of pool[page][0][0][slot][0]; -1 = skip the token
  int pos;
};

// The shared copy of append_indptr is dynamic (batch + 1 ints, none past kIndptrSmemCap) so that a
// small launch fits beside a resident decode CTA and can start under programmatic dependent launch.
template <int D>
__global__ void __launch_bounds__(kThreads) append_rope_kernel(AppendParams p) {
  extern __shared__ int s_indptr[];
  __shared__ TokenSlot s_tok[kTokensPerCta];
  __shared__ float2 s_cs[kTokensPerCta][D / 2];  // (cos, sin) rows of the CTA's tokens
  pdl_launch_dependents();

  const int t0 = blockIdx.x * kTokensPerCta;
  const bool indptr_in_smem = p.batch <= kIndptrSmemCap;
  if (indptr_in_smem) {
    for (int i = threadIdx.x; i <= p.batch; i += kThreads) s_indptr[i] = p.append_indptr[i];
  }
  __syncthreads();
  const int* indptr = indptr_in_smem ? s_indptr : p.append_indptr;

  if (threadIdx.x < kTokensPerCta) {
    const int t = t0 + threadIdx.x;
    TokenSlot ts{-1, 0};
    if (t < p.num_tokens) {
      // sequence of token t: the last s with indptr[s] <= t
      int lo = 0, hi = p.batch;  // invariant: indptr[lo] <= t < indptr[hi] when t is in range
      if (indptr[0] <= t && t < indptr[p.batch]) {
        while (hi - lo > 1) {
          const int mid = (lo + hi) >> 1;
          if (indptr[mid] <= t) lo = mid; else hi = mid;
        }
        const int s = lo;
        const int pos = p.pos_map[t];
        const int first = p.page_indptr[s];
        const int n_pages = p.page_indptr[s + 1] - first;
        if (pos < 0 || pos >= p.max_position || (pos >> 4) >= n_pages) {
          atomicOr(p.status, kFlagBadPosition);
        } else {
          const int page = p.page_indices[first + (pos >> 4)];
          if (page < 0 || page >= p.num_pages) {
            atomicOr(p.status, kFlagBadPage);
          } else {
            ts.k_off = ((long long)page * 2 * p.hkv * kPageSize + (pos & 15)) * D;
            ts.pos = pos;
          }
        }
      } else {
        atomicOr(p.status, kFlagBadSequence);
      }
    }
    s_tok[threadIdx.x] = ts;
  }
  __syncthreads();
  // The RoPE table is written once at cache creation, so its rows can be staged before the wait.
  for (int i = threadIdx.x; i < kTokensPerCta * (D / 2); i += kThreads) {
    const int tk = i / (D / 2), e = i - tk * (D / 2);
    const TokenSlot ts = s_tok[tk];
    if (ts.k_off >= 0) s_cs[tk][e] = p.rope[(long long)ts.pos * (D / 2) + e];
  }
  __syncthreads();
  pdl_wait();  // q, k, v and the pool may be produced or read by the preceding kernel

  constexpr int kRopeUnits = D / 16;  // 8-element blocks in the first half of a head
  constexpr int kVUnits = D / 8;
  const int q_units = p.hq * kRopeUnits;
  const int k_units = p.hkv * kRopeUnits;
  const int v_units = p.hkv * kVUnits;
  const int per_token = q_units + k_units + v_units;
  const long long head_stride = (long long)kPageSize * D;  // pool elements between heads

  for (int idx = threadIdx.x; idx < kTokensPerCta * per_token; idx += kThreads) {
    const int tk = idx / per_token;
    const int u = idx - tk * per_token;
    const int t = t0 + tk;
    const TokenSlot ts = s_tok[tk];
    if (ts.k_off < 0) continue;
    if (u < q_units + k_units) {
      const bool is_q = u < q_units;
      const int uu = is_q ? u : u - q_units;
      const int h = uu / kRopeUnits;
      const int i0 = (uu - h * kRopeUnits) * 8;
      const __half* src = is_q ? p.q + ((long long)t * p.hq + h) * D : p.k + ((long long)t * p.hkv + h) * D;
      const uint4 lo = *reinterpret_cast<const uint4*>(src + i0);
      const uint4 hi = *reinterpret_cast<const uint4*>(src + i0 + D / 2);
      uint4 ylo, yhi;
      rope8(lo, hi, &s_cs[tk][i0], ylo, yhi);
      __half* dst = is_q ? p.q_out + ((long long)t * p.hq + h) * D : p.pool + ts.k_off + h * head_stride;
      *reinterpret_cast<uint4*>(dst + i0) = ylo;
      *reinterpret_cast<uint4*>(dst + i0 + D / 2) = yhi;
    } else {
      const int uu = u - q_units - k_units;
      const int h = uu / kVUnits;
      const int i0 = (uu - h * kVUnits) * 8;
      const uint4 val = *reinterpret_cast<const uint4*>(p.v + ((long long)t * p.hkv + h) * D + i0);
      __half* dst = p.pool + ts.k_off + (long long)p.hkv * head_stride + h * head_stride;  // V block
      *reinterpret_cast<uint4*>(dst + i0) = val;
    }
  }
}

}  // namespace

cudaError_t append_prepare() {
  const void* k[] = {(const void*)&append_rope_kernel<64>, (const void*)&append_rope_kernel<96>,
                     (const void*)&append_rope_kernel<128>};
  for (const void* f : k) {
    const cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout,
                                               cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_append(const AppendParams& p, cudaStream_t stream, bool pdl) {
  if (p.num_tokens <= 0 || p.batch <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((p.num_tokens + kTokensPerCta - 1) / kTokensPerCta);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = p.batch <= kIndptrSmemCap ? (size_t)(p.batch + 1) * sizeof(int) : 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  switch (p.head_dim) {
    case 64: return cudaLaunchKernelEx(&cfg, append_rope_kernel<64>, p);
    case 96: return cudaLaunchKernelEx(&cfg, append_rope_kernel<96>, p);
    case 128: return cudaLaunchKernelEx(&cfg, append_rope_kernel<128>, p);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pkv

// ------------------------------------------------------------------------------------------------
// The append into an int8 cache (PKV_OPT_INT8_KV).  Layout per layer: uint8 blocks
// [num_pages][2][Hkv][16 * d + 64], a block holding the 16 slots' int8 codes, each stored as the
// byte code + 128, and then their fp32 scales [16]; K codes are slot-major [16][d], V codes
// dim-major [d][16] (the layouts the decode's tensor-core fragments read four codes at a time
// from).  Row quantizer: amax = max |x_i| of the row's fp16 values (K after RoPE and its fp16
// rounding, as the fp16 cache stores it; V as given), s = amax / 127 (fp32 division),
// code_i = clamp(rint_even(x_i / s), -127, 127) (fp32 division), amax = 0 giving s = 0 and codes 0.
// One warp per (token, row): Hq query rows (rotated to q_out, fp16), Hkv K rows, Hkv V rows.

namespace pkv {
namespace {

constexpr int kQ8Warps = 8;

template <int D>
__global__ void __launch_bounds__(kQ8Warps * 32) append_rope_q8_kernel(AppendParams p) {
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int rows_per_token = p.hq + 2 * p.hkv;
  const long long job = (long long)blockIdx.x * kQ8Warps + (threadIdx.x >> 5);
  if (job >= (long long)p.num_tokens * rows_per_token) return;
  const int t = (int)(job / rows_per_token);
  const int row = (int)(job - (long long)t * rows_per_token);
  // token -> sequence -> page slot (the fp16 append's checks; the first row of a token reports)
  long long blk_page = -1;
  int pos = 0;
  {
    int lo = 0, hi = p.batch;
    if (p.append_indptr[0] <= t && t < p.append_indptr[p.batch]) {
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (p.append_indptr[mid] <= t) lo = mid; else hi = mid;
      }
      pos = p.pos_map[t];
      const int first = p.page_indptr[lo];
      const int n_pages = p.page_indptr[lo + 1] - first;
      if (pos < 0 || pos >= p.max_position || (pos >> 4) >= n_pages) {
        if (row == 0 && lane == 0) atomicOr(p.status, kFlagBadPosition);
      } else {
        const int page = p.page_indices[first + (pos >> 4)];
        if (page < 0 || page >= p.num_pages) {
          if (row == 0 && lane == 0) atomicOr(p.status, kFlagBadPage);
        } else {
          blk_page = page;
        }
      }
    } else if (row == 0 && lane == 0) {
      atomicOr(p.status, kFlagBadSequence);
    }
  }
  pdl_wait();  // q, k, v and the pool may be produced or read by the preceding kernel
  if (blk_page < 0) return;

  const bool is_q = row < p.hq;
  const bool is_k = !is_q && row < p.hq + p.hkv;
  const int head = is_q ? row : is_k ? row - p.hq : row - p.hq - p.hkv;
  const __half* src = is_q ? p.q + ((long long)t * p.hq + head) * D
                    : (is_k ? p.k : p.v) + ((long long)t * p.hkv + head) * D;
  const float2* cs = p.rope + (long long)pos * (D / 2);
  // the row's values as the fp16 cache would hold them: pairs (j, j + D/2), j = lane, lane + 32
  constexpr int kPairs = (D / 2 + 31) / 32;
  __half lo_v[kPairs], hi_v[kPairs];
#pragma unroll
  for (int u = 0; u < kPairs; ++u) {
    const int j = lane + 32 * u;
    if (j < D / 2) {
      __half a = src[j], b = src[j + D / 2];
      if (!(row >= p.hq + p.hkv)) {  // q and k rows are rotated
        float ra, rb;
        rope_pair(__half2float(a), __half2float(b), cs[j], ra, rb);
        a = __float2half_rn(ra);
        b = __float2half_rn(rb);
      }
      lo_v[u] = a;
      hi_v[u] = b;
    }
  }
  if (is_q) {
    __half* dst = p.q_out + ((long long)t * p.hq + head) * D;
#pragma unroll
    for (int u = 0; u < kPairs; ++u) {
      const int j = lane + 32 * u;
      if (j < D / 2) {
        dst[j] = lo_v[u];
        dst[j + D / 2] = hi_v[u];
      }
    }
    return;
  }
  float amax = 0.f;
#pragma unroll
  for (int u = 0; u < kPairs; ++u)
    if (lane + 32 * u < D / 2) amax = fmaxf(amax, fmaxf(fabsf(__half2float(lo_v[u])), fabsf(__half2float(hi_v[u]))));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float s = amax / 127.0f;
  const int kv = is_k ? 0 : 1;
  unsigned char* blk = p.pool8 + ((blk_page * 2 + kv) * p.hkv + head) * (long long)(16 * D + 64);
  const int slot = pos & 15;
  auto code = [&](__half h) -> unsigned char {  // the stored byte: code + 128
    if (s == 0.f) return 128;
    const float q = rintf(__half2float(h) / s);
    return (unsigned char)(128 + (int)fminf(127.f, fmaxf(-127.f, q)));
  };
#pragma unroll
  for (int u = 0; u < kPairs; ++u) {
    const int j = lane + 32 * u;
    if (j < D / 2) {
      if (is_k) {
        blk[slot * D + j] = code(lo_v[u]);
        blk[slot * D + j + D / 2] = code(hi_v[u]);
      } else {
        blk[j * 16 + slot] = code(lo_v[u]);
        blk[(j + D / 2) * 16 + slot] = code(hi_v[u]);
      }
    }
  }
  if (lane == 0) *reinterpret_cast<float*>(blk + 16 * D + 4 * slot) = s;
}

}  // namespace

cudaError_t launch_append_q8(const AppendParams& p, cudaStream_t stream, bool pdl) {
  if (p.num_tokens <= 0 || p.batch <= 0) return cudaSuccess;
  const long long jobs = (long long)p.num_tokens * (p.hq + 2 * p.hkv);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((jobs + kQ8Warps - 1) / kQ8Warps));
  cfg.blockDim = dim3(kQ8Warps * 32);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  switch (p.head_dim) {
    case 64: return cudaLaunchKernelEx(&cfg, append_rope_q8_kernel<64>, p);
    case 96: return cudaLaunchKernelEx(&cfg, append_rope_q8_kernel<96>, p);
    case 128: return cudaLaunchKernelEx(&cfg, append_rope_q8_kernel<128>, p);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pkv
