// QKV projection with Q4F16_1 weights, fused with RoPE and the KV append (Zero TVM
// Documentation, "Decode loop": the QKV matmul, RoPE and the KV-append in one dispatch; "Q4F16
// quantization format": eight int4 values per uint32, element i in bits 4i..4i+3, one fp16 scale
// per 32 weights, weight value f16(nibble - 7) * scale evaluated in fp16).
//
// Weights are row-major by output feature and packed along the input: w[n][k / 8] holds input k
// of output n in nibble k % 8, scales[n][k / 32].  Output rows are [q heads | k heads | v heads],
// head_dim rows each.
//
// Work decomposition.  A CTA owns 16 output rows of one head, the rope pairs 8b + i and
// head_dim/2 + 8b + i (i < 8), so it can rotate what it computes.  Its warps split the rows in
// two halves of 8 and the input into parts of 1024 (a lane takes 32 consecutive inputs: one
// 16-byte weight load and one scale per row); every lane loads its 8 rows' weights up front.  Per
// word the eight nibbles become four half2 pairs {i, i+4} with mask-and-or (1024 + nibble as an
// fp16), an exact subtraction of 1031 and an fp16 multiply by the scale (the format's fp16
// product, rounded to nearest); the input is stored in shared memory in the same pair order and
// the products accumulate in fp32.  The warps' partial sums are reduced in a fixed order, rounded
// to fp16 (the projection's value), rotated with the append kernel's arithmetic and written: q
// rows to q_out, k and v rows into the pool.  Tokens are processed two at a time (one: a kernel
// specialised for a single token).  The token slots are looked up before the programmatic
// dependent launch wait (page tables and positions are not produced by the preceding kernel).
#include <algorithm>

#include "pkv_internal.h"
#include "ptx.cuh"
#include "rope.cuh"

namespace pkv {
namespace {

constexpr int kTokMax = 2;     // tokens per pass of the multi-token kernel (1 for a single token)
constexpr int kPartIn = 1024;  // inputs per warp (32 lanes x 32)

struct QkvSlot {
  long long k_off;  // pool element offset of [page][0][0][slot][0]; -1 = skip the token
  int pos;
};


// acc += a.lo * b.lo + a.hi * b.hi (fp16 operands, fp32 accumulation)
__device__ __forceinline__ float fma2(uint32_t a, uint32_t b, float acc) {
  asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
      "mov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
      "fma.rn.f32.f16 %0, al, bl, %0;\n\tfma.rn.f32.f16 %0, ah, bh, %0;\n\t}"
      : "+f"(acc) : "r"(a), "r"(b));
  return acc;
}

// Weights of the eight nibbles of `word` as four fp16 pairs {j, j+4}: f16(nibble - 7) * scale.
// (word >> 4j) & 0x000F000F | 0x64006400 is the fp16 pair {1024 + n_j, 1024 + n_j+4}; subtracting
// 1031 is exact, the multiply by the scale pair is the format's fp16 product, rounded to nearest.
__device__ __forceinline__ void dequant_word(uint32_t word, uint32_t scale2, uint32_t (&wp)[4]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    asm("{\n\t.reg .b32 t;\n\t"
        "lop3.b32 t, %1, 0x000F000F, 0x64006400, 0xEA;\n\t"
        "sub.rn.f16x2 t, t, %2;\n\t"
        "mul.rn.f16x2 %0, t, %3;\n\t}"
        : "=r"(wp[j])
        : "r"(word >> (4 * j)), "r"(0x64076407u), "r"(scale2));
  }
}

// Sum of acc[r][t] over the 32 lanes for the 8 rows r at once: each exchange halves the rows a
// lane keeps (lane bit 4 keeps rows 4..7, bit 3 the upper half of those, bit 2 the upper one),
// so lane l ends with row (l >> 2) & 7; 9 shuffles instead of 40.
template <int kTok>
__device__ __forceinline__ float reduce8(const float (&acc)[8][kTok], int t, int lane) {
  const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
  float v4[4];
#pragma unroll
  for (int a = 0; a < 4; ++a)
    v4[a] = (b4 ? acc[a + 4][t] : acc[a][t]) + __shfl_xor_sync(0xffffffffu, b4 ? acc[a][t] : acc[a + 4][t], 16);
  float v2[2];
#pragma unroll
  for (int a = 0; a < 2; ++a) v2[a] = (b3 ? v4[a + 2] : v4[a]) + __shfl_xor_sync(0xffffffffu, b3 ? v4[a] : v4[a + 2], 8);
  float v1 = (b2 ? v2[1] : v2[0]) + __shfl_xor_sync(0xffffffffu, b2 ? v2[0] : v2[1], 4);
  v1 += __shfl_xor_sync(0xffffffffu, v1, 2);
  return v1 + __shfl_xor_sync(0xffffffffu, v1, 1);
}

// ------------------------------------------------------------------------------------------------
// Several tokens: the projection on tensor cores (mma.sync m16n8k16, fp16 weights and inputs, fp32
// accumulation).  A CTA owns the same 16 rows (M: row g = element 8b + g of the head, row g + 8 its
// RoPE partner D/2 + 8b + g) and takes the tokens 8, 16 or 32 at a time (one to four n-tiles of N =
// 8).  Its weight rows are copied once into shared memory (rows padded by 16 bytes) before the launch
// wait.  The inputs are split over the warps in blocks of 64 (8 words of a row); within a block the
// sum runs over the inputs in a permuted order that leaves it unchanged: at k-step s, lane (g, c)
// takes word 2c + s/2 of the block and its nibble pairs {2(s%2), +4} and {2(s%2) + 1, +4}, which one
// mask-and-or per pair dequantizes, for rows g and g + 8 (the A fragment), and the same input pairs
// of token g, read from the 16 bytes of that word's inputs (the B fragment).  Each weight is
// dequantized once per pass, the format's fp16 product as in the CUDA-core kernel.  The warps'
// fragments are summed in a fixed order, rounded to fp16, rotated and written like the CUDA-core
// kernel's.
constexpr int kMmaWarps = 8;

template <int NT>
struct QkvMmaSmem {
  // bytes of the shared layout for `hidden` inputs: barrier, weight rows, scales, warp fragments
  static size_t bytes(int hidden) {
    const size_t w = (size_t)16 * (hidden / 2 + 16);
    const size_t sc = ((size_t)16 * (hidden / 32) * 2 + 15) & ~(size_t)15;
    const size_t red = (size_t)kMmaWarps * NT * 16 * 8 * 4;
    return 16 + w + sc + red;
  }
};

template <int D, int NT>
__global__ void __launch_bounds__(kMmaWarps * 32) qkv_mma_kernel(QkvParams p) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int groups = p.hidden / 32;
  const int wstride = p.hidden / 2 + 16;  // bytes per staged weight row
  const int tok_cap = min(8 * NT, p.num_tokens);
  uint64_t* wbar = reinterpret_cast<uint64_t*>(smem);
  unsigned char* ws = smem + 16;
  __half* scs = reinterpret_cast<__half*>(ws + 16 * wstride);
  float* red = reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(scs) + ((16 * groups * 2 + 15) & ~15));
  // [warp][NT][16][8]
  __shared__ QkvSlot slots[8 * NT];
  __shared__ float2 cs[8 * NT][8];
  pdl_launch_dependents();

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int blocks_per_head = D / 16;
  const int hh = blockIdx.x / blocks_per_head;
  const int b = blockIdx.x - hh * blocks_per_head;
  const int N = (p.hq + 2 * p.hkv) * D;
  auto row_of = [&](int r) -> long long { return (long long)hh * D + (r < 8 ? 8 * b + r : D / 2 + 8 * b + r - 8); };

  // the CTA's 16 weight rows and their scales: inputs of the weights, copied before the wait
  if (tid == 0) {
    mbar_init(wbar, 1);
    fence_mbarrier_init();
    mbar_arrive_expect_tx(wbar, (uint32_t)(16 * (p.hidden / 2)));
  }
  __syncthreads();
  if (tid < 16)
    bulk_load(ws + tid * wstride, reinterpret_cast<const unsigned char*>(p.w) + row_of(tid) * (p.hidden / 2),
              (uint32_t)(p.hidden / 2), wbar);
  for (int i = tid; i < 16 * groups; i += blockDim.x) {
    const int r = i / groups, k = i - r * groups;
    scs[i] = p.scales[row_of(r) * groups + k];
  }
  auto lookup_slot = [&](int t, int i) {
    QkvSlot ts{-1, 0};
    if (t < p.num_tokens && p.pool != nullptr) {
      int lo = 0, hi = p.batch;
      if (p.append_indptr[0] <= t && t < p.append_indptr[p.batch]) {
        while (hi - lo > 1) {
          const int mid = (lo + hi) >> 1;
          if (p.append_indptr[mid] <= t) lo = mid; else hi = mid;
        }
        const int pos = p.pos_map[t];
        const int first = p.page_indptr[lo];
        const int n_pages = p.page_indptr[lo + 1] - first;
        if (pos < 0 || pos >= p.max_position || (pos >> 4) >= n_pages) {
          atomicOr(p.status, kFlagBadPosition);
        } else {
          const int page = p.page_indices[first + (pos >> 4)];
          if (page < 0 || page >= p.num_pages) {
            atomicOr(p.status, kFlagBadPage);
          } else {
            ts.k_off = ((long long)page * 2 * p.hkv * kPageSize + (pos & 15)) * D;
            ts.pos = pos;
#pragma unroll
            for (int e = 0; e < 8; ++e) cs[i][e] = p.rope[(long long)pos * (D / 2) + 8 * b + e];
          }
        }
      } else {
        atomicOr(p.status, kFlagBadSequence);
      }
    }
    slots[i] = ts;
  };
  if (tid < tok_cap) lookup_slot(tid, tid);  // the first tokens, before the wait
  pdl_wait();  // the input rows and the pool may come from the preceding kernel
  const bool weights_ok = mbar_wait_bounded(wbar, 0, kWaitLimitNs);
  if (!weights_ok) {
    if (tid == 0) atomicOr(p.status, kFlagTimeout);
    mbar_wait_bounded(wbar, 0, kDrainLimitNs);  // the copies may still land: wait (bounded) before leaving
    return;
  }

  const int nblk = p.hidden / 64;          // whole blocks of 64 inputs
  const bool tail = (p.hidden & 63) != 0;  // a last half block of 32 inputs
  for (int t0 = 0; t0 < p.num_tokens; t0 += 8 * NT) {
    const int nt = min(8 * NT, p.num_tokens - t0);
    if (t0 > 0 && tid < nt) lookup_slot(t0 + tid, tid);
    __syncthreads();

    float acc[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
    // A of one k-step: the word's nibble pairs {j0, +4} and {j0 + 1, +4} of rows g and g + 8
    auto afrag = [&](int wglob, int j0, uint32_t (&a)[4]) {
      const uint32_t wg = *reinterpret_cast<const uint32_t*>(ws + g * wstride + 4 * wglob);
      const uint32_t wg8 = *reinterpret_cast<const uint32_t*>(ws + (g + 8) * wstride + 4 * wglob);
      const int grp = wglob >> 2;
      const uint32_t s0 = __half_as_ushort(scs[g * groups + grp]), s1 = __half_as_ushort(scs[(g + 8) * groups + grp]);
      const uint32_t sh[4] = {wg >> (4 * j0), wg8 >> (4 * j0), wg >> (4 * j0 + 4), wg8 >> (4 * j0 + 4)};
      const uint32_t sc2[4] = {s0 | (s0 << 16), s1 | (s1 << 16), s0 | (s0 << 16), s1 | (s1 << 16)};
#pragma unroll
      for (int i = 0; i < 4; ++i)
        asm("{\n\t.reg .b32 t;\n\t"
            "lop3.b32 t, %1, 0x000F000F, 0x64006400, 0xEA;\n\tsub.rn.f16x2 t, t, %3;\n\tmul.rn.f16x2 %0, t, %2;\n\t}"
            : "=r"(a[i]) : "r"(sh[i]), "r"(sc2[i]), "r"(0x64076407u));
    };
    // one word of the block: its two k-steps (pairs {0, 1}, then {2, 3}) for every n-tile; B is the
    // word's eight inputs of token 8n + g, rearranged into the pairs {x_j, x_j+4}
    auto word_steps = [&](int wglob, int nsteps) {
      uint4 xv[NT];
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        const int t = 8 * n + g;
        xv[n] = t < nt ? *reinterpret_cast<const uint4*>(p.x + (long long)(t0 + t) * p.hidden + 8 * wglob)
                       : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int s2 = 0; s2 < 2; ++s2) {
        if (s2 >= nsteps) break;
        uint32_t a[4];
        afrag(wglob, 2 * s2, a);
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          const uint32_t lo = s2 == 0 ? xv[n].x : xv[n].y, hi = s2 == 0 ? xv[n].z : xv[n].w;
          mma_16816(acc[n], a[0], a[1], a[2], a[3], __byte_perm(lo, hi, 0x5410), __byte_perm(lo, hi, 0x7632));
        }
      }
    };
    for (int blk = warp; blk < nblk; blk += kMmaWarps) {
      word_steps(8 * blk + 2 * c, 2);
      word_steps(8 * blk + 2 * c + 1, 2);
    }
    if (tail && warp == nblk % kMmaWarps) word_steps(8 * nblk + c, 2);  // the last 32 inputs: word c
    // the warps' fragments, then their sum in a fixed order
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      float* rw = red + ((size_t)(warp * NT + n) * 16) * 8;
      rw[g * 8 + 2 * c] = acc[n][0];
      rw[g * 8 + 2 * c + 1] = acc[n][1];
      rw[(g + 8) * 8 + 2 * c] = acc[n][2];
      rw[(g + 8) * 8 + 2 * c + 1] = acc[n][3];
    }
    __syncthreads();
    for (int i = tid; i < nt * 8; i += blockDim.x) {
      const int t = i >> 3, r = i & 7;
      const int n = t >> 3, tc = t & 7;
      float ylo = 0.f, yhi = 0.f;
      for (int w = 0; w < kMmaWarps; ++w) {
        const float* rw = red + ((size_t)(w * NT + n) * 16) * 8;
        ylo += rw[r * 8 + tc];
        yhi += rw[(r + 8) * 8 + tc];
      }
      const __half hlo = __float2half_rn(ylo), hhi = __float2half_rn(yhi);
      const int e = 8 * b + r;
      const long long tok = t0 + t;
      if (p.y_out != nullptr) {
        p.y_out[tok * N + hh * D + e] = hlo;
        p.y_out[tok * N + hh * D + D / 2 + e] = hhi;
        continue;
      }
      const QkvSlot ts = slots[t];
      if (ts.k_off < 0) continue;
      __half olo = hlo, ohi = hhi;
      if (hh < p.hq + p.hkv) {
        float ra, rb;
        rope_pair(__half2float(hlo), __half2float(hhi), cs[t][r], ra, rb);
        olo = __float2half_rn(ra);
        ohi = __float2half_rn(rb);
      }
      __half* dst = hh < p.hq ? p.q_out + (tok * p.hq + hh) * D
                              : p.pool + ts.k_off + (long long)(hh - p.hq) * kPageSize * D;  // K or V block
      dst[e] = olo;
      dst[D / 2 + e] = ohi;
    }
    __syncthreads();
  }
}

template <int D, int kTok>
__global__ void __launch_bounds__(256, kTok == 1 ? 3 : 2) qkv_append_kernel(QkvParams p) {
  extern __shared__ __align__(16) unsigned char smem[];
  __half* xs = reinterpret_cast<__half*>(smem);                       // [kTok][hidden], pair order
  float* red = reinterpret_cast<float*>(smem + (size_t)kTok * p.hidden * 2);  // [parts][kTok][16]
  __shared__ QkvSlot slots[kTokMax];
  __shared__ float2 cs[kTokMax][8];  // (cos, sin) of elements 8b .. 8b + 7 at each token's position
  pdl_launch_dependents();

  const int lane = threadIdx.x & 31;
  const int parts = blockDim.x >> 6;                 // warps per row half
  const int half = (threadIdx.x >> 5) / parts;       // 0: rows 8b + i, 1: rows D/2 + 8b + i
  const int warp = (threadIdx.x >> 5) - half * parts;  // input part
  const int blocks_per_head = D / 16;
  const int hh = blockIdx.x / blocks_per_head;  // head among q, k, v heads
  const int b = blockIdx.x - hh * blocks_per_head;
  const int N = (p.hq + 2 * p.hkv) * D;
  const int words = p.hidden / 8, groups = p.hidden / 32;
  const int group = warp * 32 + lane;  // this lane's 32 inputs
  const bool active = group < groups;

  // this warp's rows: hh * D + half * D/2 + 8b + r, r < 8
  const long long row0 = (long long)hh * D + half * (D / 2) + 8 * b;

  // weights and scales of the 8 rows: inputs of the weights, no wait needed
  uint4 wv[8];
  uint32_t sc2[8];  // the row's scale as an fp16 pair
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const long long row = row0 + r;
    if (active) {
      wv[r] = *reinterpret_cast<const uint4*>(p.w + row * words + group * 4);
      const uint32_t h = __half_as_ushort(p.scales[row * groups + group]);
      sc2[r] = h | (h << 16);
    } else {
      wv[r] = make_uint4(0, 0, 0, 0);
      sc2[r] = 0u;
    }
  }
  // token t -> sequence -> page slot, into slots[i] (the append kernel's checks)
  auto lookup_slot = [&](int t, int i) {
    QkvSlot ts{-1, 0};
    if (t < p.num_tokens && p.pool != nullptr) {
      int lo = 0, hi = p.batch;
      if (p.append_indptr[0] <= t && t < p.append_indptr[p.batch]) {
        while (hi - lo > 1) {
          const int mid = (lo + hi) >> 1;
          if (p.append_indptr[mid] <= t) lo = mid; else hi = mid;
        }
        const int pos = p.pos_map[t];
        const int first = p.page_indptr[lo];
        const int n_pages = p.page_indptr[lo + 1] - first;
        if (pos < 0 || pos >= p.max_position || (pos >> 4) >= n_pages) {
          atomicOr(p.status, kFlagBadPosition);
        } else {
          const int page = p.page_indices[first + (pos >> 4)];
          if (page < 0 || page >= p.num_pages) {
            atomicOr(p.status, kFlagBadPage);
          } else {
            ts.k_off = ((long long)page * 2 * p.hkv * kPageSize + (pos & 15)) * D;
            ts.pos = pos;
#pragma unroll
            for (int e = 0; e < 8; ++e) cs[i][e] = p.rope[(long long)pos * (D / 2) + 8 * b + e];
          }
        }
      } else {
        atomicOr(p.status, kFlagBadSequence);
      }
    }
    slots[i] = ts;
  };
  if (threadIdx.x < kTok) lookup_slot(threadIdx.x, threadIdx.x);  // the first tokens, before the wait
  pdl_wait();  // the input rows and the pool may come from the preceding kernel

  for (int t0 = 0; t0 < p.num_tokens; t0 += kTok) {
    const int nt = min(kTok, p.num_tokens - t0);
    // the tokens' input rows, each word's eight values stored as the pairs {j, j+4}
    for (int i = threadIdx.x; i < nt * words; i += blockDim.x) {
      const int t = i / words, m = i - t * words;
      const uint4 v = *reinterpret_cast<const uint4*>(p.x + (long long)(t0 + t) * p.hidden + 8 * m);
      const uint32_t e[4] = {v.x, v.y, v.z, v.w};  // pairs (0,1), (2,3), (4,5), (6,7)
      uint4 o;
      o.x = __byte_perm(e[0], e[2], 0x5410);  // {x0, x4}
      o.y = __byte_perm(e[0], e[2], 0x7632);  // {x1, x5}
      o.z = __byte_perm(e[1], e[3], 0x5410);  // {x2, x6}
      o.w = __byte_perm(e[1], e[3], 0x7632);  // {x3, x7}
      *reinterpret_cast<uint4*>(xs + (size_t)t * p.hidden + 8 * m) = o;
    }
    if (t0 > 0 && threadIdx.x < kTok) lookup_slot(t0 + threadIdx.x, threadIdx.x);
    __syncthreads();

    // partial sums: acc[r][t] over this lane's 32 inputs, then over the warp
    float acc[8][kTok];
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
      for (int t = 0; t < kTok; ++t) acc[r][t] = 0.f;
    if (active) {
      // the lane's 32 inputs of each token (four words' worth, in pair order)
      uint4 xw[kTok][4];
#pragma unroll
      for (int t = 0; t < kTok; ++t)
#pragma unroll
        for (int q = 0; q < 4; ++q)
          xw[t][q] = t < nt ? *reinterpret_cast<const uint4*>(xs + (size_t)t * p.hidden + 32 * group + 8 * q)
                            : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int r = 0; r < 8; ++r) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t word = q == 0 ? wv[r].x : q == 1 ? wv[r].y : q == 2 ? wv[r].z : wv[r].w;
          uint32_t wp[4];
          dequant_word(word, sc2[r], wp);
#pragma unroll
          for (int t = 0; t < kTok; ++t) {
            float a = acc[r][t];
            a = fma2(wp[0], xw[t][q].x, a);
            a = fma2(wp[1], xw[t][q].y, a);
            a = fma2(wp[2], xw[t][q].z, a);
            a = fma2(wp[3], xw[t][q].w, a);
            acc[r][t] = a;
          }
        }
      }
    }
    // transposing butterfly: after it lanes 4r .. 4r + 3 hold row r summed over the warp
#pragma unroll
    for (int t = 0; t < kTok; ++t) {
      if (t < nt) {
        const float sum = reduce8<kTok>(acc, t, lane);
        if ((lane & 3) == 0) red[(warp * kTok + t) * 16 + 8 * half + ((lane >> 2) & 7)] = sum;
      }
    }
    __syncthreads();

    // the projection (fp16), then RoPE and the append for the CTA's rows
    for (int i = threadIdx.x; i < nt * 8; i += blockDim.x) {
      const int t = i >> 3, r = i & 7;
      float ylo = 0.f, yhi = 0.f;
      for (int w = 0; w < parts; ++w) {
        ylo += red[(w * kTok + t) * 16 + r];
        yhi += red[(w * kTok + t) * 16 + 8 + r];
      }
      const __half hlo = __float2half_rn(ylo), hhi = __float2half_rn(yhi);
      const int e = 8 * b + r;  // element of the head's first half
      const long long tok = t0 + t;
      if (p.y_out != nullptr) {
        p.y_out[tok * N + hh * D + e] = hlo;
        p.y_out[tok * N + hh * D + D / 2 + e] = hhi;
        continue;
      }
      const QkvSlot ts = slots[t];
      if (ts.k_off < 0) continue;
      __half olo = hlo, ohi = hhi;
      if (hh < p.hq + p.hkv) {
        // rotate-half RoPE of the pair (e, e + D/2) at the token's position
        float ra, rb;
        rope_pair(__half2float(hlo), __half2float(hhi), cs[t][r], ra, rb);
        olo = __float2half_rn(ra);
        ohi = __float2half_rn(rb);
      }
      __half* dst;
      if (hh < p.hq) {
        dst = p.q_out + (tok * p.hq + hh) * D;
      } else if (hh < p.hq + p.hkv) {
        dst = p.pool + ts.k_off + (long long)(hh - p.hq) * kPageSize * D;  // K block of head hh - hq
      } else {
        dst = p.pool + ts.k_off + (long long)(hh - p.hq) * kPageSize * D;  // V block: (hkv + g) blocks in
      }
      dst[e] = olo;
      dst[D / 2 + e] = ohi;
    }
    __syncthreads();
  }
}

}  // namespace

cudaError_t qkv_prepare() {
  const void* k[] = {(const void*)&qkv_append_kernel<64, 1>, (const void*)&qkv_append_kernel<96, 1>,
                     (const void*)&qkv_append_kernel<128, 1>};
  for (const void* f : k) {
    cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, kQkvMaxSmem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
  }
  const void* km[] = {(const void*)&qkv_mma_kernel<64, 1>, (const void*)&qkv_mma_kernel<96, 1>,
                      (const void*)&qkv_mma_kernel<128, 1>, (const void*)&qkv_mma_kernel<64, 2>,
                      (const void*)&qkv_mma_kernel<96, 2>, (const void*)&qkv_mma_kernel<128, 2>,
                      (const void*)&qkv_mma_kernel<64, 4>, (const void*)&qkv_mma_kernel<96, 4>,
                      (const void*)&qkv_mma_kernel<128, 4>};
  for (const void* f : km) {
    // at most QkvMmaSmem<4>::bytes(4096) (~53 KB); the kernel's static shared memory comes on top
    cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, 64 * 1024);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

size_t qkv_smem_bytes(int hidden, int parts, int tok) {
  return (size_t)tok * hidden * 2 + (size_t)parts * tok * 16 * sizeof(float);
}

cudaError_t launch_qkv(const QkvParams& p, cudaStream_t stream, bool pdl) {
  if (p.num_tokens <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((p.hq + 2 * p.hkv) * (p.head_dim / 16)));
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (p.num_tokens == 1) {
    // one token: the CUDA-core kernel (every weight is used once; nothing to share across tokens)
    const int parts = (p.hidden + kPartIn - 1) / kPartIn;
    cfg.blockDim = dim3(64 * parts);
    cfg.dynamicSmemBytes = qkv_smem_bytes(p.hidden, parts, 1);
    switch (p.head_dim) {
      case 64: return cudaLaunchKernelEx(&cfg, qkv_append_kernel<64, 1>, p);
      case 96: return cudaLaunchKernelEx(&cfg, qkv_append_kernel<96, 1>, p);
      case 128: return cudaLaunchKernelEx(&cfg, qkv_append_kernel<128, 1>, p);
      default: return cudaErrorInvalidValue;
    }
  }
  // several tokens: tensor cores, 8, 16 or 32 tokens per pass
  cfg.blockDim = dim3(kMmaWarps * 32);
  const int nt = p.num_tokens <= 8 ? 1 : p.num_tokens <= 16 ? 2 : 4;
  cfg.dynamicSmemBytes = nt == 1 ? QkvMmaSmem<1>::bytes(p.hidden) : nt == 2 ? QkvMmaSmem<2>::bytes(p.hidden)
                                                                            : QkvMmaSmem<4>::bytes(p.hidden);
  auto pick = [&](auto k1, auto k2, auto k4) {
    return nt == 1 ? cudaLaunchKernelEx(&cfg, k1, p) : nt == 2 ? cudaLaunchKernelEx(&cfg, k2, p)
                                                               : cudaLaunchKernelEx(&cfg, k4, p);
  };
  switch (p.head_dim) {
    case 64: return pick(qkv_mma_kernel<64, 1>, qkv_mma_kernel<64, 2>, qkv_mma_kernel<64, 4>);
    case 96: return pick(qkv_mma_kernel<96, 1>, qkv_mma_kernel<96, 2>, qkv_mma_kernel<96, 4>);
    case 128: return pick(qkv_mma_kernel<128, 1>, qkv_mma_kernel<128, 2>, qkv_mma_kernel<128, 4>);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pkv
