// Split-K partial attention over paged KV (Zero TVM Documentation, "How it works": attention
// split over KV chunks, then a combine; "KV cache": 16-slot pages behind a page table; "Port to
// Phi-4-mini or Qwen3": query head h reads KV head h / (Hq / Hkv)).
//
// Work decomposition.  A work item is (sequence s, chunk j, KV head g): the pages
// [j*c, min((j+1)*c, n_s)) of s for one KV head and all G = Hq/Hkv query heads that read it, so
// every KV page is fetched once per KV head; with the exact page total the chunks are the pieces
// of a page-balanced partition instead.  Items are enumerated sequence-major through a prefix sum
// of items per sequence that each CTA builds in shared memory from page_indptr.  The grid is
// persistent (one or two CTAs per SM); every warp owns items gw, gw + W, gw + 2W, ... (W = warps
// in the grid) or one run of the balanced partition, and works alone: no CTA-wide barrier after
// the prologue.
//
// Memory pipeline.  Each warp has a private ring of `nstage` shared-memory stages.  Lane 0 is the
// producer: for each page it issues the copies of the page's K and V blocks of one KV head (two
// plain bulk copies on the CUDA-core path, swizzled 4-D tensor boxes on the tensor-core path),
// plus, with the first page of an item, a bulk copy of the item's G query rows into one of two
// per-warp item slots, all completing on the stage's mbarrier.  The same warp consumes stages in
// order and refills the ring at the top of its loop, so nstage pages per warp are in flight.
// Per-stage metadata (sequence, chunk, head, valid slots, first/last flags) travels through shared
// memory with the barrier's release/acquire order.
//
// Compute.  G = 1 runs on CUDA cores: a half-warp covers one 16-slot row pair, each lane owns
// head_dim/16 dimensions; q.k partials of 8 rows are reduced with a transposing butterfly (one
// shuffle per row), the online softmax runs in the log2 domain, and P.V reuses the lane's
// dimensions.  G >= 2 runs q.K^T and P.V on tensor cores with mma.sync m16n8k16 (fp16 in, fp32
// accumulate): the G query heads are rows of A (padded to 16), the 16 slots of a page are two
// n-blocks, and the score accumulators are re-used directly as the A operand of P.V.  K/V boxes
// use the 128-byte (64-byte for head_dim 96) TMA swizzle so the ldmatrix row reads are free of
// bank conflicts.  An int8 cache (template flag Q8) stages two pages of an item per stage and
// computes from the codes: on CUDA cores with the fp16 arrangement for G = 1 (GroupOneQ8), on
// tensor cores with the page's slots as the MMA rows for G >= 2 (GroupQ8).  The CUDA-core path
// has a wide form (template flag WIDE: 12 warps per SM, at most 168 registers) for large batches.
//
// One-launch mode (template flag FUSED) also performs the append of a decode step: the first
// stage of an item brings the new token's raw k and v and its (cos, sin) row, the consumer
// rotates q and k there, and the staged copy of the page that holds the token is patched (and the
// pool written) before it is used.
//
// Every wait is bounded (2 s of global time unless pkv_set_wait_limit sets another limit); on
// expiry the warp flags PKV_FLAG_TIMEOUT, waits a fixed bounded time for its own copies in flight
// (so none lands in the shared memory of a finished block) and returns.  The test setting
// pkv_set_stage_stall makes every stage's phase wait for an arrival that nothing makes, so that
// the waits run out on a healthy GPU.
#include <algorithm>

#include "merge.cuh"
#include "pkv_internal.h"
#include "ptx.cuh"
#include "rope.cuh"

namespace pkv {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLazyRescale = 8.f;  // raise the running max only when a score exceeds it by 2^8

constexpr int kMetaValid = 0x1f;
constexpr int kMetaFirst = 1 << 5;
constexpr int kMetaLast = 1 << 6;
constexpr int kMetaLastChunk = 1 << 7;
constexpr int kMetaEmpty = 1 << 8;
constexpr int kMetaNew = 1 << 9;     // one-launch mode: the stage also carries the new token's k and v
constexpr int kMetaPatch = 1 << 10;  // one-launch mode: the page holds the new token (slot in bits 11..14)
constexpr int kMetaSlotShift = 11;
constexpr int kMetaValid2Shift = 9;  // int8 cache (never one-launch): valid slots of the stage's second page
constexpr int kMetaChunkShift = 16;  // bits 16..31: chunks of the item's sequence

// Stage metadata: sequence, chunk, KV head and (low half of gl's high bits) the first attended slot
// of the page (a sliding window's start inside its first visible page), flags.
struct __align__(16) StageMeta {
  int s, j, gl, flags;
  __device__ int g() const { return gl & 0xffff; }
  __device__ int lo() const { return gl >> 16; }
};

// Dynamic shared memory budget: the 227 KB per-block opt-in maximum less room for the kernel's
// static shared memory (128 bytes).
constexpr int kSmemBudget = 232448 - 256;

// Shared memory of one SM, and the CTAs per SM the decode grid prefers.
constexpr int kSmemPerSm = 233472;
constexpr int kCtasPerSm = 2;

// Alignment of the shared-memory base: 1024 bytes on the tensor-core path (its swizzled boxes), 128
// bytes on the CUDA-core path.  The kernel aligns its base by the same rule and the layout reserves
// that much slack.
__host__ __device__ constexpr bool uses_mma(int group, bool q8) {
  (void)q8;  // an int8 cache takes the same path as an fp16 one: tensor cores for G >= 2
  return group >= 2;
}
__host__ __device__ constexpr int smem_align(bool mma) { return mma ? 1024 : 128; }

struct Layout {
  int stage_bytes, ring_off, qslot_bytes, q_off, patch_off, bar_off, meta_off, pid_off, defer_off, prefix_off,
      indptr_off, aptr_off, wstart_off, total;
};

// Items whose query rows may be in flight at once, per warp (one item slot each).
constexpr int kItemSlots = 2;

// Shared memory: the stage ring, then per warp kItemSlots item slots (the item's query rows;
// one-launch mode also the query position's (cos, sin) row and the new token's raw k and v rows)
// and (one-launch mode) the rotated K and V rows of the new token, the mbarriers, the stage
// metadata, (one-launch mode) the page id of each stage, and per sequence the work prefix, the
// page ranges, (one-launch mode) the new-token ranges and (sliding window) the first visible page
// and its first attended slot.
__host__ __device__ inline Layout make_layout(int warps, int nstage, int head_dim, int group, int batch,
                                              bool fused, bool windowed = false, bool q8 = false) {
  Layout L;
  const int n = warps * nstage;
  // K and V of one page for one KV head (int8 cache: the two int8 blocks as stored, of two pages)
  L.stage_bytes = q8 ? 4 * int8_block_bytes(head_dim) : 64 * head_dim;
  L.ring_off = 0;
  L.qslot_bytes = (group * head_dim * 2 + (fused ? 8 * head_dim : 0) + 15) & ~15;
  L.q_off = L.ring_off + n * L.stage_bytes;
  L.patch_off = L.q_off + warps * kItemSlots * L.qslot_bytes;
  L.bar_off = L.patch_off + (fused ? warps * 4 * head_dim : 0);
  L.meta_off = L.bar_off + n * 8;
  L.meta_off = (L.meta_off + 15) & ~15;
  L.pid_off = L.meta_off + n * 16;
  L.defer_off = (L.pid_off + (fused ? n * 4 : 0) + 15) & ~15;  // 16-byte entries are stored as vectors
  L.prefix_off = L.defer_off + (fused ? n * 32 : 0);
  L.indptr_off = L.prefix_off + (batch + 1) * 4;
  L.aptr_off = L.indptr_off + (batch + 1) * 4;
  L.wstart_off = L.aptr_off + (fused ? (batch + 1) * 4 : 0);
  L.total = L.wstart_off + (windowed ? batch * 4 : 0) + smem_align(uses_mma(group, q8));  // + slack to align the base
  return L;
}

// Rotated element i of a head row x (rotate-half RoPE with the row's (cos, sin) table cs), with
// the same fp32 operations and rounding order as the append kernel.
template <int D>
__device__ __forceinline__ float rope_element(const __half* x, const float2* cs, int i) {
  if (i < D / 2) {
    const float a = __half2float(x[i]), b = __half2float(x[i + D / 2]);
    return __fmaf_rn(a, cs[i].x, -__fmul_rn(b, cs[i].y));
  }
  const int ii = i - D / 2;
  const float a = __half2float(x[ii]), b = __half2float(x[i]);
  return __fmaf_rn(b, cs[ii].x, __fmul_rn(a, cs[ii].y));
}

// Chunks of a sequence with n pages; c receives the chunk size.  Returns 0 for an invalid n.
__device__ __forceinline__ int seq_chunks(const DecodeParams& p, int n, int& c) {
  if (n < 0 || n > p.max_pages) return 0;
  if (n == 0) {
    c = 1;
    return 1;
  }
  c = p.chunk_pages > 0 ? p.chunk_pages : (n + p.splits - 1) / p.splits;
  const int nch = (n + c - 1) / c;
  return nch <= p.splits ? nch : 0;
}

// ------------------------------------------------------------------------------------------------
// CUDA-core compute for one query head per KV head.

template <int D>
struct GroupOne {
  static constexpr int DPL = D / 16;  // dimensions per lane
  static constexpr int HPL = DPL / 2; // half2 pairs per lane
  uint32_t q2[HPL];                   // the lane's query dimensions, fp16 pairs
  float o[DPL], m, l, scale_log2;
  int lane, half, li;

  __device__ void init(int lane_) {
    lane = lane_;
    half = lane >> 4;
    li = lane & 15;
  }

  // Shared-memory address of 16-byte chunk c (elements 8c..8c+7) of row t of K (kv 0) or V (kv 1).
  __device__ static uint32_t row_chunk(uint32_t stage, int kv, int t, int c) {
    return stage + (uint32_t)((kv * kPageSize + t) * D * 2 + 16 * c);
  }

  // The lane's DPL consecutive fp16 values of a row, as half2 pairs.
  __device__ static void load_row(const unsigned char* row, int li, uint32_t (&x)[HPL]) {
    if constexpr (D == 128) {
      const uint4 v = *reinterpret_cast<const uint4*>(row + li * 16);
      x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
    } else if constexpr (D == 96) {
      const uint32_t* b = reinterpret_cast<const uint32_t*>(row + li * 12);
      x[0] = b[0]; x[1] = b[1]; x[2] = b[2];
    } else {
      const uint2 v = *reinterpret_cast<const uint2*>(row + li * 8);
      x[0] = v.x; x[1] = v.y;
    }
  }

  // acc + a.lo * b.lo + a.hi * b.hi with fp16 operands and fp32 accumulation (the fp16 products
  // are exact in fp32, so this equals converting first and using fp32 fused multiply-adds).
  __device__ static float fma2(uint32_t a, uint32_t b, float acc) {
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
        "mov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.f16 %0, al, bl, %0;\n\tfma.rn.f32.f16 %0, ah, bh, %0;\n\t}"
        : "+f"(acc) : "r"(a), "r"(b));
    return acc;
  }

  // o + p * v for both halves of v (p already an fp16 value held in the low half of pp).
  __device__ static void fma_pv(uint16_t p16, uint32_t v, float& o0, float& o1) {
    asm("{\n\t.reg .b16 vl, vh;\n\t"
        "mov.b32 {vl, vh}, %2;\n\t"
        "fma.rn.f32.f16 %0, %3, vl, %0;\n\tfma.rn.f32.f16 %1, %3, vh, %1;\n\t}"
        : "+f"(o0), "+f"(o1) : "r"(v), "h"(p16));
  }

  // Fused mode: rotate the raw query row in the slot with the (cos, sin) row that follows it.
  __device__ void begin_rotate(const unsigned char* qslot, float scale_log2_) {
    const __half* x = reinterpret_cast<const __half*>(qslot);
    const float2* cs = reinterpret_cast<const float2*>(qslot + D * 2);
#pragma unroll
    for (int e = 0; e < HPL; ++e) {
      const int i = li * DPL + 2 * e;
      const __half2 h = __floats2half2_rn(rope_element<D>(x, cs, i), rope_element<D>(x, cs, i + 1));
      q2[e] = *reinterpret_cast<const uint32_t*>(&h);
    }
#pragma unroll
    for (int e = 0; e < DPL; ++e) o[e] = 0.f;
    m = -INFINITY;
    l = 0.f;
    scale_log2 = scale_log2_;
  }

  // Store the rotated query (fused mode) as the q_out row of head `row` of the query token.
  __device__ void store_query(__half* q_out_row) const {
    if (half == 0) {
      uint32_t* dst = reinterpret_cast<uint32_t*>(q_out_row + li * DPL);
#pragma unroll
      for (int e = 0; e < HPL; ++e) dst[e] = q2[e];
    }
  }

  __device__ void begin(const unsigned char* qslot, float scale_log2_) {
    load_row(qslot, li, q2);
#pragma unroll
    for (int e = 0; e < DPL; ++e) o[e] = 0.f;
    m = -INFINITY;
    l = 0.f;
    scale_log2 = scale_log2_;
  }

  // q.k partial of the lane's 8 rows of one page.
  __device__ void dots(const unsigned char* Kb, float (&acc)[8]) const {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      uint32_t x[HPL];
      load_row(Kb + (2 * i + half) * D * 2, li, x);
      float a = 0.f;
#pragma unroll
      for (int e = 0; e < HPL; ++e) a = fma2(q2[e], x[e], a);
      acc[i] = a;
    }
  }

  // Transposing butterfly over the 16 lanes of each half for NP pages (8*NP row partials per
  // lane): halving exchanges at xor 8, 4, 2 leave NP values per lane, the row pair-sums of rows
  // 2*(li>>1)+half of each page; the xor-1 exchange completes them.
  template <int NP>
  __device__ void reduce_rows(float (&acc)[8 * NP], float (&sc)[NP]) const {
    const bool b3 = li & 8, b2 = li & 4, b1 = li & 2;
    constexpr int N = 8 * NP;
    float t4[N / 2];
#pragma unroll
    for (int a = 0; a < N / 2; ++a) {
      // the kept half alternates in blocks of 4 so each page keeps its own rows
      const int lo = (a / 4) * 8 + (a % 4), hi = lo + 4;
      const float send = b3 ? acc[lo] : acc[hi];
      const float keep = b3 ? acc[hi] : acc[lo];
      t4[a] = keep + __shfl_xor_sync(kFull, send, 8);
    }
    float t2[N / 4];
#pragma unroll
    for (int a = 0; a < N / 4; ++a) {
      const int lo = (a / 2) * 4 + (a % 2), hi = lo + 2;
      const float send = b2 ? t4[lo] : t4[hi];
      const float keep = b2 ? t4[hi] : t4[lo];
      t2[a] = keep + __shfl_xor_sync(kFull, send, 4);
    }
#pragma unroll
    for (int pg = 0; pg < NP; ++pg) {
      const float t1 = (b1 ? t2[2 * pg + 1] : t2[2 * pg]) +
                       __shfl_xor_sync(kFull, b1 ? t2[2 * pg] : t2[2 * pg + 1], 2);
      sc[pg] = (t1 + __shfl_xor_sync(kFull, t1, 1)) * scale_log2;
    }
  }

  // Online-softmax update for NP pages' scores (log2 domain).  The running max m is only raised,
  // with a warp-wide reduction and a rescale of o and l, when some score exceeds it by more than
  // 2^8; otherwise the page's probabilities exp2(s - m) stay below 256 and the stale max is kept
  // (the final normalisation by l makes the result independent of m).
  template <int NP>
  __device__ void softmax(float (&sc)[NP], uint16_t (&pbits)[NP]) {
    bool need = false;
#pragma unroll
    for (int pg = 0; pg < NP; ++pg) need |= sc[pg] > m + kLazyRescale;
    if (__any_sync(kFull, need)) {
      float mx = sc[0];
#pragma unroll
      for (int pg = 1; pg < NP; ++pg) mx = fmaxf(mx, sc[pg]);
      mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 16));
      mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 4));
      mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
      const float m_new = fmaxf(m, mx);
      const float alpha = exp2f(m - m_new);
      l *= alpha;
#pragma unroll
      for (int e = 0; e < DPL; ++e) o[e] *= alpha;
      m = m_new;
    }
    // probabilities rounded to fp16 for the P.V products; l sums the same rounded values
#pragma unroll
    for (int pg = 0; pg < NP; ++pg) {
      const __half pr16 = __float2half_rn(exp2f(sc[pg] - m));
      pbits[pg] = __half_as_ushort(pr16);
      l += (li & 1) ? 0.f : __half2float(pr16);
    }
  }

  // Slots past the sequence end may hold anything (even NaN): zero their V rows so that p = 0
  // times V adds exactly nothing.
  __device__ void zero_v_tail(unsigned char* Vb, int nvalid) const {
    if (nvalid < kPageSize) {
      constexpr int kChunksPerRow = D / 8;
      const int n = (kPageSize - nvalid) * kChunksPerRow;
      const uint32_t base = smem_u32(Vb + nvalid * D * 2);
      for (int i = lane; i < n; i += 32)
        asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(base + 16 * i), "r"(0u) : "memory");
      __syncwarp();
    }
  }

  __device__ void pv(const unsigned char* Vb, uint16_t pbits) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint16_t pi = (uint16_t)__shfl_sync(kFull, (uint32_t)pbits, (lane & 16) | (2 * i));
      uint32_t x[HPL];
      load_row(Vb + (2 * i + half) * D * 2, li, x);
#pragma unroll
      for (int e = 0; e < HPL; ++e) fma_pv(pi, x[e], o[2 * e], o[2 * e + 1]);
    }
  }

  // Rows outside [lo, nvalid) do not take part (lo: a sliding window's first slot, usually 0).
  __device__ float mask(float sc, int lo, int nvalid) const {
    const int row = 2 * ((li >> 1) & 7) + half;
    return (row >= lo && row < nvalid) ? sc : -INFINITY;
  }

  __device__ void page(unsigned char* stage, int lo, int nvalid) {
    zero_v_tail(stage + kPageSize * D * 2, nvalid);
    float acc[8];
    dots(stage, acc);
    float sc[1];
    reduce_rows<1>(acc, sc);
    sc[0] = mask(sc[0], lo, nvalid);
    uint16_t pb[1];
    softmax<1>(sc, pb);
    pv(stage + kPageSize * D * 2, pb[0]);
  }

  // Two consecutive pages of one item at once: independent q.k work for both, one softmax update.
  __device__ void page2(unsigned char* sa, int la, int na, unsigned char* sb, int nb) {
    zero_v_tail(sa + kPageSize * D * 2, na);
    zero_v_tail(sb + kPageSize * D * 2, nb);
    float acc[16];
    float (&a0)[8] = *reinterpret_cast<float(*)[8]>(&acc[0]);
    float (&a1)[8] = *reinterpret_cast<float(*)[8]>(&acc[8]);
    dots(sa, a0);
    dots(sb, a1);
    float sc[2];
    reduce_rows<2>(acc, sc);
    sc[0] = mask(sc[0], la, na);
    sc[1] = mask(sc[1], 0, nb);
    uint16_t pb[2];
    softmax<2>(sc, pb);
    pv(sa + kPageSize * D * 2, pb[0]);
    pv(sb + kPageSize * D * 2, pb[1]);
  }

  // Writes the item's partial; returns false when nothing was accumulated.
  __device__ bool finish(float* po, float* pl, long long row_base, int S, int j) {
    float lt = l;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) lt += __shfl_xor_sync(kFull, lt, off);
#pragma unroll
    for (int e = 0; e < DPL; ++e) o[e] += __shfl_xor_sync(kFull, o[e], 16);
    if (!(lt > 0.f)) return false;
    const float inv = 1.f / lt;
    if (half == 0) {
      float* dst = po + (row_base * S + j) * D + li * DPL;
#pragma unroll
      for (int e = 0; e < DPL; ++e) dst[e] = o[e] * inv;
    }
    if (lane == 0) pl[row_base * S + j] = (m + log2f(lt)) * kLn2;
    return true;
  }

  // The item is its sequence's only chunk: write the final output (the merge of one split gives
  // the same bits, since its weight is exactly 1).
  __device__ void finish_out(__half* out, float* lse_out, long long row) {
    float lt = l;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) lt += __shfl_xor_sync(kFull, lt, off);
#pragma unroll
    for (int e = 0; e < DPL; ++e) o[e] += __shfl_xor_sync(kFull, o[e], 16);
    const bool any = lt > 0.f;
    const float inv = any ? 1.f / lt : 0.f;
    if (half == 0) {
      __half* dst = out + row * D + li * DPL;
#pragma unroll
      for (int e = 0; e < DPL; ++e) dst[e] = __float2half_rn(any ? o[e] * inv : 0.f);
    }
    if (lse_out != nullptr && lane == 0) lse_out[row] = any ? (m + log2f(lt)) * kLn2 : -INFINITY;
  }
};

// ------------------------------------------------------------------------------------------------
// int8 cache, one query head per KV head, on CUDA cores: GroupOne's arrangement over the codes.
// q.k: a half-warp covers one key row, each lane D/16 dimensions; the lane's codes of the row (the
// stored bytes, code + 128) become exact fp16 values (byte in the mantissa of 1024, minus 1152) and
// meet the query in fp16 x fp16 -> fp32 fused multiply-adds; the transposing butterfly leaves each
// lane one row's sum, which takes the row's K scale.  P V: each half-warp takes eight of the
// page's slots, each lane D/16 dimensions, whose eight codes are one 8-byte run of the dim-major V
// block; the probabilities carry the V scales relative to a lazily raised reference (as in the
// tensor-core int8 form), and the two halves' sums are added at the end.  A stage holds one or two
// pages of the item.
template <int D>
struct GroupOneQ8 : GroupOne<D> {
  using Base = GroupOne<D>;
  using Base::DPL;
  using Base::HPL;
  static constexpr int kBlk = int8_block_bytes(D);
  float vref, vinv;

  // Four stored bytes -> their codes as fp16 pairs: bytes 0, 1 in lo, bytes 2, 3 in hi.
  __device__ static void codes_to_half(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const __half2 bias = __half2half2(__ushort_as_half((unsigned short)0x6480));  // 1152
    const uint32_t a = __byte_perm(w, 0x64646464u, 0x5140), b = __byte_perm(w, 0x64646464u, 0x5342);
    const __half2 x = __hsub2(*reinterpret_cast<const __half2*>(&a), bias);
    const __half2 y = __hsub2(*reinterpret_cast<const __half2*>(&b), bias);
    lo = *reinterpret_cast<const uint32_t*>(&x);
    hi = *reinterpret_cast<const uint32_t*>(&y);
  }

  __device__ void begin8(const unsigned char* qslot) {
    Base::load_row(qslot, this->li, this->q2);
#pragma unroll
    for (int e = 0; e < DPL; ++e) this->o[e] = 0.f;
    this->m = -1e30f;  // a finite floor: a fully masked page gives exp2(-inf) = 0
    this->l = 0.f;
    vref = 0.f;
    vinv = 0.f;
  }

  // The lane's D/16 codes of a key row as fp16 pairs.
  __device__ void row_codes(const unsigned char* row, uint32_t (&x)[HPL]) const {
    const unsigned char* src = row + this->li * DPL;
    if constexpr (D == 128) {
      const uint2 w = *reinterpret_cast<const uint2*>(src);
      codes_to_half(w.x, x[0], x[1]);
      codes_to_half(w.y, x[2], x[3]);
    } else if constexpr (D == 96) {
      const uint16_t* h = reinterpret_cast<const uint16_t*>(src);
      const uint32_t w0 = (uint32_t)h[0] | ((uint32_t)h[1] << 16), w1 = (uint32_t)h[2];
      uint32_t unused;
      codes_to_half(w0, x[0], x[1]);
      codes_to_half(w1, x[2], unused);
    } else {
      codes_to_half(*reinterpret_cast<const uint32_t*>(src), x[0], x[1]);
    }
  }

  template <int NP>
  __device__ void page8(const unsigned char* stage, int lo, int nv0, int nv1, float scale_log2) {
    const int half = this->half, li = this->li;
    this->scale_log2 = scale_log2;  // the butterfly's scaling of the row sums
    // q.k partials of the lane's 8 rows of each page, then the rows' sums (log2 domain)
    float acc[8 * NP];
#pragma unroll
    for (int pg = 0; pg < NP; ++pg) {
      const unsigned char* kb = stage + pg * 2 * kBlk;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        uint32_t x[HPL];
        row_codes(kb + (2 * i + half) * D, x);
        float a = 0.f;
#pragma unroll
        for (int e = 0; e < HPL; ++e) a = Base::fma2(this->q2[e], x[e], a);
        acc[8 * pg + i] = a;
      }
    }
    float sc[NP];
    this->template reduce_rows<NP>(acc, sc);
    const int row = 2 * ((li >> 1) & 7) + half;  // the row this lane holds
    bool valid[NP];
    float v[NP];
    bool need = false, vneed = false;
#pragma unroll
    for (int pg = 0; pg < NP; ++pg) {
      const unsigned char* kb = stage + pg * 2 * kBlk;
      const float* ksc = reinterpret_cast<const float*>(kb + 16 * D);
      const float* vsc = reinterpret_cast<const float*>(kb + kBlk + 16 * D);
      valid[pg] = row >= (pg == 0 ? lo : 0) && row < (pg == 0 ? nv0 : nv1);
      sc[pg] = valid[pg] ? sc[pg] * ksc[row] : -INFINITY;
      v[pg] = valid[pg] ? vsc[row] : 0.f;
      need |= sc[pg] > this->m + kLazyRescale;
      vneed |= v[pg] > vref * 128.f;
    }
    // the running max, raised (with a rescale) only when a score exceeds it by more than 2^8
    if (__any_sync(kFull, need)) {
      float mx = sc[0];
#pragma unroll
      for (int pg = 1; pg < NP; ++pg) mx = fmaxf(mx, sc[pg]);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, off));
      if (mx > this->m + kLazyRescale) {
        const float alpha = exp2f(this->m - mx);
        this->l *= alpha;
#pragma unroll
        for (int e = 0; e < DPL; ++e) this->o[e] *= alpha;
        this->m = mx;
      }
    }
    // the V-scale reference, raised only when a scale exceeds it by more than 2^7
    if (__any_sync(kFull, vneed)) {
      float vm = v[0];
#pragma unroll
      for (int pg = 1; pg < NP; ++pg) vm = fmaxf(vm, v[pg]);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) vm = fmaxf(vm, __shfl_xor_sync(kFull, vm, off));
      if (vm > vref * 128.f) {
        const float alpha = vref / vm;
#pragma unroll
        for (int e = 0; e < DPL; ++e) this->o[e] *= alpha;
        vref = vm;
        vinv = 1.f / vm;
      }
    }
#pragma unroll
    for (int pg = 0; pg < NP; ++pg) {
      const float ex = exp2f(sc[pg] - this->m);
      // the row sum adds the fp16-rounded probability (each row sits in two lanes)
      this->l += (li & 1) ? 0.f : __half2float(__float2half_rn(ex));
      const uint32_t pbits = (uint32_t)__half_as_ushort(__float2half_rn(ex * (v[pg] * vinv)));
      // this half-warp's slots 8 half + k come from the lanes holding those rows
      uint32_t pk[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int s0 = 8 * half + 2 * k;  // slots s0 (even) and s0 + 1 (odd)
        const uint32_t a = __shfl_sync(kFull, pbits, 2 * (s0 >> 1));
        const uint32_t b = __shfl_sync(kFull, pbits, 16 + 2 * (s0 >> 1));
        pk[k] = a | (b << 16);
      }
      const unsigned char* vb = stage + pg * 2 * kBlk + kBlk;
#pragma unroll
      for (int e = 0; e < DPL; ++e) {
        const uint2 w = *reinterpret_cast<const uint2*>(vb + (li * DPL + e) * 16 + 8 * half);
        uint32_t c01, c23, c45, c67;
        codes_to_half(w.x, c01, c23);
        codes_to_half(w.y, c45, c67);
        float a = this->o[e];
        a = Base::fma2(pk[0], c01, a);
        a = Base::fma2(pk[1], c23, a);
        a = Base::fma2(pk[2], c45, a);
        a = Base::fma2(pk[3], c67, a);
        this->o[e] = a;
      }
    }
  }

  __device__ bool finish(float* po, float* pl, long long row_base, int S, int j) {
    float lt = this->l;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) lt += __shfl_xor_sync(kFull, lt, off);
#pragma unroll
    for (int e = 0; e < DPL; ++e) this->o[e] += __shfl_xor_sync(kFull, this->o[e], 16);
    if (!(lt > 0.f)) return false;
    const float inv = (vref > 0.f ? vref : 1.f) / lt;
    if (this->half == 0) {
      float* dst = po + (row_base * S + j) * D + this->li * DPL;
#pragma unroll
      for (int e = 0; e < DPL; ++e) dst[e] = this->o[e] * inv;
    }
    if (this->lane == 0) pl[row_base * S + j] = (this->m + log2f(lt)) * kLn2;
    return true;
  }

  __device__ void finish_out(__half* out, float* lse_out, long long row) {
    float lt = this->l;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) lt += __shfl_xor_sync(kFull, lt, off);
#pragma unroll
    for (int e = 0; e < DPL; ++e) this->o[e] += __shfl_xor_sync(kFull, this->o[e], 16);
    const bool any = lt > 0.f;
    const float inv = any ? (vref > 0.f ? vref : 1.f) / lt : 0.f;
    if (this->half == 0) {
      __half* dst = out + row * D + this->li * DPL;
#pragma unroll
      for (int e = 0; e < DPL; ++e) dst[e] = __float2half_rn(any ? this->o[e] * inv : 0.f);
    }
    if (lse_out != nullptr && this->lane == 0) lse_out[row] = any ? (this->m + log2f(lt)) * kLn2 : -INFINITY;
  }
};

// ------------------------------------------------------------------------------------------------
// Tensor-core compute for a group of G in [2, 8] query heads per KV head.

template <int D>
struct GroupMma {
  static constexpr int E = (D == 96) ? 32 : 64;  // TMA box extent along head_dim
  static constexpr int REGION = 64 * E;          // bytes of one box: [2][16][E] fp16
  static constexpr int SWZ = (E == 64) ? 7 : 3;  // 128-byte or 64-byte swizzle
  static constexpr int KS = D / 16;              // k-steps of q.K^T
  static constexpr int NB = D / 8;               // n-blocks of P.V
  uint32_t qa[KS][2];
  float acc[NB][4];
  float m, l;
  int lane, h, group;

  __device__ void init(int lane_, int group_) {
    lane = lane_;
    h = lane >> 2;
    group = group_;
  }

  // Shared-memory address of the 16-byte chunk holding (kv, slot t, dims dim..dim+7).
  __device__ static uint32_t chunk_addr(uint32_t stage, int kv, int t, int dim) {
    const int u = dim / E;
    const uint32_t off = (uint32_t)((kv * kPageSize + t) * (E * 2) + (dim % E) * 2);
    return stage + u * REGION + (off ^ (((off >> 7) & SWZ) << 4));
  }

  __device__ static uint32_t row_chunk(uint32_t stage, int kv, int t, int c) { return chunk_addr(stage, kv, t, 8 * c); }

  // Fused mode: fragments of the rotated query rows (raw rows in the slot, then the (cos, sin) row).
  __device__ void begin_rotate(const unsigned char* qslot) {
    const int c = 2 * (lane & 3);
    const float2* cs = reinterpret_cast<const float2*>(qslot + group * D * 2);
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      if (h < group) {
        const __half* x = reinterpret_cast<const __half*>(qslot) + h * D;
        const int i = ks * 16 + c;
        const __half2 lo = __floats2half2_rn(rope_element<D>(x, cs, i), rope_element<D>(x, cs, i + 1));
        const __half2 hi = __floats2half2_rn(rope_element<D>(x, cs, i + 8), rope_element<D>(x, cs, i + 9));
        qa[ks][0] = *reinterpret_cast<const uint32_t*>(&lo);
        qa[ks][1] = *reinterpret_cast<const uint32_t*>(&hi);
      } else {
        qa[ks][0] = 0u;
        qa[ks][1] = 0u;
      }
    }
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) acc[nb][0] = acc[nb][1] = acc[nb][2] = acc[nb][3] = 0.f;
    m = -INFINITY;
    l = 0.f;
  }

  // Store the rotated query rows (fused mode): q_out_rows points at head g*G of the query token.
  __device__ void store_query(__half* q_out_rows) const {
    if (h < group) {
      const int c = 2 * (lane & 3);
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        uint32_t* dst = reinterpret_cast<uint32_t*>(q_out_rows + h * D + ks * 16 + c);
        dst[0] = qa[ks][0];
        dst[4] = qa[ks][1];
      }
    }
  }

  __device__ void begin(const unsigned char* qslot) {
    const int c = 2 * (lane & 3);
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      if (h < group) {
        const __half* qr = reinterpret_cast<const __half*>(qslot) + h * D + ks * 16 + c;
        qa[ks][0] = *reinterpret_cast<const uint32_t*>(qr);
        qa[ks][1] = *reinterpret_cast<const uint32_t*>(qr + 8);
      } else {
        qa[ks][0] = 0u;
        qa[ks][1] = 0u;
      }
    }
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) acc[nb][0] = acc[nb][1] = acc[nb][2] = acc[nb][3] = 0.f;
    m = -INFINITY;
    l = 0.f;
  }

  __device__ void page(unsigned char* stage_ptr, int lo, int nvalid, float scale_log2) {
    const uint32_t stage = smem_u32(stage_ptr);
    if (nvalid < kPageSize) {
      // Slots past the sequence end may hold anything (even NaN): zero their V rows so that
      // P = 0 times V stays 0 inside the tensor-core product.
      constexpr int kChunksPerRow = D / 8;
      const int n = (kPageSize - nvalid) * kChunksPerRow;
      for (int i = lane; i < n; i += 32) {
        const int t = nvalid + i / kChunksPerRow;
        const int dim = (i % kChunksPerRow) * 8;
        const uint32_t a = chunk_addr(stage, 1, t, dim);
        asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0u) : "memory");
      }
      __syncwarp();
    }
    // scores S^T[h][t] = q_h . K_t : rows = query heads, columns = slots (two n-blocks)
    float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    {
      const int mi = lane >> 3, r = lane & 7;
      const int t = (mi >> 1) * 8 + r;
      const int dsub = (mi & 1) * 8;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4(chunk_addr(stage, 0, t, ks * 16 + dsub), b0, b1, b2, b3);
        mma_16816(sc[0], qa[ks][0], 0u, qa[ks][1], 0u, b0, b1);
        mma_16816(sc[1], qa[ks][0], 0u, qa[ks][1], 0u, b2, b3);
      }
    }
    const int c = 2 * (lane & 3);
    float s[4] = {sc[0][0] * scale_log2, sc[0][1] * scale_log2, sc[1][0] * scale_log2, sc[1][1] * scale_log2};
    s[0] = (c >= lo && c < nvalid) ? s[0] : -INFINITY;
    s[1] = (c + 1 >= lo && c + 1 < nvalid) ? s[1] : -INFINITY;
    s[2] = (c + 8 >= lo && c + 8 < nvalid) ? s[2] : -INFINITY;
    s[3] = (c + 9 >= lo && c + 9 < nvalid) ? s[3] : -INFINITY;
    float mx = fmaxf(fmaxf(s[0], s[1]), fmaxf(s[2], s[3]));
    mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
    // Raise the head's running max (and rescale) only when a score exceeds it by more than 2^8;
    // otherwise the probabilities exp2(s - m) stay below 256 (the final division by l makes
    // the result independent of m).
    if (mx > m + kLazyRescale) {
      const float alpha = exp2f(m - mx);
      l *= alpha;
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        acc[nb][0] *= alpha;
        acc[nb][1] *= alpha;
      }
      m = mx;
    }
    const float e0 = exp2f(s[0] - m), e1 = exp2f(s[1] - m), e2 = exp2f(s[2] - m), e3 = exp2f(s[3] - m);
    const __half2 p01 = __floats2half2_rn(e0, e1);
    const __half2 p23 = __floats2half2_rn(e2, e3);
    const float2 f01 = __half22float2(p01), f23 = __half22float2(p23);
    l += (f01.x + f01.y) + (f23.x + f23.y);
    const uint32_t pa0 = *reinterpret_cast<const uint32_t*>(&p01);
    const uint32_t pa2 = *reinterpret_cast<const uint32_t*>(&p23);
    {
      const int mi = lane >> 3, r = lane & 7;
      const int t = (mi & 1) * 8 + r;
      const int dsub = (mi >> 1) * 8;
#pragma unroll
      for (int mm = 0; mm < D / 16; ++mm) {
        uint32_t v0, v1, v2, v3;
        ldmatrix_x4_trans(chunk_addr(stage, 1, t, mm * 16 + dsub), v0, v1, v2, v3);
        mma_16816(acc[2 * mm], pa0, 0u, pa2, 0u, v0, v1);
        mma_16816(acc[2 * mm + 1], pa0, 0u, pa2, 0u, v2, v3);
      }
    }
  }

  __device__ bool finish(float* po, float* pl, long long head_row0, int S, int j) {
    float lt = l;
    lt += __shfl_xor_sync(kFull, lt, 1);
    lt += __shfl_xor_sync(kFull, lt, 2);
    const bool any = __shfl_sync(kFull, lt, 0) > 0.f;  // every head row saw the same tokens
    if (!any) return false;
    if (h < group) {
      const float inv = 1.f / lt;
      const long long row = head_row0 + h;
      float* dst = po + (row * S + j) * D + 2 * (lane & 3);
#pragma unroll
      for (int nb = 0; nb < NB; ++nb)
        *reinterpret_cast<float2*>(dst + nb * 8) = make_float2(acc[nb][0] * inv, acc[nb][1] * inv);
      if ((lane & 3) == 0) pl[row * S + j] = (m + log2f(lt)) * kLn2;
    }
    return true;
  }

  __device__ void finish_out(__half* out, float* lse_out, long long head_row0) {
    float lt = l;
    lt += __shfl_xor_sync(kFull, lt, 1);
    lt += __shfl_xor_sync(kFull, lt, 2);
    if (h < group) {
      const bool any = lt > 0.f;
      const float inv = any ? 1.f / lt : 0.f;
      const long long row = head_row0 + h;
      __half* dst = out + row * D + 2 * (lane & 3);
#pragma unroll
      for (int nb = 0; nb < NB; ++nb)
        *reinterpret_cast<__half2*>(dst + nb * 8) =
            __floats2half2_rn(any ? acc[nb][0] * inv : 0.f, any ? acc[nb][1] * inv : 0.f);
      if (lse_out != nullptr && (lane & 3) == 0) lse_out[row] = any ? (m + log2f(lt)) * kLn2 : -INFINITY;
    }
  }
};

// ------------------------------------------------------------------------------------------------
// int8 cache, every group size (G <= 8 query heads of one KV head): the page is computed from its
// codes on the tensor cores with the slots, not the heads, as the 16 rows of each product, so no
// row is padding:
//   S^T = K q^T      rows = the page's 16 slots, columns = the G heads (8 wide), k = head dims
//   O^T += V^T P^T   rows = 16 head dims per product, columns = the heads, k = the 16 slots
// The head dimensions are taken in a permuted order (the sums are the same): at k-step ks, lane
// (g, c) takes dimensions D/4 c + 4 ks + {0, 1, 2, 3} of q and of the K codes, so the four codes of
// one 32-bit word are its A fragment pair.  The 16 slots are permuted too: row r of S^T is slot
// sigma(r), r = 2c + e -> 4c + e and r = 8 + 2c + e -> 4c + 2 + e, which makes the P V fragment of a
// dimension the word c (slots 4c .. 4c + 3) of the dim-major V block, and the transpose of S^T's
// 8x8 halves (movmatrix) exactly the B fragments of P^T.  A stored byte (code + 128) placed in the
// mantissa of 1024 is the exact fp16 value 1152 + code, from which 1152 is subtracted.  K scales multiply the scores and V scales the probabilities,
// relative to a reference vref raised lazily (by 2^7) so that the scaled probabilities stay inside
// fp16; the output is acc * vref / l.  A stage holds one or two pages of the item.
template <int D>
struct GroupQ8 {
  static constexpr int KS = D / 16;  // k-steps of S^T (head dims)
  static constexpr int MB = D / 16;  // 16-dim row blocks of O^T
  static constexpr int kBlk = int8_block_bytes(D);
  uint32_t qb[KS][2];  // B fragments of q^T: head g, dims D/4 c + 4 ks + {0, 1} and {2, 3}
  float acc[MB][4];    // O^T: dims 16 i + g and 16 i + g + 8, heads 2c and 2c + 1
  float m0, m1;        // running max (log2 domain) of heads 2c and 2c + 1
  float l0, l1;        // this lane's share (its two slots of every page) of the row sums of those heads
  float vref, vinv;
  int lane, g, c, group;

  __device__ void init(int lane_, int group_) {
    lane = lane_;
    g = lane >> 2;
    c = lane & 3;
    group = group_;
  }

  // Four stored bytes (codes + 128) -> their codes as fp16 pairs: bytes 0, 1 in lo, bytes 2, 3 in hi.
  __device__ static void codes_to_half(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const __half2 bias = __half2half2(__ushort_as_half((unsigned short)0x6480));  // 1152
    const uint32_t a = __byte_perm(w, 0x64646464u, 0x5140), b = __byte_perm(w, 0x64646464u, 0x5342);
    const __half2 x = __hsub2(*reinterpret_cast<const __half2*>(&a), bias);
    const __half2 y = __hsub2(*reinterpret_cast<const __half2*>(&b), bias);
    lo = *reinterpret_cast<const uint32_t*>(&x);
    hi = *reinterpret_cast<const uint32_t*>(&y);
  }

  __device__ void begin8(const unsigned char* qslot) {
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      if (g < group) {
        const uint2 w = *reinterpret_cast<const uint2*>(qslot + (g * D + (D / 4) * c + 4 * ks) * 2);
        qb[ks][0] = w.x;
        qb[ks][1] = w.y;
      } else {
        qb[ks][0] = 0u;
        qb[ks][1] = 0u;
      }
    }
#pragma unroll
    for (int i = 0; i < MB; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    // a finite floor: a fully masked page before the first attended slot gives exp2(-inf) = 0
    m0 = m1 = -1e30f;
    l0 = l1 = 0.f;
    vref = 0.f;
    vinv = 0.f;
  }

  // The D/4 codes of key row `row` this lane contracts: words w[ks] = dims D/4 c + 4 ks .. + 3.
  __device__ void key_words(const unsigned char* kb, int row, uint32_t (&w)[KS]) const {
    const unsigned char* src = kb + row * D + (D / 4) * c;
    if constexpr (D == 96) {
#pragma unroll
      for (int i = 0; i < 3; ++i) {
        const uint2 v = *reinterpret_cast<const uint2*>(src + 8 * i);
        w[2 * i] = v.x;
        w[2 * i + 1] = v.y;
      }
    } else {
#pragma unroll
      for (int i = 0; i < KS / 4; ++i) {
        const uint4 v = *reinterpret_cast<const uint4*>(src + 16 * i);
        w[4 * i] = v.x;
        w[4 * i + 1] = v.y;
        w[4 * i + 2] = v.z;
        w[4 * i + 3] = v.w;
      }
    }
  }

  // NP pages of one stage: page 0 with valid slots [lo, nv0), page 1 (NP == 2) with [0, nv1).  Each
  // page is the K block (codes [16][D] slot-major, then 16 fp32 scales) and the V block (codes
  // [D][16] dim-major, then 16 fp32 scales) as stored.  Codes of masked slots are finite and meet
  // P = 0; their scales are never used.
  template <int NP>
  __device__ void page8(const unsigned char* stage, int lo, int nv0, int nv1, float scale_log2) {
    const int rA = 4 * (g >> 1) + (g & 1), rB = rA + 2;  // slots of S^T rows g and g + 8
    float x[NP][4];   // scores (log2 domain): slot rA heads 2c, 2c+1; slot rB heads 2c, 2c+1
    bool va[NP], vb[NP];
#pragma unroll
    for (int pg = 0; pg < NP; ++pg) {
      const unsigned char* kb = stage + pg * 2 * kBlk;
      uint32_t wa[KS], wb[KS];
      key_words(kb, rA, wa);
      key_words(kb, rB, wb);
      // even and odd k-steps accumulate apart: two independent MMA chains
      float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        uint32_t a0, a1, a2, a3;
        codes_to_half(wa[ks], a0, a2);
        codes_to_half(wb[ks], a1, a3);
        mma_16816_nv((ks & 1) ? s1 : s0, a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
      }
      const int first = pg == 0 ? lo : 0, nv = pg == 0 ? nv0 : nv1;
      va[pg] = rA >= first && rA < nv;
      vb[pg] = rB >= first && rB < nv;
      const float* ksc = reinterpret_cast<const float*>(kb + 16 * D);
      const float fa = ksc[rA] * scale_log2, fb = ksc[rB] * scale_log2;
      x[pg][0] = va[pg] ? (s0[0] + s1[0]) * fa : -INFINITY;
      x[pg][1] = va[pg] ? (s0[1] + s1[1]) * fa : -INFINITY;
      x[pg][2] = vb[pg] ? (s0[2] + s1[2]) * fb : -INFINITY;
      x[pg][3] = vb[pg] ? (s0[3] + s1[3]) * fb : -INFINITY;
    }
    // Raise a head's running max (and rescale) only when one of its scores exceeds it by more than
    // 2^8; the common case costs one vote.
    bool need = false;
#pragma unroll
    for (int pg = 0; pg < NP; ++pg)
      need |= fmaxf(x[pg][0], x[pg][2]) > m0 + kLazyRescale || fmaxf(x[pg][1], x[pg][3]) > m1 + kLazyRescale;
    if (__any_sync(kFull, need)) {
      float mx0 = fmaxf(x[0][0], x[0][2]), mx1 = fmaxf(x[0][1], x[0][3]);
#pragma unroll
      for (int pg = 1; pg < NP; ++pg) {
        mx0 = fmaxf(mx0, fmaxf(x[pg][0], x[pg][2]));
        mx1 = fmaxf(mx1, fmaxf(x[pg][1], x[pg][3]));
      }
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {  // over the slots (g); lanes of one c hold the same heads
        mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, o));
        mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, o));
      }
      float a0 = 1.f, a1 = 1.f;
      if (mx0 > m0 + kLazyRescale) {
        a0 = exp2f(m0 - mx0);
        m0 = mx0;
      }
      if (mx1 > m1 + kLazyRescale) {
        a1 = exp2f(m1 - mx1);
        m1 = mx1;
      }
      l0 *= a0;
      l1 *= a1;
#pragma unroll
      for (int i = 0; i < MB; ++i) {
        acc[i][0] *= a0;
        acc[i][2] *= a0;
        acc[i][1] *= a1;
        acc[i][3] *= a1;
      }
    }
    float e[NP][4];
#pragma unroll
    for (int pg = 0; pg < NP; ++pg) {
      e[pg][0] = exp2f(x[pg][0] - m0);
      e[pg][1] = exp2f(x[pg][1] - m1);
      e[pg][2] = exp2f(x[pg][2] - m0);
      e[pg][3] = exp2f(x[pg][3] - m1);
      // the row sums add the fp16-rounded probabilities
      const float2 fa = __half22float2(__floats2half2_rn(e[pg][0], e[pg][1]));
      const float2 fb = __half22float2(__floats2half2_rn(e[pg][2], e[pg][3]));
      l0 += fa.x + fb.x;
      l1 += fa.y + fb.y;
    }
    // V scales of this lane's slots (0 where masked); the reference rises when one exceeds 2^7 vref
    float v[NP][2];
    bool vneed = false;
#pragma unroll
    for (int pg = 0; pg < NP; ++pg) {
      const float* vsc = reinterpret_cast<const float*>(stage + pg * 2 * kBlk + kBlk + 16 * D);
      v[pg][0] = va[pg] ? vsc[rA] : 0.f;
      v[pg][1] = vb[pg] ? vsc[rB] : 0.f;
      vneed |= fmaxf(v[pg][0], v[pg][1]) > vref * 128.f;
    }
    if (__any_sync(kFull, vneed)) {
      float vm = fmaxf(v[0][0], v[0][1]);
#pragma unroll
      for (int pg = 1; pg < NP; ++pg) vm = fmaxf(vm, fmaxf(v[pg][0], v[pg][1]));
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) vm = fmaxf(vm, __shfl_xor_sync(kFull, vm, o));
      if (vm > vref * 128.f) {  // the same answer on every lane (slots depend on g only)
        const float alpha = vref / vm;
#pragma unroll
        for (int i = 0; i < MB; ++i) {
          acc[i][0] *= alpha;
          acc[i][1] *= alpha;
          acc[i][2] *= alpha;
          acc[i][3] *= alpha;
        }
        vref = vm;
        vinv = 1.f / vm;
      }
    }
#pragma unroll
    for (int pg = 0; pg < NP; ++pg) {
      const float wa = v[pg][0] * vinv, wb = v[pg][1] * vinv;
      // P^T fragments: the 8x8 halves of P (slot rows, head columns) transposed
      const uint32_t b0 = movmatrix_trans(pack_half2(e[pg][0] * wa, e[pg][1] * wa));
      const uint32_t b1 = movmatrix_trans(pack_half2(e[pg][2] * wb, e[pg][3] * wb));
      const unsigned char* vblk = stage + pg * 2 * kBlk + kBlk;
#pragma unroll
      for (int i = 0; i < MB; ++i) {
        const uint32_t w0 = *reinterpret_cast<const uint32_t*>(vblk + (16 * i + g) * 16 + 4 * c);
        const uint32_t w1 = *reinterpret_cast<const uint32_t*>(vblk + (16 * i + g + 8) * 16 + 4 * c);
        uint32_t a0, a1, a2, a3;
        codes_to_half(w0, a0, a2);
        codes_to_half(w1, a1, a3);
        mma_16816_nv(acc[i], a0, a1, a2, a3, b0, b1);
      }
    }
  }

  // Row sums of heads 2c and 2c + 1 over the warp's slots (every lane of a c holds the totals).
  __device__ void row_sums(float& t0, float& t1) const {
    t0 = l0;
    t1 = l1;
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      t0 += __shfl_xor_sync(kFull, t0, o);
      t1 += __shfl_xor_sync(kFull, t1, o);
    }
  }

  __device__ bool finish(float* po, float* pl, long long head_row0, int S, int j) {
    float t0, t1;
    row_sums(t0, t1);
    const bool any = __shfl_sync(kFull, t0, 0) > 0.f;  // every head saw the same slots
    if (!any) return false;
    const float sc = vref > 0.f ? vref : 1.f;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int h = 2 * c + e;
      if (h < group) {
        const float lt = e ? t1 : t0;
        const float inv = sc / lt;
        const long long row = head_row0 + h;
        float* dst = po + (row * S + j) * D + g;
#pragma unroll
        for (int i = 0; i < MB; ++i) {
          dst[16 * i] = acc[i][e] * inv;
          dst[16 * i + 8] = acc[i][2 + e] * inv;
        }
        if (g == 0) pl[row * S + j] = ((e ? m1 : m0) + log2f(lt)) * kLn2;
      }
    }
    return true;
  }

  __device__ void finish_out(__half* out, float* lse_out, long long head_row0) {
    float t0, t1;
    row_sums(t0, t1);
    const float sc = vref > 0.f ? vref : 1.f;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int h = 2 * c + e;
      if (h < group) {
        const float lt = e ? t1 : t0;
        const bool any = lt > 0.f;
        const float inv = any ? sc / lt : 0.f;
        const long long row = head_row0 + h;
        __half* dst = out + row * D + g;
#pragma unroll
        for (int i = 0; i < MB; ++i) {
          dst[16 * i] = __float2half_rn(any ? acc[i][e] * inv : 0.f);
          dst[16 * i + 8] = __float2half_rn(any ? acc[i][2 + e] * inv : 0.f);
        }
        if (lse_out != nullptr && g == 0) lse_out[row] = any ? ((e ? m1 : m0) + log2f(lt)) * kLn2 : -INFINITY;
      }
    }
  }
};

// ------------------------------------------------------------------------------------------------

__device__ __forceinline__ int find_sequence(const int* prefix, int batch, int w) {
  int lo = 0, hi = batch;  // prefix[lo] <= w < prefix[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= w) lo = mid; else hi = mid;
  }
  return lo;
}

// One work item as the producer sees it (lane-uniform except `window`, which holds the page id
// of page win_base + lane).
struct Item {
  int s, j, g, first, n, nch, p0, p1, pnext, win_base, window, last, q0, q1;
  bool active;
  bool drop;  // balanced mode: a piece of a sequence with more pieces than partial slots
  // one-launch mode: the position of the sequence's single new token (also the query position),
  // and whether its page lies in this item
  int qpos;
  bool has_new;
  // sliding window: the first visible page of the sequence (page ordinals of the item count from
  // it) and the first attended slot of that page
  int f, lo;
};

// Locate item w and start the global loads it needs (last-page length, query row, the first 32
// page ids).  The loaded values are consumed later by activate(), so the loads overlap other work.
__device__ __forceinline__ void issue_item_loads(Item& it, const DecodeParams& p, int lane);

__device__ __forceinline__ void prepare_item(Item& it, int w, const DecodeParams& p, const int* prefix,
                                             const int* indptr, const int* wstart, int lane) {
  const int s = find_sequence(prefix, p.batch, w);
  const int r = w - prefix[s];
  it.s = s;
  it.j = r / p.hkv;
  it.g = r - it.j * p.hkv;
  it.first = indptr[s];
  it.n = indptr[s + 1] - it.first;
  it.f = 0;
  it.lo = 0;
  if (wstart != nullptr) {
    // sliding window: the item's pages are the sequence's visible pages
    const int ws = wstart[s];
    it.f = ws & 0xffffff;
    it.lo = ws >> 24;
    it.first += it.f;
    it.n -= it.f;
  }
  int c = 1;
  it.nch = seq_chunks(p, it.n, c);
  if (it.nch > 0 && it.n > 0) {
    it.p0 = it.j * c;
    it.p1 = min(it.p0 + c, it.n);
  } else {
    it.p0 = it.p1 = 0;
  }
  it.drop = false;
  issue_item_loads(it, p, lane);
}

// First warp of the balanced partition whose run contains unit b.
__device__ __forceinline__ long long first_run(long long b, long long U, long long W) {
  return ((b + 1) * W + U - 1) / U - 1;
}

// Balanced mode: the piece of warp gw that starts at unit u of its run [u, u_end); U units in PW
// runs.  Under a sliding window the units are the visible pages (wstart non-null).
__device__ __forceinline__ void prepare_piece(Item& it, long long u, long long u_end, int gw, const DecodeParams& p,
                                              const int* prefix, const int* indptr, const int* wstart,
                                              long long U, long long PW, int lane) {
  const int s = find_sequence(prefix, p.batch, (int)u);
  int f = 0, lo = 0;
  if (wstart != nullptr) {
    f = wstart[s] & 0xffffff;
    lo = wstart[s] >> 24;
  }
  const int n = indptr[s + 1] - indptr[s] - f;
  const long long r = u - prefix[s];
  const int g = (int)(r / n);
  const int page = (int)(r - (long long)g * n);
  it.s = s;
  it.g = g;
  it.first = indptr[s] + f;
  it.n = n;
  it.f = f;
  it.lo = lo;
  it.p0 = page;
  it.p1 = (int)min((long long)n, (long long)page + (u_end - u));
  const long long b = (long long)prefix[s] + (long long)g * n;  // first unit of the segment
  const long long wf = first_run(b, U, PW);
  const long long wl = first_run(b + n - 1, U, PW);
  it.j = (int)(gw - wf);
  it.nch = (int)(wl - wf + 1);
  it.drop = false;
  issue_item_loads(it, p, lane);
}

__device__ __forceinline__ void issue_item_loads(Item& it, const DecodeParams& p, int lane) {
  const int s = it.s;
  it.pnext = it.p0;
  it.win_base = it.p0;
  const int idx = it.p0 + lane;
  it.window = idx < it.p1 ? p.page_indices[it.first + idx] : 0;
  it.last = it.n > 0 ? p.last_page_len[s] : kPageSize;
  if (p.q_indptr != nullptr && it.n > 0) {
    it.q0 = p.q_indptr[s];
    it.q1 = p.q_indptr[s + 1];
  } else {
    it.q0 = s;
    it.q1 = s + 1;
  }
  it.active = true;
}

// One-launch mode: the sequence's new-token range (from the shared copy of append_indptr) and the
// new token's position.
__device__ __forceinline__ void issue_fused_loads(Item& it, const DecodeParams& p, const int* aptr) {
  it.q0 = aptr[it.s];
  it.q1 = aptr[it.s + 1];
  it.qpos = it.q1 == it.q0 + 1 ? p.pos_map[it.q0] : -1;
}

// One-launch mode, at activation: every sequence appends exactly one token; a position past the
// cache or the sequence's pages is reported by the first piece of each (sequence, KV head).
// Returns false when the query cannot be rotated (no single token or position out of the table).
__device__ __forceinline__ bool activate_fused(Item& it, const DecodeParams& p, int lane) {
  const bool single = it.q1 == it.q0 + 1;
  const bool in_table = single && it.qpos >= 0 && it.qpos < p.max_position;
  const int vpage = (it.qpos >> 4) - it.f;  // among the item's (visible) pages
  const bool in_pages = in_table && vpage >= 0 && vpage < it.n;
  if (single && !in_pages && it.j == 0 && lane == 0) atomicOr(p.status, kFlagBadPosition);
  it.has_new = in_pages && vpage >= it.p0 && vpage < it.p1;
  return in_table;
}

// One-launch mode: rotate the new token's raw k row (cs: its (cos, sin) row) and keep it with the
// raw v row as the patch rows [K][V] of the item (the same arithmetic as the append kernel).
template <int D>
__device__ __forceinline__ void make_patch(const unsigned char* cs_row, const unsigned char* kv_raw,
                                           unsigned char* patch, int lane) {
  constexpr int kUnits = D / 16;  // rope units: chunk u pairs with chunk u + D/16
  constexpr int kChunks = D / 8;  // 16-byte chunks of a row
  if (lane < kUnits) {
    const uint4 lo = *reinterpret_cast<const uint4*>(kv_raw + 16 * lane);
    const uint4 hi = *reinterpret_cast<const uint4*>(kv_raw + 16 * (lane + kUnits));
    uint4 ylo, yhi;
    rope8(lo, hi, reinterpret_cast<const float2*>(cs_row) + 8 * lane, ylo, yhi);
    *reinterpret_cast<uint4*>(patch + 16 * lane) = ylo;
    *reinterpret_cast<uint4*>(patch + 16 * (lane + kUnits)) = yhi;
  } else if (lane < kUnits + kChunks) {
    const int c = lane - kUnits;
    *reinterpret_cast<uint4*>(patch + 2 * D + 16 * c) = *reinterpret_cast<const uint4*>(kv_raw + 2 * D + 16 * c);
  }
  __syncwarp();
}

// One-launch mode: write the patch rows into slot r of a staged page (layout of Compute) and into
// the pool (page pid, KV head g), so later launches read the appended token from the cache.
template <int D, class Compute>
__device__ __forceinline__ void apply_patch(unsigned char* stage, const unsigned char* patch, int r, int pid, int g,
                                            const DecodeParams& p, int lane) {
  constexpr int kChunks = D / 8;
  if (lane < 2 * kChunks) {
    const int kv = lane >= kChunks ? 1 : 0;
    const int c = lane - kv * kChunks;
    const uint4 v = *reinterpret_cast<const uint4*>(patch + 16 * lane);
    const uint32_t a = Compute::row_chunk(smem_u32(stage), kv, r, c);
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
    __half* dst = p.pool + ((((long long)pid * 2 + kv) * p.hkv + g) * kPageSize + r) * D + 8 * c;
    *reinterpret_cast<uint4*>(dst) = v;
  }
  __syncwarp();
}

// Validate an item whose loads have been issued; an invalid or empty sequence becomes one empty
// item per KV head (its chunks are reported as -inf).
__device__ __forceinline__ void activate_item(Item& it, const DecodeParams& p, int lane) {
  bool ok = it.nch > 0;
  if (it.n > 0) ok = ok && it.last >= 1 && it.last <= kPageSize && it.q1 > it.q0;
  it.has_new = false;
  if (p.fused && it.n > 0) ok = activate_fused(it, p, lane) && ok;
  if (p.balanced && it.nch > p.splits) {
    // more pieces than partial slots (more pages than declared): the first piece reports the
    // sequence empty, the others are dropped
    ok = false;
    it.drop = it.j != 0;
    it.j = 0;
    it.nch = 1;
  }
  if (!ok) {
    if (lane == 0) atomicOr(p.status, kFlagBadSequence);
    it.p0 = it.p1 = it.pnext = 0;
    it.has_new = false;
  }
}

template <int D, bool MMA, bool FUSED, bool Q8, bool WIDE>
__global__ void __launch_bounds__(WIDE ? 384 : 256, 1) decode_kernel(const __grid_constant__ CUtensorMap map, DecodeParams p) {
  extern __shared__ unsigned char smem_raw[];
  // aligned (smem_align) by an offset from the shared array itself, so that every access below is
  // compiled as a shared-memory access
  constexpr uint32_t kAlign = smem_align(MMA);
  unsigned char* base = smem_raw + ((kAlign - (smem_u32(smem_raw) & (kAlign - 1))) & (kAlign - 1));
  const Layout L = make_layout(p.warps, p.nstage, D, p.group, p.batch, FUSED, p.window > 0, Q8);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + L.bar_off);
  StageMeta* metas = reinterpret_cast<StageMeta*>(base + L.meta_off);
  int* prefix = reinterpret_cast<int*>(base + L.prefix_off);
  int* indptr = reinterpret_cast<int*>(base + L.indptr_off);
  int* aptr = reinterpret_cast<int*>(base + L.aptr_off);  // fused mode: append_indptr
  const bool windowed = p.window > 0;
  // sliding window: per sequence, first visible page | first attended slot << 24
  int* wstart = windowed ? reinterpret_cast<int*>(base + L.wstart_off) : nullptr;
  __shared__ int warp_sums[32];

  pdl_launch_dependents();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) prefetch_tensormap(&map);
  // one arrival (the producer's) completes a stage's phase; the test setting pkv_set_stage_stall
  // asks for a second one, which nothing makes
  for (int i = tid; i < p.warps * p.nstage; i += blockDim.x) mbar_init(&bars[i], p.stall ? 2 : 1);
  fence_mbarrier_init();

  // Page ranges of every sequence, then items per sequence and their exclusive prefix sum (chunk
  // mode) or the first page unit of every sequence (balanced mode).
  for (int i = tid; i <= p.batch; i += blockDim.x) {
    indptr[i] = p.page_indptr[i];
    if constexpr (FUSED) aptr[i] = p.q_indptr[i];
  }
  __syncthreads();
  if (windowed) {
    // the query at position len - 1 attends to [len - window, len): pages from (len - window) / 16
    for (int s = tid; s < p.batch; s += blockDim.x) {
      const int n = indptr[s + 1] - indptr[s];
      int ws = 0;
      if (n > 0) {
        const int last = p.last_page_len[s];
        const int len = (n - 1) * kPageSize + last;
        if (last >= 1 && last <= kPageSize && len > p.window) ws = len - p.window;
      }
      wstart[s] = (ws >> 4) | ((ws & 15) << 24);
    }
    __syncthreads();
  }
  // pages an item walks: the sequence's pages, or its visible pages under a window
  auto seq_pages = [&](int s) {
    const int n = indptr[s + 1] - indptr[s];
    return windowed ? n - (wstart[s] & 0xffffff) : n;
  };
  if (p.balanced && !windowed) {
    for (int i = tid; i <= p.batch; i += blockDim.x) prefix[i] = p.hkv * indptr[i];
  } else {
    // exclusive scan of the units (balanced: visible page units) or items (chunk mode) per sequence
    const int per = (p.batch + blockDim.x - 1) / blockDim.x;
    const int s0 = min(p.batch, tid * per), s1 = min(p.batch, s0 + per);
    int local = 0;
    auto units_of = [&](int s) {
      if (p.balanced) return p.hkv * seq_pages(s);
      int c;
      const int nch = seq_chunks(p, seq_pages(s), c);
      return p.hkv * (nch > 0 ? nch : 1);
    };
    for (int s = s0; s < s1; ++s) local += units_of(s);
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(kFull, incl, off);
      if (lane >= off) incl += v;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    int warp_base = 0;
    for (int w = 0; w < warp; ++w) warp_base += warp_sums[w];
    int run = warp_base + incl - local;
    for (int s = s0; s < s1; ++s) {
      prefix[s] = run;
      run += units_of(s);
    }
    if (tid == blockDim.x - 1) prefix[p.batch] = run;
  }
  __syncthreads();

  const int total = prefix[p.batch];
  const int W = gridDim.x * p.warps;
  const int nst = p.nstage;
  uint64_t* bar = bars + warp * nst;
  StageMeta* meta = metas + warp * nst;
  unsigned char* stages = base + L.ring_off + (size_t)warp * nst * L.stage_bytes;
  unsigned char* qslots = base + L.q_off + (size_t)warp * kItemSlots * L.qslot_bytes;
  const uint32_t q_bytes = (uint32_t)(p.group * D * 2);
  const uint32_t cs_bytes = FUSED ? (uint32_t)(4 * D) : 0u;  // the query position's (cos, sin) row
  const uint32_t kv_bytes = FUSED ? (uint32_t)(4 * D) : 0u;  // the new token's raw k and v rows
  unsigned char* patch = base + L.patch_off + (size_t)warp * 4 * D;
  int* meta_pid = reinterpret_cast<int*>(base + L.pid_off) + warp * p.nstage;
  constexpr int kBlk = int8_block_bytes(D);
  const uint32_t page_bytes = Q8 ? (uint32_t)(2 * kBlk) : (uint32_t)(64 * D);
  const uint64_t policy = l2_policy_evict_first();

  // Producer state: the item being issued (cur) and the next one, whose loads are in flight.
  const int gw = blockIdx.x * p.warps + warp;
  int w_next = gw;
  // balanced mode: U page units in PW runs (under a window both come from the visible pages)
  const long long U = windowed ? (long long)total : p.units;
  const long long PW = windowed ? min((long long)W, U) : (long long)p.part_warps;
  long long u_next = 0, u_end = 0;  // balanced mode: the rest of this warp's run of page units
  if (p.balanced && gw < PW) {
    u_next = (long long)gw * U / PW;
    u_end = (long long)(gw + 1) * U / PW;
  }
  auto prepare_next = [&](Item& it) -> bool {
    if (p.balanced) {
      if (u_next >= u_end) return false;
      prepare_piece(it, u_next, u_end, gw, p, prefix, indptr, wstart, U, PW, lane);
      u_next += it.p1 - it.p0;
    } else {
      if (w_next >= total) return false;
      prepare_item(it, w_next, p, prefix, indptr, wstart, lane);
      w_next += W;
    }
    if constexpr (FUSED) issue_fused_loads(it, p, aptr);
    return true;
  };
  Item cur, nxt;
  cur.active = false;
  nxt.active = false;
  if (p.balanced && !windowed && prefix[p.batch] != p.units) {
    if (tid == 0) atomicOr(p.status, kFlagBadSequence);  // declared page total differs: nothing runs
  } else {
    prepare_next(nxt);  // index loads only: allowed before the wait
  }
  // One-launch mode with early pages: the ring is filled before the launch wait (the cache's pages
  // of earlier steps are not written by the preceding kernel), the items' rows after it.
  bool waited = !(FUSED && p.early);
  int ndefer = 0;
  int* defer = reinterpret_cast<int*>(base + L.defer_off) + warp * p.nstage * 8;
  if (waited) pdl_wait();  // q_rope and the pool pages come from the preceding kernel
  int issued = 0, consumed = 0;
  // Items whose first stage was issued / consumed: the first stage of item i brings its query rows
  // into item slot i % kItemSlots, so at most kItemSlots items may be issued and not yet begun.
  int items_issued = 0, items_begun = 0;
  // ring slot and barrier phase parity of `issued` and of `consumed`
  int ik = 0, ck = 0;
  uint32_t iph = 0, cph = 0;
  auto advance = [&](int& k, uint32_t& ph) {
    if (++k == nst) {
      k = 0;
      ph ^= 1u;
    }
  };

  // early: called before the launch wait.  Then the last two pages of a sequence, which hold the
  // 16 positions before its new token (written by the decode steps just before this one, which
  // may still be running under programmatic dependent launch), are not copied: the early fill
  // stops there and the copy is issued after the wait.
  auto produce = [&](bool early) -> bool {
    while (!cur.active) {
      if (!nxt.active) return false;
      cur = nxt;
      activate_item(cur, p, lane);
      nxt.active = false;
      prepare_next(nxt);
      if (cur.drop) cur.active = false;
    }
    if (cur.p1 != cur.p0 && cur.pnext == cur.p0 && items_issued - items_begun >= kItemSlots)
      return false;  // both item slots are taken: wait until the consumer begins an item
    if (early && cur.p1 != cur.p0 && cur.pnext >= cur.n - 2) return false;
    const int k = ik;
    StageMeta mt;
    mt.s = cur.s;
    mt.j = cur.j;
    mt.gl = cur.g;
    if (cur.p1 == cur.p0) {
      const int nch = max(cur.nch, 1);
      mt.flags = kMetaFirst | kMetaLast | kMetaEmpty | (cur.j >= nch - 1 ? kMetaLastChunk : 0) |
                 (nch << kMetaChunkShift);
      st_shared_v4_if(lane == 0, &meta[k], mt.s, mt.j, mt.gl, mt.flags);
      mbar_arrive_if(lane == 0, &bar[k]);
      cur.active = false;
    } else {
      // int8 cache: a stage takes two consecutive pages of the item when it has them
      const bool pair = Q8 && cur.pnext + 1 < cur.p1;
      const bool first = cur.pnext == cur.p0, lastp = cur.pnext + (pair ? 2 : 1) >= cur.p1;
      if (cur.pnext - cur.win_base >= (Q8 ? 31 : 32)) {
        cur.win_base = cur.pnext;
        const int idx = cur.pnext + lane;
        cur.window = idx < cur.p1 ? p.page_indices[cur.first + idx] : 0;
      }
      const int pid = __shfl_sync(kFull, cur.window, cur.pnext - cur.win_base);
      const bool page_ok = pid >= 0 && pid < p.num_pages;
      const int nvalid = page_ok ? ((cur.pnext == cur.n - 1) ? cur.last : kPageSize) : 0;
      const bool lastchunk = cur.j == cur.nch - 1;
      mt.flags = nvalid | (first ? kMetaFirst : 0) | (lastp ? kMetaLast : 0) | (lastchunk ? kMetaLastChunk : 0) |
                 (cur.nch << kMetaChunkShift);
      int pid2 = 0;
      bool page2_ok = false;
      if constexpr (Q8) {
        pid2 = __shfl_sync(kFull, cur.window, (cur.pnext + 1 - cur.win_base) & 31);
        page2_ok = pair && pid2 >= 0 && pid2 < p.num_pages;
        const int nvalid2 = page2_ok ? ((cur.pnext + 1 == cur.n - 1) ? cur.last : kPageSize) : 0;
        mt.flags |= nvalid2 << kMetaValid2Shift;
        if (pair && !page2_ok && lane == 0) atomicOr(p.status, kFlagBadPage);
      }
      if constexpr (FUSED) {
        // The first stage also brings the new token's raw k and v; the consumer patches the page
        // that holds the token in shared memory (the copy of that slot from the pool is stale).
        if (first && cur.has_new) mt.flags |= kMetaNew;
        if (cur.has_new && page_ok && cur.pnext == (cur.qpos >> 4) - cur.f) {
          mt.flags |= kMetaPatch | ((cur.qpos & 15) << kMetaSlotShift);
          st_shared_u32_if(lane == 0, &meta_pid[k], pid);
        }
      }
      if (!page_ok && lane == 0) atomicOr(p.status, kFlagBadPage);
      // lane 0 publishes the stage: metadata, then the barrier's byte count, then the copies (all
      // predicated on the lane, no branch)
      const bool l0 = lane == 0;
      if (cur.pnext == 0) mt.gl |= cur.lo << 16;  // a window's first attended slot
      st_shared_v4_if(l0, &meta[k], mt.s, mt.j, mt.gl, mt.flags);
      const uint32_t bytes = (page_ok ? page_bytes : 0u) + (page2_ok ? page_bytes : 0u) +
                             (first ? q_bytes + cs_bytes : 0u) + ((mt.flags & kMetaNew) ? kv_bytes : 0u);
      mbar_arrive_expect_tx_if(l0 && bytes != 0u, &bar[k], bytes);
      mbar_arrive_if(l0 && bytes == 0u, &bar[k]);
      if (first) {
        // the item's query rows (one-launch mode: with the (cos, sin) row and the new k and v)
        const int qslot_off = (items_issued % kItemSlots) * L.qslot_bytes;
        unsigned char* qslot = qslots + qslot_off;
        ++items_issued;
        if (FUSED && !waited) {
          // before the launch wait (early pages): the page copy goes now, the item's rows, which the
          // preceding kernel may write, right after the wait (the stage's byte count includes them)
          int* e = defer + ndefer * 8;
          st_shared_v4_if(l0, e, k, qslot_off, cur.q1 - 1, cur.g);
          st_shared_v4_if(l0, e + 4, cur.qpos, mt.flags, cur.q0, 0);
          ++ndefer;
        } else {
          const __half* qsrc = p.q + ((long long)(cur.q1 - 1) * p.hq + (long long)cur.g * p.group) * D;
          bulk_load_if(l0, qslot, qsrc, q_bytes, &bar[k]);
          if constexpr (FUSED) {
            bulk_load_if(l0, qslot + q_bytes, p.rope + (long long)cur.qpos * (D / 2), cs_bytes, &bar[k]);
            const bool kv = l0 && (mt.flags & kMetaNew);
            const long long row = ((long long)cur.q0 * p.hkv + cur.g) * D;
            bulk_load_if(kv, qslot + q_bytes + cs_bytes, p.k_new + row, kv_bytes / 2, &bar[k]);
            bulk_load_if(kv, qslot + q_bytes + cs_bytes + kv_bytes / 2, p.v_new + row, kv_bytes / 2, &bar[k]);
          }
        }
      }
      unsigned char* dst = stages + (size_t)k * L.stage_bytes;
      if constexpr (Q8) {
        // the page's int8 K block and V block of this KV head, as stored
        const unsigned char* kb = p.pool8 + (((long long)pid * 2) * p.hkv + cur.g) * kBlk;
        bulk_load_hint_if(l0 && page_ok, dst, kb, kBlk, &bar[k], policy);
        bulk_load_hint_if(l0 && page_ok, dst + kBlk, kb + (long long)p.hkv * kBlk, kBlk, &bar[k], policy);
        const unsigned char* kb2 = p.pool8 + (((long long)pid2 * 2) * p.hkv + cur.g) * kBlk;
        bulk_load_hint_if(l0 && page2_ok, dst + 2 * kBlk, kb2, kBlk, &bar[k], policy);
        bulk_load_hint_if(l0 && page2_ok, dst + 3 * kBlk, kb2 + (long long)p.hkv * kBlk, kBlk, &bar[k], policy);
      } else if constexpr (MMA) {
        constexpr int E = GroupMma<D>::E;
#pragma unroll
        for (int u = 0; u < D / E; ++u)
          tma_load_4d_if(l0 && page_ok, dst + u * GroupMma<D>::REGION, &map, &bar[k], u * E, 0, cur.g, 2 * pid,
                         policy);
      } else {
        // the page's K block and V block of this KV head are each contiguous in the pool
        const __half* kb = p.pool + (((long long)pid * 2 * p.hkv + cur.g) * kPageSize) * D;
        bulk_load_hint_if(l0 && page_ok, dst, kb, page_bytes / 2, &bar[k], policy);
        bulk_load_hint_if(l0 && page_ok, dst + page_bytes / 2, kb + (long long)p.hkv * kPageSize * D, page_bytes / 2,
                          &bar[k], policy);
      }
      cur.pnext += pair ? 2 : 1;
      if (lastp) cur.active = false;
    }
    ++issued;
    advance(ik, iph);
    return true;
  };

  using Compute = typename std::conditional<
      Q8, typename std::conditional<MMA, GroupQ8<D>, GroupOneQ8<D>>::type,
      typename std::conditional<MMA, GroupMma<D>, GroupOne<D>>::type>::type;
  Compute cmp;
  if constexpr (MMA) {
    cmp.init(lane, p.group);
  } else {
    cmp.init(lane);
  }

  if (!waited) {
    while (issued < min(nst, p.early) && produce(true)) {
    }
    pdl_wait();  // the new token's q, k, v come from the preceding kernel
    waited = true;
    __syncwarp();
    if (lane == 0) {
      for (int i = 0; i < ndefer; ++i) {
        const int* e = defer + i * 8;
        const int k = e[0], row_q = e[2], g = e[3], qpos = e[4], flags = e[5], q0 = e[6];
        unsigned char* qslot = qslots + e[1];
        bulk_load(qslot, p.q + ((long long)row_q * p.hq + (long long)g * p.group) * D, q_bytes, &bar[k]);
        bulk_load(qslot + q_bytes, p.rope + (long long)qpos * (D / 2), cs_bytes, &bar[k]);
        if (flags & kMetaNew) {
          const long long row = ((long long)q0 * p.hkv + g) * D;
          bulk_load(qslot + q_bytes + cs_bytes, p.k_new + row, kv_bytes / 2, &bar[k]);
          bulk_load(qslot + q_bytes + cs_bytes + kv_bytes / 2, p.v_new + row, kv_bytes / 2, &bar[k]);
        }
      }
    }
    __syncwarp();
  }

  if (p.balanced && gw == 0) {
    // sequences without pages own no page units: report them empty here
    for (int s = 0; s < p.batch; ++s) {
      if (indptr[s + 1] != indptr[s]) continue;
      const long long row0 = (long long)s * p.hq;
      if (p.merged) {
        for (int i = lane; i < p.hq * D; i += 32) p.out[row0 * D + i] = __float2half_rn(0.f);
        if (p.lse_out != nullptr)
          for (int i = lane; i < p.hq; i += 32)
            p.lse_out[row0 + i] = p.sinks != nullptr ? p.sinks[i] : -INFINITY;  // no token: the sink alone
      } else {
        for (int i = lane; i < p.hq * p.splits; i += 32) p.partial_lse[row0 * p.splits + i] = -INFINITY;
      }
    }
  }

  // Bounded wait for stage number c (ring slot k, phase parity ph), called by the whole warp in
  // step; on expiry flag a timeout and drain (bounded) the copies in flight, stage c's included
  // (stage c may be the merge's copy, numbered `issued` before it is counted).
  auto wait_stage = [&](int c, int k, uint32_t ph) -> bool {
    if (mbar_wait_bounded(&bar[k], ph, p.wait_ns)) return true;
    if (lane == 0) atomicOr(p.status, kFlagTimeout);
    for (int d = c; d < max(issued, c + 1); ++d)
      mbar_wait_bounded(&bar[d % nst], (uint32_t)((d / nst) & 1), kDrainLimitNs);
    __syncwarp();
    return false;
  };

  bool pending_merge = false;
  long long pm_row0 = 0;
  int pm_nch = 0, pm_head0 = 0;  // pm_head0: the group's first query head in the layer
  int* pm_counter = nullptr;

  // Finish an item: write its partial (or, merged, its output / its share of the merge).
  auto finish_item = [&](const StageMeta& mt) {
    const long long head_row0 = (long long)mt.s * p.hq + (long long)mt.g() * p.group;
    if (!p.merged) {
      bool wrote = false;
      if (!(mt.flags & kMetaEmpty)) wrote = cmp.finish(p.partial_o, p.partial_lse, head_row0, p.splits, mt.j);
      // -inf for this chunk when nothing was accumulated, and for every chunk after the last one
      const int j0 = wrote ? mt.j + 1 : mt.j;
      const int j1 = (mt.flags & kMetaLastChunk) ? p.splits : mt.j + 1;
      const int cnt = j1 - j0;
      for (int i = lane; i < p.group * cnt && cnt > 0; i += 32) {
        const int hh = i / cnt, jj = j0 + i % cnt;
        p.partial_lse[(head_row0 + hh) * p.splits + jj] = -INFINITY;
      }
      return;
    }
    const int nch = (mt.flags >> kMetaChunkShift) & 0xffff;
    // With sinks a single chunk also takes the merge path, so that its result is the combine's.
    if (nch == 1 && (mt.flags & kMetaEmpty) && p.sinks == nullptr) {
      for (int i = lane; i < p.group * D; i += 32) p.out[head_row0 * D + i] = __float2half_rn(0.f);
      if (p.lse_out != nullptr && lane < p.group) p.lse_out[head_row0 + lane] = -INFINITY;
    } else if (nch == 1 && p.sinks == nullptr) {
      cmp.finish_out(p.out, p.lse_out, head_row0);
    } else {
      const bool wrote =
          !(mt.flags & kMetaEmpty) && cmp.finish(p.partial_o, p.partial_lse, head_row0, p.splits, mt.j);
      if (!wrote && lane < p.group) p.partial_lse[(head_row0 + lane) * p.splits + mt.j] = -INFINITY;
      // Publish this chunk, then count it; the chunk that completes the count merges them all.
      // The warp barrier orders every lane's partial writes before lane 0's release; lane 0's
      // acquire, then the barrier of the shuffle, order the merge's reads after the other chunks'.
      __syncwarp();
      int* counter = p.counters + (long long)mt.s * p.hkv + mt.g();
      int done = 0;
      if (lane == 0) done = atom_add_acq_rel_gpu(counter, 1) + 1;
      done = __shfl_sync(kFull, done, 0);
      if (done == nch) {
        // this chunk completed the group: merge once this warp's stages are released
        pending_merge = true;
        pm_row0 = head_row0;
        pm_head0 = mt.g() * p.group;
        pm_nch = nch;
        pm_counter = counter;
      }
    }
  };

  // Merge a completed group.  With the ring empty (the usual case at the end of a warp's run) the
  // group's partial rows arrive in one bulk copy into the ring; otherwise they are read directly.
  auto run_merge = [&]() {
    const int rows_bytes = pm_nch * D * 4;
    // the group's partial rows, then its split LSEs, 64 per head
    const bool smem_ok = issued == consumed && pm_nch <= 64 &&
                         p.group * (rows_bytes + 256) <= nst * L.stage_bytes;
    if (smem_ok) {
      fence_proxy_async_global();  // the partials were written through the generic proxy
      const int k = ik;
      if (lane == 0) {
        mbar_arrive_expect_tx(&bar[k], (uint32_t)(p.group * rows_bytes));
        for (int hh = 0; hh < p.group; ++hh)
          bulk_load(stages + hh * rows_bytes, p.partial_o + (pm_row0 + hh) * p.splits * D, rows_bytes, &bar[k]);
      }
      // split LSEs: lane l loads splits l and l + 32 of each head (all loads in flight at once) and
      // parks them behind the rows
      constexpr int kHeads = MMA ? kMaxGroup : 1;
      float la[kHeads], lb[kHeads];
#pragma unroll
      for (int hh = 0; hh < kHeads; ++hh) {
        const float* lrow = p.partial_lse + (pm_row0 + hh) * p.splits;
        la[hh] = (hh < p.group && lane < pm_nch) ? lrow[lane] : -INFINITY;
        lb[hh] = (hh < p.group && lane + 32 < pm_nch) ? lrow[lane + 32] : -INFINITY;
      }
      float* lse_s = reinterpret_cast<float*>(stages + p.group * rows_bytes);
#pragma unroll
      for (int hh = 0; hh < kHeads; ++hh) {
        if (hh < p.group) {
          lse_s[hh * 64 + lane] = la[hh];
          lse_s[hh * 64 + 32 + lane] = lb[hh];
        }
      }
      if (!wait_stage(issued, ik, iph)) return false;
      ++issued;
      ++consumed;
      advance(ik, iph);
      advance(ck, cph);
      __syncwarp();
#pragma unroll 1
      for (int hh = 0; hh < p.group; ++hh) {
        const long long row = pm_row0 + hh;
        merge_rows<D>(lse_s + hh * 64, reinterpret_cast<const float*>(stages + hh * rows_bytes), pm_nch, lane,
                      p.out + row * D, p.lse_out != nullptr ? p.lse_out + row : nullptr,
                      p.sinks != nullptr ? p.sinks[pm_head0 + hh] : -INFINITY);
      }
      fence_proxy_async_smem();  // the reads above before later copies into the ring
      __syncwarp();
    } else {
      merge_group<D>(p.partial_lse, p.partial_o, pm_row0, p.group, p.splits, pm_nch, lane, p.out, p.lse_out,
                     p.sinks, pm_head0);
    }
    if (lane == 0) *pm_counter = 0;  // ready for the next launch
    pending_merge = false;
    return true;
  };

  // The ring is filled (and refilled after every step) at the top of the loop, the one place that
  // issues copies, so the producer code exists once.
  while (true) {
    while (issued - consumed < nst && produce(false)) {
    }
    if (consumed == issued) break;
    const int k = ck;
    if (!wait_stage(consumed, ck, cph)) return;
    const StageMeta mt = meta[k];
    StageMeta fin = mt;  // the last stage consumed in this step
    int used = 1;
    if (!(mt.flags & kMetaEmpty)) {
      if (mt.flags & kMetaFirst) {
        const unsigned char* qs = qslots + (items_begun % kItemSlots) * L.qslot_bytes;
        ++items_begun;  // the slot is read below, before this warp issues another copy
        if constexpr (FUSED) {
          if constexpr (MMA) {
            cmp.begin_rotate(qs);
          } else {
            cmp.begin_rotate(qs, p.scale_log2);
          }
          if (mt.j == 0) {
            // the first piece of each (sequence, KV head) writes the rotated query rows (q_out)
            const int qrow = aptr[mt.s];
            cmp.store_query(p.q_out + ((long long)qrow * p.hq + (long long)mt.g() * p.group) * D);
          }
          if (mt.flags & kMetaNew) make_patch<D>(qs + q_bytes, qs + q_bytes + cs_bytes, patch, lane);
        } else if constexpr (Q8) {
          cmp.begin8(qs);
        } else if constexpr (MMA) {
          cmp.begin(qs);
        } else {
          cmp.begin(qs, p.scale_log2);
        }
      }
      const int nvalid = mt.flags & kMetaValid;
      unsigned char* s1 = stages + (size_t)k * L.stage_bytes;
      if constexpr (Q8) {
        // an int8 stage holds one or two pages of the item (never the one-launch layout)
        const int nvalid2 = (mt.flags >> kMetaValid2Shift) & kMetaValid;
        if (nvalid2 > 0) {
          cmp.template page8<2>(s1, mt.lo(), nvalid, nvalid2, p.scale_log2);
        } else if (nvalid > 0) {
          cmp.template page8<1>(s1, mt.lo(), nvalid, 0, p.scale_log2);
        }
      } else if constexpr (!MMA) {
        // two pages of the same item at once when the next one is already in flight
        int n2 = 0;
        unsigned char* s2 = s1;
        if (!(mt.flags & kMetaLast) && consumed + 1 < issued) {
          int k2 = ck;
          uint32_t ph2 = cph;
          advance(k2, ph2);
          if (!wait_stage(consumed + 1, k2, ph2)) return;
          fin = meta[k2];
          n2 = fin.flags & kMetaValid;
          s2 = stages + (size_t)k2 * L.stage_bytes;
          used = 2;
          if constexpr (FUSED) {
            if (fin.flags & kMetaPatch)
              apply_patch<D, Compute>(s2, patch, (fin.flags >> kMetaSlotShift) & 15, meta_pid[k2], fin.g(), p, lane);
          }
        }
        if constexpr (FUSED) {
          if (mt.flags & kMetaPatch)
            apply_patch<D, Compute>(s1, patch, (mt.flags >> kMetaSlotShift) & 15, meta_pid[k], mt.g(), p, lane);
        }
        if (nvalid > 0 && n2 > 0) {
          cmp.page2(s1, mt.lo(), nvalid, s2, n2);
        } else if (nvalid + n2 > 0) {
          cmp.page(nvalid > 0 ? s1 : s2, nvalid > 0 ? mt.lo() : 0, nvalid > 0 ? nvalid : n2);
        }
      } else {
        if constexpr (FUSED) {
          if (mt.flags & kMetaPatch)
            apply_patch<D, Compute>(s1, patch, (mt.flags >> kMetaSlotShift) & 15, meta_pid[k], mt.g(), p, lane);
        }
        if (nvalid > 0) cmp.page(s1, mt.lo(), nvalid, p.scale_log2);
      }
    }
    if (fin.flags & kMetaLast) finish_item(fin);
    consumed += used;
    for (int u = 0; u < used; ++u) advance(ck, cph);
    fence_proxy_async_smem();  // this lane's reads/writes of the stages before their TMA refill
    __syncwarp();
    if (pending_merge && !run_merge()) return;
  }
}

template <int D, bool MMA, bool FUSED, bool Q8, bool WIDE = false>
void* kernel_ptr() {
  return reinterpret_cast<void*>(&decode_kernel<D, MMA, FUSED, Q8, WIDE>);
}

// The kernel of a head dim and layout: the tensor-core path, or the CUDA-core path in its 8-warp
// or its wide (12-warp, at most 168 registers) form; int8 caches run separate launches only.
template <int D, bool FUSED, bool Q8>
void* select_kernel_d(bool mma, bool wide) {
  if (mma) return kernel_ptr<D, true, FUSED, Q8>();
  return wide ? kernel_ptr<D, false, FUSED, Q8, true>() : kernel_ptr<D, false, FUSED, Q8>();
}

template <bool FUSED, bool Q8>
void* select_kernel_t(int head_dim, bool mma, bool wide) {
  switch (head_dim) {
    case 64: return select_kernel_d<64, FUSED, Q8>(mma, wide);
    case 96: return select_kernel_d<96, FUSED, Q8>(mma, wide);
    case 128: return select_kernel_d<128, FUSED, Q8>(mma, wide);
    default: return nullptr;
  }
}

void* select_kernel(int head_dim, bool mma, bool fused, bool q8, bool wide) {
  if (q8) return fused ? nullptr : select_kernel_t<false, true>(head_dim, mma, wide);
  return fused ? select_kernel_t<true, false>(head_dim, mma, wide) : select_kernel_t<false, false>(head_dim, mma, wide);
}

}  // namespace

// Deepest ring (at most 8, at least 2, else 0) of a CTA of `warps` warps within `budget` bytes.
int ring_depth(int warps, int head_dim, int group, int batch, bool fused, bool windowed, int budget, bool q8 = false) {
  int n = 8;
  while (n >= 2 && make_layout(warps, n, head_dim, group, batch, fused, windowed, q8).total > budget) --n;
  return n >= 2 ? n : 0;
}

// Dynamic shared memory a CTA may use when `ctas` CTAs share an SM (228 KB, 1 KB of it reserved per
// resident CTA, and the kernel's static shared memory).
int cta_budget(int ctas) { return std::min(kSmemBudget, (kSmemPerSm - ctas * 1024) / ctas - 256); }

DecodeConfig decode_config(int group, int head_dim, int batch, bool fused, bool windowed, bool q8) {
  DecodeConfig c;
  c.q8 = q8;
  c.mma = uses_mma(group, q8);
  c.fused = fused;
  // Warps per SM: the most stages in flight per SM (warps x ring depth) that fit the plain layout
  // in one CTA, on a tie the more warps (the CUDA-core path always runs 8 warps, the tensor-core
  // path 6 to 8).  Eight warps put two on each of the SM's four schedulers; six leave two
  // schedulers with one warp and two with two, and the warps that share a scheduler finish their
  // equal runs later (measured: mixed serving 659.5 -> 648.0 us, window 2 048 + sinks 54.6 -> 51.1 us
  // per layer, GQA long context unchanged, each with 24 stages in flight per SM).  Both layouts run
  // the same warps per SM, so they partition the work alike and give the same bits; each takes the
  // ring depth that fits.
  int sm_warps = 8, best = 0;
  for (int w = c.mma ? 6 : 8; w <= kMaxDecodeWarps; ++w) {
    const int n = ring_depth(w, head_dim, group, batch, false, false, kSmemBudget);
    if (n >= 2 && w * n >= best) {
      best = w * n;
      sm_warps = w;
    }
  }
  // The int8 cache's stages (two pages) are as large as the fp16 ones, and its page computation
  // decides its speed: it runs the most warps the registers allow (8 per SM on the tensor-core
  // path).  The CUDA-core path (one query head per KV head, fp16 or int8 pages) runs 12 warps (at
  // most 168 registers) when there are enough sequences; with few, more warps only cut the segments
  // into more pieces, whose merge ends the launch.  Measured: ragged batch of 64, int8 232 -> 191
  // and fp16 263.7 -> 255.4 us per layer with 12 warps; single stream (int8), 15.4 -> 18.9 us.
  if (q8) sm_warps = kMaxDecodeWarps;
  const bool wide = !c.mma && batch >= kWideBatch;
  if (wide) sm_warps = kWideWarps;
  c.wide = wide;
  c.warps = sm_warps;
  c.ctas_per_sm = 1;
  c.nstage = ring_depth(sm_warps, head_dim, group, batch, fused, windowed, kSmemBudget, q8);
  // The SM's warps split over kCtasPerSm CTAs when the ring stays as deep: a CTA that is still
  // merging at the end of a launch then holds only its share of the SM, and the next launch's CTAs
  // start (and run their prologue) in the rest.  The wide layout always splits (two stages per warp
  // still keep ~150 KB per SM in flight).
  if (kCtasPerSm > 1 && sm_warps % kCtasPerSm == 0) {
    const int w = sm_warps / kCtasPerSm;
    const int n = ring_depth(w, head_dim, group, batch, fused, windowed, cta_budget(kCtasPerSm), q8);
    if ((n >= c.nstage || wide) && n >= 2) {
      c.warps = w;
      c.ctas_per_sm = kCtasPerSm;
      c.nstage = n;
    }
  }
  const int nstage = c.nstage;
  c.smem_bytes =
      nstage >= 2 ? (size_t)make_layout(c.warps, nstage, head_dim, group, batch, fused, windowed, q8).total : 0;
  // The pool's tensor map always has the swizzled boxes the tensor-core layouts read (the
  // CUDA-core path copies plain runs instead; the prefill kernel uses the map for every group).
  c.box_inner = head_dim == 96 ? 32 : 64;
  c.swizzle_bytes = head_dim == 96 ? 64 : 128;
  return c;
}

cudaError_t decode_prepare(const DecodeConfig& cfg, int head_dim) {
  // both forms of the CUDA-core kernel: the batch of a launch chooses between them
  for (int w = 0; w < (cfg.mma ? 1 : 2); ++w) {
    void* k = select_kernel(head_dim, cfg.mma, cfg.fused, cfg.q8, w == 1);
    if (k == nullptr) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBudget);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_decode(const DecodeParams& p, const CUtensorMap& map, const DecodeConfig& cfg, int head_dim,
                          int grid, cudaStream_t stream, bool pdl) {
  void* k = select_kernel(head_dim, cfg.mma, cfg.fused, cfg.q8, cfg.wide);
  if (k == nullptr || cfg.smem_bytes == 0) return cudaErrorInvalidValue;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(grid);
  lc.blockDim = dim3(cfg.warps * 32);
  lc.dynamicSmemBytes = cfg.smem_bytes;
  lc.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = pdl ? 1 : 0;
  void* args[] = {const_cast<CUtensorMap*>(&map), const_cast<DecodeParams*>(&p)};
  return cudaLaunchKernelExC(&lc, k, args);
}

}  // namespace pkv
