// Chunked-prefill attention over the paged KV cache on the 5th-generation tensor cores: every
// appended token of a sequence attends causally to the positions up to its own (Zero TVM
// Documentation, "How it works": prefill in chunks; "Decode loop": a token attends to itself and
// to the earlier positions of its sequence; "KV cache": 16-slot pages behind a page table; "Port
// to Phi-4-mini or Qwen3": query head h reads KV head h / (Hq / Hkv)).  With many tokens per
// sequence this is a dense contraction, S = Q K^T and O = P V, run with tcgen05.mma.
//
// Work decomposition.  A tile is (sequence s, KV head g, 128 / G consecutive appended tokens of s):
// 128 query rows, row r = token r / G of the tile and query head g * G + r % G, so a page of KV
// head g is read once for all G heads that use it.  A key block is 8 pages (128 keys).  Tiles are
// ordered longest sequence first (tiles of one sequence last tile first) and taken in that order by
// the CTAs of a persistent grid (one per SM) from a shared counter whenever a CTA is free (the
// longest-first greedy schedule: a fixed deal left the CTAs of long histories working while
// others idled).
//
// One CTA, seven warps:
//   warps 0 and 6  producers: the tile's key blocks, each page's K (warp 0) and V (warp 6) of KV
//           head g copied as one box by the tensor-memory-access unit into rings of three K and two
//           V stages (128-byte swizzle, 64-byte for head_dim 96), each with its own barriers, so a K
//           stage is refilled as soon as its S MMA has completed while a V stage waits for its
//           P V MMA;
//   warp 1  MMA issuer (one thread): S_j = Q K_j^T into one of two tensor-memory buffers (128
//           fp32 columns each), then O += P_j V_j into a third (head_dim columns), P read from
//           tensor memory where the softmax left it (in S_j's buffer) and V MN-major straight from
//           the staged pages; every MMA group commits to a barrier;
//   warps 2-5  softmax (thread = query row = tensor-memory lane): stage the tile's queries in
//           shared memory, then per block read the row of S, mask it (the row's causal range
//           [window start, position], pages not loaded), an online softmax in the log2 domain
//           whose running max is raised only when a score exceeds it by 2^8 (then the row of O is
//           rescaled in tensor memory), P rounded to fp16 over the scores in tensor memory (the
//           row sum adds the same rounded values); the score loops run as eight independent chains,
//           since one warp per scheduler has little else to hide latencies with;
//           finally the row of O divided by the row sum (sinks join the denominator), written in
//           fp16 with its LSE.
// S is double-buffered, so the softmax of block j overlaps the MMA of block j + 1.  V rows of keys
// past the sequence end or in pages not loaded are zeroed in shared memory before P V (P = 0 times
// a NaN would be NaN).
//
// Every wait is bounded (2 s of global time unless pkv_set_wait_limit sets another limit), with
// one answer per warp; on expiry the warp flags PKV_FLAG_TIMEOUT and the CTA winds down: the
// producer drains its copies in flight, the MMA thread waits for its MMAs, the tensor memory is
// freed and the CTA returns.
#include "pkv_internal.h"
#include "ptx.cuh"
#include "tcgen05.cuh"

namespace pkv {
namespace {

constexpr unsigned kAll = 0xffffffffu;
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLazy = 8.f;

constexpr int kRows = 128;           // query rows of a tile (M)
constexpr int kKeys = 128;           // keys of a block (N of S, K of P V)
constexpr int kBlockPages = kKeys / kPageSize;
constexpr int kKStages = 3;          // key blocks whose K is in flight
constexpr int kVStages = 2;          // and whose V is
constexpr int kThreads = 224;        // K producer, MMA issuer, four softmax warps, V producer
constexpr int kTmemCols = 512;       // S0 [0,128), S1 [128,256), O [256, 256 + head_dim)
constexpr int kMaxSortedBatch = 512; // longest-first order of sequences up to this batch
constexpr int kItemSlots = 8;        // work items taken ahead by the K producer, published to the other warps
constexpr int kItemReaders = 6;      // V producer, MMA issuer, four softmax warps

template <int D>
struct Geo {
  static constexpr int E = (D == 96) ? 32 : 64;  // elements per swizzle row (TMA box extent)
  static constexpr int SW = 2 * E;               // bytes per swizzle row
  static constexpr int NA = D / E;               // atoms along head_dim
  static constexpr int KV_BYTES = kKeys * D * 2; // K (or V) of one block
  static constexpr int K_OFF = 0;                // K stages, then V stages, then the queries
  static constexpr int V_OFF = kKStages * KV_BYTES;
  static constexpr int Q_OFF = V_OFF + kVStages * KV_BYTES;
  static constexpr int BAR_OFF = Q_OFF + kRows * D * 2;
  // K and V stages hold a block as [8-key group][atom][8 keys][one swizzle row], a page (two
  // groups) as one copy lands: a swizzle atom of 8 rows, GROUP bytes, then the atoms of the
  // group's head dimensions, ROWGRP bytes per 8 keys
  static constexpr int GROUP = 8 * SW;
  static constexpr int ROWGRP = NA * GROUP;
  static constexpr int PAGE_BYTES = 2 * ROWGRP;
  static constexpr uint32_t IDESC_S = tc::idesc_f16(kRows, kKeys, false);
  static constexpr uint32_t IDESC_O = tc::idesc_f16(kRows, D, true);
};

// The tile of work item w: sequence, KV head, first token and token count.
struct Tile {
  int s, g, t0, nt, first, n, last, len;
  bool seq_ok;
};

// A work item as the K producer takes it: the item number (-1: none left), its tile and the
// tile's page range (pmax < 0: nothing to attend).
struct ItemInfo {
  int w, pmin, pmax;
  Tile t;
};

// Barriers and small shared state after the operand regions.
struct Shared {
  uint64_t k_full[kKStages], k_empty[kKStages], v_full[kVStages], v_empty[kVStages];
  uint64_t s_full[2], p_full, o_done, q_full, drain;
  uint64_t item_full[kItemSlots], item_empty[kItemSlots];
  uint32_t tmem_base;
  int abort_flag;
  int warp_sums[8];
  ItemInfo item_ring[kItemSlots];  // the CTA's i-th work item in slot i % kItemSlots
};

// 2^x with the special-function unit's approximation (relative error about 2^-22; subnormal results
// flush to zero, 2^-inf = 0); the probabilities it gives are rounded to fp16.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ int find_pos(const int* prefix, int n, int w) {
  int lo = 0, hi = n;  // prefix[lo] <= w < prefix[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= w) lo = mid; else hi = mid;
  }
  return lo;
}

__device__ __forceinline__ Tile tile_of(int w, const PrefillParams& p, const int* prefix, const int* order, int nseq,
                                        int tb) {
  Tile t;
  const int i = find_pos(prefix, nseq, w);
  t.s = order != nullptr ? order[i] : i;
  const int a0 = p.append_indptr[t.s], a1 = p.append_indptr[t.s + 1];
  const int ntiles = (a1 - a0 + tb - 1) / tb;
  const int r = w - prefix[i];
  const int rank = r / p.hkv;
  t.g = r - rank * p.hkv;
  const int tile = ntiles - 1 - rank;  // a sequence's later tokens see more keys: last tile first
  t.t0 = a0 + tile * tb;
  t.nt = min(tb, a1 - t.t0);
  t.first = p.page_indptr[t.s];
  t.n = p.page_indptr[t.s + 1] - t.first;
  t.last = t.n > 0 ? p.last_page_len[t.s] : 0;
  t.seq_ok = t.n > 0 && t.last >= 1 && t.last <= kPageSize;
  t.len = t.seq_ok ? (t.n - 1) * kPageSize + t.last : 0;
  return t;
}

// Page range [pmin, pmax] the tile's valid tokens attend to (every lane of the calling warp gets it).
__device__ __forceinline__ void tile_pages(const Tile& t, const PrefillParams& p, int lane, int& pmin, int& pmax) {
  pmin = 0x7fffffff;
  pmax = -1;
  for (int i = lane; i < t.nt; i += 32) {
    const int pos = t.seq_ok ? p.pos_map[t.t0 + i] : -1;
    if (pos >= 0 && pos < t.len) {
      const int st = (p.window > 0 && pos + 1 > p.window) ? pos + 1 - p.window : 0;
      pmin = min(pmin, st >> 4);
      pmax = max(pmax, pos >> 4);
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    pmin = min(pmin, __shfl_xor_sync(kAll, pmin, off));
    pmax = max(pmax, __shfl_xor_sync(kAll, pmax, off));
  }
}

// The page ids of a tile's key blocks, read ahead in groups of four blocks (one coalesced load per
// group, four blocks before its first use, so no wait for a page id sits in a warp's per-block
// loop): lane 8 i + l of `cur` holds page l of block bq + i (of `nxt`, of block bq + 4 + i), or -1
// outside the tile's page range [pmin, pmax].  Every lane of the warp calls it.
struct BlockIds {
  int cur, nxt, bq;
  const int* ids;
  int pmin, pmax;
  __device__ __forceinline__ int load(int b, int lane) const {
    const int ord = b * kBlockPages + lane;
    return (ord >= pmin && ord <= pmax) ? ids[ord] : -1;
  }
  __device__ __forceinline__ void start(const int* tile_ids, int b0, int lo, int hi, int lane) {
    ids = tile_ids;
    pmin = lo;
    pmax = hi;
    bq = b0;
    cur = load(b0, lane);
    nxt = load(b0 + 4, lane);
  }
  // Called once per block, b increasing from the start block: page l of block b on lane l < 8, -1
  // on the other lanes.
  __device__ __forceinline__ int page(int b, int lane) {
    if (b >= bq + 4) {
      bq += 4;
      cur = nxt;
      nxt = load(bq + 4, lane);
    }
    const int v = __shfl_sync(kAll, cur, 8 * (b - bq) + (lane & 7));
    return lane < kBlockPages ? v : -1;
  }
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(const __grid_constant__ CUtensorMap map, PrefillParams p) {
  using G = Geo<D>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Shared& sh = *reinterpret_cast<Shared*>(base + G::BAR_OFF);
  int* prefix = reinterpret_cast<int*>(base + G::BAR_OFF + sizeof(Shared));  // [batch + 1]
  int* order = prefix + p.batch + 1;                                          // [batch] (sorted batches)
  int* lens = order + p.batch;                                                // [batch] (sorted batches)
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int tb = kRows / p.group;  // tokens per tile
  volatile int* abort_flag = &sh.abort_flag;

  pdl_launch_dependents();
  if (tid == 0) {
    prefetch_tensormap(&map);
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(&sh.k_full[i], 1);
      // K of a stage is free when its S MMA has completed (only the MMA thread waits for K)
      mbar_init(&sh.k_empty[i], 1);
    }
    for (int i = 0; i < kVStages; ++i) {
      mbar_init(&sh.v_full[i], 1);
      mbar_init(&sh.v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) mbar_init(&sh.s_full[i], 1);
    mbar_init(&sh.p_full, kRows);
    mbar_init(&sh.o_done, 1);
    mbar_init(&sh.q_full, kRows);
    mbar_init(&sh.drain, 1);
    for (int i = 0; i < kItemSlots; ++i) {
      mbar_init(&sh.item_full[i], 1);
      mbar_init(&sh.item_empty[i], kItemReaders);
    }
    sh.abort_flag = 0;
  }
  fence_mbarrier_init();
  if (warp == 1) tc::alloc(&sh.tmem_base, kTmemCols);

  // Sequences longest first (when the batch is small enough to sort here), then the work prefix
  // (tiles x KV heads per sequence, in that order).
  const bool sorted = p.batch <= kMaxSortedBatch;
  auto seq_len = [&](int s) {
    const int n = p.page_indptr[s + 1] - p.page_indptr[s];
    return n > 0 ? (n - 1) * kPageSize + p.last_page_len[s] : 0;
  };
  if (sorted) {
    for (int s = tid; s < p.batch; s += kThreads) lens[s] = seq_len(s);
    __syncthreads();
    for (int s = tid; s < p.batch; s += kThreads) {
      const int ls = lens[s];
      int rank = 0;
      for (int u = 0; u < p.batch; ++u) {
        const int lu = lens[u];
        rank += (lu > ls || (lu == ls && u < s)) ? 1 : 0;
      }
      order[rank] = s;
    }
  }
  __syncthreads();
  {
    const int per = (p.batch + kThreads - 1) / kThreads;
    const int i0 = min(p.batch, tid * per), i1 = min(p.batch, i0 + per);
    auto items_of = [&](int i) {
      const int s = sorted ? order[i] : i;
      const int c = p.append_indptr[s + 1] - p.append_indptr[s];
      return c > 0 ? p.hkv * ((c + tb - 1) / tb) : 0;
    };
    int local = 0;
    for (int i = i0; i < i1; ++i) local += items_of(i);
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(kAll, incl, off);
      if (lane >= off) incl += v;
    }
    if (lane == 31) sh.warp_sums[warp] = incl;
    __syncthreads();
    int run = incl - local;
    for (int w = 0; w < warp; ++w) run += sh.warp_sums[w];
    for (int i = i0; i < i1; ++i) {
      prefix[i] = run;
      run += items_of(i);
    }
    if (tid == kThreads - 1) prefix[p.batch] = run;
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const int total = prefix[p.batch];
  const int* ord = sorted ? order : nullptr;
  const uint32_t tmem = sh.tmem_base;
  const uint32_t sbase = smem_u32(base);

  pdl_wait();  // q and the pool (the append) come from the preceding kernel

  // A bounded warp-wide wait; on expiry the CTA winds down.
  auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
    if (warp_wait_bounded(bar, parity, p.wait_ns)) return true;
    if (lane == 0) {
      atomicOr(p.status, kFlagTimeout);
      *abort_flag = 1;
    }
    __syncwarp();
    return false;
  };

  // Work items are taken in order from the launch's shared counter, so each CTA starts the longest
  // remaining item whenever it is free (the longest-first greedy schedule).  The K producer takes
  // them (a counter value past the last item means none is left) and publishes each in the item
  // ring with its tile and page range, so that the other warps, which read them from there in the
  // same order, do no global load to learn them.
  int item_i = 0;  // items this warp has taken or read
  auto no_item = []() {
    ItemInfo it;
    it.w = -1;
    it.pmin = 0;
    it.pmax = -1;
    return it;
  };
  auto take_item = [&]() -> ItemInfo {
    const int slot = item_i % kItemSlots;
    ItemInfo it = no_item();
    if (item_i >= kItemSlots && !wait(&sh.item_empty[slot], (uint32_t)(((item_i / kItemSlots) - 1) & 1))) return it;
    int w = 0;
    if (lane == 0) w = atomicAdd(p.work, 1);
    w = __shfl_sync(kAll, w, 0);
    if (w < total) {
      it.w = w;
      it.t = tile_of(w, p, prefix, ord, p.batch, tb);
      tile_pages(it.t, p, lane, it.pmin, it.pmax);
    }
    if (lane == 0) {
      sh.item_ring[slot] = it;
      mbar_arrive(&sh.item_full[slot]);
    }
    ++item_i;
    return it;
  };
  auto read_item = [&]() -> ItemInfo {
    const int slot = item_i % kItemSlots;
    if (!wait(&sh.item_full[slot], (uint32_t)((item_i / kItemSlots) & 1))) return no_item();
    const ItemInfo it = sh.item_ring[slot];
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.item_empty[slot]);
    ++item_i;
    return it;
  };

  if (warp == 0 || warp == 6) {
    // ---------------------------------------------------------------- producers (K: warp 0, V: warp 6)
    const bool is_k = warp == 0;
    const uint64_t policy = l2_policy_evict_last();  // a block's pages serve the tiles of its heads
    uint64_t* full = is_k ? sh.k_full : sh.v_full;
    uint64_t* empty = is_k ? sh.k_empty : sh.v_empty;
    const int kv = is_k ? 0 : 1;
    const int nst = is_k ? kKStages : kVStages;
    const int region = is_k ? G::K_OFF : G::V_OFF;
    int kv_it = 0;
    while (!*abort_flag) {
      const ItemInfo it = is_k ? take_item() : read_item();
      if (it.w < 0) break;
      const Tile& t = it.t;
      const int pmin = it.pmin, pmax = it.pmax;
      if (pmax < 0) continue;
      bool ok = true;
      BlockIds bid;
      bid.start(p.page_indices + t.first, pmin / kBlockPages, pmin, pmax, lane);
      for (int b = pmin / kBlockPages; b <= pmax / kBlockPages && ok; ++b, ++kv_it) {
        const int st = kv_it % nst;
        const int pid = bid.page(b, lane);  // lane l < 8: page 8b + l of the block
        // K of a stage is free once the S MMA that read it has completed, V once the P V MMA has
        if (kv_it >= nst && !(ok = wait(&empty[st], (uint32_t)(((kv_it / nst) - 1) & 1)))) break;
        const int ord_pg = b * kBlockPages + lane;
        const bool in_range = pid >= 0 && pid < p.num_pages;
        if (is_k && lane < kBlockPages && ord_pg >= pmin && ord_pg <= pmax && !in_range)
          atomicOr(p.status, kFlagBadPage);
        const unsigned loaded = __ballot_sync(kAll, in_range) & 0xffu;
        const uint32_t bytes = (uint32_t)__popc(loaded) * kPageSize * D * 2u;  // K (or V) of the loaded pages
        if (lane == 0) {
          if (bytes != 0u) {
            mbar_arrive_expect_tx(&full[st], bytes);
          } else {
            mbar_arrive(&full[st]);
          }
        }
        __syncwarp();
        if (in_range) {
          unsigned char* dst = base + region + st * G::KV_BYTES + lane * G::PAGE_BYTES;
          tma_load_5d(dst, &map, &full[st], 0, 0, 0, 0, (2 * pid + kv) * p.hkv + t.g, policy);
        }
      }
      if (!ok) break;
    }
    if (*abort_flag) {
      // wait (bounded) for the copies in flight of the last stages before leaving
      for (int i = max(0, kv_it - nst); i < kv_it; ++i)
        mbar_wait_bounded(&full[i % nst], (uint32_t)((i / nst) & 1), kDrainLimitNs);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    int kvc = 0, sc = 0, pc = 0, qi = 0;  // blocks, S MMAs, P V MMAs, tiles
    const bool leader = lane == 0;
    // O += P_j V_j for the block in stage `st`; `first` starts the accumulator
    // O += P V for block number vit: P in the block's S buffer of tensor memory (two fp16 per
    // column, written by the softmax over the scores it read), V from its stage.  MMAs execute in
    // issue order, so this one reads P before the S MMA two blocks on overwrites the buffer.
    auto issue_pv = [&](int vit, bool first) -> bool {
      const int st = vit % kVStages;
      if (!wait(&sh.p_full, (uint32_t)(pc & 1))) return false;
      if (!wait(&sh.v_full[st], (uint32_t)((vit / kVStages) & 1))) return false;
      ++pc;
      tc::fence_after_sync();
      if (leader) {
        const uint32_t vbase = sbase + G::V_OFF + st * G::KV_BYTES;
        const uint32_t pbase = tmem + 128 * (vit & 1);
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk) {
          const uint64_t bd = tc::smem_desc(vbase + (uint32_t)(2 * kk * G::ROWGRP), G::GROUP, G::ROWGRP,
                                            tc::layout_for(G::E));
          tc::mma_f16_ts(tmem + 256, pbase + 8 * kk, bd, G::IDESC_O, !(first && kk == 0));
        }
        tc::commit(&sh.v_empty[st]);
        tc::commit(&sh.o_done);
      }
      __syncwarp();
      return true;
    };
    bool ok = true;
    while (ok && !*abort_flag) {
      const ItemInfo it = read_item();
      if (it.w < 0) break;
      const int pmin = it.pmin, pmax = it.pmax;
      if (pmax < 0) continue;
      if (!(ok = wait(&sh.q_full, (uint32_t)(qi & 1)))) break;
      ++qi;
      const int nb = pmax / kBlockPages - pmin / kBlockPages + 1;
      for (int j = 0; j < nb; ++j, ++kvc, ++sc) {
        // S buffer sb held P of block kvc - 2, whose P V MMA was issued in the previous iteration
        const int st = kvc % kKStages, sb = sc & 1;
        if (!(ok = wait(&sh.k_full[st], (uint32_t)((kvc / kKStages) & 1)))) break;
        tc::fence_after_sync();
        if (leader) {
          const uint32_t kbase = sbase + G::K_OFF + st * G::KV_BYTES;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t u = (uint32_t)((16 * kk) / G::E), col = (uint32_t)((32 * kk) % G::SW);
            const uint64_t ad = tc::smem_desc(sbase + G::Q_OFF + u * kRows * G::SW + col, 16, 8 * G::SW,
                                              tc::layout_for(G::E));
            const uint64_t bd = tc::smem_desc(kbase + u * G::GROUP + col, 16, G::ROWGRP, tc::layout_for(G::E));
            tc::mma_f16(tmem + 128 * sb, ad, bd, G::IDESC_S, kk > 0);
          }
          tc::commit(&sh.s_full[sb]);
          tc::commit(&sh.k_empty[st]);
        }
        __syncwarp();
        if (j > 0 && !(ok = issue_pv(kvc - 1, j == 1))) break;
      }
      if (ok) ok = issue_pv(kvc - 1, nb == 1);
    }
    // before the tensor memory is freed: every MMA this thread issued has completed
    if (leader) tc::commit(&sh.drain);
    __syncwarp();
    mbar_wait_bounded(&sh.drain, 0, kDrainLimitNs);
  } else {
    // ---------------------------------------------------------------- softmax warps
    const int quarter = warp & 3;              // the tensor-memory lanes this warp may access
    const int r = 32 * quarter + lane;         // query row = tensor-memory lane
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * quarter) << 16);
    int kvs = 0, ss = 0, pw = 0;
    bool ok = true;
    // the tile's queries, row r, into the K-major swizzled Q region: asynchronously (rows outside
    // the tile are zero-filled); the caller waits for the copies and publishes them (q_full)
    auto copy_queries = [&](const Tile& t) {
      const int tk = r / p.group;
      const bool row_ok = t.seq_ok && tk < t.nt;
      const __half* src = p.q + ((long long)(row_ok ? t.t0 + tk : 0) * p.hq + t.g * p.group + r % p.group) * D;
#pragma unroll
      for (int c = 0; c < D / 8; ++c)
        cp_async16(base + G::Q_OFF + tc::kmajor_offset(kRows, G::E, r, 8 * c), src + 8 * c, row_ok ? 16u : 0u);
    };
    // the next item that has pages (all warps skip the others), or none
    auto next_item = [&]() -> ItemInfo {
      while (true) {
        const ItemInfo in = read_item();
        if (in.w < 0 || in.pmax >= 0) return in;
      }
    };
    ItemInfo it = read_item();
    bool q_ready = false;  // the item's queries were copied during the previous item and published
    while (ok && !*abort_flag && it.w >= 0) {
      const Tile t = it.t;
      // this row's token and query head, its position and the first position it attends to
      const int tk = r / p.group;
      const int tok = t.t0 + tk;
      const int head = t.g * p.group + r % p.group;
      bool valid = t.seq_ok && tk < t.nt;
      int pos = valid ? p.pos_map[tok] : 0;
      if (valid && (pos < 0 || pos >= t.len)) {
        atomicOr(p.status, kFlagBadPosition);  // the row is left unwritten
        valid = false;
      }
      if (!t.seq_ok && r == 0 && t.g == 0 && t.nt > 0) atomicOr(p.status, kFlagBadSequence);
      const int pmin = it.pmin, pmax = it.pmax;
      if (pmax < 0) {
        it = read_item();
        continue;
      }
      const int start = (valid && p.window > 0 && pos + 1 > p.window) ? pos + 1 - p.window : 0;
      if (!valid) pos = -1;  // attends to nothing

      if (!q_ready) {  // the first item (later ones are copied during the item before)
        copy_queries(t);
        cp_async_wait_all();
        fence_proxy_async_smem();
        mbar_arrive(&sh.q_full);
      }
      ItemInfo in = no_item();  // the next item, taken during this one's last block

      float m = -INFINITY, l = 0.f;
      const int b0 = pmin / kBlockPages, nb = pmax / kBlockPages - b0 + 1;
      BlockIds bid;
      bid.start(p.page_indices + t.first, b0, pmin, pmax, lane);
      for (int j = 0; j < nb; ++j, ++kvs, ++ss) {
        const int b = b0 + j, vst = kvs % kVStages, sb = ss & 1;
        // the block's pages the producers load (bit l = page 8b + l), decided as they decide it
        const int bpid = bid.page(b, lane);
        const int loaded = (int)(__ballot_sync(kAll, bpid >= 0 && bpid < p.num_pages) & 0xffu);
        if (!(ok = wait(&sh.s_full[sb], (uint32_t)((ss >> 1) & 1)))) break;
        tc::fence_after_sync();
        if (j == nb - 1) {
          // the item's last S MMA has completed, so the Q region is free: start copying the next
          // item's queries, which land while this block's softmax runs
          in = next_item();
          if (in.w >= 0) copy_queries(in.t);
        }
        uint32_t sv[4][32];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) tc::ld32(lane_addr + 128 * sb + 32 * q4, sv[q4]);
        tc::wait_ld();
        const int k0 = b * kKeys;  // position of the block's first key
        float x[kKeys];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
#pragma unroll
          for (int e = 0; e < 32; ++e) x[32 * q4 + e] = __uint_as_float(sv[q4][e]);
        // keys outside the row's range [start, pos] or in pages not loaded take no part (the warp
        // skips the test when every row of it sees the whole block)
        const bool whole = loaded == 0xff && k0 >= start && k0 + kKeys - 1 <= pos;
        if (!__all_sync(kAll, whole)) {
          const int lo = start - k0, hi = pos - k0;
#pragma unroll
          for (int c = 0; c < kKeys; ++c)
            x[c] = (((loaded >> (c >> 4)) & 1) && c >= lo && c <= hi) ? x[c] : -INFINITY;
        }
        // row max of the raw scores (eight independent chains), then scaled: sm_scale > 0
        float mx[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[i] = x[i];
#pragma unroll
        for (int c = 8; c < kKeys; ++c) mx[c & 7] = fmaxf(mx[c & 7], x[c]);
        const float mraw = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])), fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
        const float mb = mraw * p.scale_log2;  // -inf stays -inf
        // raise the running max only when a score exceeds it by more than 2^8
        const bool raise = mb > m + kLazy;
        const float m_new = raise ? mb : m;
        const float alpha = raise ? ex2(m - m_new) : 1.f;  // 0 on the first raise (m = -inf)
        const float m_use = m_new == -INFINITY ? 0.f : m_new;  // a row that sees no key yet: every P is 0
        float sums[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        uint32_t pk[kKeys / 2];
#pragma unroll
        for (int c = 0; c < kKeys; c += 2) {
          const float p0 = ex2(fmaf(x[c], p.scale_log2, -m_use));  // exp2(-inf) = 0 for masked keys
          const float p1 = ex2(fmaf(x[c + 1], p.scale_log2, -m_use));
          const __half2 h = __floats2half2_rn(p0, p1);
          const float2 f = __half22float2(h);  // the denominator adds the rounded values P V uses
          sums[(c >> 1) & 7] += f.x + f.y;
          pk[c / 2] = *reinterpret_cast<const uint32_t*>(&h);
        }
        const float sum = ((sums[0] + sums[1]) + (sums[2] + sums[3])) + ((sums[4] + sums[5]) + (sums[6] + sums[7]));
        l = l * alpha + sum;
        m = m_new;
        // P into the block's S buffer (the scores were read above), two fp16 per column
        tc::st32(lane_addr + 128 * sb, *reinterpret_cast<const uint32_t(*)[32]>(&pk[0]));
        tc::st32(lane_addr + 128 * sb + 32, *reinterpret_cast<const uint32_t(*)[32]>(&pk[32]));
        // key row r of the block's V: zero it when its key lies past the sequence end or in a
        // page that was not loaded (its contents are stale or a NaN sentinel)
        const bool zero_v = !(((loaded >> (r >> 4)) & 1) && k0 + r < t.len);
        if (__any_sync(kAll, zero_v)) {
          if (!(ok = wait(&sh.v_full[vst], (uint32_t)((kvs / kVStages) & 1)))) break;
          if (zero_v) {
            unsigned char* vrow = base + G::V_OFF + vst * G::KV_BYTES + (r >> 3) * G::ROWGRP + (r & 7) * G::SW;
#pragma unroll
            for (int u = 0; u < G::NA; ++u)
#pragma unroll
              for (int c = 0; c < G::SW / 16; ++c)
                *reinterpret_cast<uint4*>(vrow + u * G::GROUP + 16 * c) = make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
        }
        // O is quiescent once the previous block's P V has completed: rescale it then, if the
        // running max was raised
        if (j > 0) {
          if (!(ok = wait(&sh.o_done, (uint32_t)(pw & 1)))) break;
          ++pw;
          tc::fence_after_sync();
          if (__any_sync(kAll, raise)) {  // tensor-memory loads and stores are warp-wide (alpha = 1 elsewhere)
#pragma unroll 1
            for (int c = 0; c < D; c += 32) {
              uint32_t ov[32];
              tc::ld32(lane_addr + 256 + c, ov);
              tc::wait_ld();
#pragma unroll
              for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
              tc::st32(lane_addr + 256 + c, ov);
            }
          }
        }
        tc::wait_st();
        tc::fence_before_sync();
        mbar_arrive(&sh.p_full);
      }
      if (!ok) break;
      // publish the next item's queries, so that its first S MMA can run during this epilogue
      if (in.w >= 0) {
        cp_async_wait_all();
        fence_proxy_async_smem();
        mbar_arrive(&sh.q_full);
      }
      // the last block's P V, then the row of O
      if (!(ok = wait(&sh.o_done, (uint32_t)(pw & 1)))) break;
      ++pw;
      tc::fence_after_sync();
      float mm = m, scale = 1.f, lt = l;
      if (p.sinks != nullptr && valid) {
        const float sl = p.sinks[head] * kLog2e;
        const float M2 = fmaxf(mm, sl);
        scale = exp2f(mm - M2);
        lt = lt * scale + exp2f(sl - M2);
        mm = M2;
      }
      const bool any = lt > 0.f;
      const float inv = any ? scale / lt : 0.f;
      __half* dst = p.out + ((long long)tok * p.hq + head) * D;
#pragma unroll 1
      for (int c = 0; c < D; c += 32) {
        uint32_t ov[32];
        tc::ld32(lane_addr + 256 + c, ov);
        tc::wait_ld();
        if (valid) {
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            uint4 o;
            o.x = pack_half2(__uint_as_float(ov[e]) * inv, __uint_as_float(ov[e + 1]) * inv);
            o.y = pack_half2(__uint_as_float(ov[e + 2]) * inv, __uint_as_float(ov[e + 3]) * inv);
            o.z = pack_half2(__uint_as_float(ov[e + 4]) * inv, __uint_as_float(ov[e + 5]) * inv);
            o.w = pack_half2(__uint_as_float(ov[e + 6]) * inv, __uint_as_float(ov[e + 7]) * inv);
            *reinterpret_cast<uint4*>(dst + c + e) = o;
          }
        }
      }
      if (valid && p.lse != nullptr) p.lse[(long long)tok * p.hq + head] = any ? (mm + log2f(lt)) * kLn2 : -INFINITY;
      tc::fence_before_sync();  // the O reads above come before the next tile's first P V
      it = in;
      q_ready = in.w >= 0;
    }
    cp_async_wait_all();  // (after a timeout) no query copy may land in a finished CTA's memory
  }
  tc::fence_before_sync();
  __syncthreads();
  // the last CTA to finish (every CTA has taken its last item) resets the work counter for the
  // next launch, which reads it only after its launch wait
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(p.work + 1, 1) == (int)gridDim.x - 1) {
      atomicExch(p.work, 0);
      atomicExch(p.work + 1, 0);
    }
  }
  if (warp == 1) {
    tc::fence_after_sync();
    tc::dealloc(tmem, kTmemCols);
  }
}

template <int D>
size_t prefill_smem(int batch) {
  // operand regions, the barriers, the work prefix and the sort order, and the alignment slack;
  // at least 120 KB, so that two CTAs (each holding all tensor-memory columns) never share an SM
  const size_t need = 1024 + Geo<D>::BAR_OFF + sizeof(Shared) + (size_t)(batch + 1) * 4 +
                      (batch <= kMaxSortedBatch ? (size_t)(2 * batch) * 4 : 0);
  return need < 122880 ? 122880 : need;
}

}  // namespace

PrefillConfig prefill_config(int head_dim, int batch) {
  PrefillConfig c;
  const size_t budget = 232448 - 1024;
  c.smem_bytes = head_dim == 64 ? prefill_smem<64>(batch) : head_dim == 96 ? prefill_smem<96>(batch)
                                                                            : prefill_smem<128>(batch);
  c.nstage = c.smem_bytes <= budget ? kKStages : 0;
  if (c.nstage == 0) c.smem_bytes = 0;
  return c;
}

cudaError_t prefill_prepare() {
  const void* k[] = {(const void*)&prefill_kernel<64>, (const void*)&prefill_kernel<96>,
                     (const void*)&prefill_kernel<128>};
  for (const void* f : k) {
    cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448 - 1024);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_prefill(const PrefillParams& p, const CUtensorMap& map, const PrefillConfig& cfg, int head_dim,
                           int grid, cudaStream_t stream, bool pdl) {
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(grid);
  lc.blockDim = dim3(kThreads);
  lc.dynamicSmemBytes = cfg.smem_bytes;
  lc.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = pdl ? 1 : 0;
  void* args[] = {const_cast<CUtensorMap*>(&map), const_cast<PrefillParams*>(&p)};
  const void* k = head_dim == 64 ? (const void*)&prefill_kernel<64>
                  : head_dim == 96 ? (const void*)&prefill_kernel<96>
                                   : (const void*)&prefill_kernel<128>;
  return cudaLaunchKernelExC(&lc, k, args);
}

}  // namespace pkv
