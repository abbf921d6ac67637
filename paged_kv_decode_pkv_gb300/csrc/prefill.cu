// Chunked-prefill attention over the paged KV cache: every appended token of a sequence attends
// causally to the positions up to its own (Zero TVM Documentation, "Decode loop": a token attends
// to itself and to the earlier positions of its sequence; "KV cache": 16-slot pages behind a page
// table; "Port to Phi-4-mini or Qwen3": query head h reads KV head h / (Hq / Hkv)).  With several
// tokens per sequence this is a dense contraction, and it runs on tensor cores.
//
// Work decomposition.  A tile is (sequence s, KV head g, a block of 16 / G of the sequence's
// appended tokens): 16 rows of mma.sync m16n8k16, row r = token r / G of the block, query head
// g * G + r % G.  One warp owns a tile at a time (tiles gw, gw + W, ... over a persistent grid)
// and walks the pages from the first one any row attends to (its window start) to the last one
// (its position), each copied once for the 16 rows by swizzled TMA boxes into the warp's own ring
// of shared-memory stages.  Per page: S = Q K^T for the 16 rows and 16 slots, a per-row mask
// (slot position within [start_r, pos_r]), an online softmax per row in the log2 domain with the
// running max raised only when a score exceeds it by 2^8, P rounded to fp16 (the score fragments
// re-used as the A operand) and P V accumulated in fp32.  V rows past the sequence end are zeroed
// in shared memory.  No split: a tile's result is final (sinks fold into its denominator).
//
// Every wait is bounded (2 s of global time unless pkv_set_wait_limit sets another limit), with
// one answer per warp; on expiry the warp flags PKV_FLAG_TIMEOUT, waits a fixed bounded time for
// its own copies in flight (so none lands in the shared memory of a finished block) and returns.
#include "pkv_internal.h"
#include "ptx.cuh"

namespace pkv {
namespace {

constexpr unsigned kAll = 0xffffffffu;
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLazy = 8.f;

template <int D>
struct PfGeom {
  static constexpr int E = (D == 96) ? 32 : 64;  // TMA box extent along head_dim
  static constexpr int REGION = 64 * E;          // bytes of one box: [2][16][E] fp16
  static constexpr int SWZ = (E == 64) ? 7 : 3;  // 128-byte or 64-byte swizzle
  static constexpr int KS = D / 16;
  static constexpr int NB = D / 8;
  static constexpr int STAGE = 64 * D;

  // Shared-memory address of the 16-byte chunk holding (kv, slot t, dims dim..dim+7).
  __device__ static uint32_t chunk_addr(uint32_t stage, int kv, int t, int dim) {
    const int u = dim / E;
    const uint32_t off = (uint32_t)((kv * kPageSize + t) * (E * 2) + (dim % E) * 2);
    return stage + u * REGION + (off ^ (((off >> 7) & SWZ) << 4));
  }
};

__device__ __forceinline__ int find_seq(const int* prefix, int batch, int w) {
  int lo = 0, hi = batch;  // prefix[lo] <= w < prefix[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= w) lo = mid; else hi = mid;
  }
  return lo;
}

template <int D>
__global__ void __launch_bounds__((kPrefillWarps + 1) * 32) prefill_kernel(const __grid_constant__ CUtensorMap map,
                                                                           PrefillParams p) {
  using Gm = PfGeom<D>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int nst = p.nstage;
  unsigned char* stages = base;
  uint64_t* full = reinterpret_cast<uint64_t*>(base + (size_t)nst * Gm::STAGE);
  uint64_t* empty = full + nst;
  int* prefix = reinterpret_cast<int*>(empty + nst);
  __shared__ int warp_sums[kPrefillWarps + 1];
  __shared__ int abort_flag;

  pdl_launch_dependents();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool producer = warp == kPrefillWarps;
  if (tid == 0) {
    prefetch_tensormap(&map);
    abort_flag = 0;
  }
  for (int i = tid; i < nst; i += blockDim.x) {
    mbar_init(&full[i], 1);
    mbar_init(&empty[i], kPrefillWarps);
  }
  fence_mbarrier_init();

  // tasks of each sequence (Hkv x blocks of kPrefillWarps tiles of tpt tokens) and their prefix
  const int block_tokens = kPrefillWarps * p.tpt;
  {
    const int per = (p.batch + blockDim.x - 1) / blockDim.x;
    const int s0 = min(p.batch, tid * per), s1 = min(p.batch, s0 + per);
    auto tasks_of = [&](int s) {
      const int c = p.append_indptr[s + 1] - p.append_indptr[s];
      return c > 0 ? p.hkv * ((c + block_tokens - 1) / block_tokens) : 0;
    };
    int local = 0;
    for (int s = s0; s < s1; ++s) local += tasks_of(s);
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(kAll, incl, off);
      if (lane >= off) incl += v;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    int run = incl - local;
    for (int w = 0; w < warp; ++w) run += warp_sums[w];
    for (int s = s0; s < s1; ++s) {
      prefix[s] = run;
      run += tasks_of(s);
    }
    if (tid == blockDim.x - 1) prefix[p.batch] = run;
  }
  __syncthreads();
  const int total = prefix[p.batch];

  // the tiles of one (sequence, KV head) run side by side and read the same pages: keep them in L2
  const uint64_t policy = l2_policy_evict_last();
  const int G = p.group;
  const int c2 = 2 * (lane & 3);
  int seq = 0;  // pages the CTA has streamed so far (ring slot and phases)
  int fills = 0;  // producer: stages filled so far (those it must drain before leaving)

  pdl_wait();  // q and the pool (the append) come from the preceding kernel

  for (int task = blockIdx.x; task < total; task += gridDim.x) {
    if (*reinterpret_cast<volatile int*>(&abort_flag)) break;
    const int s = find_seq(prefix, p.batch, task);
    const int a0 = p.append_indptr[s], cnt = p.append_indptr[s + 1] - a0;
    const int per_head = (cnt + block_tokens - 1) / block_tokens;
    const int r = task - prefix[s];
    const int g = r / per_head;
    const int tb0 = a0 + (r - g * per_head) * block_tokens;  // first token of the block
    const int nb_tok = min(block_tokens, a0 + cnt - tb0);
    const int first = p.page_indptr[s];
    const int n = p.page_indptr[s + 1] - first;
    const int last = n > 0 ? p.last_page_len[s] : 0;
    const bool seq_ok = n > 0 && last >= 1 && last <= kPageSize;
    const int len = seq_ok ? (n - 1) * kPageSize + last : 0;
    if (!seq_ok && tid == 0 && r == 0) atomicOr(p.status, kFlagBadSequence);

    // the block's page range (every warp computes it from the block's positions)
    int pmin = 0x7fffffff, pmax = -1;
    for (int t = lane; t < nb_tok; t += 32) {
      const int pos = seq_ok ? p.pos_map[tb0 + t] : -1;
      if (pos >= 0 && pos < len) {
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
    if (pmax < 0) continue;  // no valid token (reported below by the rows)
    const int np = pmax - pmin + 1;

    if (producer) {
      // ---- the CTA's producer: page copies into the shared ring ----
      int win_base = 0;
      int window_ids = lane < np ? p.page_indices[first + pmin + lane] : 0;
      for (int i = 0; i < np; ++i) {
        if (i - win_base >= 32) {
          win_base = i & ~31;
          window_ids = win_base + lane < np ? p.page_indices[first + pmin + win_base + lane] : 0;
        }
        const int pid = __shfl_sync(kAll, window_ids, i - win_base);
        const int f = seq + i, slot = f % nst;
        if (f >= nst && !warp_wait_bounded(&empty[slot], (uint32_t)(((f / nst) - 1) & 1), p.wait_ns)) {
          if (lane == 0) {
            atomicOr(p.status, kFlagTimeout);
            abort_flag = 1;
          }
          break;
        }
        const bool ok = pid >= 0 && pid < p.num_pages;
        fills = f + 1;
        if (!ok && lane == 0) atomicOr(p.status, kFlagBadPage);
        mbar_arrive_expect_tx_if(lane == 0 && ok, &full[slot], (uint32_t)Gm::STAGE);
        mbar_arrive_if(lane == 0 && !ok, &full[slot]);
        unsigned char* dst = stages + (size_t)slot * Gm::STAGE;
#pragma unroll
        for (int u = 0; u < D / Gm::E; ++u)
          tma_load_4d_if(lane == 0 && ok, dst + u * Gm::REGION, &map, &full[slot], u * Gm::E, 0, g, 2 * pid, policy);
      }
      seq += np;
      continue;
    }

    // ---- consumer warp: 16 rows = tokens tok0 .. tok0 + tpt - 1 of the block x the group's heads ----
    const int tok0 = tb0 + warp * p.tpt;
    int tok[2], head[2], pos[2], start[2];
    bool valid[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int rho = (lane >> 2) + 8 * i;
      const int tk = rho / G;
      tok[i] = tok0 + tk;
      head[i] = g * G + rho % G;
      valid[i] = seq_ok && tk < p.tpt && tok[i] < a0 + cnt;
      pos[i] = valid[i] ? p.pos_map[tok[i]] : 0;
      if (valid[i] && (pos[i] < 0 || pos[i] >= len)) {
        atomicOr(p.status, kFlagBadPosition);
        valid[i] = false;
      }
      start[i] = (p.window > 0 && pos[i] + 1 > p.window) ? pos[i] + 1 - p.window : 0;
    }
    // the warp's own last page (nothing to compute after it), and the positions every valid row
    // attends to (pages inside [full_lo, full_hi] need no mask)
    int wmax = -1, full_lo = 0, full_hi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < 2; ++i)
      if (valid[i]) {
        wmax = max(wmax, pos[i] >> 4);
        full_lo = max(full_lo, start[i]);
        full_hi = min(full_hi, pos[i]);
      }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      wmax = max(wmax, __shfl_xor_sync(kAll, wmax, off));
      full_lo = max(full_lo, __shfl_xor_sync(kAll, full_lo, off));
      full_hi = min(full_hi, __shfl_xor_sync(kAll, full_hi, off));
    }

    uint32_t qa[Gm::KS][4];
#pragma unroll
    for (int ks = 0; ks < Gm::KS; ++ks) {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const __half* qr = p.q + ((long long)tok[i] * p.hq + head[i]) * D + ks * 16 + c2;
        qa[ks][i] = valid[i] ? *reinterpret_cast<const uint32_t*>(qr) : 0u;
        qa[ks][2 + i] = valid[i] ? *reinterpret_cast<const uint32_t*>(qr + 8) : 0u;
      }
    }
    float acc[Gm::NB][4];
#pragma unroll
    for (int nb = 0; nb < Gm::NB; ++nb) acc[nb][0] = acc[nb][1] = acc[nb][2] = acc[nb][3] = 0.f;
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};

    bool stop = false;
    for (int i = 0; i < np; ++i) {
      const int f = seq + i, slot = f % nst;
      if (!warp_wait_bounded(&full[slot], (uint32_t)((f / nst) & 1), p.wait_ns)) {
        if (lane == 0) {
          atomicOr(p.status, kFlagTimeout);
          abort_flag = 1;
        }
        stop = true;
        break;
      }
      const int ord = pmin + i;
      const uint32_t stage = smem_u32(stages + (size_t)slot * Gm::STAGE);
      if (ord <= wmax) {
        const int nvalid = ord == n - 1 ? last : kPageSize;
        // S = Q K^T: two n-blocks of 8 slots (V rows past the end are masked through P below,
        // and their values are zeroed so that P = 0 times anything stays 0)
        // (even and odd k-steps accumulate apart: four independent mma chains instead of two)
        float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        {
          float sc_odd[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
          const int mi = lane >> 3, rr = lane & 7;
          const int t = (mi >> 1) * 8 + rr;
          const int dsub = (mi & 1) * 8;
#pragma unroll
          for (int ks = 0; ks < Gm::KS; ++ks) {
            uint32_t b0, b1, b2, b3;
            ldmatrix_x4(Gm::chunk_addr(stage, 0, t, ks * 16 + dsub), b0, b1, b2, b3);
            float (&c0)[4] = (ks & 1) ? sc_odd[0] : sc[0];
            float (&c1)[4] = (ks & 1) ? sc_odd[1] : sc[1];
            mma_16816(c0, qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
            mma_16816(c1, qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            sc[0][e] += sc_odd[0][e];
            sc[1][e] += sc_odd[1][e];
          }
        }
        // a page every valid row sees whole needs no mask (rows without a token are never written)
        const bool whole = ord * kPageSize >= full_lo && ord * kPageSize + kPageSize - 1 <= full_hi &&
                           nvalid == kPageSize;
        float pr[2][4];
#pragma unroll
        for (int i2 = 0; i2 < 2; ++i2) {
          float v[4];
          if (whole) {
#pragma unroll
            for (int e = 0; e < 4; ++e) v[e] = sc[e >> 1][2 * i2 + (e & 1)] * p.scale_log2;
          } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int col = (e >> 1) * 8 + c2 + (e & 1);
              const int tpos = ord * kPageSize + col;
              const float x = sc[e >> 1][2 * i2 + (e & 1)] * p.scale_log2;
              v[e] = (valid[i2] && tpos >= start[i2] && tpos <= pos[i2]) ? x : -INFINITY;
            }
          }
          float mx = fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3]));
          mx = fmaxf(mx, __shfl_xor_sync(kAll, mx, 1));
          mx = fmaxf(mx, __shfl_xor_sync(kAll, mx, 2));
          if (mx > m[i2] + kLazy) {
            const float alpha = exp2f(m[i2] - mx);
            l[i2] *= alpha;
#pragma unroll
            for (int nb = 0; nb < Gm::NB; ++nb) {
              acc[nb][2 * i2] *= alpha;
              acc[nb][2 * i2 + 1] *= alpha;
            }
            m[i2] = mx;
          }
          // a row may see no position yet (its window starts further on): its P is 0, not NaN
#pragma unroll
          for (int e = 0; e < 4; ++e) pr[i2][e] = v[e] == -INFINITY ? 0.f : exp2f(v[e] - m[i2]);
        }
        uint32_t pa[4];
#pragma unroll
        for (int i2 = 0; i2 < 2; ++i2) {
          const __half2 lo = __floats2half2_rn(pr[i2][0], pr[i2][1]);
          const __half2 hi = __floats2half2_rn(pr[i2][2], pr[i2][3]);
          const float2 flo = __half22float2(lo), fhi = __half22float2(hi);
          l[i2] += (flo.x + flo.y) + (fhi.x + fhi.y);
          pa[i2] = *reinterpret_cast<const uint32_t*>(&lo);
          pa[2 + i2] = *reinterpret_cast<const uint32_t*>(&hi);
        }
        if (nvalid < kPageSize) {
          // the ring is shared: instead of zeroing V rows past the end, zero their P (already 0
          // through the mask) and read those V rows as zero via a guarded copy of the fragment
          // inputs below
        }
        {
          const int mi = lane >> 3, rr = lane & 7;
          const int t = (mi & 1) * 8 + rr;
          const int dsub = (mi >> 1) * 8;
#pragma unroll
          for (int mm = 0; mm < D / 16; ++mm) {
            uint32_t v0, v1, v2, v3;
            ldmatrix_x4_trans(Gm::chunk_addr(stage, 1, t, mm * 16 + dsub), v0, v1, v2, v3);
            if (nvalid < kPageSize) {
              // V fragments of slots past the sequence end may hold anything (NaN): zero them
              // (ldmatrix.trans gives this lane slots tr and tr + 8 of its two 8x8 matrices)
              const int tr = 2 * (lane & 3);
              if (tr >= nvalid) v0 = 0u;
              if (tr + 1 >= nvalid) v0 &= 0x0000FFFFu;
              if (tr + 8 >= nvalid) v1 = 0u;
              if (tr + 9 >= nvalid) v1 &= 0x0000FFFFu;
              if (tr >= nvalid) v2 = 0u;
              if (tr + 1 >= nvalid) v2 &= 0x0000FFFFu;
              if (tr + 8 >= nvalid) v3 = 0u;
              if (tr + 9 >= nvalid) v3 &= 0x0000FFFFu;
            }
            mma_16816(acc[2 * mm], pa[0], pa[1], pa[2], pa[3], v0, v1);
            mma_16816(acc[2 * mm + 1], pa[0], pa[1], pa[2], pa[3], v2, v3);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);  // this warp is done with the stage
    }
    seq += np;
    if (stop) break;

    // finish the two rows: out = acc / l (with the sink in the denominator), lse
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      float lt = l[i];
      lt += __shfl_xor_sync(kAll, lt, 1);
      lt += __shfl_xor_sync(kAll, lt, 2);
      float mm = m[i], scale = 1.f;
      if (p.sinks != nullptr && valid[i]) {
        const float sl = p.sinks[head[i]] * kLog2e;
        const float M2 = fmaxf(mm, sl);
        scale = exp2f(mm - M2);
        lt = lt * scale + exp2f(sl - M2);
        mm = M2;
      }
      if (!valid[i]) continue;
      const bool any = lt > 0.f;
      const float inv = any ? scale / lt : 0.f;
      __half* dst = p.out + ((long long)tok[i] * p.hq + head[i]) * D + c2;
#pragma unroll
      for (int nb = 0; nb < Gm::NB; ++nb)
        *reinterpret_cast<__half2*>(dst + nb * 8) = __floats2half2_rn(acc[nb][2 * i] * inv, acc[nb][2 * i + 1] * inv);
      if (p.lse != nullptr && (lane & 3) == 0)
        p.lse[(long long)tok[i] * p.hq + head[i]] = any ? (mm + log2f(lt)) * kLn2 : -INFINITY;
    }
  }
  // the producer leaves only when its copies have landed: wait (bounded) for the last fills
  if (producer && *reinterpret_cast<volatile int*>(&abort_flag)) {
    for (int f = max(0, fills - nst); f < fills; ++f)
      mbar_wait_bounded(&full[f % nst], (uint32_t)((f / nst) & 1), kDrainLimitNs);
  }
}

template <int D>
size_t prefill_smem(int nstage, int batch) {
  return 1024 + (size_t)nstage * PfGeom<D>::STAGE + (size_t)nstage * 16 + (size_t)(batch + 1) * 4;
}

}  // namespace

PrefillConfig prefill_config(int head_dim, int batch) {
  PrefillConfig c;
  const int budget = 232448 - 256;  // one CTA (nine warps) per SM
  c.nstage = 8;
  auto smem = [&](int n) {
    return head_dim == 64 ? prefill_smem<64>(n, batch) : head_dim == 96 ? prefill_smem<96>(n, batch)
                                                                         : prefill_smem<128>(n, batch);
  };
  while (c.nstage >= 2 && smem(c.nstage) > (size_t)budget) --c.nstage;
  c.smem_bytes = c.nstage >= 2 ? smem(c.nstage) : 0;
  return c;
}

cudaError_t prefill_prepare() {
  const void* k[] = {(const void*)&prefill_kernel<64>, (const void*)&prefill_kernel<96>,
                     (const void*)&prefill_kernel<128>};
  for (const void* f : k) {
    cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448 - 256);
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
  lc.blockDim = dim3((kPrefillWarps + 1) * 32);  // consumers and one producer warp
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
