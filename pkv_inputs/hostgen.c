/*
 * Seeded synthetic inputs, host side.
 *
 * This file is shared input generation: it holds none of the attention
 * method's arithmetic (no RoPE, no paging, no softmax).  The device twin in
 * devgen.cu implements the very same definitions so that a tensor filled on
 * the GPU is bit-identical to the one filled here.
 *
 * Definitions (both files implement exactly these):
 *
 *   mix64(z)        SplitMix64 output finaliser (Steele, Lea, Flood, "Fast
 *                   splittable pseudorandom number generators", OOPSLA 2014;
 *                   constants of Vigna's public-domain splitmix64.c).
 *   key(seed, tag)  = mix64(seed ^ mix64(tag))
 *   word(key, i)    = mix64(key + (i + 1) * 0x9e3779b97f4a7c15)
 *                   i.e. the i-th output of a SplitMix64 generator whose state
 *                   starts at `key` (counter-based: any i can be computed
 *                   directly, in any order, on any thread).
 *   normal(key, i)  Irwin-Hall approximation of N(0,1): the twelve 16-bit
 *                   halves of word(key,3i), word(key,3i+1), word(key,3i+2)
 *                   are summed; x = (sum - 393210) * 2^-16 exactly in fp32
 *                   (mean 0, variance 1 - 2^-32, support [-6, 6]).
 *   value(i)        f = x * (outlier(i) ? 8 : 1)      exact in fp32
 *                   f = f * scale                     one fp32 rounding
 *                   fp16 = round-to-nearest-even(f)
 *   outlier(i)      when enabled: row r = i / row_len is an outlier row iff
 *                   word(okey, r) % 100 < pct.
 */
#include <stdint.h>
#include <string.h>

#define PKVGEN_GAMMA 0x9e3779b97f4a7c15ULL

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ULL;
  z = (z ^ (z >> 27)) * 0x94d049bb133111ebULL;
  return z ^ (z >> 31);
}

uint64_t pkvgen_key(uint64_t seed, uint64_t tag) { return mix64(seed ^ mix64(tag)); }

uint64_t pkvgen_word(uint64_t key, uint64_t i) { return mix64(key + (i + 1) * PKVGEN_GAMMA); }

static inline float normal_f32(uint64_t key, uint64_t i) {
  int32_t sum = 0;
  for (int w = 0; w < 3; ++w) {
    uint64_t u = pkvgen_word(key, 3 * i + (uint64_t)w);
    sum += (int32_t)(u & 0xffff) + (int32_t)((u >> 16) & 0xffff) + (int32_t)((u >> 32) & 0xffff) +
           (int32_t)(u >> 48);
  }
  return (float)(sum - 393210) * (1.0f / 65536.0f);
}

static inline uint16_t f32_to_f16_bits(float f) {
  _Float16 h = (_Float16)f; /* IEEE binary16, round to nearest even */
  uint16_t b;
  memcpy(&b, &h, 2);
  return b;
}

static inline uint16_t value_bits(uint64_t key, uint64_t i, float scale, uint64_t okey,
                                  uint64_t row_len, int pct) {
  float f = normal_f32(key, i);
  if (pct > 0 && (pkvgen_word(okey, i / row_len) % 100u) < (uint64_t)pct) f = f * 8.0f;
  return f32_to_f16_bits(f * scale); /* one fp32 rounding, then one fp16 rounding */
}

/* dst[j] = value(first + j), j in [0, n).  pct = 0 disables outliers. */
void pkvgen_fill_range(uint16_t* dst, int64_t n, uint64_t key, int64_t first, float scale,
                       uint64_t okey, int64_t row_len, int pct) {
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < n; ++j)
    dst[j] = value_bits(key, (uint64_t)(first + j), scale, okey, (uint64_t)row_len, pct);
}

/* Gathered fill: for each listed block b, dst[b][e] = value(blocks[b]*block_elems + e).
 * Used to regenerate only some pages of a large pool. */
void pkvgen_fill_blocks(uint16_t* dst, const int64_t* blocks, int64_t nblocks, int64_t block_elems,
                        uint64_t key, float scale, uint64_t okey, int64_t row_len, int pct) {
#pragma omp parallel for schedule(static)
  for (int64_t b = 0; b < nblocks; ++b) {
    uint64_t base = (uint64_t)blocks[b] * (uint64_t)block_elems;
    for (int64_t e = 0; e < block_elems; ++e)
      dst[b * block_elems + e] = value_bits(key, base + (uint64_t)e, scale, okey, (uint64_t)row_len, pct);
  }
}

/* Raw 64-bit words, for seeded integer draws (lengths, permutations). */
void pkvgen_words(uint64_t* dst, int64_t n, uint64_t key, int64_t first) {
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < n; ++j) dst[j] = pkvgen_word(key, (uint64_t)(first + j));
}
