/*
 * ORACLE for the decode-step paged-KV attention path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
 * CPU-baseline / reference arm load this library; the product path (the CUDA
 * library and its Python binding) never does, and it shares no code with it.
 *
 * Plain, slow, obviously correct: fp64 arithmetic from fp16 inputs, one loop
 * per definition, OpenMP only across independent (sequence, head) pairs.
 *
 * What it follows (page title, section):
 *  - Zero TVM Documentation, "KV cache": fixed pages of 16 slots, a page table
 *    mapping logical positions to physical pages, K rotated by RoPE before the
 *    cache write (a page is valid only at the positions it was written at).
 *  - Zero TVM Documentation, "Decode loop": per-step position map, page range
 *    per sequence, sequence length = position + 1 (the new token attends to
 *    itself); QKV + RoPE + KV-append in one dispatch, which also writes the
 *    rotated query (binding order q_out, k_out, v_out, qkv, posMap, "Debugging
 *    tips").
 *  - Zero TVM Documentation, "How it works": split-K attention over KV chunks
 *    followed by a combine dispatch per layer.
 *  - Zero TVM Documentation, "Port to Phi-4-mini or Qwen3": when KV heads are
 *    fewer than query heads, KV heads are repeated (query head h reads KV head
 *    h / (Hq/Hkv)).
 *
 * Readings where the pages are silent (each one is listed in the design notes):
 *  - RoPE is the rotate-half form over the whole head: element i pairs with
 *    i + d/2, inverse frequency theta^(-2i/d), angle = position * frequency.
 *  - Pool layout per layer: [page][K=0,V=1][kv_head][slot][dim], fp16.
 *  - softmax scale 1/sqrt(d); split chunks are page-aligned and contiguous;
 *    a chunk with no token gives o = 0 and lse = -inf (natural log); the
 *    combine of all-empty chunks gives out = 0 and lse = -inf.
 *  - fp16 results are rounded to nearest, ties to even.
 *  - Sliding window (Splash models page, the families' sliding_window and layer_types; Zero TVM
 *    Documentation, "Decode loop": the unused fields of lengthInfo): a layer with window W > 0
 *    lets the query at position len-1 attend to positions [max(0, len-W), len), the W most recent
 *    tokens including itself; W = 0 is full attention.
 *  - Attention sinks (Splash models page, a layer's attn_sinks, F32): one logit per query head,
 *    in the units of the scaled scores, that joins the softmax's denominator and carries no
 *    value: out = sum_t e^s_t V_t / (sum_t e^s_t + e^sink), lse = ln(sum_t e^s_t + e^sink).
 *    Split partials are unaffected; the sink enters the combine.  -inf means no sink.
 */
#include <math.h>
#include <omp.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_PAGE 16

enum { ORC_OK = 0, ORC_INVALID = 1, ORC_OUT_OF_RANGE = 3, ORC_DUPLICATE = 5 };

typedef struct {
  int num_pages;
  int num_qo_heads;
  int num_kv_heads;
  int head_dim;
  int max_position;
  double rope_theta;
} orc_geom;

/* ------------------------------------------------------------------------------------------ */
/* IEEE 754 binary16 <-> binary64, written from the format's definition.                       */

double orc_f16_to_f64(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int m = h & 0x3ff;
  double v;
  if (e == 0) {
    v = ldexp((double)m, -24); /* zero or subnormal: m * 2^-24 */
  } else if (e == 31) {
    v = m ? NAN : INFINITY;
  } else {
    v = ldexp((double)(1024 + m), e - 25); /* (1 + m/1024) * 2^(e-15) */
  }
  return sign ? -v : v;
}

/* Round to nearest binary16, ties to even. */
uint16_t orc_f64_to_f16(double x) {
  uint16_t sign = signbit(x) ? 0x8000 : 0;
  if (isnan(x)) return 0x7e00;
  double a = fabs(x);
  if (isinf(a)) return sign | 0x7c00;
  if (a == 0.0) return sign;
  int e2;
  frexp(a, &e2);    /* a = f * 2^e2, f in [0.5, 1) */
  int E = e2 - 1;   /* floor(log2 a) */
  if (E < -14) E = -14; /* subnormal range shares the quantum 2^-24 */
  double quantum = ldexp(1.0, E - 10);
  double n = nearbyint(a / quantum); /* exact division; nearbyint rounds ties to even */
  double r = n * quantum;
  if (r >= 65536.0) return sign | 0x7c00; /* overflow */
  if (r < ldexp(1.0, -14)) return sign | (uint16_t)(r / ldexp(1.0, -24)); /* subnormal */
  int er;
  frexp(r, &er);
  int Er = er - 1;
  uint16_t mant = (uint16_t)(r / ldexp(1.0, Er - 10) - 1024.0);
  return sign | (uint16_t)((Er + 15) << 10) | mant;
}

/* Threads the OpenMP loops below use (reported with CPU timings). */
int orc_threads(void) { return omp_get_max_threads(); }

static double g_f16_table[65536];
static int g_table_ready = 0;

/* Fill the decode cache (a table of orc_f16_to_f64 for every bit pattern). */
void orc_init(void) {
  if (g_table_ready) return;
  for (int i = 0; i < 65536; ++i) g_f16_table[i] = orc_f16_to_f64((uint16_t)i);
  g_table_ready = 1;
}

static inline double dec(uint16_t h) { return g_f16_table[h]; }

void orc_f16_decode_array(const uint16_t* in, double* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_f16_to_f64(in[i]);
}

void orc_f16_encode_array(const double* in, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_f64_to_f16(in[i]);
}

/* ------------------------------------------------------------------------------------------ */
/* RoPE (rotate-half), fp64.                                                                   */

void orc_rope(const double* x, double* y, int d, int64_t pos, double theta) {
  int half = d / 2;
  for (int i = 0; i < half; ++i) {
    double inv_freq = pow(theta, -2.0 * (double)i / (double)d);
    double phi = (double)pos * inv_freq;
    double c = cos(phi), s = sin(phi);
    double a = x[i], b = x[i + half];
    y[i] = a * c - b * s;
    y[i + half] = b * c + a * s;
  }
}

/* ------------------------------------------------------------------------------------------ */
/* Append: rotate q and k at their positions, write k and v into the page slots.               */

static int64_t pool_row(const orc_geom* g, int64_t page, int kv, int head, int slot) {
  /* element offset of pool[page][kv][head][slot][0] */
  return (((page * 2 + kv) * g->num_kv_heads + head) * (int64_t)ORC_PAGE + slot) * g->head_dim;
}

static int cmp_i32(const void* a, const void* b) {
  int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
  return (x > y) - (x < y);
}

int orc_append(const orc_geom* g, const uint16_t* q, const uint16_t* k, const uint16_t* v, int T,
               const int32_t* pos_map, const int32_t* append_indptr, int B,
               const int32_t* page_indptr, const int32_t* page_indices, uint16_t* pool,
               uint16_t* q_out) {
  orc_init();
  const int d = g->head_dim, Hq = g->num_qo_heads, Hkv = g->num_kv_heads;
  if (d <= 0 || d % 2 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || T < 0 || B < 0) return ORC_INVALID;
  if (append_indptr[0] != 0 || append_indptr[B] != T || page_indptr[0] != 0) return ORC_INVALID;
  for (int s = 0; s < B; ++s)
    if (append_indptr[s + 1] < append_indptr[s] || page_indptr[s + 1] < page_indptr[s]) return ORC_INVALID;

  /* validate every token before writing anything */
  for (int s = 0; s < B; ++s) {
    int t0 = append_indptr[s], t1 = append_indptr[s + 1];
    int n_pages = page_indptr[s + 1] - page_indptr[s];
    for (int t = t0; t < t1; ++t) {
      int p = pos_map[t];
      if (p < 0 || p >= g->max_position) return ORC_OUT_OF_RANGE;
      if (p / ORC_PAGE >= n_pages) return ORC_OUT_OF_RANGE;
      int page = page_indices[page_indptr[s] + p / ORC_PAGE];
      if (page < 0 || page >= g->num_pages) return ORC_OUT_OF_RANGE;
    }
    if (t1 - t0 > 1) {
      int32_t* sorted = (int32_t*)malloc(sizeof(int32_t) * (size_t)(t1 - t0));
      memcpy(sorted, pos_map + t0, sizeof(int32_t) * (size_t)(t1 - t0));
      qsort(sorted, (size_t)(t1 - t0), sizeof(int32_t), cmp_i32);
      int dup = 0;
      for (int i = 1; i < t1 - t0; ++i) dup |= (sorted[i] == sorted[i - 1]);
      free(sorted);
      if (dup) return ORC_DUPLICATE;
    }
  }

  double* x = (double*)malloc(sizeof(double) * (size_t)d);
  double* y = (double*)malloc(sizeof(double) * (size_t)d);
  for (int s = 0; s < B; ++s) {
    for (int t = append_indptr[s]; t < append_indptr[s + 1]; ++t) {
      int p = pos_map[t];
      int64_t page = page_indices[page_indptr[s] + p / ORC_PAGE];
      int slot = p % ORC_PAGE;
      for (int h = 0; h < Hq; ++h) {
        const uint16_t* src = q + ((int64_t)t * Hq + h) * d;
        for (int i = 0; i < d; ++i) x[i] = dec(src[i]);
        orc_rope(x, y, d, p, g->rope_theta);
        for (int i = 0; i < d; ++i) q_out[((int64_t)t * Hq + h) * d + i] = orc_f64_to_f16(y[i]);
      }
      for (int h = 0; h < Hkv; ++h) {
        const uint16_t* ks = k + ((int64_t)t * Hkv + h) * d;
        const uint16_t* vs = v + ((int64_t)t * Hkv + h) * d;
        for (int i = 0; i < d; ++i) x[i] = dec(ks[i]);
        orc_rope(x, y, d, p, g->rope_theta);
        uint16_t* kd = pool + pool_row(g, page, 0, h, slot);
        uint16_t* vd = pool + pool_row(g, page, 1, h, slot);
        for (int i = 0; i < d; ++i) kd[i] = orc_f64_to_f16(y[i]);
        memcpy(vd, vs, sizeof(uint16_t) * (size_t)d);
      }
    }
  }
  free(x);
  free(y);
  return ORC_OK;
}

/* ------------------------------------------------------------------------------------------ */
/* int8 KV pages (Zero TVM Documentation, "The memory-bandwidth ceiling": int8 KV is exposed
 * behind a flag; the format is this library's reading).
 * Layout per layer: uint8 pool8[num_pages][2][Hkv][16 * d + 64]: a block holds the 16 slots'
 * int8 codes, each stored as the unsigned byte code + 128 (offset binary), and then their fp32
 * scales [16]; the codes of a K block are slot-major [16][d], those of a V block dim-major [d][16]
 * (the 16 slots of one dimension together).
 * Row quantizer (one row = one token, one KV head, K or V, of d fp16 values x_i; K after RoPE and
 * its fp16 rounding, as the fp16 cache stores it): amax = max |x_i|; s = fp32(amax / 127) (fp32
 * division, nearest); code_i = clamp(rint_even(fp32(x_i / s)), -127, 127); amax = 0 gives s = 0 and
 * codes 0.  The decision is taken in fp32, the precision of the kernel.  The value of a slot is
 * code * s. */
static int64_t block8(const orc_geom* g, int64_t page, int kv, int head) {
  return ((page * 2 + kv) * g->num_kv_heads + head) * (int64_t)(16 * g->head_dim + 64);
}

/* Index of the code of (slot, dimension i) inside a K (kv = 0) or V (kv = 1) block. */
static int64_t code8(int d, int kv, int slot, int i) { return kv == 0 ? (int64_t)slot * d + i : (int64_t)i * 16 + slot; }

void orc_quantize_row(const uint16_t* x, int d, int8_t* codes, float* scale);

/* Quantize one row into its block: codes at code8(), the scale after the 16 x d codes. */
static void store_row8(uint8_t* blk, int d, int kv, int slot, const uint16_t* row) {
  int8_t codes[256];
  float sc;
  orc_quantize_row(row, d, codes, &sc);
  for (int i = 0; i < d; ++i) blk[code8(d, kv, slot, i)] = (uint8_t)(codes[i] + 128);
  memcpy(blk + 16 * d + 4 * slot, &sc, 4);
}

void orc_quantize_row(const uint16_t* x, int d, int8_t* codes, float* scale) {
  orc_init();
  float amax = 0.f;
  for (int i = 0; i < d; ++i) {
    const float a = fabsf((float)dec(x[i]));
    if (a > amax) amax = a;
  }
  const float s = amax / 127.0f;
  *scale = s;
  for (int i = 0; i < d; ++i) {
    if (s == 0.f) {
      codes[i] = 0;
      continue;
    }
    float q = nearbyintf((float)dec(x[i]) / s);
    if (q > 127.f) q = 127.f;
    if (q < -127.f) q = -127.f;
    codes[i] = (int8_t)q;
  }
}

/* The append into an int8 pool: orc_append's rotation and placement, then the row quantizer. */
int orc_append_int8(const orc_geom* g, const uint16_t* q, const uint16_t* k, const uint16_t* v, int T,
                    const int32_t* pos_map, const int32_t* append_indptr, int B, const int32_t* page_indptr,
                    const int32_t* page_indices, uint8_t* pool8, uint16_t* q_out) {
  orc_init();
  const int d = g->head_dim, Hkv = g->num_kv_heads;
  /* the fp16 append into a scratch pool of the same geometry gives the rows to quantize */
  const int64_t rows = (int64_t)g->num_pages * 2 * Hkv * ORC_PAGE;
  uint16_t* scratch = (uint16_t*)calloc((size_t)rows * d, sizeof(uint16_t));
  int rc = orc_append(g, q, k, v, T, pos_map, append_indptr, B, page_indptr, page_indices, scratch, q_out);
  if (rc == ORC_OK) {
    for (int s = 0; s < B; ++s) {
      for (int t = append_indptr[s]; t < append_indptr[s + 1]; ++t) {
        const int p = pos_map[t];
        const int64_t page = page_indices[page_indptr[s] + p / ORC_PAGE];
        const int slot = p % ORC_PAGE;
        for (int h = 0; h < Hkv; ++h)
          for (int kv = 0; kv < 2; ++kv)
            store_row8(pool8 + block8(g, page, kv, h), d, kv, slot, scratch + pool_row(g, page, kv, h, slot));
      }
    }
  }
  free(scratch);
  return rc;
}

/* Quantize every slot row of an fp16 pool into an int8 pool (cache contents before a step). */
void orc_quantize_pool(const orc_geom* g, const uint16_t* pool, uint8_t* pool8) {
  orc_init();
  const int d = g->head_dim, Hkv = g->num_kv_heads;
#pragma omp parallel for schedule(static)
  for (int64_t page = 0; page < g->num_pages; ++page)
    for (int kv = 0; kv < 2; ++kv)
      for (int h = 0; h < Hkv; ++h)
        for (int slot = 0; slot < ORC_PAGE; ++slot)
          store_row8(pool8 + block8(g, page, kv, h), d, kv, slot, pool + pool_row(g, page, kv, h, slot));
}

/* Dequantize an int8 pool into fp64 rows laid out like the fp16 pool: out[page][kv][head][slot][d]. */
void orc_dequantize_pool(const orc_geom* g, const uint8_t* pool8, double* out) {
  const int d = g->head_dim, Hkv = g->num_kv_heads;
  for (int64_t page = 0; page < g->num_pages; ++page)
    for (int kv = 0; kv < 2; ++kv)
      for (int h = 0; h < Hkv; ++h) {
        const uint8_t* blk = pool8 + block8(g, page, kv, h);
        for (int slot = 0; slot < ORC_PAGE; ++slot) {
          float sc;
          memcpy(&sc, blk + 16 * d + 4 * slot, 4);
          for (int i = 0; i < d; ++i)
            out[pool_row(g, page, kv, h, slot) + i] = (double)((int)blk[code8(d, kv, slot, i)] - 128) * (double)sc;
        }
      }
}

/* ------------------------------------------------------------------------------------------ */
/* QKV projection with Q4F16_1 weights (Zero TVM Documentation, "Q4F16 quantization format": eight
 * int4 values per uint32, element i in bits 4i..4i+3, one fp16 scale per 32 weights, weight value
 * f16(nibble - 7) * scale evaluated in fp16; "Decode loop": the QKV matmul feeds RoPE and the KV
 * append in one dispatch).
 * Readings: the weight is row-major by output feature, packed along the input:
 *   w[n][k / 8] holds input k of output n in nibble k % 8, scales[n][k / 32];
 * the fp16 product (nibble - 7) * scale is rounded to nearest even (an fp16 multiply), the dot
 * product over the input is exact here (fp64), and the projection is rounded to fp16, the q, k, v
 * rows [q heads | k heads | v heads] of width head_dim that the append then takes.
 * x: fp16 [T][hidden]; y: fp16 [T][N]. */
int orc_qkv_project(const uint16_t* x, const uint32_t* w, const uint16_t* scales, int T, int hidden, int N,
                    uint16_t* y) {
  orc_init();
  if (T < 0 || hidden <= 0 || hidden % 32 || N <= 0) return ORC_INVALID;
  const int words = hidden / 8, groups = hidden / 32;
#pragma omp parallel for schedule(static)
  for (int n = 0; n < N; ++n) {
    double* wrow = (double*)malloc(sizeof(double) * (size_t)hidden);
    for (int k = 0; k < hidden; ++k) {
      const uint32_t packed = w[(int64_t)n * words + k / 8];
      const int nibble = (int)((packed >> (4 * (k % 8))) & 0xFu);
      const double scale = dec(scales[(int64_t)n * groups + k / 32]);
      wrow[k] = dec(orc_f64_to_f16((double)(nibble - 7) * scale));
    }
    for (int t = 0; t < T; ++t) {
      double acc = 0.0;
      for (int k = 0; k < hidden; ++k) acc += dec(x[(int64_t)t * hidden + k]) * wrow[k];
      y[(int64_t)t * N + n] = orc_f64_to_f16(acc);
    }
    free(wrow);
  }
  return ORC_OK;
}

/* ------------------------------------------------------------------------------------------ */
/* Attention of one query head over logical tokens [t0, t1) of sequence s.                     */

static int seq_len_of(const int32_t* page_indptr, const int32_t* last_page_len, int s, int* len) {
  int n = page_indptr[s + 1] - page_indptr[s];
  if (n < 0) return ORC_INVALID;
  if (n == 0) {
    *len = 0;
    return ORC_OK;
  }
  int last = last_page_len[s];
  if (last < 1 || last > ORC_PAGE) return ORC_OUT_OF_RANGE;
  *len = (n - 1) * ORC_PAGE + last;
  return ORC_OK;
}

/* First attended position of a sequence of length len under window W (0 = no window). */
static int window_start(int len, int window) { return (window > 0 && len > window) ? len - window : 0; }

/* Fold a sink logit into an attention result (o normalised over its tokens, lse their log-sum):
 * o *= e^lse / (e^lse + e^sink), lse = ln(e^lse + e^sink); an empty result stays o = 0 with
 * lse = sink. */
static void apply_sink(double* o, double* lse, int d, double sink) {
  if (sink == -INFINITY) return;
  if (*lse == -INFINITY) {
    *lse = sink;
    return;
  }
  const double M = *lse > sink ? *lse : sink;
  const double wa = exp(*lse - M), ws = exp(sink - M);
  for (int i = 0; i < d; ++i) o[i] = o[i] * wa / (wa + ws);
  *lse = M + log(wa + ws);
}

/* o[d] = sum_t softmax(score)_t V_t, lse = ln sum_t exp(score_t); empty range: o = 0, lse = -inf */
/* The cache the attention reads: fp16 rows, or (int8 caches) their dequantized fp64 values. */
static const double* g_pool64 = NULL; /* set only inside the int8 entry points (single-threaded setup) */

static double kv_at(const uint16_t* pool, int64_t row, int i) {
  return g_pool64 != NULL ? g_pool64[row + i] : dec(pool[row + i]);
}

static int attend(const orc_geom* g, const uint16_t* pool, const double* q, int s, int kv_head,
                  int t0, int t1, const int32_t* page_indptr, const int32_t* page_indices,
                  double sm_scale, double* o, double* lse) {
  const int d = g->head_dim;
  for (int i = 0; i < d; ++i) o[i] = 0.0;
  if (t1 <= t0) {
    *lse = -INFINITY;
    return ORC_OK;
  }
  double* score = (double*)malloc(sizeof(double) * (size_t)(t1 - t0));
  double m = -INFINITY;
  for (int t = t0; t < t1; ++t) {
    int page = page_indices[page_indptr[s] + t / ORC_PAGE];
    if (page < 0 || page >= g->num_pages) {
      free(score);
      return ORC_OUT_OF_RANGE;
    }
    const int64_t krow = pool_row(g, page, 0, kv_head, t % ORC_PAGE);
    double dot = 0.0;
    for (int i = 0; i < d; ++i) dot += q[i] * kv_at(pool, krow, i);
    score[t - t0] = sm_scale * dot;
    if (score[t - t0] > m) m = score[t - t0];
  }
  double l = 0.0;
  for (int t = t0; t < t1; ++t) {
    int page = page_indices[page_indptr[s] + t / ORC_PAGE];
    const int64_t vrow = pool_row(g, page, 1, kv_head, t % ORC_PAGE);
    double w = exp(score[t - t0] - m);
    l += w;
    for (int i = 0; i < d; ++i) o[i] += w * kv_at(pool, vrow, i);
  }
  for (int i = 0; i < d; ++i) o[i] /= l;
  *lse = m + log(l);
  free(score);
  return ORC_OK;
}

/* Full (unsplit) decode attention.  q_rope: [B][Hq][d] fp16 bits; out: [B][Hq][d]; lse: [B][Hq]. */
int orc_attention(const orc_geom* g, const uint16_t* pool, const uint16_t* q_rope, int B,
                  const int32_t* page_indptr, const int32_t* page_indices,
                  const int32_t* last_page_len, double sm_scale, int window, const double* sinks,
                  double* out, double* lse) {
  orc_init();
  const int d = g->head_dim, Hq = g->num_qo_heads, Hkv = g->num_kv_heads;
  if (d <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || B < 0) return ORC_INVALID;
  const int G = Hq / Hkv;
  int rc = ORC_OK;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t sh = 0; sh < (int64_t)B * Hq; ++sh) {
    int s = (int)(sh / Hq), h = (int)(sh % Hq);
    int len;
    int r = seq_len_of(page_indptr, last_page_len, s, &len);
    double* q = (double*)malloc(sizeof(double) * (size_t)d);
    for (int i = 0; i < d; ++i) q[i] = dec(q_rope[sh * d + i]);
    if (r == ORC_OK)
      r = attend(g, pool, q, s, h / G, window_start(len, window), len, page_indptr, page_indices, sm_scale,
                 out + sh * d, lse + sh);
    if (r == ORC_OK && sinks != NULL) apply_sink(out + sh * d, lse + sh, d, sinks[h]);
    free(q);
    if (r != ORC_OK) {
#pragma omp critical
      rc = r;
    }
  }
  return rc;
}

/* Chunked-prefill attention (the step after the append when a sequence appends several tokens;
 * Zero TVM Documentation, "How it works": prefill in chunks; "Decode loop": a token attends to itself and to every
 * earlier position of its sequence).  Token t of sequence s (append_indptr) at position
 * p = pos_map[t] attends to the positions [window_start(p + 1, W), p] of s, the cache after the
 * append holding them; sinks as in orc_attention.  q_rope: [T][Hq][d] fp16 bits; out: [T][Hq][d];
 * lse: [T][Hq].  A position outside [0, len_s) is rejected. */
int orc_prefill_attention(const orc_geom* g, const uint16_t* pool, const uint16_t* q_rope, int T, int B,
                          const int32_t* append_indptr, const int32_t* pos_map, const int32_t* page_indptr,
                          const int32_t* page_indices, const int32_t* last_page_len, double sm_scale,
                          int window, const double* sinks, double* out, double* lse) {
  orc_init();
  const int d = g->head_dim, Hq = g->num_qo_heads, Hkv = g->num_kv_heads;
  if (d <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || B < 0 || T < 0) return ORC_INVALID;
  if (append_indptr[0] != 0 || append_indptr[B] != T) return ORC_INVALID;
  const int G = Hq / Hkv;
  int* seq_of = (int*)malloc(sizeof(int) * (size_t)(T > 0 ? T : 1));
  for (int s = 0; s < B; ++s) {
    if (append_indptr[s + 1] < append_indptr[s]) {
      free(seq_of);
      return ORC_INVALID;
    }
    int len;
    if (seq_len_of(page_indptr, last_page_len, s, &len) != ORC_OK) {
      free(seq_of);
      return ORC_OUT_OF_RANGE;
    }
    for (int t = append_indptr[s]; t < append_indptr[s + 1]; ++t) {
      if (pos_map[t] < 0 || pos_map[t] >= len) {
        free(seq_of);
        return ORC_OUT_OF_RANGE;
      }
      seq_of[t] = s;
    }
  }
  int rc = ORC_OK;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t th = 0; th < (int64_t)T * Hq; ++th) {
    const int t = (int)(th / Hq), h = (int)(th % Hq);
    const int s = seq_of[t], p = pos_map[t];
    double* q = (double*)malloc(sizeof(double) * (size_t)d);
    for (int i = 0; i < d; ++i) q[i] = dec(q_rope[th * d + i]);
    int r = attend(g, pool, q, s, h / G, window_start(p + 1, window), p + 1, page_indptr, page_indices, sm_scale,
                   out + th * d, lse + th);
    if (r == ORC_OK && sinks != NULL) apply_sink(out + th * d, lse + th, d, sinks[h]);
    free(q);
    if (r != ORC_OK) {
#pragma omp critical
      rc = r;
    }
  }
  free(seq_of);
  return rc;
}

/* Split-K partial attention.  Under a window W the visible pages of sequence s are
 * [f_s, n_s) with f_s = floor(window_start / 16), n'_s = n_s - f_s of them; without one f_s = 0.
 * Chunk size in pages: chunk_pages if > 0 (uniform), otherwise ceil(n'_s / num_splits).  Chunk j
 * covers visible pages [f_s + j*c, f_s + min((j+1)*c, n'_s)), and within them the attended
 * positions only.  partial_o: [B][Hq][S][d], partial_lse: [B][Hq][S] with S = num_out_splits. */
int orc_split_attention(const orc_geom* g, const uint16_t* pool, const uint16_t* q_rope, int B,
                        const int32_t* page_indptr, const int32_t* page_indices,
                        const int32_t* last_page_len, int num_splits, int chunk_pages,
                        int num_out_splits, double sm_scale, int window, double* partial_o,
                        double* partial_lse) {
  orc_init();
  const int d = g->head_dim, Hq = g->num_qo_heads, Hkv = g->num_kv_heads, S = num_out_splits;
  if (d <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || B < 0 || S <= 0) return ORC_INVALID;
  if (chunk_pages <= 0 && num_splits <= 0) return ORC_INVALID;
  const int G = Hq / Hkv;
  for (int s = 0; s < B; ++s) {
    int len;
    if (seq_len_of(page_indptr, last_page_len, s, &len) != ORC_OK) return ORC_OUT_OF_RANGE;
    int n = page_indptr[s + 1] - page_indptr[s] - window_start(len, window) / ORC_PAGE;
    int c = chunk_pages > 0 ? chunk_pages : (n + num_splits - 1) / num_splits;
    int chunks = (c > 0) ? (n + c - 1) / c : 0;
    if (chunks > S) return ORC_INVALID;
  }
  int rc = ORC_OK;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t sh = 0; sh < (int64_t)B * Hq; ++sh) {
    int s = (int)(sh / Hq), h = (int)(sh % Hq);
    int len;
    int r = seq_len_of(page_indptr, last_page_len, s, &len);
    const int ws = window_start(len, window), f = ws / ORC_PAGE;
    int n = page_indptr[s + 1] - page_indptr[s] - f;
    int c = chunk_pages > 0 ? chunk_pages : (n + num_splits - 1) / num_splits;
    double* q = (double*)malloc(sizeof(double) * (size_t)d);
    for (int i = 0; i < d; ++i) q[i] = dec(q_rope[sh * d + i]);
    for (int j = 0; j < S && r == ORC_OK; ++j) {
      int64_t t0 = ((int64_t)f + (int64_t)j * c) * ORC_PAGE, t1 = ((int64_t)f + (int64_t)(j + 1) * c) * ORC_PAGE;
      if (t0 < ws) t0 = ws;
      if (t1 > len) t1 = len;
      if (t0 > len) t0 = len;
      r = attend(g, pool, q, s, h / G, (int)t0, (int)t1, page_indptr, page_indices, sm_scale,
                 partial_o + (sh * S + j) * d, partial_lse + sh * S + j);
    }
    free(q);
    if (r != ORC_OK) {
#pragma omp critical
      rc = r;
    }
  }
  return rc;
}

/* Split-K partial attention with the page-balanced partition: the page units of all
 * (sequence, KV head) segments, ordered sequence-major, then KV head, then page, are cut into
 * num_warps contiguous runs, run w being units [floor(w*U/W), floor((w+1)*U/W)) with
 * U = Hkv * (total pages).  Piece k of a segment is its intersection with the k-th run that
 * meets it.  Under a window W > 0 a sequence's units are its visible pages [f_s, n_s) (see
 * orc_split_attention) and U counts those.  partial_o: [B][Hq][S][d], partial_lse: [B][Hq][S];
 * slots without a piece are (0, -inf).  Requires num_warps <= U (every run non-empty). */
int orc_split_attention_balanced(const orc_geom* g, const uint16_t* pool, const uint16_t* q_rope, int B,
                                 const int32_t* page_indptr, const int32_t* page_indices,
                                 const int32_t* last_page_len, int num_warps, int num_out_splits,
                                 double sm_scale, int window, double* partial_o, double* partial_lse) {
  orc_init();
  const int d = g->head_dim, Hq = g->num_qo_heads, Hkv = g->num_kv_heads, S = num_out_splits;
  if (d <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || B < 0 || S <= 0 || num_warps <= 0) return ORC_INVALID;
  const int G = Hq / Hkv;
  /* visible pages of each sequence and their exclusive prefix */
  int64_t* vstart = (int64_t*)malloc(sizeof(int64_t) * (size_t)(B + 1));
  int* vfirst = (int*)malloc(sizeof(int) * (size_t)(B > 0 ? B : 1));
  vstart[0] = 0;
  for (int s = 0; s < B; ++s) {
    int len = 0;
    if (seq_len_of(page_indptr, last_page_len, s, &len) != ORC_OK) {
      free(vstart);
      free(vfirst);
      return ORC_OUT_OF_RANGE;
    }
    vfirst[s] = window_start(len, window) / ORC_PAGE;
    vstart[s + 1] = vstart[s] + (page_indptr[s + 1] - page_indptr[s] - vfirst[s]);
  }
  const int64_t U = (int64_t)Hkv * vstart[B];
  const int64_t W = num_warps;
  if (U > 0 && W > U) {
    free(vstart);
    free(vfirst);
    return ORC_INVALID;
  }
  int rc = ORC_OK;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t sh = 0; sh < (int64_t)B * Hq; ++sh) {
    int s = (int)(sh / Hq), h = (int)(sh % Hq), kvh = h / G;
    int len;
    int r = seq_len_of(page_indptr, last_page_len, s, &len);
    double* q = (double*)malloc(sizeof(double) * (size_t)d);
    for (int i = 0; i < d; ++i) q[i] = dec(q_rope[sh * d + i]);
    for (int j = 0; j < S; ++j) {
      for (int i = 0; i < d; ++i) partial_o[(sh * S + j) * d + i] = 0.0;
      partial_lse[sh * S + j] = -INFINITY;
    }
    const int64_t n = vstart[s + 1] - vstart[s];
    const int64_t b = (int64_t)Hkv * vstart[s] + (int64_t)kvh * n; /* first unit of the segment */
    const int64_t f = vfirst[s], ws = window_start(len, window);
    int k = 0;
    for (int64_t w = 0; w < W && r == ORC_OK && n > 0; ++w) {
      const int64_t u0 = w * U / W, u1 = (w + 1) * U / W;
      const int64_t lo = u0 > b ? u0 : b, hi = u1 < b + n ? u1 : b + n;
      if (hi <= lo) continue;
      if (k >= S) {
        r = ORC_INVALID;
        break;
      }
      int64_t t0 = (f + lo - b) * ORC_PAGE, t1 = (f + hi - b) * ORC_PAGE;
      if (t0 < ws) t0 = ws;
      if (t1 > len) t1 = len;
      if (t0 > len) t0 = len;
      r = attend(g, pool, q, s, kvh, (int)t0, (int)t1, page_indptr, page_indices, sm_scale,
                 partial_o + (sh * S + k) * d, partial_lse + sh * S + k);
      ++k;
    }
    free(q);
    if (r != ORC_OK) {
#pragma omp critical
      rc = r;
    }
  }
  free(vstart);
  free(vfirst);
  return rc;
}

/* Log-sum-exp merge of the partials: out = sum_j w_j o_j / sum_j w_j with w_j = exp(lse_j - M),
 * M = max_j lse_j, lse = M + ln sum_j w_j; with a sink (sinks[h], nullable) the merged result then
 * takes the sink into its denominator.  out_f16 (nullable) gets out rounded to fp16. */
int orc_combine(const double* partial_o, const double* partial_lse, int B, int Hq, int S, int d,
                const double* sinks, double* out, uint16_t* out_f16, double* lse) {
  if (B < 0 || Hq <= 0 || S <= 0 || d <= 0) return ORC_INVALID;
  for (int64_t sh = 0; sh < (int64_t)B * Hq; ++sh) {
    const double* L = partial_lse + sh * S;
    double M = -INFINITY;
    for (int j = 0; j < S; ++j)
      if (L[j] > M) M = L[j];
    double* o = out + sh * d;
    for (int i = 0; i < d; ++i) o[i] = 0.0;
    if (M == -INFINITY) {
      lse[sh] = -INFINITY;
    } else {
      double W = 0.0;
      for (int j = 0; j < S; ++j) {
        if (L[j] == -INFINITY) continue;
        double w = exp(L[j] - M);
        W += w;
        for (int i = 0; i < d; ++i) o[i] += w * partial_o[(sh * S + j) * d + i];
      }
      for (int i = 0; i < d; ++i) o[i] /= W;
      lse[sh] = M + log(W);
    }
    if (sinks != NULL) apply_sink(o, lse + sh, d, sinks[sh % Hq]);
    if (out_f16)
      for (int i = 0; i < d; ++i) out_f16[sh * d + i] = orc_f64_to_f16(o[i]);
  }
  return ORC_OK;
}

/* ------------------------------------------------------------------------------------------ */
/* Attention over an int8 pool: the same definitions over the dequantized values code * s. */
int orc_attention_int8(const orc_geom* g, const uint8_t* pool8, const uint16_t* q_rope, int B,
                       const int32_t* page_indptr, const int32_t* page_indices, const int32_t* last_page_len,
                       double sm_scale, int window, const double* sinks, double* out, double* lse) {
  double* p64 = (double*)malloc(sizeof(double) * (size_t)g->num_pages * 2 * g->num_kv_heads * ORC_PAGE *
                                (size_t)g->head_dim);
  orc_dequantize_pool(g, pool8, p64);
  g_pool64 = p64;
  int rc = orc_attention(g, NULL, q_rope, B, page_indptr, page_indices, last_page_len, sm_scale, window, sinks,
                         out, lse);
  g_pool64 = NULL;
  free(p64);
  return rc;
}

int orc_split_attention_int8(const orc_geom* g, const uint8_t* pool8, const uint16_t* q_rope, int B,
                             const int32_t* page_indptr, const int32_t* page_indices,
                             const int32_t* last_page_len, int num_splits, int chunk_pages, int num_out_splits,
                             double sm_scale, int window, double* partial_o, double* partial_lse) {
  double* p64 = (double*)malloc(sizeof(double) * (size_t)g->num_pages * 2 * g->num_kv_heads * ORC_PAGE *
                                (size_t)g->head_dim);
  orc_dequantize_pool(g, pool8, p64);
  g_pool64 = p64;
  int rc = orc_split_attention(g, NULL, q_rope, B, page_indptr, page_indices, last_page_len, num_splits,
                               chunk_pages, num_out_splits, sm_scale, window, partial_o, partial_lse);
  g_pool64 = NULL;
  free(p64);
  return rc;
}
