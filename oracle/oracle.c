/*
 * oracle.c -- plain CPU reference for one decode step of hierarchically pruned,
 * block-sparse attention over a paged KV cache whose keys are int8, per-channel
 * quantised.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg may load this library. The product path never
 * links, loads or calls it, and it shares no code, header, table or constant
 * with the CUDA library.
 *
 * Sources (web pages; cited by page title and section):
 *  [HiP]  "韩国通过卸载键值缓存节约英伟达GPU内存，实现18.95倍解码加速" (163.com article on
 *         InfiniteHiP), section "实现 7.24 倍的端到端解码加速": each pruning module cuts
 *         its input into fixed-length chunks, finds each chunk's top-scoring token in
 *         parallel and passes only the top-K chunks on; stacking modules refines a
 *         block-sparse attention mask.
 *  [HCA]  "HCAttention: Extreme KV cache compression via heterogeneous attention
 *         computing for LLMs" (ebiotrade.com excerpt), abstract and contribution list:
 *         keys are quantised and kept on the GPU for a global approximate scoring of
 *         every token; values are fetched late, only for the final aggregation.
 *  [KVN]  "KV Cache 与长上下文推理" (jeffliulab notes), section "KV Cache 回顾", the
 *         attention equation softmax(q K^T / sqrt(d_k)) V; section "KV Cache 量化"
 *         (INT8 keys); section "Token Eviction 与 Sparse Attention" (StreamingLLM:
 *         attention sinks plus a sliding window); section "MQA 与 GQA" (G key/value
 *         heads shared by H query heads).
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  - key scale per (sequence, kv head, channel) over the whole context:
 *      s_c = f32(amax_c / 127), code = clamp(rint_even(f32(k / s_c)), -127, 127),
 *      s_c = 0 gives code 0; the 4-bit key format (N4 variant) uses 7 in place of 127
 *      for the keys (codes in [-7, 7]), the query codes stay 8-bit;
 *  - the key scales are folded into the query, q'_{j,c} = f32(q_{j,c} * s_c), and the
 *    group of G query heads sharing a kv head is quantised with ONE scale
 *      A = max |q'|, sq = f32(A / 127), qq = clamp(rint_even(f32(q' / sq)), -127, 127);
 *  - token score g_t = max over the group of the exact integer dot qq_j . kq_t;
 *  - candidate region C = [sink, N - window); chunks and blocks are aligned to token 0
 *    and only their tokens inside C count; a chunk or block with no token in C is
 *    never selected;
 *  - ties: the lower index wins at both levels; index lists are returned ascending;
 *  - attended set T = [0, min(S,N)) u [max(N-W, min(S,N)), N) u (kept blocks n C);
 *  - the "cumulative magnitude" of a KV block ([HCA], eviction from the GPU cache) is the
 *    softmax probability its attended tokens receive, summed over the group's query heads
 *    and accumulated over the decode calls.
 *
 * Precision: attention in fp64 from the exact bf16 values. The quantisation steps
 * decide integers in IEEE fp32, emulated as ONE fp64 operation followed by a cast to
 * float: exact for a product of two floats (48 significant bits < 53) and correctly
 * rounded for a quotient of two floats (53 >= 2*24 + 2, Figueroa 1995). Build with
 * -ffp-contract=off so that no product is fused into an add.
 *
 * Pins (what ties this file to something other than itself): hand-worked examples
 * under tests/golden, brute force on tiny inputs, the closed form "two-stage top-K
 * equals the single-stage top-K2 of blocks whenever K1 >= K2", K1/K2 covering every
 * block reproducing dense attention, K1 = K2 = 0 reproducing sink + window
 * attention, the quantisation error bound, power-of-two scale invariance, and the
 * restriction identity linking sparse output, dense output and recall.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
  int32_t batch, hq, hkv, head_dim, page_size, max_pages_per_seq, num_pages;
  int32_t chunk, block, k1, k2, sink, window;
  double sm_scale; /* <= 0 means 1/sqrt(head_dim) */
  int32_t chunk0, k0; /* k0 > 0: a first module keeps the top-k0 chunks of chunk0 tokens */
  int32_t key_bits;   /* 4: 4-bit key codes (levels +-7); 0 or 8: 8-bit (levels +-127) */
  int32_t per_head;   /* 1: every query head selects its own chunks and blocks (N3 variant) */
  int32_t key_fp8;    /* 1: FP8 E4M3 key codes (scale amax / 448, real-valued scores; N4 variant) */
} oracle_dims;

/* Rows of the selection outputs per sequence: one per kv head (the group shares one
 * selection), or one per query head with per-head selection. */
static int sel_rows(const oracle_dims* d) { return d->per_head ? d->hq : d->hkv; }

/* ---------------------------------------------------------------- helpers */

static double bf16_value(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Index of element (token t, channel c) of kv head h of sequence b in a paged
 * cache laid out [page][kv head][slot in page][channel]. */
static size_t cache_index(const oracle_dims* d, const int32_t* page_table, int b, int h,
                          int64_t t, int c) {
  int64_t page = page_table[(int64_t)b * d->max_pages_per_seq + t / d->page_size];
  int64_t slot = t % d->page_size;
  return (size_t)(((page * d->hkv + h) * d->page_size + slot) * d->head_dim + c);
}

static int dims_ok(const oracle_dims* d) {
  if (!d) return 0;
  if (d->batch <= 0 || d->hq <= 0 || d->hkv <= 0 || d->head_dim <= 0) return 0;
  if (d->hq % d->hkv) return 0;
  if (d->page_size <= 0 || d->max_pages_per_seq <= 0 || d->num_pages <= 0) return 0;
  if (d->chunk <= 0 || d->block <= 0 || d->chunk % d->block) return 0;
  if (d->k1 < 0 || d->k2 < 0 || d->sink < 0 || d->window < 0) return 0;
  if (d->k0 < 0) return 0;
  if (d->k0 > 0 && (d->chunk0 < d->chunk || d->chunk0 % d->chunk)) return 0;
  if (d->key_bits != 0 && d->key_bits != 4 && d->key_bits != 8) return 0;
  if (d->key_fp8 != 0 && (d->key_fp8 != 1 || d->key_bits == 4)) return 0;
  return 1;
}

static int seq_ok(const oracle_dims* d, const int32_t* page_table, const int32_t* lens, int b) {
  int64_t n = lens[b];
  if (n < 0 || n > (int64_t)d->max_pages_per_seq * d->page_size) return 0;
  for (int64_t p = 0; p * d->page_size < n; p++) {
    int32_t pg = page_table[(int64_t)b * d->max_pages_per_seq + p];
    if (pg < 0 || pg >= d->num_pages) return 0;
  }
  return 1;
}

static int wanted(const int32_t* bh_mask, const oracle_dims* d, int b, int h) {
  return bh_mask == NULL || bh_mask[b * d->hkv + h] != 0;
}

/* fp32 round-to-nearest-even code of x / s, clamped to the symmetric range [-levels, levels]. */
static int8_t key_code(double x, float s, int levels) {
  if (s == 0.0f) return 0;
  float ratio = (float)(x / (double)s);
  double r = nearbyint((double)ratio); /* default rounding mode: half to even */
  if (r > levels) r = levels;
  if (r < -levels) r = -levels;
  return (int8_t)r;
}

static int8_t int8_code(double x, float s) { return key_code(x, s, 127); }

/* Largest key code: 127 for 8-bit keys, 7 for the 4-bit key format. */
static int key_levels(const oracle_dims* d) { return d->key_bits == 4 ? 7 : 127; }

/* ------------------------------------------------------------ FP8 keys */

/* [KVN] "KV Cache 量化" (FP8 KV caches). E4M3: sign, 4 exponent bits (bias 7), 3 mantissa
 * bits, no infinities, S.1111.111 is NaN, so the largest finite magnitude is
 * 1.75 * 2^8 = 448; exponent field 0 holds the subnormals m * 2^-9. */
static float e4m3_value(uint8_t code) {
  const int e = (code >> 3) & 15, m = code & 7;
  const double v = e == 0 ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
  return (float)((code & 0x80) ? -v : v);
}

/* The E4M3 code of x: round to nearest, ties to the even mantissa; magnitudes from 448 up
 * give 448 (saturating); a zero result keeps the sign of x. */
static uint8_t e4m3_code(float x) {
  const uint8_t sign = signbit(x) ? 0x80 : 0;
  const double a = fabs((double)x);
  if (a >= 448.0) return sign | 0x7E; /* exponent field 15, mantissa 6 */
  if (a < ldexp(1.0, -6)) {
    /* subnormal grid 2^-9; 8 steps give the smallest normal, whose code is also 8 */
    return sign | (uint8_t)nearbyint(ldexp(a, 9));
  }
  int p;
  frexp(a, &p);                              /* a = f * 2^p, f in [0.5, 1) */
  int e = p - 1;                             /* a in [2^e, 2^(e+1)) */
  double q = nearbyint(ldexp(a, 3 - e));     /* 8 .. 16, in steps of 2^(e-3) */
  if (q == 16.0) {
    q = 8.0;
    e += 1;
  }
  return sign | (uint8_t)(((e + 7) << 3) | ((int)q - 8));
}

/* The key code of x / s in the key format of d (int8 codes hold the E4M3 bits as is). */
static int8_t format_code(const oracle_dims* d, double x, float s) {
  if (!d->key_fp8) return key_code(x, s, key_levels(d));
  if (s == 0.0f) return 0;
  return (int8_t)e4m3_code((float)(x / (double)s));
}

/* Ordered integer of a float score: a < b as floats exactly when key(a) < key(b); both
 * zeros map to 0 (the block_max output of FP8 selections). */
static int32_t ordered_key(float f) {
  f = f + 0.0f; /* -0 -> +0 */
  int32_t bits;
  memcpy(&bits, &f, sizeof bits);
  return bits >= 0 ? bits : bits ^ 0x7FFFFFFF;
}

/* The same for an fp64 score: the selection ranks FP8 scores as it ranks integer scores. */
static int64_t ordered_key64(double x) {
  x = x + 0.0; /* -0 -> +0 */
  int64_t bits;
  memcpy(&bits, &x, sizeof bits);
  return bits >= 0 ? bits : bits ^ INT64_MAX;
}

/* FP8 keys: the score of head j for token t is the dot of the folded fp32 query with the
 * E4M3 values, sum_c q'_{j,c} x_{t,c}. The pages fix no precision or order for it, so the
 * oracle takes the sum itself: every product is exact in fp64 (24 + 4 significant bits)
 * and the fp64 sum of 128 of them is within 127 * 2^-53 * sum |q' x| of the exact value.
 * An fp32 evaluation with one rounding per term (a chain of fused multiply-adds, in any
 * order) is within gamma_n * sum |q' x| of the exact value (Higham, "Accuracy and Stability
 * of Numerical Algorithms", recursive summation: gamma_n = n u / (1 - n u), u = 2^-24,
 * n = the number of terms); *abs_sum receives sum |q' x|. */
static double fp8_dot(const oracle_dims* d, const float* qf_j, const int8_t* kq,
                      const int32_t* page_table, int b, int h, int64_t t, double* abs_sum) {
  double acc = 0.0, mag = 0.0;
  for (int c = 0; c < d->head_dim; c++) {
    const double p =
        (double)qf_j[c] * (double)e4m3_value((uint8_t)kq[cache_index(d, page_table, b, h, t, c)]);
    acc += p;
    mag += fabs(p);
  }
  *abs_sum = mag;
  return acc;
}

static double fp32_chain_gamma(int n) {
  const double u = ldexp(1.0, -24);
  return n * u / (1.0 - n * u);
}

/* ----------------------------------------------- key scales and int8 codes */

/* [HCA] quantised keys on the GPU; [KVN] "KV Cache 量化" (INT8 keys).
 * Full mode: per (b, h, c) amax over tokens t < N_b, then every token's code.
 * Slots of the last page past N_b get code 0. */
int oracle_quantize_keys(const oracle_dims* d, const uint16_t* k, const int32_t* page_table,
                         const int32_t* lens, const int32_t* bh_mask, int8_t* kq, float* scale) {
  if (!dims_ok(d) || !k || !page_table || !lens || !kq || !scale) return 1;
  for (int b = 0; b < d->batch; b++)
    if (!seq_ok(d, page_table, lens, b)) return 2;
  const int D = d->head_dim;
#pragma omp parallel for schedule(dynamic, 1)
  for (int bh = 0; bh < d->batch * d->hkv; bh++) {
    int b = bh / d->hkv, h = bh % d->hkv;
    if (!wanted(bh_mask, d, b, h)) continue;
    int64_t n = lens[b];
    for (int c = 0; c < D; c++) {
      double amax = 0.0;
      for (int64_t t = 0; t < n; t++) {
        double x = fabs(bf16_value(k[cache_index(d, page_table, b, h, t, c)]));
        if (x > amax) amax = x;
      }
      const double levels = d->key_fp8 ? 448.0 : (double)key_levels(d);
      float s = (float)(amax / levels);
      scale[((int64_t)b * d->hkv + h) * D + c] = s;
      for (int64_t t = 0; t < n; t++) {
        size_t i = cache_index(d, page_table, b, h, t, c);
        kq[i] = format_code(d, bf16_value(k[i]), s);
      }
      int64_t end = ((n + d->page_size - 1) / d->page_size) * d->page_size;
      for (int64_t t = n; t < end; t++) kq[cache_index(d, page_table, b, h, t, c)] = 0;
    }
  }
  return 0;
}

/* Append mode: codes of tokens [from_b, N_b) with the scales already stored;
 * from < 0 means each sequence's last token (the decode-step append). */
int oracle_quantize_append(const oracle_dims* d, const uint16_t* k, const int32_t* page_table,
                           const int32_t* lens, int32_t from, const float* scale, int8_t* kq) {
  if (!dims_ok(d) || !k || !page_table || !lens || !kq || !scale) return 1;
  for (int b = 0; b < d->batch; b++) {
    if (!seq_ok(d, page_table, lens, b)) return 2;
    int64_t n = lens[b];
    int64_t t0 = from < 0 ? n - 1 : from;
    if (t0 < 0) t0 = 0;
    for (int h = 0; h < d->hkv; h++)
      for (int64_t t = t0; t < n; t++)
        for (int c = 0; c < d->head_dim; c++) {
          size_t i = cache_index(d, page_table, b, h, t, c);
          kq[i] = format_code(d, bf16_value(k[i]),
                              scale[((int64_t)b * d->hkv + h) * d->head_dim + c]);
        }
  }
  return 0;
}

/* ------------------------------------------------------ query int8 codes */

/* [HCA] scoring against quantised keys: the key scales are folded into the query
 * (q' = q * s) and the G query heads of one kv head share one quantisation scale, so
 * that the integer scores of the group are in the same units and their max is
 * meaningful. qq: [B][Hkv][G][D]; q_scale: [B][Hkv] (sq = A / 127). */
static void query_codes_one(const oracle_dims* d, const uint16_t* q, const float* scale, int b,
                            int h, int8_t* qq, float* sq_out) {
  const int D = d->head_dim, G = d->hq / d->hkv;
  const float* s = scale + ((int64_t)b * d->hkv + h) * D;
  float* qf = (float*)malloc(sizeof(float) * (size_t)G * D);
  float amax = 0.0f;
  for (int j = 0; j < G; j++)
    for (int c = 0; c < D; c++) {
      double qv = bf16_value(q[((int64_t)b * d->hq + h * G + j) * D + c]);
      float folded = (float)(qv * (double)s[c]);
      qf[j * D + c] = folded;
      if (fabsf(folded) > amax) amax = fabsf(folded);
    }
  float sq = (float)((double)amax / 127.0);
  for (int j = 0; j < G; j++)
    for (int c = 0; c < D; c++) qq[j * D + c] = int8_code((double)qf[j * D + c], sq);
  if (sq_out) *sq_out = sq;
  free(qf);
}

/* FP8 keys: the folded query q'_{j,c} = f32(q_{j,c} * s_c) itself, [G][D], not quantised. */
static void query_folded(const oracle_dims* d, const uint16_t* q, const float* scale, int b,
                         int h, float* qf) {
  const int D = d->head_dim, G = d->hq / d->hkv;
  const float* s = scale + ((int64_t)b * d->hkv + h) * D;
  for (int j = 0; j < G; j++)
    for (int c = 0; c < D; c++)
      qf[j * D + c] = (float)(bf16_value(q[((int64_t)b * d->hq + h * G + j) * D + c]) * (double)s[c]);
}

int oracle_query_codes(const oracle_dims* d, const uint16_t* q, const float* scale, int8_t* qq,
                       float* q_scale) {
  if (!dims_ok(d) || !q || !scale || !qq) return 1;
  const int D = d->head_dim, G = d->hq / d->hkv;
  for (int b = 0; b < d->batch; b++)
    for (int h = 0; h < d->hkv; h++)
      query_codes_one(d, q, scale, b, h, qq + ((int64_t)b * d->hkv + h) * G * D,
                      q_scale ? q_scale + (int64_t)b * d->hkv + h : NULL);
  return 0;
}

/* ------------------------------------------------------ the two modules */

typedef struct {
  int64_t score;
  int64_t index;
} ranked;

/* higher score first; equal scores: lower index first */
static int by_score_then_index(const void* a, const void* b) {
  const ranked* x = (const ranked*)a;
  const ranked* y = (const ranked*)b;
  if (x->score != y->score) return x->score > y->score ? -1 : 1;
  return (x->index > y->index) - (x->index < y->index);
}

static int by_index(const void* a, const void* b) {
  const ranked* x = (const ranked*)a;
  const ranked* y = (const ranked*)b;
  return (x->index > y->index) - (x->index < y->index);
}

/* [HiP] two stacked pruning modules over the candidate region C = [S, N - W):
 *  module 1: chunks of `chunk` tokens; a chunk's score is the max token score over
 *            its tokens in C; the top-K1 chunks pass on;
 *  module 2: the kept chunks are cut into blocks of `block` tokens; a block's score is
 *            the max token score over its tokens in C; the top-K2 blocks are kept.
 * A token's score is the max over the group's query heads of the exact integer dot
 * product of the query codes with the key codes ([HCA] global approximate scoring).
 * Outputs (per (b, h)): block_max [B][Hkv][max_pages_per_seq*page_size/block]
 * (INT32_MIN where a block has no token in C; nullable), chunk_idx [B][Hkv][K1]
 * and block_idx [B][Hkv][K2] ascending and padded with -1, n_chunks / n_blocks
 * [B][Hkv] (nullable).
 * Per-head selection (d->per_head; [HiP] prunes every attention head on its own): the
 * same query codes, but every query head j ranks its own token scores qq_j . kq_t, with
 * no max over the group; the outputs then have one row per query head ([B][Hq][..]). */
int oracle_select(const oracle_dims* d, const uint16_t* q, const float* scale, const int8_t* kq,
                  const int32_t* page_table, const int32_t* lens, const int32_t* bh_mask,
                  int32_t* block_max, int32_t* chunk_idx, int32_t* n_chunks, int32_t* block_idx,
                  int32_t* n_blocks) {
  if (!dims_ok(d) || !q || !scale || !kq || !page_table || !lens || !chunk_idx || !block_idx)
    return 1;
  for (int b = 0; b < d->batch; b++)
    if (!seq_ok(d, page_table, lens, b)) return 2;
  const int D = d->head_dim, G = d->hq / d->hkv;
  const int64_t max_tokens = (int64_t)d->max_pages_per_seq * d->page_size;
  const int64_t max_blocks = (max_tokens + d->block - 1) / d->block;
  int bad = 0;
  /* one (sequence, kv head) at a time; its token scores are spread over the threads */
  for (int bh = 0; bh < d->batch * d->hkv; bh++) {
    int b = bh / d->hkv, h = bh % d->hkv;
    if (!wanted(bh_mask, d, b, h)) continue;
    int64_t n = lens[b];
    int64_t lo = d->sink, hi = n - d->window; /* C = [lo, hi) */
    int8_t* qq = (int8_t*)malloc((size_t)G * D);
    if (qq) query_codes_one(d, q, scale, b, h, qq, NULL);
    float* qf = d->key_fp8 ? (float*)malloc(sizeof(float) * (size_t)G * D) : NULL;
    if (qf) query_folded(d, q, scale, b, h, qf);
    const int nrow = d->per_head ? G : 1;
    for (int rj = 0; rj < nrow; rj++) {
      /* the output row, and the query heads whose scores it ranks: [j_lo, j_hi) */
      const int64_t row =
          d->per_head ? (int64_t)b * d->hq + h * G + rj : (int64_t)b * d->hkv + h;
      const int j_lo = d->per_head ? rj : 0, j_hi = d->per_head ? rj + 1 : G;

      int64_t n_chunk_all = (max_tokens + d->chunk - 1) / d->chunk;
      const int64_t c0 = d->k0 > 0 ? d->chunk0 : d->chunk; /* coarse chunk of module 0 */
      int64_t n_coarse_all = (max_tokens + c0 - 1) / c0;
      int64_t* cmax0 = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n_coarse_all + 1));
      char* cvalid0 = (char*)calloc((size_t)n_coarse_all + 1, 1);
      char* ckept0 = (char*)calloc((size_t)n_coarse_all + 1, 1);
      int64_t* cmax = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n_chunk_all + 1));
      int64_t* bmax = (int64_t*)malloc(sizeof(int64_t) * (size_t)(max_blocks + 1));
      char* cvalid = (char*)calloc((size_t)n_chunk_all + 1, 1);
      char* bvalid = (char*)calloc((size_t)max_blocks + 1, 1);
      if (!qq || (d->key_fp8 && !qf) || !cmax || !bmax || !cvalid || !bvalid || !cmax0 ||
          !cvalid0 || !ckept0) {
        bad = 1;
      } else {
        /* token scores, folded into the block maxima: a block is a range of tokens of its
         * own, so the blocks are scored in parallel; a chunk's maximum is then the maximum
         * of its blocks' (blocks nest in chunks, chunks in coarse chunks) */
        const int64_t kb_lo = hi > lo ? lo / d->block : 0;
        const int64_t kb_hi = hi > lo ? (hi + d->block - 1) / d->block : 0;
#pragma omp parallel for schedule(static)
        for (int64_t k = kb_lo; k < kb_hi; k++) {
          const int64_t t0 = k * d->block > lo ? k * d->block : lo;
          const int64_t t1 = (k + 1) * d->block < hi ? (k + 1) * d->block : hi;
          for (int64_t t = t0; t < t1; t++) {
            int64_t g = INT64_MIN;
            for (int j = j_lo; j < j_hi; j++) {
              int64_t dot = 0;
              if (d->key_fp8) {
                /* FP8 keys: the dot of the folded query with the E4M3 values (fp8_dot),
                 * ranked through its ordered integer */
                double mag;
                dot = ordered_key64(fp8_dot(d, qf + j * D, kq, page_table, b, h, t, &mag));
              } else {
                for (int c = 0; c < D; c++)
                  dot += (int64_t)qq[j * D + c] *
                         (int64_t)kq[cache_index(d, page_table, b, h, t, c)];
              }
              if (dot > g) g = dot;
            }
            if (!bvalid[k] || g > bmax[k]) bmax[k] = g;
            bvalid[k] = 1;
          }
        }
        for (int64_t k = kb_lo; k < kb_hi; k++) {
          if (!bvalid[k]) continue;
          const int64_t ci = k * d->block / d->chunk, c0i = k * d->block / c0;
          if (!cvalid0[c0i] || bmax[k] > cmax0[c0i]) cmax0[c0i] = bmax[k];
          cvalid0[c0i] = 1;
          if (!cvalid[ci] || bmax[k] > cmax[ci]) cmax[ci] = bmax[k];
          cvalid[ci] = 1;
        }
        if (block_max) {
          /* FP8 keys: the ordered integer of the block maximum rounded to fp32 (the exact
           * maxima and their bounds: oracle_fp8_block_scores) */
          int32_t* out = block_max + row * max_blocks;
          for (int64_t k = 0; k < max_blocks; k++) {
            int32_t v = INT32_MIN;
            if (bvalid[k] && d->key_fp8) {
              const int64_t bits = bmax[k] >= 0 ? bmax[k] : bmax[k] ^ INT64_MAX;
              double x;
              memcpy(&x, &bits, sizeof x);
              v = ordered_key((float)x);
            } else if (bvalid[k]) {
              v = (int32_t)bmax[k];
            }
            out[k] = v;
          }
        }
        ranked* list = (ranked*)malloc(sizeof(ranked) * (size_t)(n_chunk_all + max_blocks +
                                                                  n_coarse_all + 1));
        /* module 0 (stacked in front when k0 > 0): top-K0 coarse chunks, by the same order */
        if (d->k0 > 0) {
          int64_t n0 = 0;
          for (int64_t c = 0; c < n_coarse_all; c++)
            if (cvalid0[c]) {
              list[n0].score = cmax0[c];
              list[n0].index = c;
              n0++;
            }
          qsort(list, (size_t)n0, sizeof(ranked), by_score_then_index);
          int64_t keep0 = n0 < d->k0 ? n0 : d->k0;
          for (int64_t i = 0; i < keep0; i++) ckept0[list[i].index] = 1;
        }
        /* module 1: top-K1 chunks (inside the kept coarse chunks when module 0 runs) */
        int64_t nc = 0;
        for (int64_t c = 0; c < n_chunk_all; c++)
          if (cvalid[c] && (d->k0 == 0 || ckept0[c * d->chunk / c0])) {
            list[nc].score = cmax[c];
            list[nc].index = c;
            nc++;
          }
        qsort(list, (size_t)nc, sizeof(ranked), by_score_then_index);
        int64_t keep1 = nc < d->k1 ? nc : d->k1;
        qsort(list, (size_t)keep1, sizeof(ranked), by_index);
        int32_t* cout = chunk_idx + row * d->k1;
        for (int64_t i = 0; i < d->k1; i++) cout[i] = i < keep1 ? (int32_t)list[i].index : -1;
        if (n_chunks) n_chunks[row] = (int32_t)keep1;
        /* module 2: the kept chunks' blocks, top-K2 */
        ranked* blist = list + keep1;
        int64_t nb = 0;
        const int per = d->chunk / d->block;
        for (int64_t i = 0; i < keep1; i++)
          for (int64_t k = list[i].index * per; k < (list[i].index + 1) * per; k++)
            if (k < max_blocks && bvalid[k]) {
              blist[nb].score = bmax[k];
              blist[nb].index = k;
              nb++;
            }
        qsort(blist, (size_t)nb, sizeof(ranked), by_score_then_index);
        int64_t keep2 = nb < d->k2 ? nb : d->k2;
        qsort(blist, (size_t)keep2, sizeof(ranked), by_index);
        int32_t* bout = block_idx + row * d->k2;
        for (int64_t i = 0; i < d->k2; i++) bout[i] = i < keep2 ? (int32_t)blist[i].index : -1;
        if (n_blocks) n_blocks[row] = (int32_t)keep2;
        free(list);
      }
      free(cmax0);
      free(cvalid0);
      free(ckept0);
      free(cmax);
      free(bmax);
      free(cvalid);
      free(bvalid);
    }
    free(qq);
    free(qf);
  }
  return bad ? 3 : 0;
}

/* FP8 keys: for every selection row and block, the exact block score (the max over the
 * block's candidate tokens of the token score, the max over the row's query heads of
 * fp8_dot) in block_score [B][R][max_blocks] (-inf where the block has no candidate
 * token), and in block_bound the largest gamma_n * sum |q' x| over those (token, head)
 * pairs, n = head_dim: a block maximum computed from fp32 sums with one rounding per term
 * lies within block_bound of block_score (the max of perturbed values moves by at most the
 * largest perturbation). R and bh_mask as in oracle_select. */
int oracle_fp8_block_scores(const oracle_dims* d, const uint16_t* q, const float* scale,
                            const int8_t* kq, const int32_t* page_table, const int32_t* lens,
                            const int32_t* bh_mask, double* block_score, double* block_bound) {
  if (!dims_ok(d) || !d->key_fp8 || !q || !scale || !kq || !page_table || !lens ||
      !block_score || !block_bound)
    return 1;
  for (int b = 0; b < d->batch; b++)
    if (!seq_ok(d, page_table, lens, b)) return 2;
  const int D = d->head_dim, G = d->hq / d->hkv;
  const int64_t max_tokens = (int64_t)d->max_pages_per_seq * d->page_size;
  const int64_t max_blocks = (max_tokens + d->block - 1) / d->block;
  const double gamma = fp32_chain_gamma(D);
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int bh = 0; bh < d->batch * d->hkv; bh++) {
    const int b = bh / d->hkv, h = bh % d->hkv;
    if (!wanted(bh_mask, d, b, h)) continue;
    float* qf = (float*)malloc(sizeof(float) * (size_t)G * D);
    if (!qf) {
#pragma omp atomic write
      bad = 1;
      continue;
    }
    query_folded(d, q, scale, b, h, qf);
    const int64_t n = lens[b], lo = d->sink, hi = n - d->window;
    const int nrow = d->per_head ? G : 1;
    for (int rj = 0; rj < nrow; rj++) {
      const int64_t row =
          d->per_head ? (int64_t)b * d->hq + h * G + rj : (int64_t)b * d->hkv + h;
      const int j_lo = d->per_head ? rj : 0, j_hi = d->per_head ? rj + 1 : G;
      double* sc = block_score + row * max_blocks;
      double* bd = block_bound + row * max_blocks;
      for (int64_t k = 0; k < max_blocks; k++) {
        sc[k] = -HUGE_VAL;
        bd[k] = 0.0;
      }
      for (int64_t t = lo; t < hi; t++) {
        const int64_t k = t / d->block;
        for (int j = j_lo; j < j_hi; j++) {
          double mag;
          const double s = fp8_dot(d, qf + j * D, kq, page_table, b, h, t, &mag);
          if (s > sc[k]) sc[k] = s;
          if (gamma * mag > bd[k]) bd[k] = gamma * mag;
        }
      }
    }
    free(qf);
  }
  return bad ? 3 : 0;
}

/* ---------------------------------------------------------- attention */

/* Membership of token t in the attended set T of (b, h):
 * sink [0, min(S,N)), window [max(N-W, min(S,N)), N), and the kept blocks' tokens
 * inside C = [S, N-W). The three parts are disjoint. `kept` flags blocks. */
static int attended(const oracle_dims* d, int64_t n, int64_t t, const char* kept) {
  int64_t sink_end = d->sink < n ? d->sink : n;
  int64_t win_start = n - d->window;
  if (win_start < sink_end) win_start = sink_end;
  if (t < sink_end) return 1;
  if (t >= win_start) return 1;
  if (kept && t >= d->sink && t < n - d->window && kept[t / d->block]) return 1;
  return 0;
}

/* [KVN] "KV Cache 回顾": out = softmax(q K_T^T / sqrt(d)) V_T over the attended set T,
 * in fp64 from the exact bf16 values; lse = log sum_t exp(l_t). When `all` is set, T
 * is the whole context [0, N) (dense decode). When `recall` is given, the function
 * instead returns sum_{t in T} p_t with p the dense softmax over [0, N). When `mass` is
 * given, it instead returns, for every block, the softmax probability over T that the
 * block's attended tokens receive: mass [B][Hq][max_blocks]. */
static int attention_common(const oracle_dims* d, const uint16_t* q, const uint16_t* k,
                            const uint16_t* v, const int32_t* page_table, const int32_t* lens,
                            const int32_t* block_idx, const int32_t* n_blocks,
                            const int32_t* qh_mask, int all, double* out, double* lse,
                            double* recall, double* mass) {
  const int D = d->head_dim, G = d->hq / d->hkv;
  const double scale = d->sm_scale > 0 ? d->sm_scale : 1.0 / sqrt((double)D);
  const int64_t max_tokens = (int64_t)d->max_pages_per_seq * d->page_size;
  const int64_t max_blocks = (max_tokens + d->block - 1) / d->block;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int bj = 0; bj < d->batch * d->hq; bj++) {
    int b = bj / d->hq, j = bj % d->hq, h = j / G;
    if (qh_mask && !qh_mask[bj]) continue;
    int64_t n = lens[b];
    char* kept = NULL;
    if (!all) {
      kept = (char*)calloc((size_t)max_blocks + 1, 1);
      if (!kept) {
#pragma omp atomic write
        bad = 1;
        continue;
      }
      /* the selection row of query head j: its kv head's, or its own (per-head selection) */
      const int64_t row = d->per_head ? (int64_t)bj : (int64_t)b * d->hkv + h;
      int nk = n_blocks ? n_blocks[row] : d->k2;
      const int32_t* list = block_idx + row * d->k2;
      for (int i = 0; i < nk && i < d->k2; i++)
        if (list[i] >= 0 && list[i] < max_blocks) kept[list[i]] = 1;
    }
    double* logit = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    double* qv = (double*)malloc(sizeof(double) * (size_t)D);
    if (!logit || !qv) {
#pragma omp atomic write
      bad = 1;
      free(kept);
      free(logit);
      free(qv);
      continue;
    }
    for (int c = 0; c < D; c++) qv[c] = bf16_value(q[((int64_t)b * d->hq + j) * D + c]);
    int dense_for_recall = recall != NULL;
    double m = -INFINITY;
    for (int64_t t = 0; t < n; t++) {
      int in_t = all || dense_for_recall || attended(d, n, t, kept);
      if (!in_t) continue;
      double dot = 0.0;
      for (int c = 0; c < D; c++) dot += qv[c] * bf16_value(k[cache_index(d, page_table, b, h, t, c)]);
      logit[t] = dot * scale;
      if (logit[t] > m) m = logit[t];
    }
    double z = 0.0, zt = 0.0;
    for (int64_t t = 0; t < n; t++) {
      int in_t = all || attended(d, n, t, kept);
      if (!(in_t || dense_for_recall)) continue;
      double e = exp(logit[t] - m);
      z += e;
      if (in_t) zt += e;
    }
    if (recall) {
      recall[bj] = n > 0 ? zt / z : 0.0;
    } else if (mass) {
      double* row = mass + (int64_t)bj * max_blocks;
      for (int64_t i = 0; i < max_blocks; i++) row[i] = 0.0;
      for (int64_t t = 0; t < n; t++)
        if (attended(d, n, t, kept)) row[t / d->block] += exp(logit[t] - m) / z;
    } else {
      double* o = out + (int64_t)bj * D;
      for (int c = 0; c < D; c++) o[c] = 0.0;
      for (int64_t t = 0; t < n; t++) {
        if (!(all || attended(d, n, t, kept))) continue;
        double p = exp(logit[t] - m) / z;
        for (int c = 0; c < D; c++) o[c] += p * bf16_value(v[cache_index(d, page_table, b, h, t, c)]);
      }
      if (lse) lse[bj] = n > 0 ? m + log(z) : -INFINITY;
    }
    free(kept);
    free(logit);
    free(qv);
  }
  return bad ? 3 : 0;
}

/* Sparse decode attention over T (sink, window and the kept blocks inside C).
 * out [B][Hq][D], lse [B][Hq] (nullable); qh_mask [B][Hq] selects query heads
 * (nullable = all). */
int oracle_attend(const oracle_dims* d, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                  const int32_t* page_table, const int32_t* lens, const int32_t* block_idx,
                  const int32_t* n_blocks, const int32_t* qh_mask, double* out, double* lse) {
  if (!dims_ok(d) || !q || !k || !v || !page_table || !lens || !block_idx || !out) return 1;
  for (int b = 0; b < d->batch; b++)
    if (!seq_ok(d, page_table, lens, b)) return 2;
  return attention_common(d, q, k, v, page_table, lens, block_idx, n_blocks, qh_mask, 0, out, lse,
                          NULL, NULL);
}

/* Dense decode attention over the whole context [0, N). */
int oracle_dense(const oracle_dims* d, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                 const int32_t* page_table, const int32_t* lens, const int32_t* qh_mask,
                 double* out, double* lse) {
  if (!dims_ok(d) || !q || !k || !v || !page_table || !lens || !out) return 1;
  for (int b = 0; b < d->batch; b++)
    if (!seq_ok(d, page_table, lens, b)) return 2;
  return attention_common(d, q, k, v, page_table, lens, NULL, NULL, qh_mask, 1, out, lse, NULL,
                          NULL);
}

/* Attention-mass recall of T against dense attention ([HiP], latency section: recall of
 * the attention probability of the important tokens): R = sum_{t in T} p_dense(t). */
int oracle_recall(const oracle_dims* d, const uint16_t* q, const uint16_t* k,
                  const int32_t* page_table, const int32_t* lens, const int32_t* block_idx,
                  const int32_t* n_blocks, const int32_t* qh_mask, double* recall) {
  if (!dims_ok(d) || !q || !k || !page_table || !lens || !block_idx || !recall) return 1;
  for (int b = 0; b < d->batch; b++)
    if (!seq_ok(d, page_table, lens, b)) return 2;
  return attention_common(d, q, k, NULL, page_table, lens, block_idx, n_blocks, qh_mask, 0, NULL,
                          NULL, recall, NULL);
}

/* Attention mass of every block under the sparse attention of one call: mass [B][Hq][max
 * blocks], the softmax probability over T that the block's attended tokens receive from
 * query head j (zero for blocks outside T). Summed over the G query heads of a kv head and
 * accumulated over the calls, it is the cumulative magnitude by which the block cache evicts
 * ([HCA] contribution list: dynamic, reversible eviction of the least important KV pairs from
 * the GPU cache by a cumulative-magnitude criterion; the evicted pairs stay in host memory). */
int oracle_block_mass(const oracle_dims* d, const uint16_t* q, const uint16_t* k,
                      const int32_t* page_table, const int32_t* lens, const int32_t* block_idx,
                      const int32_t* n_blocks, double* mass) {
  if (!dims_ok(d) || !q || !k || !page_table || !lens || !block_idx || !mass) return 1;
  for (int b = 0; b < d->batch; b++)
    if (!seq_ok(d, page_table, lens, b)) return 2;
  return attention_common(d, q, k, NULL, page_table, lens, block_idx, n_blocks, NULL, 0, NULL,
                          NULL, NULL, mass);
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* The threads later calls may use (n >= 1); a timing of one thread sets 1, then restores. */
void oracle_set_num_threads(int n) {
#ifdef _OPENMP
  if (n >= 1) omp_set_num_threads(n);
#else
  (void)n;
#endif
}
