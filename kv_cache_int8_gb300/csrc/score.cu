// score.cu -- global scoring of every candidate token over the quantised keys.
//
// Sources: "HCAttention: Extreme KV cache compression via heterogeneous attention computing
// for LLMs", abstract and contribution list (global approximate attention scoring over the
// GPU-resident quantised keys); "KV Cache 与长上下文推理", section "MQA 与 GQA" (G query heads
// share one kv head) and section "KV Cache 量化" (INT8, INT4 and FP8 key formats);
// InfiniteHiP article (163.com), section "实现 7.24 倍的端到端解码加速" (each chunk's best
// token is what the pruning module ranks: here exact per-block and per-64-token-tile maxima
// of the token scores; every head pruned on its own with per-head selection).
//
// score_blocks_kernel (the HBM-bound scan): a persistent grid walks the flattened list of
// 64-token tiles (sequence, kv head, tile). One producer lane per CTA streams each tile's
// four (page, head) blocks into a shared-memory ring with TMA tensor copies (one 4-page copy
// where the pages are consecutive; 128-byte swizzle, so the token-per-lane reads below are
// bank-conflict free) and mbarrier transaction counts. Consumer warps own fixed ring slots;
// lane = token (two tokens per lane, the tile's two halves), dp4a gives the G exact int32
// dot products, their max is the token score and a 16-lane max gives the block maximum.
// 8-bit codes with G <= 4 keep the G x 32 packed query words in registers; 4-bit codes, G = 8
// and per-head maxima read them from a per-warp shared-memory copy, which leaves room for
// more warps. FP8 codes: fp32 scores, one fused multiply-add per channel in channel order
// from the warp's fp32 query copy, whose maxima go on as order-preserving integers.
#include <algorithm>
#include <climits>
#include <type_traits>

#include <cuda_fp16.h>

#include "append.cuh"
#include "common.cuh"
#include "internal.h"

// Tuning of the 4-bit-code instances: consumer warps per CTA, resident CTAs per SM and the
// ring of one CTA (KiB). Measured on GB300 at 1M tokens: 4 warps x 3 CTAs with a 64 KiB ring
// beats 8 x 2 (113 against 141 us); 4 x 4 with 48 KiB rings is no faster.
#ifndef HSA_SCORE_QS_WARPS
#define HSA_SCORE_QS_WARPS 4
#endif
#ifndef HSA_SCORE_QS_CTAS
#define HSA_SCORE_QS_CTAS 3
#endif
#ifndef HSA_SCORE_QS_RING_KB
#define HSA_SCORE_QS_RING_KB 64
#endif
// The same for the 8-bit-code instances that keep the query words in registers. Measured on
// GB300 (one-launch graphs, 128K / 1M): 4 warps x 2 CTAs with 64 KiB rings 27.1 / 157.7 us;
// 8 x 1 with 128 KiB 34.7 / 214.9; 4 x 2 with 96 KiB 27.3 / 165.8; 2 x 3 with 64 KiB
// 29.8 / 171.1.
#ifndef HSA_SCORE_WARPS
#define HSA_SCORE_WARPS 4
#endif
#ifndef HSA_SCORE_CTAS
#define HSA_SCORE_CTAS 2
#endif
#ifndef HSA_SCORE_RING_KB
#define HSA_SCORE_RING_KB 64
#endif

namespace hsa {
namespace {

// ------------------------------------------------------------------ scorer

constexpr int kTileBlocks = 4;                  // blocks per ring slot (64 tokens)
constexpr int kTileTokens = kTileBlocks * kPage;
constexpr int kMaxBatch = 1024;                 // sequences (the tile prefix sums in shared memory)
// 8-bit codes, up to 4 heads: short scans (at most kShortScanTiles tiles) and batches of
// several sequences run the shared-memory-query shape, more and smaller CTAs with fewer tiles
// each (128K: 43.6 against 45.4 us a step; 8 sequences of 32K-128K tokens in permuted pages:
// 122.7 against 125.8 us); one long sequence keeps the query words in registers, 2 CTAs a SM
// (1M: 194.4 against 197.8 us with the short shape).
#ifndef HSA_SCORE_SHORT_TILES
#define HSA_SCORE_SHORT_TILES 32768
#endif
constexpr long long kShortScanTiles = HSA_SCORE_SHORT_TILES;

// Key formats of the scorer instances.
constexpr int kKeyInt8 = 0;  // 8-bit integer codes
constexpr int kKeyInt4 = 1;  // 4-bit integer codes, two per byte
constexpr int kKeyFp8 = 2;   // FP8 E4M3 codes: fp32 scores

// Launch shape and shared-memory layout of one scorer instance (KF: key format; PH:
// per-head maxima, whose epilogue needs the registers the query words would take).
// The short-scan shape (8-bit codes, up to 4 heads, query in shared memory): consumer
// warps, CTAs a SM and ring KiB a CTA. Measured at 128K (step / scorer alone, us): 2 x 5 with
// 32 KiB rings 43.6 / 23.3; 3 x 4, 48 KiB 43.7 / 23.9; 4 x 3, 64 KiB 43.8 / 23.8; 2 x 4,
// 32 KiB 44.4 / 23.8; 4 x 2, 64 KiB 45.3 / 24.3.
#ifndef HSA_SCORE_Q8_WARPS
#define HSA_SCORE_Q8_WARPS 2
#endif
#ifndef HSA_SCORE_Q8_CTAS
#define HSA_SCORE_Q8_CTAS 5
#endif
#ifndef HSA_SCORE_Q8_RING_KB
#define HSA_SCORE_Q8_RING_KB 32
#endif

// FP8 codes with up to 4 heads: consumer warps, CTAs a SM and ring KiB a CTA.
#ifndef HSA_SCORE_F8_WARPS
#define HSA_SCORE_F8_WARPS 4
#endif
#ifndef HSA_SCORE_F8_CTAS
#define HSA_SCORE_F8_CTAS 3
#endif
#ifndef HSA_SCORE_F8_RING_KB
#define HSA_SCORE_F8_RING_KB 64
#endif

template <int G, int KF, bool PH, bool QS = false>
struct ScoreCfg {
  static constexpr bool KB4 = KF == kKeyInt4;
  static constexpr bool kQSmem = KF != kKeyInt8 || G > 4 || PH || QS;  // query in shared memory
  static constexpr bool kShort = QS && KF == kKeyInt8 && G <= 4 && !PH;  // the short-scan shape
  static constexpr bool kF8 = KF == kKeyFp8 && G <= 4;
  static constexpr int kWarps =
      KB4 ? HSA_SCORE_QS_WARPS
          : (kShort ? HSA_SCORE_Q8_WARPS
                    : (kF8 ? HSA_SCORE_F8_WARPS : (kQSmem ? 4 : HSA_SCORE_WARPS)));
  static constexpr int kThreads = (kWarps + 1) * 32;
  // FP8 with 8 heads: the fp32 query of 4 warps takes 16 KiB, so 2 CTAs fit per SM
  static constexpr int kCtasPerSm =
      KB4 ? HSA_SCORE_QS_CTAS
          : (kShort ? HSA_SCORE_Q8_CTAS
                    : (kF8 ? HSA_SCORE_F8_CTAS
                           : (KF == kKeyFp8 && G > 4 ? 2 : (kQSmem ? 3 : HSA_SCORE_CTAS))));
  // 8-bit codes: one 128-byte row per token; 4-bit codes: two tokens per row
  static constexpr int kRowsPerBlock = KB4 ? kPage / 2 : kPage;
  static constexpr int kBlockBytes = kRowsPerBlock * kHeadDim;
  static constexpr int kSlotBytes = kTileBlocks * kBlockBytes;
  static constexpr int kRingBytes =
      (KB4 ? HSA_SCORE_QS_RING_KB
           : (kShort ? HSA_SCORE_Q8_RING_KB
                     : (kF8 ? HSA_SCORE_F8_RING_KB : (kQSmem ? 64 : HSA_SCORE_RING_KB)))) *
      1024;  // one CTA's ring
  static constexpr int kStages = kRingBytes / kSlotBytes;
  static_assert(kStages % kWarps == 0 && kStages / kWarps >= 2,
                "every consumer warp owns at least two fixed ring slots");
  // words of a warp's query copy: G x 32 code words, or G x 128 fp32 values (FP8 keys)
  static constexpr int kQWarpWords = KF == kKeyFp8 ? G * kHeadDim : G * 32;
  static constexpr int kQWords = kQSmem ? kWarps * kQWarpWords : 0;
  static size_t smem_bytes(int batch) {
    return 1024 + kRingBytes + 2 * kStages * sizeof(uint64_t) + kQWords * sizeof(int) +
           (2 * batch + 1) * sizeof(int);
  }
};

struct ScoreArgs {
  const __nv_bfloat16* q;
  const float* k_scale;
  const int32_t* page_table;
  const int32_t* seq_lens;
  int32_t* block_max;
  int32_t* tile_max;  // nullable: max of each 64-token tile's blocks (= chunk max for chunk 64)
  // nullable: [rows][4] running range of each row's maxima, order-preserving unsigned words
  // raised with atomicMax (zero: empty): max tile, ~min tile, max block, ~min block
  unsigned* row_range;
  // nullable: the decode step's append, done by the last CTA beside the scan (the new token
  // at slot N - 1 is never a candidate: the step has a window of at least one token)
  const uint4* k_new;
  const uint4* v_new;
  __nv_bfloat16* k_cache;
  __nv_bfloat16* v_cache;
  int8_t* kq_out;
  int key_fmt;
  int* err;
  int batch, hkv, max_pages, max_tiles, num_pages, sink, window;
};

// Candidate region of one sequence in block and tile units.
struct SeqRange {
  int lo, hi;          // candidate tokens [lo, hi)
  int k_lo, k_hi;      // blocks holding a candidate token
  int tile_lo, ntile;  // tiles covering [k_lo, k_hi)
};

// From the sequence length n (read once per CTA into shared memory).
__device__ __forceinline__ SeqRange seq_range(const ScoreArgs& a, int n) {
  SeqRange r;
  r.lo = a.sink;
  r.hi = n - a.window;
  if (n < 0 || n > a.max_pages * kPage || r.hi <= r.lo) {
    r.hi = r.lo;
    r.k_lo = r.k_hi = r.tile_lo = r.ntile = 0;
    return r;
  }
  r.k_lo = r.lo / kPage;
  r.k_hi = (r.hi + kPage - 1) / kPage;
  r.tile_lo = r.k_lo / kTileBlocks;
  r.ntile = (r.k_hi + kTileBlocks - 1) / kTileBlocks - r.tile_lo;
  return r;
}

// Query folding and quantisation for (b, h), executed by one whole warp: lane l returns the
// packed codes of channels [4l, 4l+4) of each of the G heads.
template <int G>
__device__ __forceinline__ void fold_query_words(int (&word)[G], const ScoreArgs& a, int b,
                                                 int h, int lane) {
  const float4 s4 =
      *reinterpret_cast<const float4*>(a.k_scale + ((size_t)b * a.hkv + h) * kHeadDim + 4 * lane);
  float qp[G][4];
  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < G; j++) {
    const uint2 w = *reinterpret_cast<const uint2*>(
        a.q + ((size_t)b * a.hkv * G + (size_t)h * G + j) * kHeadDim + 4 * lane);
    qp[j][0] = __fmul_rn(bf16_lo(w.x), s4.x);
    qp[j][1] = __fmul_rn(bf16_hi(w.x), s4.y);
    qp[j][2] = __fmul_rn(bf16_lo(w.y), s4.z);
    qp[j][3] = __fmul_rn(bf16_hi(w.y), s4.w);
#pragma unroll
    for (int i = 0; i < 4; i++) amax = fmaxf(amax, fabsf(qp[j][i]));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  const float sq = __fdiv_rn(amax, 127.0f);
#pragma unroll
  for (int j = 0; j < G; j++) {
    int v = 0;
#pragma unroll
    for (int i = 0; i < 4; i++) v |= (int8_code(qp[j][i], sq) & 0xFF) << (8 * i);
    word[j] = v;
  }
}

// Register copy: every lane holds all G x 32 words (word c of head j = channels 4c..4c+3).
template <int G>
__device__ __forceinline__ void load_query_codes(int (&qq)[G][32], const ScoreArgs& a, int b,
                                                 int h, int lane) {
  int word[G];
  fold_query_words<G>(word, a, b, h, lane);
#pragma unroll
  for (int j = 0; j < G; j++)
#pragma unroll
    for (int c = 0; c < 32; c++) qq[j][c] = __shfl_sync(0xffffffffu, word[j], c);
}

// Shared-memory copy qs[G][32] of the warp. 8-bit keys: word c of head j = channels
// 4c..4c+3. 4-bit keys: words 0..15 hold channels 8w, 8w+2, 8w+4, 8w+6 and words 16..31
// channels 8w+1, ..., 8w+7: the even and odd channels that one word of packed key nibbles
// holds.
template <int G, bool KB4>
__device__ __forceinline__ void store_query_codes(int* qs, const ScoreArgs& a, int b, int h,
                                                  int lane) {
  int word[G];
  fold_query_words<G>(word, a, b, h, lane);
#pragma unroll
  for (int j = 0; j < G; j++) {
    int v = word[j];
    if constexpr (KB4) {
      // lane l < 16: even channels of words 2l and 2l + 1; lane l >= 16: their odd channels
      const int p = 2 * (lane & 15);
      const int w0 = __shfl_sync(0xffffffffu, v, p), w1 = __shfl_sync(0xffffffffu, v, p + 1);
      v = (int)__byte_perm(w0, w1, lane < 16 ? 0x6420 : 0x7531);
    }
    qs[j * 32 + lane] = v;
  }
}

// FP8 keys: the warp's shared-memory copy of the folded query itself, qs[G][128] fp32,
// q'_{j,c} = f32(q_{j,c} * s_c) (lane l computes channels [4l, 4l+4) of each head).
template <int G>
__device__ __forceinline__ void store_query_folded(float* qs, const ScoreArgs& a, int b, int h,
                                                   int lane) {
  const float4 s4 =
      *reinterpret_cast<const float4*>(a.k_scale + ((size_t)b * a.hkv + h) * kHeadDim + 4 * lane);
#pragma unroll
  for (int j = 0; j < G; j++) {
    const uint2 w = *reinterpret_cast<const uint2*>(
        a.q + ((size_t)b * a.hkv * G + (size_t)h * G + j) * kHeadDim + 4 * lane);
    *reinterpret_cast<float4*>(qs + j * kHeadDim + 4 * lane) =
        make_float4(__fmul_rn(bf16_lo(w.x), s4.x), __fmul_rn(bf16_hi(w.x), s4.y),
                    __fmul_rn(bf16_lo(w.y), s4.z), __fmul_rn(bf16_hi(w.y), s4.w));
  }
}

// The exact values of four E4M3 codes (byte i of w -> f[i]), through f16 (exact: every
// E4M3 value is an f16 value).
__device__ __forceinline__ void e4m3x4_to_float(uint32_t w, float* f) {
  uint32_t h01, h23;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h01) : "h"((unsigned short)(w & 0xFFFFu)));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h23) : "h"((unsigned short)(w >> 16)));
  f[0] = __half2float(__ushort_as_half((unsigned short)(h01 & 0xFFFFu)));
  f[1] = __half2float(__ushort_as_half((unsigned short)(h01 >> 16)));
  f[2] = __half2float(__ushort_as_half((unsigned short)(h23 & 0xFFFFu)));
  f[3] = __half2float(__ushort_as_half((unsigned short)(h23 >> 16)));
}

// Order-preserving integer of an fp32 score (both zeros map to 0): the block and tile maxima
// of FP8 scores are then taken, written and ranked as integers.
__device__ __forceinline__ int ordered_key(float f) {
  const int bits = __float_as_int(f + 0.0f);  // -0 -> +0
  return bits >= 0 ? bits : bits ^ 0x7FFFFFFF;
}

// 4-bit codes: a 32-bit word holds 8 channels as two's-complement nibbles. Moved into the
// high half of their bytes (the even channels shifted up by 4, the odd ones masked in place),
// the nibbles read as signed bytes equal to 16 x code, so two signed dp4a per word give 16 x
// the dot product, exactly; one arithmetic shift by 4 takes the factor off (|16 x dot| stays
// below 127 x 128 x 128 x 16 < 2^31).
__device__ __forceinline__ int nibbles_even(uint32_t w) { return (int)((w << 4) & 0xF0F0F0F0u); }
__device__ __forceinline__ int nibbles_odd(uint32_t w) { return (int)(w & 0xF0F0F0F0u); }

__device__ __forceinline__ uint32_t word_of(const uint4& v, int m) {
  return m == 0 ? v.x : m == 1 ? v.y : m == 2 ? v.z : v.w;
}

// Order-preserving unsigned image of an int (for atomicMax on the row ranges).
__device__ __forceinline__ unsigned range_key(int v) { return (unsigned)v ^ 0x80000000u; }

// PH: per-head selection, the maxima of every query head (rows b * hq + h * G + j) rather
// than of the group's token scores.
template <int G, int KF, bool PH, bool QS = false>
__global__ void __launch_bounds__(ScoreCfg<G, KF, PH, QS>::kThreads,
                                  ScoreCfg<G, KF, PH, QS>::kCtasPerSm)
    score_blocks_kernel(const __grid_constant__ CUtensorMap kq_map,
                        const __grid_constant__ CUtensorMap kq_map4, const ScoreArgs a) {
  using C = ScoreCfg<G, KF, PH, QS>;
  constexpr bool KB4 = C::KB4;
  constexpr int kStages = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kRingBytes);
  uint64_t* empty = full + kStages;
  int* qbuf = reinterpret_cast<int*>(empty + kStages);  // [consumer warp][G][32] (kQSmem)
  int* prefix = qbuf + C::kQWords;                       // [batch + 1] tiles before b
  int* lens = prefix + a.batch + 1;                      // [batch] sequence lengths

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; s++) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    fence_barrier_init();
  }
  // inputs may come from the previous kernel of the stream; then let the next one launch
  grid_dep_wait();
  grid_dep_launch();
  if (warp == C::kWarps && lane == 0) {
    tma_prefetch_descriptor(&kq_map);
    tma_prefetch_descriptor(&kq_map4);
  }
  // tiles per sequence (x hkv), exclusive prefix sum by warp 0
  if (warp == 0) {
    int carry = 0;
    for (int b0 = 0; b0 < a.batch; b0 += 32) {
      const int b = b0 + lane;
      int v = 0;
      if (b < a.batch) {
        const int n = a.seq_lens[b];
        if (n < 0 || n > a.max_pages * kPage) set_error(a.err, kDevErrCheck);
        lens[b] = n;
        v = seq_range(a, n).ntile * a.hkv;
      }
      int x = v;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
      }
      if (b < a.batch) prefix[b] = carry + x - v;
      carry += __shfl_sync(0xffffffffu, x, 31);
    }
    if (lane == 0) prefix[a.batch] = carry;
  }
  __syncthreads();

  // the CTA that appends (the last) takes about 1.5 us worth of tiles fewer
  const long long total = prefix[a.batch];
  const long long hcap = a.k_new != nullptr ? (KB4 ? 8 : 4) : 0;
  const int f0 = (int)((total + hcap) * blockIdx.x / gridDim.x);
  const int f1 = (int)min(total, (total + hcap) * (blockIdx.x + 1) / gridDim.x);
  if (a.k_new != nullptr && blockIdx.x == gridDim.x - 1 && warp < C::kWarps) {
    // the append (its producer warp is already streaming this CTA's tiles)
    const int per_seq = a.hkv * 16;
    for (int i = threadIdx.x; i < a.batch * per_seq; i += C::kWarps * 32)
      append_token(i / per_seq, i % per_seq, a.k_new, a.v_new, a.k_cache, a.v_cache, a.kq_out,
                   a.k_scale, a.page_table, a.seq_lens, a.hkv, a.max_pages, a.num_pages, a.err,
                   a.key_fmt);
  }
  if (f0 >= f1) return;

  int b = 0;
  while (prefix[b + 1] <= f0) b++;

  if (warp == C::kWarps) {
    // ------------------------------------------------------------ producer
    // The whole warp resolves the page ids of the next 32 tiles at once (one coalesced
    // round trip), then lane 0 issues their copies in order as ring slots free up: one copy
    // of the four blocks when they sit in consecutive pages, else one copy per block.
    bool ok = true;
    const uint64_t policy = l2_evict_first_policy();  // each code is read once
    int bw = b;  // sequence of tile f0 + jb (warp-uniform)
    for (int jb = 0; ok && f0 + jb < f1; jb += 32) {
      const int f = f0 + jb + lane;
      int rows[kTileBlocks];
#pragma unroll
      for (int i = 0; i < kTileBlocks; i++) rows[i] = -1;
      int run_page = -1, run_head = 0;  // first page of 4 consecutive ones, and the head
      if (f < f1) {
        int bl = bw;
        while (prefix[bl + 1] <= f) bl++;
        const SeqRange sr = seq_range(a, lens[bl]);
        const int r = f - prefix[bl];
        const int h = r / sr.ntile;
        const int tile = sr.tile_lo + r % sr.ntile;
        const int32_t* row = a.page_table + (size_t)bl * a.max_pages;
        int pg[kTileBlocks];
#pragma unroll
        for (int i = 0; i < kTileBlocks; i++) {
          const int k = tile * kTileBlocks + i;
          pg[i] = (k >= sr.k_lo && k < sr.k_hi) ? row[k] : -2;
        }
#pragma unroll
        for (int i = 0; i < kTileBlocks; i++) {
          if (pg[i] == -2) continue;
          if (pg[i] < 0 || pg[i] >= a.num_pages) {
            set_error(a.err, kDevErrCheck);
            continue;
          }
          rows[i] = (pg[i] * a.hkv + h) * C::kRowsPerBlock;
        }
        bool run = rows[0] >= 0;
#pragma unroll
        for (int i = 1; i < kTileBlocks; i++) run = run && rows[i] >= 0 && pg[i] == pg[0] + i;
        if (run) {
          run_page = pg[0];
          run_head = h;
        }
      }
      const int n = min(32, f1 - f0 - jb);
      for (int i = 0; i < n; i++) {
        int rr[kTileBlocks];
#pragma unroll
        for (int q = 0; q < kTileBlocks; q++) rr[q] = __shfl_sync(0xffffffffu, rows[q], i);
        const int rp = __shfl_sync(0xffffffffu, run_page, i);
        const int rh = __shfl_sync(0xffffffffu, run_head, i);
        if (lane == 0) {
          const int j = jb + i;
          const int s = j % kStages;
          if (j >= kStages && !mbar_wait(&empty[s], ((j / kStages) - 1) & 1)) {
            set_error(a.err, kDevErrTimeout);
            ok = false;
          } else {
            uint32_t bytes = 0;
#pragma unroll
            for (int q = 0; q < kTileBlocks; q++) bytes += rr[q] >= 0 ? C::kBlockBytes : 0;
            mbar_arrive_expect_tx(&full[s], bytes);
            uint8_t* dst = ring + s * C::kSlotBytes;
            if (rp >= 0) {
              tma_load_4d_hint(dst, &kq_map4, 0, 0, rh, rp, &full[s], policy);
            } else {
#pragma unroll
              for (int q = 0; q < kTileBlocks; q++)
                if (rr[q] >= 0)
                  tma_load_2d_hint(dst + q * C::kBlockBytes, &kq_map, 0, rr[q], &full[s], policy);
            }
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
      }
      // advance the warp's sequence cursor to the first tile of the next batch
      const int fn = f0 + jb + 32;
      while (bw + 1 < a.batch && prefix[bw + 1] <= fn) bw++;
    }
    if (!ok && lane == 0) {
      // let the copies already issued land before the CTA exits (bounded)
      const int issued = f1 - f0;
      for (int j = max(0, issued - kStages); j < issued; j++)
        mbar_wait(&full[j % kStages], (j / kStages) & 1);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  int qq[C::kQSmem ? 1 : G][32];  // register copy of the query words (8-bit codes, G <= 4)
  int* qs = qbuf + (C::kQSmem ? warp * C::kQWarpWords : 0);
  const uint32_t qs_addr = smem_addr(qs);
  int cur_b = -1, cur_h = -1;
  SeqRange sr = seq_range(a, lens[b]);
  // this lane's running range of the current (b, h)'s maxima, flushed when (b, h) changes
  constexpr int kRows = PH ? G : 1;
  unsigned rng[kRows][4];
#pragma unroll
  for (int jr = 0; jr < kRows; jr++) rng[jr][0] = rng[jr][1] = rng[jr][2] = rng[jr][3] = 0u;
  auto flush_range = [&](int fb, int fh) {
#pragma unroll
    for (int jr = 0; jr < kRows; jr++) {
      const size_t row = PH ? ((size_t)fb * a.hkv + fh) * G + jr : (size_t)fb * a.hkv + fh;
#pragma unroll
      for (int w = 0; w < 4; w++) {
        const unsigned v = __reduce_max_sync(0xffffffffu, rng[jr][w]);
        if (lane == 0 && v != 0u) atomicMax(a.row_range + row * 4 + w, v);
        rng[jr][w] = 0u;
      }
    }
  };
  for (int j = warp; f0 + j < f1; j += C::kWarps) {
    const int f = f0 + j;
    while (prefix[b + 1] <= f) {
      b++;
      sr = seq_range(a, lens[b]);
    }
    const int r = f - prefix[b];
    const int h = r / sr.ntile;
    const int tile = sr.tile_lo + r % sr.ntile;
    if (b != cur_b || h != cur_h) {
      if (a.row_range != nullptr && cur_b >= 0) flush_range(cur_b, cur_h);
      if constexpr (C::kQSmem) {
        __syncwarp();  // every lane is done reading the previous words
        if constexpr (KF == kKeyFp8)
          store_query_folded<G>(reinterpret_cast<float*>(qs), a, b, h, lane);
        else
          store_query_codes<G, KB4>(qs, a, b, h, lane);
        __syncwarp();
      } else {
        load_query_codes<G>(qq, a, b, h, lane);
      }
      cur_b = b;
      cur_h = h;
    }
    const int s = j % kStages;
    if (!mbar_wait(&full[s], (j / kStages) & 1)) {
      set_error(a.err, kDevErrTimeout);
      break;
    }
    const uint32_t sbase = smem_addr(ring + s * C::kSlotBytes);
    // both 32-token halves of the tile at once (lane = token `half * 32 + lane`)
    int acc[2][G];
#pragma unroll
    for (int half = 0; half < 2; half++)
#pragma unroll
      for (int jj = 0; jj < G; jj++) acc[half][jj] = 0;
    if constexpr (KB4) {
      // token `row` is half `row & 1` of 128-byte row `row >> 1` of the tile; the row's
      // swizzle phase (row >> 1) & 7 is the same for both halves
      const int sub = lane & 1, ph = (lane >> 1) & 7;
#pragma unroll
      for (int c = 0; c < 4; c++) {
        int ev[2][4], od[2][4];
#pragma unroll
        for (int half = 0; half < 2; half++) {
          const uint4 kv =
              lds128(sbase + (half * 16 + (lane >> 1)) * 128 + (((sub * 4 + c) ^ ph) << 4));
#pragma unroll
          for (int m = 0; m < 4; m++) {
            ev[half][m] = nibbles_even(word_of(kv, m));
            od[half][m] = nibbles_odd(word_of(kv, m));
          }
        }
#pragma unroll
        for (int jj = 0; jj < G; jj++) {
          const uint4 qe = lds128(qs_addr + (jj * 32 + 4 * c) * 4);
          const uint4 qo = lds128(qs_addr + (jj * 32 + 16 + 4 * c) * 4);
#pragma unroll
          for (int m = 0; m < 4; m++)
#pragma unroll
            for (int half = 0; half < 2; half++) {
              acc[half][jj] = __dp4a(ev[half][m], (int)word_of(qe, m), acc[half][jj]);
              acc[half][jj] = __dp4a(od[half][m], (int)word_of(qo, m), acc[half][jj]);
            }
        }
      }
#pragma unroll
      for (int half = 0; half < 2; half++)
#pragma unroll
        for (int jj = 0; jj < G; jj++) acc[half][jj] >>= 4;
    } else if constexpr (KF == kKeyFp8) {
      // fp32 scores: one fused multiply-add per channel, in channel order, of the folded
      // query with the exact values of the E4M3 codes; then their order-preserving integers
      float facc[2][G];
#pragma unroll
      for (int half = 0; half < 2; half++)
#pragma unroll
        for (int jj = 0; jj < G; jj++) facc[half][jj] = 0.0f;
#pragma unroll 1
      for (int c = 0; c < 8; c++) {  // channels 16c .. 16c + 15
        float x[2][16];
#pragma unroll
        for (int half = 0; half < 2; half++) {
          const uint4 kv =
              lds128(sbase + (half * 32 + lane) * kHeadDim + ((c ^ (lane & 7)) << 4));
#pragma unroll
          for (int m = 0; m < 4; m++) e4m3x4_to_float(word_of(kv, m), &x[half][4 * m]);
        }
#pragma unroll
        for (int jj = 0; jj < G; jj++) {
#pragma unroll
          for (int i4 = 0; i4 < 4; i4++) {
            const uint4 q4 = lds128(qs_addr + (jj * kHeadDim + 16 * c + 4 * i4) * 4);
            const float qv[4] = {__uint_as_float(q4.x), __uint_as_float(q4.y),
                                 __uint_as_float(q4.z), __uint_as_float(q4.w)};
#pragma unroll
            for (int i = 0; i < 4; i++)
#pragma unroll
              for (int half = 0; half < 2; half++)
                facc[half][jj] = __fmaf_rn(qv[i], x[half][4 * i4 + i], facc[half][jj]);
          }
        }
      }
#pragma unroll
      for (int half = 0; half < 2; half++)
#pragma unroll
        for (int jj = 0; jj < G; jj++) acc[half][jj] = ordered_key(facc[half][jj]);
    } else {
#pragma unroll
      for (int c = 0; c < 8; c++) {
        uint4 kv[2];
#pragma unroll
        for (int half = 0; half < 2; half++)
          kv[half] = lds128(sbase + (half * 32 + lane) * kHeadDim + ((c ^ (lane & 7)) << 4));
#pragma unroll
        for (int jj = 0; jj < G; jj++) {
          uint4 qv;
          if constexpr (C::kQSmem) {
            qv = lds128(qs_addr + (jj * 32 + 4 * c) * 4);
          } else {
            qv = make_uint4(qq[jj][4 * c], qq[jj][4 * c + 1], qq[jj][4 * c + 2], qq[jj][4 * c + 3]);
          }
#pragma unroll
          for (int half = 0; half < 2; half++)
#pragma unroll
            for (int m = 0; m < 4; m++)
              acc[half][jj] = __dp4a((int)word_of(kv[half], m), (int)word_of(qv, m), acc[half][jj]);
        }
      }
    }
    // block and tile maxima of the token scores (the max over the group's heads), or of each
    // head's own dot products with per-head selection
#pragma unroll
    for (int jr = 0; jr < kRows; jr++) {
      const size_t row = PH ? ((size_t)b * a.hkv + h) * G + jr : (size_t)b * a.hkv + h;
      int tmax = INT_MIN;
#pragma unroll
      for (int half = 0; half < 2; half++) {
        const int t = tile * kTileTokens + half * 32 + lane;
        int g = acc[half][PH ? jr : 0];
        if constexpr (!PH) {
#pragma unroll
          for (int jj = 1; jj < G; jj++) g = max(g, acc[half][jj]);
        }
        if (t < sr.lo || t >= sr.hi) g = INT_MIN;
        g = max(g, __shfl_xor_sync(0xffffffffu, g, 8));
        g = max(g, __shfl_xor_sync(0xffffffffu, g, 4));
        g = max(g, __shfl_xor_sync(0xffffffffu, g, 2));
        g = max(g, __shfl_xor_sync(0xffffffffu, g, 1));
        if ((lane & 15) == 0) {
          const int k = tile * kTileBlocks + half * 2 + (lane >> 4);
          if (k >= sr.k_lo && k < sr.k_hi) {
            a.block_max[row * a.max_pages + k] = g;
            rng[jr][2] = max(rng[jr][2], range_key(g));
            rng[jr][3] = max(rng[jr][3], ~range_key(g));
          }
        }
        tmax = max(tmax, g);
      }
      tmax = max(tmax, __shfl_xor_sync(0xffffffffu, tmax, 16));
      if (a.tile_max != nullptr && lane == 0) a.tile_max[row * a.max_tiles + tile] = tmax;
      if (lane == 0) {
        rng[jr][0] = max(rng[jr][0], range_key(tmax));
        rng[jr][1] = max(rng[jr][1], ~range_key(tmax));
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
  if (a.row_range != nullptr && cur_b >= 0) flush_range(cur_b, cur_h);
}

}  // namespace

int score_max_tiles(const Shape& s) { return (s.max_pages + kTileBlocks - 1) / kTileBlocks; }

cudaError_t launch_score_blocks(const Shape& s, const CUtensorMap& kq_map,
                                const CUtensorMap& kq_map4, const void* q,
                                const float* k_scale, const int32_t* page_table,
                                const int32_t* seq_lens, int32_t* block_max, int32_t* tile_max,
                                unsigned* row_range, const AppendArgs* app, int* err,
                                int num_sms, cudaStream_t st) {
  if (s.batch > kMaxBatch) return cudaErrorInvalidValue;
  ScoreArgs a;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.k_scale = k_scale;
  a.page_table = page_table;
  a.seq_lens = seq_lens;
  a.block_max = block_max;
  a.tile_max = tile_max;
  a.row_range = row_range;
  a.k_new = app ? static_cast<const uint4*>(app->k_new) : nullptr;
  a.v_new = app ? static_cast<const uint4*>(app->v_new) : nullptr;
  a.k_cache = app ? static_cast<__nv_bfloat16*>(app->k_cache) : nullptr;
  a.v_cache = app ? static_cast<__nv_bfloat16*>(app->v_cache) : nullptr;
  a.kq_out = app ? app->kq : nullptr;
  a.key_fmt = s.key_fp8 ? append_detail::kFmtFp8 : s.key_bits;
  a.err = err;
  a.batch = s.batch;
  a.hkv = s.hkv;
  a.max_pages = s.max_pages;
  a.max_tiles = score_max_tiles(s);
  a.num_pages = s.num_pages;
  a.sink = s.sink;
  a.window = s.window;
  // upper bound of the tile count; the kernel splits the true count evenly
  const long long tiles_max =
      (long long)s.batch * s.hkv * ((s.max_pages + kTileBlocks - 1) / kTileBlocks + 1);
  auto go = [&](auto kernel, auto cfg) {
    using C = decltype(cfg);
    const size_t smem = C::smem_bytes(s.batch);
    const int grid = (int)std::min<long long>(tiles_max, (long long)C::kCtasPerSm * num_sms);
    cudaError_t e = set_kernel_smem(kernel, smem);
    if (e != cudaSuccess) return e;
    return launch_kernel(kernel, dim3(grid), dim3(C::kThreads), smem, st, true, kq_map, kq_map4,
                         a);
  };
  const int kf = s.key_fp8 ? kKeyFp8 : (s.key_bits == 4 ? kKeyInt4 : kKeyInt8);
  auto go_kf = [&](auto g_, auto ph_) {
    constexpr int g = decltype(g_)::value;
    constexpr bool ph = decltype(ph_)::value;
    switch (kf) {
      case kKeyInt4:
        return go(score_blocks_kernel<g, kKeyInt4, ph>, ScoreCfg<g, kKeyInt4, ph>{});
      case kKeyFp8:
        return go(score_blocks_kernel<g, kKeyFp8, ph>, ScoreCfg<g, kKeyFp8, ph>{});
      default:
        if constexpr (g <= 4 && !ph) {
          if (tiles_max <= kShortScanTiles || s.batch > 1)
            return go(score_blocks_kernel<g, kKeyInt8, ph, true>, ScoreCfg<g, kKeyInt8, ph, true>{});
        }
        return go(score_blocks_kernel<g, kKeyInt8, ph>, ScoreCfg<g, kKeyInt8, ph>{});
    }
  };
#define HSA_SCORE_CASE(g)                                                    \
  case g:                                                                    \
    e = s.per_head ? go_kf(std::integral_constant<int, g>{}, std::true_type{}) \
                   : go_kf(std::integral_constant<int, g>{}, std::false_type{}); \
    break;
  cudaError_t e;
  switch (s.group) {
    HSA_SCORE_CASE(1)
    HSA_SCORE_CASE(2)
    HSA_SCORE_CASE(4)
    HSA_SCORE_CASE(8)
    default:
      return cudaErrorInvalidValue;
  }
#undef HSA_SCORE_CASE
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace hsa
