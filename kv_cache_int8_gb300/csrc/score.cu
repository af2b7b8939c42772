// score.cu -- global int8 scoring of every candidate token.
//
// Sources: "HCAttention: Extreme KV cache compression via heterogeneous attention computing
// for LLMs", abstract and contribution list (global approximate attention scoring over the
// GPU-resident quantised keys); "KV Cache 与长上下文推理", section "MQA 与 GQA" (G query heads
// share one kv head); InfiniteHiP article (163.com), section "实现 7.24 倍的端到端解码加速"
// (each chunk's best token is what the pruning module ranks: here exact per-block and
// per-64-token-tile maxima of the token scores).
//
// score_blocks_kernel (the HBM-bound scan): a persistent grid walks the flattened list of
// 64-token tiles (sequence, kv head, tile). One producer lane per CTA streams each tile's
// four 2 KiB (page, head) blocks into a shared-memory ring with TMA tensor copies
// (128-byte swizzle, so the token-per-lane reads below are bank-conflict free) and
// mbarrier transaction counts. Consumer warps own fixed ring slots; lane = token, the
// G x 32 packed int8 query words sit in registers, dp4a gives the G exact int32 dot
// products, their max is the token score and a 16-lane max gives the block maximum.
#include <algorithm>
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace hsa {
namespace {

// ------------------------------------------------------------------ scorer

constexpr int kTileBlocks = 4;                             // blocks per ring slot (64 tokens)
constexpr int kTileTokens = kTileBlocks * kPage;
constexpr int kStageBytes = kTileBlocks * kBlockBytesI8;   // 8 KiB
constexpr int kScoreWarps = 4;                             // consumer warps
constexpr int kScoreStages = 8;                            // ring slots (multiple of kScoreWarps)
constexpr int kScoreThreads = (kScoreWarps + 1) * 32;
constexpr int kMaxBatch = 1024;
static_assert(kScoreStages % kScoreWarps == 0, "each consumer warp owns fixed ring slots");

struct ScoreArgs {
  const __nv_bfloat16* q;
  const float* k_scale;
  const int32_t* page_table;
  const int32_t* seq_lens;
  int32_t* block_max;
  int32_t* tile_max;  // nullable: max of each 64-token tile's blocks (= chunk max for chunk 64)
  int* err;
  int batch, hkv, max_pages, max_tiles, num_pages, sink, window;
};

// Candidate region of one sequence in block and tile units.
struct SeqRange {
  int lo, hi;          // candidate tokens [lo, hi)
  int k_lo, k_hi;      // blocks holding a candidate token
  int tile_lo, ntile;  // tiles covering [k_lo, k_hi)
};

__device__ __forceinline__ SeqRange seq_range(const ScoreArgs& a, int b) {
  SeqRange r;
  const int n = a.seq_lens[b];
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

// Query folding and quantisation for (b, h), executed by one whole warp. Lane l computes
// channels [4l, 4l+4) of each of the G heads; the packed code words are then broadcast so
// that every lane holds all G x 32 words (uniform registers of the dot-product loop).
template <int G>
__device__ __forceinline__ void load_query_codes(int (&qq)[G][32], const ScoreArgs& a, int b,
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
    int word = 0;
#pragma unroll
    for (int i = 0; i < 4; i++) word |= (int8_code(qp[j][i], sq) & 0xFF) << (8 * i);
#pragma unroll
    for (int c = 0; c < 32; c++) qq[j][c] = __shfl_sync(0xffffffffu, word, c);
  }
}

// The query code words of the 4-bit key format: word w of head j becomes the codes of
// channels 8w, 8w+2, 8w+4, 8w+6 (qq[j][w]) and 8w+1, ..., 8w+7 (qq[j][16 + w]), the even and
// odd channels that one word of packed key nibbles holds.
template <int G>
__device__ __forceinline__ void split_query_codes(int (&qq)[G][32]) {
#pragma unroll
  for (int j = 0; j < G; j++) {
    int o[16];
#pragma unroll
    for (int w = 0; w < 16; w++) {
      // reads words 2w and 2w + 1, never yet overwritten (only words below w are)
      const int e = (int)__byte_perm(qq[j][2 * w], qq[j][2 * w + 1], 0x6420);
      o[w] = (int)__byte_perm(qq[j][2 * w], qq[j][2 * w + 1], 0x7531);
      qq[j][w] = e;
    }
#pragma unroll
    for (int w = 0; w < 16; w++) qq[j][16 + w] = o[w];
  }
}

// KB4: 4-bit key codes. Two tokens share a 128-byte row of the TMA box (a block is 8 rows,
// 1 KiB); each 32-bit word holds 8 channels as two's-complement nibbles. Moved into the high
// half of their bytes (the even channels shifted up by 4, the odd ones masked in place), the
// nibbles read as signed bytes equal to 16 x code, so two signed dp4a per word give 16 x the
// dot product, exactly; one arithmetic shift by 4 takes the factor off (|16 x dot| stays
// below 127 x 128 x 128 x 16 < 2^31).
template <int G, bool KB4>
__global__ void __launch_bounds__(kScoreThreads, 2)
    score_blocks_kernel(const __grid_constant__ CUtensorMap kq_map, const ScoreArgs a) {
  constexpr int kRowsPerBlock = KB4 ? kPage / 2 : kPage;  // rows of the TMA box per block
  constexpr int kBlockBytes = KB4 ? kBlockBytesI8 / 2 : kBlockBytesI8;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kScoreStages * kStageBytes);
  uint64_t* empty = full + kScoreStages;
  int* prefix = reinterpret_cast<int*>(empty + kScoreStages);  // [batch + 1] tiles before b

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kScoreStages; s++) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    fence_barrier_init();
  }
  // inputs may come from the previous kernel of the stream; then let the next one launch
  grid_dep_wait();
  grid_dep_launch();
  if (warp == kScoreWarps && lane == 0) tma_prefetch_descriptor(&kq_map);
  // tiles per sequence (x hkv), exclusive prefix sum by warp 0
  if (warp == 0) {
    int carry = 0;
    for (int b0 = 0; b0 < a.batch; b0 += 32) {
      const int b = b0 + lane;
      int v = 0;
      if (b < a.batch) {
        const int n = a.seq_lens[b];
        if (n < 0 || n > a.max_pages * kPage) set_error(a.err, kDevErrCheck);
        v = seq_range(a, b).ntile * a.hkv;
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

  const long long total = prefix[a.batch];
  const int f0 = (int)(total * blockIdx.x / gridDim.x);
  const int f1 = (int)(total * (blockIdx.x + 1) / gridDim.x);
  if (f0 >= f1) return;

  int b = 0;
  while (prefix[b + 1] <= f0) b++;

  if (warp == kScoreWarps) {
    // ------------------------------------------------------------ producer
    // The whole warp resolves the page ids of the next 32 tiles at once (one coalesced
    // round trip), then lane 0 issues their copies in order as ring slots free up.
    bool ok = true;
    const uint64_t policy = l2_evict_first_policy();  // each code is read once
    int bw = b;  // sequence of tile f0 + jb (warp-uniform)
    for (int jb = 0; ok && f0 + jb < f1; jb += 32) {
      const int f = f0 + jb + lane;
      int rows[kTileBlocks];
#pragma unroll
      for (int i = 0; i < kTileBlocks; i++) rows[i] = -1;
      if (f < f1) {
        int bl = bw;
        while (prefix[bl + 1] <= f) bl++;
        const SeqRange sr = seq_range(a, bl);
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
          rows[i] = (pg[i] * a.hkv + h) * kRowsPerBlock;
        }
      }
      const int n = min(32, f1 - f0 - jb);
      for (int i = 0; i < n; i++) {
        int rr[kTileBlocks];
#pragma unroll
        for (int q = 0; q < kTileBlocks; q++) rr[q] = __shfl_sync(0xffffffffu, rows[q], i);
        if (lane == 0) {
          const int j = jb + i;
          const int s = j % kScoreStages;
          if (j >= kScoreStages && !mbar_wait(&empty[s], ((j / kScoreStages) - 1) & 1)) {
            set_error(a.err, kDevErrTimeout);
            ok = false;
          } else {
            uint32_t bytes = 0;
#pragma unroll
            for (int q = 0; q < kTileBlocks; q++) bytes += rr[q] >= 0 ? kBlockBytes : 0;
            mbar_arrive_expect_tx(&full[s], bytes);
#pragma unroll
            for (int q = 0; q < kTileBlocks; q++)
              if (rr[q] >= 0)
                tma_load_2d_hint(ring + s * kStageBytes + q * kBlockBytes, &kq_map, 0, rr[q],
                                 &full[s], policy);
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
      for (int j = max(0, issued - kScoreStages); j < issued; j++)
        mbar_wait(&full[j % kScoreStages], (j / kScoreStages) & 1);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  int qq[G][32];
  int cur_b = -1, cur_h = -1;
  SeqRange sr = seq_range(a, b);
  for (int j = warp; f0 + j < f1; j += kScoreWarps) {
    const int f = f0 + j;
    while (prefix[b + 1] <= f) {
      b++;
      sr = seq_range(a, b);
    }
    const int r = f - prefix[b];
    const int h = r / sr.ntile;
    const int tile = sr.tile_lo + r % sr.ntile;
    if (b != cur_b || h != cur_h) {
      load_query_codes<G>(qq, a, b, h, lane);
      if constexpr (KB4) split_query_codes<G>(qq);
      cur_b = b;
      cur_h = h;
    }
    const int s = j % kScoreStages;
    if (!mbar_wait(&full[s], (j / kScoreStages) & 1)) {
      set_error(a.err, kDevErrTimeout);
      break;
    }
    const uint32_t sbase = smem_addr(ring + s * kStageBytes);
    int32_t* out = a.block_max + ((size_t)b * a.hkv + h) * a.max_pages;
    int tmax = INT_MIN;
#pragma unroll
    for (int half = 0; half < 2; half++) {
      const int row = half * 32 + lane;           // token within the tile
      const int t = tile * kTileTokens + row;
      const uint32_t rbase = sbase + row * kHeadDim;
      int acc[G];
#pragma unroll
      for (int jj = 0; jj < G; jj++) acc[jj] = 0;
      if constexpr (KB4) {
        // token `row` is half `row & 1` of 128-byte row `row >> 1` of the tile
        const int r = row >> 1, sub = row & 1;
        const uint32_t rb = sbase + r * 128;
#pragma unroll
        for (int c = 0; c < 4; c++) {
          const uint4 kv = lds128(rb + (((sub * 4 + c) ^ (r & 7)) << 4));
          const uint32_t wv[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
          for (int m = 0; m < 4; m++) {
            const int ev = (int)((wv[m] << 4) & 0xF0F0F0F0u), od = (int)(wv[m] & 0xF0F0F0F0u);
#pragma unroll
            for (int jj = 0; jj < G; jj++) {
              acc[jj] = __dp4a(ev, qq[jj][4 * c + m], acc[jj]);
              acc[jj] = __dp4a(od, qq[jj][16 + 4 * c + m], acc[jj]);
            }
          }
        }
#pragma unroll
        for (int jj = 0; jj < G; jj++) acc[jj] >>= 4;
      } else {
#pragma unroll
        for (int c = 0; c < 8; c++) {
          const uint4 kv = lds128(rbase + ((c ^ (row & 7)) << 4));
#pragma unroll
          for (int jj = 0; jj < G; jj++) {
            acc[jj] = __dp4a((int)kv.x, qq[jj][4 * c + 0], acc[jj]);
            acc[jj] = __dp4a((int)kv.y, qq[jj][4 * c + 1], acc[jj]);
            acc[jj] = __dp4a((int)kv.z, qq[jj][4 * c + 2], acc[jj]);
            acc[jj] = __dp4a((int)kv.w, qq[jj][4 * c + 3], acc[jj]);
          }
        }
      }
      int g = acc[0];
#pragma unroll
      for (int jj = 1; jj < G; jj++) g = max(g, acc[jj]);
      if (t < sr.lo || t >= sr.hi) g = INT_MIN;
      g = max(g, __shfl_xor_sync(0xffffffffu, g, 8));
      g = max(g, __shfl_xor_sync(0xffffffffu, g, 4));
      g = max(g, __shfl_xor_sync(0xffffffffu, g, 2));
      g = max(g, __shfl_xor_sync(0xffffffffu, g, 1));
      if ((lane & 15) == 0) {
        const int k = tile * kTileBlocks + half * 2 + (lane >> 4);
        if (k >= sr.k_lo && k < sr.k_hi) out[k] = g;
      }
      tmax = max(tmax, g);
    }
    tmax = max(tmax, __shfl_xor_sync(0xffffffffu, tmax, 16));
    if (a.tile_max != nullptr && lane == 0)
      a.tile_max[((size_t)b * a.hkv + h) * a.max_tiles + tile] = tmax;
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
}

size_t score_smem_bytes(int batch) {
  return 1024 + kScoreStages * kStageBytes + 2 * kScoreStages * sizeof(uint64_t) +
         (batch + 1) * sizeof(int);
}

}  // namespace

int score_max_tiles(const Shape& s) { return (s.max_pages + kTileBlocks - 1) / kTileBlocks; }

cudaError_t launch_score_blocks(const Shape& s, const CUtensorMap& kq_map, const void* q,
                                const float* k_scale, const int32_t* page_table,
                                const int32_t* seq_lens, int32_t* block_max, int32_t* tile_max,
                                int* err, int num_sms, cudaStream_t st) {
  if (s.batch > kMaxBatch) return cudaErrorInvalidValue;
  ScoreArgs a;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.k_scale = k_scale;
  a.page_table = page_table;
  a.seq_lens = seq_lens;
  a.block_max = block_max;
  a.tile_max = tile_max;
  a.err = err;
  a.batch = s.batch;
  a.hkv = s.hkv;
  a.max_pages = s.max_pages;
  a.max_tiles = score_max_tiles(s);
  a.num_pages = s.num_pages;
  a.sink = s.sink;
  a.window = s.window;
  const size_t smem = score_smem_bytes(s.batch);
  // upper bound of the tile count; the kernel splits the true count evenly
  const long long tiles_max =
      (long long)s.batch * s.hkv * ((s.max_pages + kTileBlocks - 1) / kTileBlocks + 1);
  const int grid = (int)std::min<long long>(tiles_max, 2LL * num_sms);
  const bool kb4 = s.key_bits == 4;
  auto go = [&](auto kernel) {
    cudaError_t e = set_kernel_smem(kernel, smem);
    if (e != cudaSuccess) return e;
    return launch_kernel(kernel, dim3(grid), dim3(kScoreThreads), smem, st, true, kq_map, a);
  };
  cudaError_t e;
  switch (s.group) {
    case 1: e = kb4 ? go(score_blocks_kernel<1, true>) : go(score_blocks_kernel<1, false>); break;
    case 2: e = kb4 ? go(score_blocks_kernel<2, true>) : go(score_blocks_kernel<2, false>); break;
    case 4: e = kb4 ? go(score_blocks_kernel<4, true>) : go(score_blocks_kernel<4, false>); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace hsa
