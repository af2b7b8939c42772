// select.cu -- global int8 scoring of every candidate token and the two pruning modules.
//
// Sources: "HCAttention: Extreme KV cache compression via heterogeneous attention computing
// for LLMs", abstract and contribution list (global approximate attention scoring over the
// GPU-resident quantised keys); InfiniteHiP article (163.com), section "实现 7.24 倍的端到端
// 解码加速" (a pruning module cuts the context into fixed-length chunks, finds each chunk's
// best token in parallel and passes the top-K chunks on; stacked modules refine a
// block-sparse mask); "KV Cache 与长上下文推理", section "MQA 与 GQA" (G query heads share
// one kv head).
//
// score_blocks_kernel (the HBM-bound scan): a persistent grid walks the flattened list of
// 64-token tiles (sequence, kv head, tile). One producer lane per CTA streams each tile's
// four 2 KiB (page, head) blocks into a shared-memory ring with TMA tensor copies
// (128-byte swizzle, so the token-per-lane reads below are bank-conflict free) and
// mbarrier transaction counts. Consumer warps own fixed ring slots; lane = token, the
// G x 32 packed int8 query words sit in registers, dp4a gives the G exact int32 dot
// products, their max is the token score and a 16-lane max gives the block maximum.
//
// prune_kernel: one CTA per (sequence, kv head). Chunk scores (the scorer's per-tile maxima
// for 64-token chunks, else the max of their blocks' maxima) are staged in shared memory;
// the K-th largest value is found by radix selection on 8-bit digits of (value - min) with
// per-warp histograms; ties at the threshold are broken toward lower indices by ballots
// over warp-contiguous ranges, which also write the kept indices in ascending order.
// Module 2 repeats this on the blocks of the kept chunks.
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

template <int G>
__global__ void __launch_bounds__(kScoreThreads, 2)
    score_blocks_kernel(const __grid_constant__ CUtensorMap kq_map, const ScoreArgs a) {
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
          rows[i] = (pg[i] * a.hkv + h) * kPage;
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
            for (int q = 0; q < kTileBlocks; q++) bytes += rr[q] >= 0 ? kBlockBytesI8 : 0;
            mbar_arrive_expect_tx(&full[s], bytes);
#pragma unroll
            for (int q = 0; q < kTileBlocks; q++)
              if (rr[q] >= 0)
                tma_load_2d_hint(ring + s * kStageBytes + q * kBlockBytesI8, &kq_map, 0, rr[q],
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

// -------------------------------------------------------------------- prune

#ifndef HSA_PRUNE_THREADS
#define HSA_PRUNE_THREADS 512
#endif
constexpr int kPruneThreads = HSA_PRUNE_THREADS;  // overridable at build time for tuning
constexpr int kPruneWarps = kPruneThreads / 32;
constexpr int kDigitBins = 256;
constexpr int kMaxChunks = 53248;
constexpr size_t kSmemLimit = 227 * 1024;

struct PruneArgs {
  const int32_t* seq_lens;
  const int32_t* block_max;
  const int32_t* tile_max;  // nullable; used when chunks are 64 tokens
  int max_tiles;
  int32_t* chunk_idx;
  int32_t* n_chunks;
  int32_t* block_idx;
  int32_t* n_blocks;
  const int32_t* page_table;  // with sel_pages: the page of every kept block is written too
  int32_t* sel_pages;         // nullable, [B][Hkv][K2] beside block_idx
  int* err;
  int hkv, max_pages, chunk_blocks, k1, k2, sink, window, vals_cap, cand_cap;
};

// Shared scratch of the selection: per-warp digit histograms and per-warp totals.
struct SelectScratch {
  unsigned hist[kPruneWarps][kDigitBins];
  int w_a[kPruneWarps], w_b[kPruneWarps];
  int red[kPruneWarps];
  int decided[4];
};

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Min of the entries that are not INT_MIN (placeholders), or INT_MAX if none.
__device__ int block_min_valid(const int* vals, int n, SelectScratch& ss) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int m = INT_MAX;
  for (int i = threadIdx.x; i < n; i += kPruneThreads)
    if (vals[i] != INT_MIN) m = min(m, vals[i]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = min(m, __shfl_xor_sync(0xffffffffu, m, off));
  if (lane == 0) ss.red[warp] = m;
  __syncthreads();
  int r = ss.red[0];
#pragma unroll
  for (int w = 1; w < kPruneWarps; w++) r = min(r, ss.red[w]);
  __syncthreads();
  return r;
}

// Order-preserving key of a value relative to the smallest valid value; placeholders get 0.
__device__ __forceinline__ unsigned rel_key(int v, int vmin) {
  return v == INT_MIN ? 0u : (unsigned)((long long)v - vmin) + 1u;
}

// The K-th largest value T of vals[0..n) (0 < K < number of valid entries) by radix
// selection on 8-bit digits of the keys, from the highest digit in which they differ;
// need_eq = K - #(values > T), i.e. how many of the entries equal to T are kept (the
// lowest-index ones). Two CTA barriers per digit.
__device__ void kth_largest(const int* vals, int n, int K, SelectScratch& ss, int& T,
                            int& need_eq) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int vmin = block_min_valid(vals, n, ss);
  unsigned kmax = 0;
  for (int i = threadIdx.x; i < n; i += kPruneThreads) kmax = max(kmax, rel_key(vals[i], vmin));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, off));
  if (lane == 0) ss.red[warp] = (int)kmax;
  __syncthreads();
  kmax = 0;
#pragma unroll
  for (int w = 0; w < kPruneWarps; w++) kmax = max(kmax, (unsigned)ss.red[w]);
  int shift = kmax > 0 ? ((31 - __clz(kmax)) / 8) * 8 : 0;
  unsigned prefix = 0;  // decided high bits of T's key
  int above = 0;        // entries known to lie above T
  for (;;) {
    unsigned* hist = ss.hist[warp];
#pragma unroll
    for (int q = 0; q < kDigitBins / 32; q++) hist[lane * (kDigitBins / 32) + q] = 0;
    __syncwarp();
    const int hi_shift = shift + 8;
    for (int i = threadIdx.x; i < n; i += kPruneThreads) {
      const unsigned key = rel_key(vals[i], vmin);
      const bool match = hi_shift >= 32 || (key >> hi_shift) == (prefix >> hi_shift);
      if (match) atomicAdd(&hist[(key >> shift) & 0xFF], 1u);
    }
    __syncthreads();
    if (warp == 0) {
      // lane owns digits [8 lane, 8 lane + 8); counts summed over the warps
      unsigned c[8];
      unsigned mine = 0;
#pragma unroll
      for (int q = 0; q < 8; q++) {
        unsigned t = 0;
#pragma unroll
        for (int w = 0; w < kPruneWarps; w++) t += ss.hist[w][lane * 8 + q];
        c[q] = t;
        mine += t;
      }
      // entries in the digits of higher lanes
      unsigned incl = mine;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const unsigned y = __shfl_down_sync(0xffffffffu, incl, off);
        if (lane + off < 32) incl += y;
      }
      unsigned higher = above + (incl - mine);
#pragma unroll
      for (int q = 7; q >= 0; q--) {
        if (higher < (unsigned)K && higher + c[q] >= (unsigned)K) {
          ss.decided[0] = lane * 8 + q;
          ss.decided[1] = (int)higher;
        }
        higher += c[q];
      }
    }
    __syncthreads();
    prefix |= (unsigned)ss.decided[0] << shift;
    above = ss.decided[1];
    if (shift == 0) break;
    shift -= 8;
  }
  T = (int)((long long)vmin + (long long)prefix - 1);
  need_eq = K - above;
  __syncthreads();
}

// Emits, in ascending index order, every i with vals[i] > T plus the first need_eq indices
// with vals[i] == T, calling emit(position, i); returns how many. Warp w owns a contiguous
// range, scanned 32 entries at a time with ballots (conflict-free, one CTA barrier).
template <typename Emit>
__device__ int collect(const int* vals, int n, int T, int need_eq, SelectScratch& ss, Emit emit) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int per = ((n + kPruneWarps * 32 - 1) / (kPruneWarps * 32)) * 32;
  const int w0 = min(n, warp * per), w1 = min(n, w0 + per);
  int n_gt = 0, n_eq = 0;
  for (int i = w0 + lane; i < w1; i += 32) {
    n_gt += vals[i] > T;
    n_eq += vals[i] == T;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    n_gt += __shfl_xor_sync(0xffffffffu, n_gt, off);
    n_eq += __shfl_xor_sync(0xffffffffu, n_eq, off);
  }
  if (lane == 0) {
    ss.w_a[warp] = n_gt;
    ss.w_b[warp] = n_eq;
  }
  __syncthreads();
  // per warp: entries kept = all above T plus the ties still allowed after the earlier warps
  int eq_acc = 0, pos = 0, total = 0, eq_base = 0;
  for (int w = 0; w < kPruneWarps; w++) {
    const int kept_w = ss.w_a[w] + min(max(need_eq - eq_acc, 0), ss.w_b[w]);
    if (w == warp) {
      pos = total;
      eq_base = eq_acc;
    }
    total += kept_w;
    eq_acc += ss.w_b[w];
  }
  const unsigned lt = lanemask_lt();
  for (int i0 = w0; i0 < w1; i0 += 32) {
    const int i = i0 + lane;
    const int v = i < w1 ? vals[i] : INT_MIN;
    const bool gt = i < w1 && v > T, eq = i < w1 && v == T;
    const unsigned eqm = __ballot_sync(0xffffffffu, eq);
    const bool take = gt || (eq && eq_base + __popc(eqm & lt) < need_eq);
    const unsigned tm = __ballot_sync(0xffffffffu, take);
    if (take) emit(pos + __popc(tm & lt), i);
    eq_base += __popc(eqm);
    pos += __popc(tm);
  }
  __syncthreads();
  return total;
}

template <int UNROLL>
__device__ __forceinline__ void gather_strided(int* dst, const int32_t* __restrict__ src, int n) {
  for (int i0 = threadIdx.x; i0 < n; i0 += UNROLL * kPruneThreads) {
    int v[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; u++) {
      const int i = i0 + u * kPruneThreads;
      v[u] = i < n ? __ldg(src + i) : 0;
    }
#pragma unroll
    for (int u = 0; u < UNROLL; u++) {
      const int i = i0 + u * kPruneThreads;
      if (i < n) dst[i] = v[u];
    }
  }
}

// At most 40 registers a thread (three 512-thread CTAs' worth per SM): a prune CTA and a
// CTA of the sparse attend, which is launched while the prune runs, then fit on one SM
// together, and no attend CTA has to wait for the prune to leave its SM.
__global__ void __launch_bounds__(kPruneThreads, 1536 / kPruneThreads) prune_kernel(const PruneArgs a) {
  extern __shared__ __align__(16) int psmem[];
  SelectScratch& ss = *reinterpret_cast<SelectScratch*>(psmem);
  int* vals = psmem + sizeof(SelectScratch) / sizeof(int);  // vals_cap
  int* cand = vals + a.vals_cap;                            // cand_cap block ids of module 2
  int* kept_chunks = cand + a.cand_cap;                     // k1
  int* cand_page = kept_chunks + a.k1;                      // cand_cap pages (with sel_pages)

  const int h = blockIdx.x, b = blockIdx.y;
  grid_dep_wait();  // the scores come from the previous kernel
  grid_dep_launch();
  const int n = a.seq_lens[b];
  const int P = a.chunk_blocks;
  int lo = a.sink, hi = n - a.window;
  if (n < 0 || n > a.max_pages * kPage) {
    if (threadIdx.x == 0) set_error(a.err, kDevErrCheck);
    hi = lo;
  }
  int k_lo = 0, k_hi = 0, c_lo = 0, n1 = 0;
  if (hi > lo) {
    k_lo = lo / kPage;
    k_hi = (hi + kPage - 1) / kPage;
    c_lo = k_lo / P;
    n1 = (k_hi + P - 1) / P - c_lo;
  }
  const int32_t* bm = a.block_max + ((size_t)b * a.hkv + h) * a.max_pages;
  const size_t bh = (size_t)b * a.hkv + h;

  // ---- module 1: chunk scores, top-K1
  if (a.tile_max != nullptr && P == 4) {
    gather_strided<8>(vals, a.tile_max + bh * a.max_tiles + c_lo, n1);
  } else {
    for (int i = threadIdx.x; i < n1; i += kPruneThreads) vals[i] = INT_MIN;
    __syncthreads();
    // every candidate block once (independent, coalesced loads); max into its chunk
#pragma unroll 4
    for (int k = k_lo + threadIdx.x; k < k_hi; k += kPruneThreads)
      atomicMax(&vals[k / P - c_lo], __ldg(bm + k));
  }
  __syncthreads();
  const int keep1 = min(a.k1, n1);
  int T = INT_MIN, need_eq = 0;
  if (keep1 < n1 && keep1 > 0) kth_largest(vals, n1, keep1, ss, T, need_eq);
  int got1 = 0;
  if (keep1 > 0) {
    got1 = collect(vals, n1, T, need_eq, ss, [&](int pos, int i) {
      kept_chunks[pos] = c_lo + i;
      if (a.chunk_idx) a.chunk_idx[bh * a.k1 + pos] = c_lo + i;
    });
  }
  if (a.chunk_idx)
    for (int i = got1 + threadIdx.x; i < a.k1; i += kPruneThreads) a.chunk_idx[bh * a.k1 + i] = -1;
  if (a.n_chunks && threadIdx.x == 0) a.n_chunks[bh] = got1;
  __syncthreads();

  // ---- module 2: the kept chunks' blocks (P per chunk, ascending; blocks outside the
  // candidate region are INT_MIN placeholders that are never kept), top-K2
  const int n2 = got1 * P;
  // with sel_pages, each candidate's page id is loaded beside its block maximum (same round
  // trip), so the next kernel reads the pages of the kept blocks directly
  const int32_t* prow = a.sel_pages ? a.page_table + (size_t)b * a.max_pages : nullptr;
  int valid_local = 0;
  for (int x0 = threadIdx.x; x0 < n2; x0 += 4 * kPruneThreads) {
    int v[4], kk[4], pg[4];
#pragma unroll
    for (int u = 0; u < 4; u++) {
      const int x = x0 + u * kPruneThreads;
      kk[u] = x < n2 ? kept_chunks[x / P] * P + x % P : -1;
      const bool in = kk[u] >= k_lo && kk[u] < k_hi;
      v[u] = in ? __ldg(bm + kk[u]) : INT_MIN;
      pg[u] = (in && prow) ? __ldg(prow + kk[u]) : -1;
    }
#pragma unroll
    for (int u = 0; u < 4; u++) {
      const int x = x0 + u * kPruneThreads;
      if (x < n2) {
        cand[x] = kk[u];
        vals[x] = v[u];
        if (prow) cand_page[x] = pg[u];
        valid_local += v[u] != INT_MIN;
      }
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) valid_local += __shfl_xor_sync(0xffffffffu, valid_local, off);
  if ((threadIdx.x & 31) == 0) ss.red[threadIdx.x >> 5] = valid_local;
  __syncthreads();
  int n2_valid = 0;
#pragma unroll
  for (int w = 0; w < kPruneWarps; w++) n2_valid += ss.red[w];
  __syncthreads();
  const int keep2 = min(a.k2, n2_valid);
  T = INT_MIN;
  need_eq = 0;
  if (keep2 < n2_valid && keep2 > 0) kth_largest(vals, n2, keep2, ss, T, need_eq);
  int got2 = 0;
  if (keep2 > 0) {
    got2 = collect(vals, n2, T, need_eq, ss, [&](int pos, int i) {
      a.block_idx[bh * a.k2 + pos] = cand[i];
      if (prow) a.sel_pages[bh * a.k2 + pos] = cand_page[i];
    });
  }
  for (int i = got2 + threadIdx.x; i < a.k2; i += kPruneThreads) a.block_idx[bh * a.k2 + i] = -1;
  if (threadIdx.x == 0) a.n_blocks[bh] = got2;
}

int prune_caps(const Shape& s, int& vals_cap, int& cand_cap) {
  const int P = s.chunk / kPage;
  const long long n1max = ((long long)s.max_pages + P - 1) / P;
  const long long keep1 = std::min<long long>(s.k1, n1max);
  const long long n2max = keep1 * P;
  if (n1max > kMaxChunks) return -1;
  vals_cap = (int)std::max(n1max, n2max);
  cand_cap = (int)n2max;
  return 0;
}

}  // namespace

int prune_max_chunks() { return kMaxChunks; }

size_t prune_smem_bytes(const Shape& s) {
  int vals_cap, cand_cap;
  if (prune_caps(s, vals_cap, cand_cap) != 0) return ~size_t(0);
  return sizeof(SelectScratch) + sizeof(int) * ((size_t)vals_cap + 2 * (size_t)cand_cap + s.k1);
}

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
  cudaError_t e;
  switch (s.group) {
    case 1:
      e = set_kernel_smem(score_blocks_kernel<1>, smem);
      if (e != cudaSuccess) return e;
      e = launch_kernel(score_blocks_kernel<1>, dim3(grid), dim3(kScoreThreads), smem, st, true,
                        kq_map, a);
      if (e != cudaSuccess) return e;
      break;
    case 2:
      e = set_kernel_smem(score_blocks_kernel<2>, smem);
      if (e != cudaSuccess) return e;
      e = launch_kernel(score_blocks_kernel<2>, dim3(grid), dim3(kScoreThreads), smem, st, true,
                        kq_map, a);
      if (e != cudaSuccess) return e;
      break;
    case 4:
      e = set_kernel_smem(score_blocks_kernel<4>, smem);
      if (e != cudaSuccess) return e;
      e = launch_kernel(score_blocks_kernel<4>, dim3(grid), dim3(kScoreThreads), smem, st, true,
                        kq_map, a);
      if (e != cudaSuccess) return e;
      break;
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_prune(const Shape& s, const int32_t* seq_lens, const int32_t* block_max,
                         const int32_t* tile_max, int32_t* chunk_idx, int32_t* n_chunks,
                         int32_t* block_idx, int32_t* n_blocks, const int32_t* page_table,
                         int32_t* sel_pages, int* err, cudaStream_t st) {
  if (sel_pages != nullptr && page_table == nullptr) return cudaErrorInvalidValue;
  PruneArgs a;
  if (prune_caps(s, a.vals_cap, a.cand_cap) != 0) return cudaErrorInvalidValue;
  const size_t smem = prune_smem_bytes(s);
  if (smem > kSmemLimit) return cudaErrorInvalidValue;
  a.seq_lens = seq_lens;
  a.block_max = block_max;
  a.tile_max = tile_max;
  a.max_tiles = score_max_tiles(s);
  a.chunk_idx = chunk_idx;
  a.n_chunks = n_chunks;
  a.block_idx = block_idx;
  a.n_blocks = n_blocks;
  a.page_table = page_table;
  a.sel_pages = sel_pages;
  a.err = err;
  a.hkv = s.hkv;
  a.max_pages = s.max_pages;
  a.chunk_blocks = s.chunk / kPage;
  a.k1 = s.k1;
  a.k2 = s.k2;
  a.sink = s.sink;
  a.window = s.window;
  cudaError_t e = set_kernel_smem(prune_kernel, smem);
  if (e != cudaSuccess) return e;
  return launch_kernel(prune_kernel, dim3(s.hkv, s.batch), dim3(kPruneThreads), smem, st, true, a);
}

}  // namespace hsa
