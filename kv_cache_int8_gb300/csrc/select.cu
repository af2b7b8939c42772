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
// prune_kernel: one CTA per (sequence, kv head). Chunk scores (max of their blocks'
// maxima) are staged in shared memory; the K-th largest value is found by histogram
// refinement over the value range (2048 bins per pass), ties at the threshold are broken
// toward lower indices with a block-wide prefix count, and the kept indices are written
// in ascending order. Module 2 repeats this on the blocks of the kept chunks.
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
  int* err;
  int batch, hkv, max_pages, num_pages, sink, window;
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
    if (lane != 0) return;
    SeqRange sr = seq_range(a, b);
    bool ok = true;
    for (int j = 0; f0 + j < f1; j++) {
      const int f = f0 + j;
      const int s = j % kScoreStages;
      if (j >= kScoreStages && !mbar_wait(&empty[s], ((j / kScoreStages) - 1) & 1)) {
        set_error(a.err, kDevErrTimeout);
        ok = false;
        break;
      }
      while (prefix[b + 1] <= f) {
        b++;
        sr = seq_range(a, b);
      }
      const int r = f - prefix[b];
      const int h = r / sr.ntile;
      const int tile = sr.tile_lo + r % sr.ntile;
      int rows[kTileBlocks];
      uint32_t bytes = 0;
#pragma unroll
      for (int i = 0; i < kTileBlocks; i++) {
        const int k = tile * kTileBlocks + i;
        rows[i] = -1;
        if (k < sr.k_lo || k >= sr.k_hi) continue;
        const int page = a.page_table[(size_t)b * a.max_pages + k];
        if (page < 0 || page >= a.num_pages) {
          set_error(a.err, kDevErrCheck);
          continue;
        }
        rows[i] = (page * a.hkv + h) * kPage;
        bytes += kBlockBytesI8;
      }
      mbar_arrive_expect_tx(&full[s], bytes);
#pragma unroll
      for (int i = 0; i < kTileBlocks; i++)
        if (rows[i] >= 0)
          tma_load_2d(ring + s * kStageBytes + i * kBlockBytesI8, &kq_map, 0, rows[i], &full[s]);
    }
    if (!ok) {
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
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
}

size_t score_smem_bytes(int batch) {
  return 1024 + kScoreStages * kStageBytes + 2 * kScoreStages * sizeof(uint64_t) +
         (batch + 1) * sizeof(int);
}

// -------------------------------------------------------------------- prune

constexpr int kPruneThreads = 512;
constexpr int kPruneWarps = kPruneThreads / 32;
constexpr int kBins = 2048;
constexpr int kBinsPerThread = kBins / kPruneThreads;
constexpr int kMaxChunks = 53248;
constexpr size_t kSmemLimit = 227 * 1024;

struct PruneArgs {
  const int32_t* seq_lens;
  const int32_t* block_max;
  int32_t* chunk_idx;
  int32_t* n_chunks;
  int32_t* block_idx;
  int32_t* n_blocks;
  int* err;
  int hkv, max_pages, chunk_blocks, k1, k2, sink, window, vals_cap, cand_cap;
};

// Exclusive prefix sum over the CTA; `total` receives the sum. All threads must call.
__device__ int block_exclusive_scan(int v, int* scratch, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kPruneWarps ? scratch[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w += y;
    }
    if (lane < kPruneWarps) scratch[lane] = w;
  }
  __syncthreads();
  const int base = warp > 0 ? scratch[warp - 1] : 0;
  total = scratch[kPruneWarps - 1];
  __syncthreads();
  return base + x - v;
}

__device__ int block_min_max(int v, bool want_max, int* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const int y = __shfl_xor_sync(0xffffffffu, v, off);
    v = want_max ? max(v, y) : min(v, y);
  }
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  int r = scratch[0];
  for (int w = 1; w < kPruneWarps; w++) r = want_max ? max(r, scratch[w]) : min(r, scratch[w]);
  __syncthreads();
  return r;
}

// Contiguous ownership: thread t owns [t m, min((t+1) m, n)).
__device__ __forceinline__ void own_range(int n, int& i0, int& i1) {
  const int m = (n + kPruneThreads - 1) / kPruneThreads;
  i0 = min(n, (int)threadIdx.x * m);
  i1 = min(n, i0 + m);
}

// Finds T, the K-th largest of vals[0..n) (0 < K < n), and need_eq = how many of the
// values equal to T are kept (the lowest-index ones): K - #(values > T).
__device__ void kth_largest(const int* vals, int n, int K, int* hist, int* scratch, int& T,
                            int& need_eq) {
  int i0, i1;
  own_range(n, i0, i1);
  int lmin = INT_MAX, lmax = INT_MIN;
  for (int i = i0; i < i1; i++) {
    lmin = min(lmin, vals[i]);
    lmax = max(lmax, vals[i]);
  }
  long long lo = block_min_max(lmin, false, scratch);
  long long hi = block_min_max(lmax, true, scratch);
  int above = 0;  // values known to lie above the current range
  while (lo < hi) {
    const unsigned long long range = (unsigned long long)(hi - lo);
    int bits = 64 - __clzll(range);
    const int shift = max(0, bits - 11);
    const int nb = (int)(range >> shift) + 1;
    for (int i = threadIdx.x; i < nb; i += kPruneThreads) hist[i] = 0;
    __syncthreads();
    for (int i = i0; i < i1; i++) {
      const long long v = vals[i];
      if (v >= lo && v <= hi) atomicAdd(&hist[(int)((unsigned long long)(v - lo) >> shift)], 1);
    }
    __syncthreads();
    int local = 0;
#pragma unroll
    for (int q = 0; q < kBinsPerThread; q++) {
      const int bin = threadIdx.x * kBinsPerThread + q;
      if (bin < nb) local += hist[bin];
    }
    int tot;
    const int before = block_exclusive_scan(local, scratch, tot);
    int higher = above + (tot - before - local);  // values in bins of later threads
    for (int q = kBinsPerThread - 1; q >= 0; q--) {
      const int bin = threadIdx.x * kBinsPerThread + q;
      if (bin >= nb) continue;
      const int c = hist[bin];
      if (higher < K && higher + c >= K) {
        scratch[40] = bin;
        scratch[41] = higher;
      }
      higher += c;
    }
    __syncthreads();
    const int bin = scratch[40];
    above = scratch[41];
    lo = lo + ((long long)bin << shift);
    hi = min(hi, lo + ((1LL << shift) - 1));
    __syncthreads();
  }
  T = (int)lo;
  need_eq = K - above;
}

// Writes, in ascending index order, every i with vals[i] > T plus the first need_eq
// indices with vals[i] == T, calling emit(position, i). Returns the number kept.
template <typename Emit>
__device__ int collect(const int* vals, int n, int T, int need_eq, int* scratch, Emit emit) {
  int i0, i1;
  own_range(n, i0, i1);
  int n_eq = 0;
  for (int i = i0; i < i1; i++) n_eq += vals[i] == T;
  int tot;
  int eq_rank = block_exclusive_scan(n_eq, scratch, tot);
  const int eq_rank0 = eq_rank;
  int n_take = 0;
  for (int i = i0; i < i1; i++) {
    const int v = vals[i];
    if (v > T || (v == T && eq_rank++ < need_eq)) n_take++;
  }
  int kept;
  int pos = block_exclusive_scan(n_take, scratch, kept);
  eq_rank = eq_rank0;
  for (int i = i0; i < i1; i++) {
    const int v = vals[i];
    if (v > T || (v == T && eq_rank++ < need_eq)) emit(pos++, i);
  }
  __syncthreads();
  return kept;
}

__global__ void __launch_bounds__(kPruneThreads) prune_kernel(const PruneArgs a) {
  extern __shared__ int psmem[];
  int* vals = psmem;                     // vals_cap
  int* cand = vals + a.vals_cap;         // cand_cap block ids of module 2
  int* kept_chunks = cand + a.cand_cap;  // k1
  int* hist = kept_chunks + a.k1;        // kBins
  int* scratch = hist + kBins;           // 64

  const int h = blockIdx.x, b = blockIdx.y;
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
  for (int i = threadIdx.x; i < n1; i += kPruneThreads) {
    const int c = c_lo + i;
    const int kb0 = max(c * P, k_lo), kb1 = min(c * P + P, k_hi);
    int m = INT_MIN;
    for (int k = kb0; k < kb1; k++) m = max(m, bm[k]);
    vals[i] = m;
  }
  __syncthreads();
  const int keep1 = min(a.k1, n1);
  int T = INT_MIN, need_eq = n1;
  if (keep1 < n1 && keep1 > 0) kth_largest(vals, n1, keep1, hist, scratch, T, need_eq);
  int got1 = 0;
  if (keep1 > 0) {
    got1 = collect(vals, n1, T, need_eq, scratch, [&](int pos, int i) {
      kept_chunks[pos] = c_lo + i;
      if (a.chunk_idx) a.chunk_idx[bh * a.k1 + pos] = c_lo + i;
    });
  }
  if (a.chunk_idx)
    for (int i = got1 + threadIdx.x; i < a.k1; i += kPruneThreads) a.chunk_idx[bh * a.k1 + i] = -1;
  if (a.n_chunks && threadIdx.x == 0) a.n_chunks[bh] = got1;
  __syncthreads();

  // ---- module 2: the kept chunks' blocks, top-K2
  int i0, i1;
  own_range(got1, i0, i1);
  int mine = 0;
  for (int i = i0; i < i1; i++) {
    const int c = kept_chunks[i];
    mine += min(c * P + P, k_hi) - max(c * P, k_lo);
  }
  int n2;
  int off = block_exclusive_scan(mine, scratch, n2);
  for (int i = i0; i < i1; i++) {
    const int c = kept_chunks[i];
    for (int k = max(c * P, k_lo); k < min(c * P + P, k_hi); k++) {
      cand[off] = k;
      vals[off] = bm[k];
      off++;
    }
  }
  __syncthreads();
  const int keep2 = min(a.k2, n2);
  T = INT_MIN;
  need_eq = n2;
  if (keep2 < n2 && keep2 > 0) kth_largest(vals, n2, keep2, hist, scratch, T, need_eq);
  int got2 = 0;
  if (keep2 > 0) {
    got2 = collect(vals, n2, T, need_eq, scratch, [&](int pos, int i) {
      a.block_idx[bh * a.k2 + pos] = cand[i];
    });
  }
  for (int i = got2 + threadIdx.x; i < a.k2; i += kPruneThreads) a.block_idx[bh * a.k2 + i] = -1;
  if (threadIdx.x == 0) a.n_blocks[bh] = got2;
}

int prune_caps(const Shape& s, int& vals_cap, int& cand_cap) {
  const int P = s.chunk / kPage;
  const long long n1max = ((long long)s.max_pages + P - 1) / P;
  const long long keep1 = std::min<long long>(s.k1, n1max);
  const long long n2max = std::min<long long>(keep1 * P, s.max_pages);
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
  return sizeof(int) * ((size_t)vals_cap + cand_cap + s.k1 + kBins + 64);
}

cudaError_t launch_score_blocks(const Shape& s, const CUtensorMap& kq_map, const void* q,
                                const float* k_scale, const int32_t* page_table,
                                const int32_t* seq_lens, int32_t* block_max, int* err,
                                int num_sms, cudaStream_t st) {
  if (s.batch > kMaxBatch) return cudaErrorInvalidValue;
  ScoreArgs a;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.k_scale = k_scale;
  a.page_table = page_table;
  a.seq_lens = seq_lens;
  a.block_max = block_max;
  a.err = err;
  a.batch = s.batch;
  a.hkv = s.hkv;
  a.max_pages = s.max_pages;
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
      e = cudaFuncSetAttribute(score_blocks_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem);
      if (e != cudaSuccess) return e;
      score_blocks_kernel<1><<<grid, kScoreThreads, smem, st>>>(kq_map, a);
      break;
    case 2:
      e = cudaFuncSetAttribute(score_blocks_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem);
      if (e != cudaSuccess) return e;
      score_blocks_kernel<2><<<grid, kScoreThreads, smem, st>>>(kq_map, a);
      break;
    case 4:
      e = cudaFuncSetAttribute(score_blocks_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem);
      if (e != cudaSuccess) return e;
      score_blocks_kernel<4><<<grid, kScoreThreads, smem, st>>>(kq_map, a);
      break;
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_prune(const Shape& s, const int32_t* seq_lens, const int32_t* block_max,
                         int32_t* chunk_idx, int32_t* n_chunks, int32_t* block_idx,
                         int32_t* n_blocks, int* err, cudaStream_t st) {
  PruneArgs a;
  if (prune_caps(s, a.vals_cap, a.cand_cap) != 0) return cudaErrorInvalidValue;
  const size_t smem = prune_smem_bytes(s);
  if (smem > kSmemLimit) return cudaErrorInvalidValue;
  a.seq_lens = seq_lens;
  a.block_max = block_max;
  a.chunk_idx = chunk_idx;
  a.n_chunks = n_chunks;
  a.block_idx = block_idx;
  a.n_blocks = n_blocks;
  a.err = err;
  a.hkv = s.hkv;
  a.max_pages = s.max_pages;
  a.chunk_blocks = s.chunk / kPage;
  a.k1 = s.k1;
  a.k2 = s.k2;
  a.sink = s.sink;
  a.window = s.window;
  cudaError_t e =
      cudaFuncSetAttribute(prune_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  prune_kernel<<<dim3(s.hkv, s.batch), kPruneThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace hsa
