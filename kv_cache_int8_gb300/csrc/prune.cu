// prune.cu -- the two pruning modules: top-K1 chunks, then top-K2 blocks of those chunks.
//
// Source: InfiniteHiP article (163.com), section "实现 7.24 倍的端到端解码加速" (a pruning
// module cuts the context into fixed-length chunks, finds each chunk's best token in
// parallel and passes the top-K chunks on; stacked modules refine a block-sparse mask).
//
// prune_kernel: one CTA per (sequence, kv head). Chunk scores (the scorer's per-tile maxima
// for 64-token chunks, else the max of their blocks' maxima) are staged in shared memory
// with bulk copies, and so are the whole row of block maxima and page ids when they fit;
// the K-th largest value is found by counting (select.cuh: a histogram of the values' top
// 11 bits above the row's minimum, usually one level); ties at the threshold are broken
// toward lower indices by ballots over warp-contiguous ranges, which also write the kept
// indices in ascending order. Module 2 repeats this on the blocks of the kept chunks.
#include <algorithm>
#include <climits>

#include "common.cuh"
#include "internal.h"
#include "select.cuh"

namespace hsa {
namespace {

// -------------------------------------------------------------------- prune

#ifndef HSA_PRUNE_THREADS
#define HSA_PRUNE_THREADS 512
#endif
constexpr int kPruneThreads = HSA_PRUNE_THREADS;  // overridable at build time for tuning
constexpr int kPruneWarps = kPruneThreads / 32;
constexpr int kPrunePeel = 8;  // module 2's threshold form: most candidates dropped one a round
// 1: without chunk outputs and with K1 >= K2, module 2 ranks only the kept chunks' blocks at
// or above module 1's threshold (see prune_kernel)
#ifndef HSA_PRUNE_THRESHOLD
#define HSA_PRUNE_THRESHOLD 1
#endif
#ifndef HSA_PRUNE_RANGE
#define HSA_PRUNE_RANGE 1
#endif
constexpr int kMaxChunks = 53248;
constexpr int kRowCap = 16384;  // block-maxima rows up to this many blocks are staged whole
constexpr size_t kSmemLimit = 227 * 1024;
static_assert(kPruneThreads >= kSelScan && kPruneThreads % 32 == 0, "selection threads");

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
  unsigned* row_range;        // nullable, [rows][4]: the scorer's range of the maxima
  int* err;
  int hkv, max_pages, chunk_blocks, k1, k2, sink, window;
  int k0, coarse_chunks;  // module 0: top-k0 coarse chunks of coarse_chunks chunks each
  int vals_cap, cand_cap, kept_cap, row_cap, prow_cap, sel_cap;  // shared-memory array sizes
  int n0_cap, k0_cap, c1_cap;                                     // module 0's (0 without it)
};

// Shared scratch of the selection.
struct PruneShared {
  SelectShared sel;  // histogram, per-warp scratch (select.cuh)
  uint64_t bar[2];   // staging copies: [0] module 1's, [1] the rest
  int wcnt[4][kPruneWarps];  // module 2's threshold form: blocks kept by each warp and pass
};

// Issue (thread 0) and tail of a planned row; returns where src[0] lands.
__device__ __forceinline__ int* stage(const StagedRow& r, uint64_t* bar) {
  if (threadIdx.x == 0) issue_row(r, bar);
  tail_row<kPruneThreads>(r);
  return r.dst();
}

// At most 64 registers a thread (two 512-thread CTAs' worth per SM).
//
// Shared memory: PruneShared, vals [vals_cap + 4], cand [cand_cap] (module 2's block ids),
// cand_page [cand_cap] (with
// sel_pages), kept [kept_cap], row [row_cap + 4] (the sequence's block maxima, staged whole
// when they fit), prow [prow_cap + 4] (its page ids, with sel_pages), sel_pos [sel_cap]
// (module 2's kept positions in cand).
__global__ void __launch_bounds__(kPruneThreads, 1024 / kPruneThreads) prune_kernel(const PruneArgs a) {
  extern __shared__ __align__(16) unsigned char psmem_raw[];
  PruneShared& ps = *reinterpret_cast<PruneShared*>(psmem_raw);
  int* arr = reinterpret_cast<int*>(psmem_raw + ((sizeof(PruneShared) + 15) / 16) * 16);
  int* vals_base = arr;                              // vals_cap + 4
  int* cand = vals_base + a.vals_cap + 4;            // cand_cap
  int* cand_page = cand + a.cand_cap;                // cand_cap
  int* kept_chunks = cand_page + a.cand_cap;         // kept_cap
  int* row_base = kept_chunks + a.kept_cap;          // row_cap + 4 (16-byte aligned)
  int* prow_base = row_base + (a.row_cap > 0 ? a.row_cap + 4 : 0);  // prow_cap + 4
  int* sel_pos = prow_base + (a.prow_cap > 0 ? a.prow_cap + 4 : 0);  // sel_cap
  int* vals0 = sel_pos + a.sel_cap;  // module 0 (k0 > 0): n0_cap coarse scores,
  int* kept0 = vals0 + a.n0_cap;     // k0_cap kept coarse chunks,
  int* vals1 = kept0 + a.k0_cap;     // c1_cap scores of their fine chunks
  int* cand1 = vals1 + a.c1_cap;     // and c1_cap fine chunk ids

  const int h = blockIdx.x, b = blockIdx.y;
  const int tid = threadIdx.x;
  if (tid == 0) {
    mbar_init(&ps.bar[0], 1);
    mbar_init(&ps.bar[1], 1);
    fence_barrier_init();
  }
  sel_init<kPruneThreads>(ps.sel);
  // the sequence length is an input of the step, not written by the previous kernel: it is
  // read before the wait
  const int n = a.seq_lens[b];
  grid_dep_wait();  // the scores come from the previous kernel
  grid_dep_launch();
  const int P = a.chunk_blocks;
  int lo = a.sink, hi = n - a.window;
  if (n < 0 || n > a.max_pages * kPage) {
    if (tid == 0) set_error(a.err, kDevErrCheck);
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
  // the scorer's range of the row's tile maxima (zero: not recorded); cleared once read
  uint4 rr = make_uint4(0u, 0u, 0u, 0u);
  if (a.row_range != nullptr) rr = __ldcg(reinterpret_cast<const uint4*>(a.row_range) + bh);
  __syncthreads();  // the barrier's initialisation is visible; every thread has read rr
  if (a.row_range != nullptr && tid == 0)
    *reinterpret_cast<uint4*>(a.row_range + bh * 4) = make_uint4(0u, 0u, 0u, 0u);
  // module 1's values lie in the range of the tile maxima (64-token chunks: they are the
  // tile maxima) or else in that of the block maxima (a chunk's score is its best block's)
  const bool c64 = a.chunk_blocks == 4;
  const unsigned r_hi = c64 ? rr.x : rr.z, r_lo = c64 ? rr.y : rr.w;
  const bool t_range = HSA_PRUNE_RANGE && r_hi != 0u && r_lo != 0u;
  const int t_max = (int)(r_hi ^ 0x80000000u), t_min = (int)(~r_lo ^ 0x80000000u);

  // ---- stage the scores: the 64-token tile maxima when the scorer wrote them (chunk c of 64
  // tokens == tile c) on barrier 0, the whole row of block maxima and of page ids when they
  // fit on barrier 1 (module 2 needs them only later); whatever is not staged is gathered
  // from global memory
  const bool use_tiles = a.tile_max != nullptr && P == 4;
  const bool use_row = a.row_cap > 0;
  const bool use_prow = a.prow_cap > 0 && a.sel_pages != nullptr;
  const int32_t* t_src = a.tile_max + bh * a.max_tiles + c_lo;
  const int32_t* p_src = a.page_table + (size_t)b * a.max_pages + k_lo;
  // each barrier's bytes are announced before its first copy is issued
  const uint32_t bytes0 = use_tiles ? plan_row(vals_base, t_src, n1).bytes() : 0u;
  const uint32_t bytes1 = (use_row ? plan_row(row_base, bm + k_lo, k_hi - k_lo).bytes() : 0u) +
                          (use_prow ? plan_row(prow_base, p_src, k_hi - k_lo).bytes() : 0u);
  if (tid == 0 && bytes0 > 0) mbar_arrive_expect_tx(&ps.bar[0], bytes0);
  if (tid == 0 && bytes1 > 0) mbar_arrive_expect_tx(&ps.bar[1], bytes1);
  int* vals = use_tiles ? stage(plan_row(vals_base, t_src, n1), &ps.bar[0]) : vals_base;
  const int* row =  // row[k - k_lo] = block maximum of block k
      use_row ? stage(plan_row(row_base, bm + k_lo, k_hi - k_lo), &ps.bar[1]) : nullptr;
  const int* prow_s =  // prow_s[k - k_lo] = page of block k
      use_prow ? stage(plan_row(prow_base, p_src, k_hi - k_lo), &ps.bar[1]) : nullptr;
  // module 1 reads the tiles, or the block row when it reduces chunks itself
  const bool need1_now = !use_tiles && use_row;
  bool ok1 = true;
  if (bytes0 > 0 && !mbar_wait(&ps.bar[0], 0)) ok1 = false;
  if (need1_now && bytes1 > 0 && !mbar_wait(&ps.bar[1], 0)) ok1 = false;
  if (!ok1) set_error(a.err, kDevErrTimeout);
  __syncthreads();  // the plain-load tails are visible
  if (!use_tiles && use_row) {
    for (int c = tid; c < n1; c += kPruneThreads) {
      const int k0 = max((c_lo + c) * P, k_lo), k1 = min((c_lo + c) * P + P, k_hi);
      int m = INT_MIN;
      for (int k = k0; k < k1; k++) m = max(m, row[k - k_lo]);
      vals[c] = m;
    }
    __syncthreads();
  } else if (!use_tiles) {
    for (int i = tid; i < n1; i += kPruneThreads) vals[i] = INT_MIN;
    __syncthreads();
    // every candidate block once (independent, coalesced loads); max into its chunk
#pragma unroll 4
    for (int k = k_lo + tid; k < k_hi; k += kPruneThreads)
      atomicMax(&vals[k / P - c_lo], __ldg(bm + k));
    __syncthreads();
  }

  int T = INT_MIN, need_eq = 0, eq_total = 0;
  int got1 = 0;
  if (a.k0 > 0) {
    // ---- module 0 (stacked in front): coarse chunks of R fine chunks, scored by the max of
    // their fine chunks' scores; top-K0, ascending
    const int R = a.coarse_chunks;
    const int g_lo = c_lo / R;
    const int n0 = n1 > 0 ? (c_lo + n1 - 1) / R - g_lo + 1 : 0;
    for (int j = tid; j < n0; j += kPruneThreads) {
      const int f0 = max((g_lo + j) * R, c_lo) - c_lo;
      const int f1 = min((g_lo + j) * R + R, c_lo + n1) - c_lo;
      int m = INT_MIN;
      for (int i = f0; i < f1; i++) m = max(m, vals[i]);
      vals0[j] = m;
    }
    __syncthreads();
    const int keep0 = min(a.k0, n0);
    if (keep0 < n0) {
      const int3 r = sel_kth_largest<kPruneThreads>(vals0, n0, keep0, ps.sel, false, 0, 0);
      T = r.x;
      need_eq = r.y;
      eq_total = r.z;
    }
    const int got0 =
        keep0 > 0
            ? sel_collect<kPruneThreads>(vals0, n0, T, need_eq, eq_total, ps.sel, kept0, g_lo)
            : 0;
    // ---- module 1 over the kept coarse chunks' fine chunks (ascending; those outside the
    // candidate region are placeholders), top-K1
    const int n1c = got0 * R;
    int valid = 0;
    for (int x = tid; x < n1c; x += kPruneThreads) {
      const int c = kept0[x / R] * R + x % R;
      const bool in = c >= c_lo && c < c_lo + n1;
      vals1[x] = in ? vals[c - c_lo] : INT_MIN;
      cand1[x] = c;
      valid += in;
    }
    const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) valid += __shfl_xor_sync(0xffffffffu, valid, off);
    if (lane == 0) ps.sel.wsum[warp] = valid;
    __syncthreads();
    int n1_valid = 0;
#pragma unroll
    for (int w = 0; w < kPruneWarps; w++) n1_valid += ps.sel.wsum[w];
    __syncthreads();
    const int keep1 = min(a.k1, n1_valid);
    T = INT_MIN;
    need_eq = 0;
    eq_total = 0;
    if (keep1 < n1_valid && keep1 > 0) {
      const int3 r = sel_kth_largest<kPruneThreads>(vals1, n1c, keep1, ps.sel, false, 0, 0);
      T = r.x;
      need_eq = r.y;
      eq_total = r.z;
    }
    if (keep1 > 0) {
      // positions in vals1
      got1 = sel_collect<kPruneThreads>(vals1, n1c, T, need_eq, eq_total, ps.sel, kept_chunks, 0);
      for (int i = tid; i < got1; i += kPruneThreads) kept_chunks[i] = cand1[kept_chunks[i]];
      __syncthreads();
    }
  } else {
    // ---- module 1: top-K1 chunks (within the recorded range when there is one)
    const int keep1 = min(a.k1, n1);
    if (keep1 < n1 && keep1 > 0) {
      const int3 r = sel_kth_largest<kPruneThreads>(vals, n1, keep1, ps.sel, t_range, t_min, t_max);
      T = r.x;
      need_eq = r.y;
      eq_total = r.z;
    }
    if (keep1 > 0)
      got1 = sel_collect<kPruneThreads>(vals, n1, T, need_eq, eq_total, ps.sel, kept_chunks, c_lo);
  }
  if (a.chunk_idx)
    for (int i = tid; i < a.k1; i += kPruneThreads)
      a.chunk_idx[bh * a.k1 + i] = i < got1 ? kept_chunks[i] : -1;
  if (a.n_chunks && tid == 0) a.n_chunks[bh] = got1;
  __syncthreads();

  // ---- module 2: the kept chunks' blocks (P per chunk, ascending; blocks outside the
  // candidate region are INT_MIN placeholders that are never kept), top-K2. With sel_pages,
  // each candidate's page id is loaded beside its block maximum, so the next kernel reads
  // the pages of the kept blocks directly.
  const int n2 = got1 * P;
  const int32_t* prow = a.sel_pages ? a.page_table + (size_t)b * a.max_pages : nullptr;
  if (!need1_now && bytes1 > 0 && !mbar_wait(&ps.bar[1], 0)) set_error(a.err, kDevErrTimeout);
  const int lane = tid & 31, warp = tid >> 5;
  // Threshold form (no chunk ids are output, K1 >= K2): module 1's threshold T, the K1-th
  // largest chunk score, is at most the K2-th largest, and the top K2 chunks each hold a block
  // equal to their score, so every kept block reaches T. Only the blocks >= T take part: laid
  // out in order (positions by ballots, one barrier), and when a few more than K2 of them
  // remain, the lowest ranked are taken one a round by warp 0.
  const bool thr = HSA_PRUNE_THRESHOLD && a.k0 == 0 && a.chunk_idx == nullptr &&
                   a.n_chunks == nullptr && a.k1 >= a.k2 && a.k2 > 0 &&
                   n2 <= 4 * kPruneThreads;
  int valid_local = 0, mn2 = INT_MAX, mx2 = INT_MIN;
  int n2c = n2;  // entries in vals / cand (/ cand_page)
  if (thr) {
    int v[4], kk[4], pg[4];
    unsigned bal[4];
#pragma unroll
    for (int u = 0; u < 4; u++) {
      const int x = tid + u * kPruneThreads;
      kk[u] = x < n2 ? kept_chunks[x / P] * P + x % P : -1;
      const bool in = kk[u] >= k_lo && kk[u] < k_hi;
      v[u] = in ? (use_row ? row[kk[u] - k_lo] : __ldg(bm + kk[u])) : INT_MIN;
      pg[u] = (in && prow) ? (prow_s ? prow_s[kk[u] - k_lo] : __ldg(prow + kk[u])) : -1;
    }
#pragma unroll
    for (int u = 0; u < 4; u++) {
      if (v[u] < T) v[u] = INT_MIN;
      bal[u] = __ballot_sync(0xffffffffu, v[u] != INT_MIN);
      if (lane == 0) ps.wcnt[u][warp] = __popc(bal[u]);
      if (v[u] != INT_MIN) {
        mn2 = min(mn2, v[u]);
        mx2 = max(mx2, v[u]);
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      mn2 = min(mn2, __shfl_xor_sync(0xffffffffu, mn2, off));
      mx2 = max(mx2, __shfl_xor_sync(0xffffffffu, mx2, off));
    }
    if (lane == 0) {
      ps.sel.mn[warp] = mn2;
      ps.sel.mx[warp] = mx2;
    }
    __syncthreads();  // (module 1's collect is done with vals: it ended on a barrier)
    // lane l of every warp reads the counts of warp l & 15 (passes 0-1 in lanes 0-15, 2-3
    // in lanes 16-31); warp sums give each pass's total and the warps before this one
    static_assert(kPruneWarps == 16, "two lanes a warp: 16 warps");
    const int cw = lane & 15, u0 = lane >> 4;
    const int c0 = ps.wcnt[2 * u0][cw], c1 = ps.wcnt[2 * u0 + 1][cw];
    mn2 = min(ps.sel.mn[cw], __shfl_xor_sync(0xffffffffu, ps.sel.mn[cw], 16));
    mx2 = max(ps.sel.mx[cw], __shfl_xor_sync(0xffffffffu, ps.sel.mx[cw], 16));
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) {
      mn2 = min(mn2, __shfl_xor_sync(0xffffffffu, mn2, off));
      mx2 = max(mx2, __shfl_xor_sync(0xffffffffu, mx2, off));
    }
    int tot[4], pre[4];
#pragma unroll
    for (int u = 0; u < 4; u++) {
      const int c = (u >> 1) == u0 ? ((u & 1) ? c1 : c0) : 0;
      tot[u] = __reduce_add_sync(0xffffffffu, c);
      pre[u] = __reduce_add_sync(0xffffffffu, cw < warp ? c : 0);
    }
    n2c = tot[0] + tot[1] + tot[2] + tot[3];
    const unsigned lt = (1u << lane) - 1u;
    int before_u = 0;
#pragma unroll
    for (int u = 0; u < 4; u++) {
      if (v[u] != INT_MIN) {
        const int pos = before_u + pre[u] + __popc(bal[u] & lt);
        vals[pos] = v[u];
        cand[pos] = kk[u];
        if (prow) cand_page[pos] = pg[u];
      }
      before_u += tot[u];
    }
    __syncthreads();
    const int drop = n2c - a.k2;
    if (drop <= kPrunePeel) {
      if (drop > 0 && warp == 0) sel_peel_lowest(vals, n2c, drop, ps.sel.cand_i);
      if (drop > 0) __syncthreads();
      const int got2 = min(a.k2, n2c);
      for (int i = tid; i < n2c; i += kPruneThreads) {
        int before = 0;
        bool dropped = false;
        for (int e = 0; e < drop; e++) {
          const int de = ps.sel.cand_i[e];
          before += de < i ? 1 : 0;
          dropped = dropped || de == i;
        }
        if (!dropped) {
          a.block_idx[bh * a.k2 + i - before] = cand[i];
          if (prow) a.sel_pages[bh * a.k2 + i - before] = cand_page[i];
        }
      }
      for (int i = got2 + tid; i < a.k2; i += kPruneThreads) a.block_idx[bh * a.k2 + i] = -1;
      if (tid == 0) a.n_blocks[bh] = got2;
      return;
    }
    valid_local = tid == 0 ? n2c : 0;  // the general selection over the n2c laid-out blocks
  } else {
    for (int x0 = tid; x0 < n2; x0 += 4 * kPruneThreads) {
      int v[4], kk[4], pg[4];
#pragma unroll
      for (int u = 0; u < 4; u++) {
        const int x = x0 + u * kPruneThreads;
        kk[u] = x < n2 ? kept_chunks[x / P] * P + x % P : -1;
        const bool in = kk[u] >= k_lo && kk[u] < k_hi;
        v[u] = in ? (use_row ? row[kk[u] - k_lo] : __ldg(bm + kk[u])) : INT_MIN;
        pg[u] = (in && prow) ? (prow_s ? prow_s[kk[u] - k_lo] : __ldg(prow + kk[u])) : -1;
      }
#pragma unroll
      for (int u = 0; u < 4; u++) {
        const int x = x0 + u * kPruneThreads;
        if (x < n2) {
          cand[x] = kk[u];
          vals[x] = v[u];
          if (prow) cand_page[x] = pg[u];
          if (v[u] != INT_MIN) {
            valid_local++;
            mn2 = min(mn2, v[u]);
            mx2 = max(mx2, v[u]);
          }
        }
      }
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    valid_local += __shfl_xor_sync(0xffffffffu, valid_local, off);
    mn2 = min(mn2, __shfl_xor_sync(0xffffffffu, mn2, off));
    mx2 = max(mx2, __shfl_xor_sync(0xffffffffu, mx2, off));
  }
  if (lane == 0) {
    ps.sel.wsum[warp] = valid_local;
    ps.sel.mn[warp] = mn2;
    ps.sel.mx[warp] = mx2;
  }
  __syncthreads();
  int n2_valid = 0;
#pragma unroll
  for (int w = 0; w < kPruneWarps; w++) {
    n2_valid += ps.sel.wsum[w];
    mn2 = min(mn2, ps.sel.mn[w]);
    mx2 = max(mx2, ps.sel.mx[w]);
  }
  __syncthreads();
  const int keep2 = min(a.k2, n2_valid);
  T = INT_MIN;
  need_eq = 0;
  eq_total = 0;
  if (keep2 < n2_valid && keep2 > 0) {
    const int3 r = sel_kth_largest<kPruneThreads>(vals, n2c, keep2, ps.sel, true, mn2, mx2);
    T = r.x;
    need_eq = r.y;
    eq_total = r.z;
  }
  int got2 = 0;
  if (keep2 > 0) {
    got2 = sel_collect<kPruneThreads>(vals, n2c, T, need_eq, eq_total, ps.sel, sel_pos, 0);
  }
  for (int i = tid; i < a.k2; i += kPruneThreads) {
    const int x = i < got2 ? sel_pos[i] : -1;
    a.block_idx[bh * a.k2 + i] = x >= 0 ? cand[x] : -1;
    if (prow && x >= 0) a.sel_pages[bh * a.k2 + i] = cand_page[x];
  }
  if (tid == 0) a.n_blocks[bh] = got2;
}

// stage_pages: also stage the page-table row (only with sel_pages and a 16-byte-aligned page
// table).
int prune_caps(const Shape& s, PruneArgs& a, bool stage_pages) {
  const int P = s.chunk / kPage;
  const long long n1max = ((long long)s.max_pages + P - 1) / P;
  const long long keep1 = std::min<long long>(s.k1, n1max);
  const long long n2max = keep1 * P;
  if (n1max > kMaxChunks) return -1;
  // every array a multiple of 4 ints, so that each one starts 16-byte aligned
  auto up4 = [](long long x) { return (int)((x + 3) / 4 * 4); };
  a.vals_cap = up4(std::max(n1max, n2max));
  a.cand_cap = up4(n2max);
  a.kept_cap = up4(std::max<long long>(keep1, 1));
  a.row_cap = s.max_pages <= kRowCap ? up4(s.max_pages) : 0;
  a.prow_cap = stage_pages ? a.row_cap : 0;
  a.sel_cap = up4(std::max<long long>(std::min<long long>(s.k2, n2max), 1));
  a.n0_cap = a.k0_cap = a.c1_cap = 0;
  if (s.k0 > 0) {
    const long long R = s.chunk0 / s.chunk;
    const long long n0max = (n1max + R - 1) / R + 1;
    const long long k0cap = std::min<long long>(s.k0, n0max);
    a.n0_cap = up4(n0max);
    a.k0_cap = up4(k0cap);
    a.c1_cap = up4(k0cap * R);
  }
  return 0;
}

size_t prune_smem(const PruneArgs& a) {
  return ((sizeof(PruneShared) + 15) / 16) * 16 +
         sizeof(int) * ((size_t)a.vals_cap + 4 + 2 * (size_t)a.cand_cap + a.kept_cap +
                        (a.row_cap > 0 ? a.row_cap + 4 : 0) +
                        (a.prow_cap > 0 ? a.prow_cap + 4 : 0) + a.sel_cap + a.n0_cap +
                        a.k0_cap + 2 * (size_t)a.c1_cap);
}


// ------------------------------------------------------- GPU block cache plan

// A device cache of (page, kv head) K/V blocks in front of K/V in host memory (InfiniteHiP
// article: the GPU keeps recently used blocks, least recently used first out, and the rest
// of the cache lives in host memory). One plan per attention call, in one CTA:
//  - the call's segments (sink pages, window pages, kept blocks of every (sequence, kv
//    head), in the attention's order) are looked up; hits are stamped with the call's
//    step number; the page that holds the sequence's last token is always copied again
//    (an append may have changed it) into the slot it has;
//  - the misses, in segment order, take the slots not used by this call with the oldest
//    stamps (ties: lower slot), found by the prune's selection over -stamp;
//  - every segment's slot goes to seg_slot, every slot to fill goes to the fill list.
struct CachePlanArgs {
  const int32_t* seq_lens;
  const int32_t* page_table;
  const int32_t* block_idx;  // [B][Hkv][k2] (k2 > 0)
  const int32_t* n_blocks;   // [B][Hkv]
  int32_t* header;           // [0]: step counter
  int32_t* slot_of;          // [num_pages * hkv]: slot + 1, 0 when absent
  int32_t* slot_key;         // [capacity]: page * hkv + head + 1, 0 when free
  int32_t* slot_stamp;       // [capacity]: last step that used the slot, 0 never
  const float* mass;         // nullable: [num_pages * hkv] cumulative attention mass; victims
                             // by least mass instead of least recent use
  int32_t* seg_slot;         // [B][Hkv][seg_stride]: slot of each segment, -1 empty
  int4* fill;                // [B * Hkv * seg_stride]: (slot, page, head) to copy in
  int32_t* n_fill;
  int* err;
  int batch, hkv, max_pages, num_pages, k2, sink, window, seg_stride, capacity;
};

struct CachePlanShared {
  SelectShared ps;
  int warp_cnt[kPruneWarps];  // per-warp counts of one 512-entry chunk
  int step, n_miss, n_refresh;
};

// Segment i of (b, h): block k, or -1 when empty (same order and clipping as the attention).
__device__ int cache_segment_block(const CachePlanArgs& a, int b, int h, int i, int n) {
  const int sink_end = min(a.sink, n);
  const int n_sink = (sink_end + kPage - 1) / kPage;
  const int cand_hi = n - a.window;
  const int n_sel_max = cand_hi > a.sink ? a.k2 : 0;
  const int w0 = max(n - a.window, sink_end);
  const int win_k0 = w0 / kPage;
  const int n_win = w0 < n ? (n + kPage - 1) / kPage - win_k0 : 0;
  if (i < n_sink) return i;
  if (i < n_sink + n_win) return win_k0 + (i - n_sink);
  const int r = i - n_sink - n_win;
  if (r >= n_sel_max) return -1;
  const int nsel = max(0, min(a.n_blocks[(size_t)b * a.hkv + h], n_sel_max));
  if (r >= nsel) return -1;
  const int k = a.block_idx[((size_t)b * a.hkv + h) * a.k2 + r];
  if (k < 0 || k >= (n + kPage - 1) / kPage) return -1;
  // a kept block is attended only inside the candidate region
  if (max(k * kPage, a.sink) >= min(k * kPage + kPage, cand_hi)) return -1;
  return k;
}

// A block can be two segments of one call: the sink's last page or the window's first page
// when either is partial, and a kept block (or the other of the two). Returns the index of
// the earlier segment of (b, h) holding block k of segment i, or -1: the later one takes the
// earlier one's slot and is neither looked up nor filled on its own.
__device__ int cache_segment_alias(const CachePlanArgs& a, int i, int n, int k) {
  const int sink_end = min(a.sink, n);
  const int n_sink = (sink_end + kPage - 1) / kPage;
  const int w0 = max(n - a.window, sink_end);
  const int n_win = w0 < n ? (n + kPage - 1) / kPage - w0 / kPage : 0;
  if (i < n_sink) return -1;
  if (n_sink > 0 && k == n_sink - 1) return n_sink - 1;
  if (i < n_sink + n_win) return -1;
  if (n_win > 0 && k == w0 / kPage) return n_sink;
  return -1;
}

__global__ void __launch_bounds__(kPruneThreads) cache_plan_kernel(const CachePlanArgs a) {
  extern __shared__ __align__(16) unsigned char csmem_raw[];
  CachePlanShared& cs = *reinterpret_cast<CachePlanShared*>(csmem_raw);
  int* vals = reinterpret_cast<int*>(csmem_raw + ((sizeof(CachePlanShared) + 15) / 16) * 16);
  int* miss_f = vals + a.capacity;              // [B * Hkv * seg_stride] segment of miss j
  int* victims = miss_f + a.batch * a.hkv * a.seg_stride;  // same size
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  sel_init<kPruneThreads>(cs.ps);
  grid_dep_wait();  // the selection and the cache state come from earlier kernels
  grid_dep_launch();
  if (tid == 0) {
    cs.step = a.header[0] + 1;
    a.header[0] = cs.step;
    cs.n_miss = 0;
    cs.n_refresh = 0;
  }
  __syncthreads();
  const int step = cs.step;

  // ---- lookups. Thread t takes the segments [t per, (t + 1) per) (per <= 64: the capacity,
  // at most 32768, holds every segment of a call), eight at a time with their dependent
  // loads (length, block id, page, slot) issued together; then one scan orders the misses.
  const int F = a.batch * a.hkv * a.seg_stride;
  const int per = (F + kPruneThreads - 1) / kPruneThreads;
  const int f_lo = min(F, tid * per), f_hi = min(F, f_lo + per);
  unsigned long long miss_mask = 0ull;
  int my_miss = 0;
  for (int fb = f_lo; fb < f_hi; fb += 8) {
    int k[8], page[8], slot[8], n[8];
#pragma unroll
    for (int u = 0; u < 8; u++) {
      const int f = fb + u;
      n[u] = f < f_hi ? a.seq_lens[(f / a.seg_stride) / a.hkv] : 0;
    }
    int alias[8];
#pragma unroll
    for (int u = 0; u < 8; u++) {
      const int f = fb + u;
      const int bh = f / a.seg_stride;
      if (n[u] < 0 || n[u] > a.max_pages * kPage) n[u] = 0;
      k[u] = (f < f_hi && n[u] > 0) ? cache_segment_block(a, bh / a.hkv, bh % a.hkv,
                                                          f % a.seg_stride, n[u])
                                    : -1;
      alias[u] = k[u] >= 0 ? cache_segment_alias(a, f % a.seg_stride, n[u], k[u]) : -1;
      if (alias[u] >= 0) k[u] = -1;  // resolved after the victims are placed
    }
#pragma unroll
    for (int u = 0; u < 8; u++) {
      const int b = ((fb + u) / a.seg_stride) / a.hkv;
      page[u] = k[u] >= 0 ? a.page_table[(size_t)b * a.max_pages + k[u]] : -1;
      if (k[u] >= 0 && (page[u] < 0 || page[u] >= a.num_pages)) {
        set_error(a.err, kDevErrCheck);
        k[u] = -1;
      }
    }
#pragma unroll
    for (int u = 0; u < 8; u++) {
      const int h = ((fb + u) / a.seg_stride) % a.hkv;
      slot[u] = k[u] >= 0 ? a.slot_of[page[u] * a.hkv + h] - 1 : -1;
    }
#pragma unroll
    for (int u = 0; u < 8; u++) {
      const int f = fb + u;
      if (f >= f_hi) continue;
      if (k[u] >= 0 && slot[u] >= 0) {
        a.slot_stamp[slot[u]] = step;
        if (k[u] == (n[u] - 1) / kPage) {  // the last token's page: copy it again
          const int j = atomicAdd(&cs.n_refresh, 1);
          a.fill[j] = make_int4(slot[u], page[u], (f / a.seg_stride) % a.hkv, 0);
        }
      } else if (k[u] >= 0) {
        miss_mask |= 1ull << (f - f_lo);
        my_miss++;
      }
      // misses are overwritten below; an alias holds -2 - (its segment's index)
      a.seg_slot[f] = k[u] >= 0 ? slot[u] : (alias[u] >= 0 ? -2 - alias[u] : -1);
    }
  }
  // exclusive scan of the per-thread miss counts, then each thread lists its misses in order
  int incl = my_miss;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  if (lane == 31) cs.warp_cnt[warp] = incl;
  __syncthreads();
  int base = incl - my_miss;
  for (int w = 0; w < warp; w++) base += cs.warp_cnt[w];
  if (tid == kPruneThreads - 1) cs.n_miss = base + my_miss;
  for (int o = 0; miss_mask != 0ull; o++) {
    const int bit = __ffsll((long long)miss_mask) - 1;
    miss_mask &= miss_mask - 1;
    miss_f[base + o] = f_lo + bit;
  }
  __syncthreads();
  const int M = cs.n_miss, R = cs.n_refresh;

  // ---- victims: the M slots not used by this call with the oldest stamps (lower slot
  // first), ascending by slot; the fill list holds the refreshes, then the misses. With the
  // mass policy: the free slots, then the least cumulative attention mass (the masses are
  // non-negative, so their fp32 bits order them; a free slot ranks above every block).
  int got = 0;
  if (M > 0) {
    int valid = 0;
    for (int s = tid; s < a.capacity; s += kPruneThreads) {
      const int st = a.slot_stamp[s];
      int v = -st;
      if (a.mass) {
        const int key = a.slot_key[s] - 1;
        const float w = key >= 0 ? a.mass[key] : 0.0f;
        v = key < 0 ? 1 : -(w > 0.0f ? min(__float_as_int(w), 0x7F800000) : 0);
      }
      vals[s] = st < step ? v : INT_MIN;
      valid += st < step;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) valid += __shfl_xor_sync(0xffffffffu, valid, off);
    if (lane == 0) cs.ps.wsum[warp] = valid;
    __syncthreads();
    int n_valid = 0;
    for (int w = 0; w < kPruneWarps; w++) n_valid += cs.ps.wsum[w];
    __syncthreads();
    if (n_valid < M) {
      if (tid == 0) set_error(a.err, kDevErrCheck);  // capacity below the call's working set
    } else {
      int T = INT_MIN, need_eq = 0, eq_total = 0;
      if (M < n_valid) {
        const int3 r = sel_kth_largest<kPruneThreads>(vals, a.capacity, M, cs.ps, false, 0, 0);
        T = r.x;
        need_eq = r.y;
        eq_total = r.z;
      }
      got = sel_collect<kPruneThreads>(vals, a.capacity, T, need_eq, eq_total, cs.ps, victims, 0);
    }
  }
  // evict the victims' old keys first (none of them is looked up by this call)
  for (int j = tid; j < got; j += kPruneThreads) {
    const int old = a.slot_key[victims[j]] - 1;
    if (old >= 0) a.slot_of[old] = 0;
  }
  __syncthreads();
  for (int j = tid; j < got; j += kPruneThreads) {
    const int v = victims[j], f = miss_f[j];
    const int bh = f / a.seg_stride, i = f % a.seg_stride;
    const int b = bh / a.hkv, h = bh % a.hkv;
    const int k = cache_segment_block(a, b, h, i, a.seq_lens[b]);
    const int page = a.page_table[(size_t)b * a.max_pages + k];
    const int key = page * a.hkv + h;
    a.slot_of[key] = v + 1;
    a.slot_key[v] = key + 1;
    a.slot_stamp[v] = step;
    a.seg_slot[f] = v;
    a.fill[R + j] = make_int4(v, page, h, 0);
  }
  __syncthreads();
  // every alias takes the slot of the segment it repeats (a hit's, or a miss's just placed)
  for (int f = f_lo; f < f_hi; f++) {
    const int sv = a.seg_slot[f];
    if (sv <= -2) a.seg_slot[f] = a.seg_slot[(f / a.seg_stride) * a.seg_stride + (-2 - sv)];
  }
  // two segments of one call on the same (page, head) otherwise (pages shared between
  // sequences) are not supported: reported through the error word
  for (int j = tid; j < got; j += kPruneThreads) {
    const int v = victims[j];
    if (a.slot_of[a.slot_key[v] - 1] != v + 1) set_error(a.err, kDevErrCheck);
  }
  if (tid == 0) *a.n_fill = R + got;
}

int cache_plan_seg_stride(const Shape& s) {
  return (s.sink + kPage - 1) / kPage + (s.window + kPage - 1) / kPage + 1 + s.k2;
}

size_t cache_plan_smem(const Shape& s, int capacity) {
  const size_t F = (size_t)s.batch * s.hkv * cache_plan_seg_stride(s);
  return ((sizeof(CachePlanShared) + 15) / 16) * 16 + sizeof(int) * ((size_t)capacity + 2 * F);
}

}  // namespace

int prune_max_chunks() { return kMaxChunks; }

int block_cache_seg_stride(const Shape& s) { return cache_plan_seg_stride(s); }

size_t block_cache_plan_smem(const Shape& s, int capacity) { return cache_plan_smem(s, capacity); }

cudaError_t launch_cache_plan(const Shape& s, const int32_t* seq_lens, const int32_t* page_table,
                              const int32_t* block_idx, const int32_t* n_blocks,
                              const BlockCache& c, int32_t* seg_slot, void* fill,
                              int32_t* n_fill, int* err, cudaStream_t st) {
  CachePlanArgs a;
  a.seq_lens = seq_lens;
  a.page_table = page_table;
  a.block_idx = block_idx;
  a.n_blocks = n_blocks;
  a.header = c.header;
  a.slot_of = c.slot_of;
  a.slot_key = c.slot_key;
  a.slot_stamp = c.slot_stamp;
  a.mass = s.cache_policy == 1 ? c.mass : nullptr;
  a.seg_slot = seg_slot;
  a.fill = static_cast<int4*>(fill);
  a.n_fill = n_fill;
  a.err = err;
  a.batch = s.batch;
  a.hkv = s.hkv;
  a.max_pages = s.max_pages;
  a.num_pages = s.num_pages;
  a.k2 = s.k2;
  a.sink = s.sink;
  a.window = s.window;
  a.seg_stride = cache_plan_seg_stride(s);
  a.capacity = c.capacity;
  const size_t smem = cache_plan_smem(s, c.capacity);
  if (smem > kSmemLimit) return cudaErrorInvalidValue;
  const cudaError_t e = set_kernel_smem(cache_plan_kernel, smem);
  if (e != cudaSuccess) return e;
  return launch_kernel(cache_plan_kernel, dim3(1), dim3(kPruneThreads), smem, st, true, a);
}

size_t prune_smem_bytes(const Shape& s) {
  PruneArgs a;
  if (prune_caps(s, a, true) != 0) return ~size_t(0);
  return prune_smem(a);
}

cudaError_t launch_prune(const Shape& s, const int32_t* seq_lens, const int32_t* block_max,
                         const int32_t* tile_max, int32_t* chunk_idx, int32_t* n_chunks,
                         int32_t* block_idx, int32_t* n_blocks, const int32_t* page_table,
                         int32_t* sel_pages, int* err, cudaStream_t st, unsigned* row_range) {
  if (sel_pages != nullptr && page_table == nullptr) return cudaErrorInvalidValue;
  if (row_range != nullptr && (reinterpret_cast<uintptr_t>(row_range) & 15) != 0)
    return cudaErrorInvalidValue;
  PruneArgs a;
  const bool stage_pages =
      sel_pages != nullptr && (reinterpret_cast<uintptr_t>(page_table) & 15) == 0;
  if (prune_caps(s, a, stage_pages) != 0) return cudaErrorInvalidValue;
  const size_t smem = prune_smem(a);
  if (smem > kSmemLimit) return cudaErrorInvalidValue;
  // the staging copies start from the 16-byte boundary at or below a row's first entry
  if ((reinterpret_cast<uintptr_t>(block_max) & 15) != 0 ||
      (reinterpret_cast<uintptr_t>(tile_max) & 15) != 0)
    return cudaErrorInvalidValue;
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
  a.row_range = row_range;
  a.err = err;
  a.hkv = s.hkv;
  a.max_pages = s.max_pages;
  a.chunk_blocks = s.chunk / kPage;
  a.k1 = s.k1;
  a.k2 = s.k2;
  a.sink = s.sink;
  a.window = s.window;
  a.k0 = s.k0;
  a.coarse_chunks = s.k0 > 0 ? s.chunk0 / s.chunk : 1;
  cudaError_t e = set_kernel_smem(prune_kernel, smem);
  if (e != cudaSuccess) return e;
  return launch_kernel(prune_kernel, dim3(s.hkv, s.batch), dim3(kPruneThreads), smem, st, true, a);
}

}  // namespace hsa
