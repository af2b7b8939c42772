// select.cuh -- exact top-K selection inside one CTA, shared by the pruning kernel, the
// block-cache plan and the sparse attention that runs the pruning modules itself.
//
// Source: InfiniteHiP article (163.com), section "实现 7.24 倍的端到端解码加速" (each pruning
// module keeps the top-K chunks by their best token's score); ties go to the lower index
// (kept lists ascending).
//
// kth_largest finds the K-th largest value T of a shared-memory row by counting: a 2048-bin
// histogram of the values' top 11 bits above the row's minimum, scaled to the row's own value
// range (so that the values spread over the bins: the chunk maxima of a 128K-token row leave
// one to three values in the bin holding T), one scan that locates T's bin, and then either
// the exact value (bin width 1), one warp ranking the few values of that bin, or the next 11
// bits of the values in it. collect then writes, in ascending index order, every index whose
// value is above T plus the lowest-index ones equal to T.
#pragma once

#include <climits>

#include "common.cuh"

// Out-of-line by default; a build may define HSA_SEL_NOINLINE to choose.
#ifndef HSA_SEL_NOINLINE
#define HSA_SEL_NOINLINE __noinline__
#endif

namespace hsa {

constexpr int kSelDigitBits = 11;
constexpr int kSelBins = 1 << kSelDigitBits;  // 2048 histogram bins
constexpr int kSelScan = 256;                 // threads of the locate phase, 8 bins each
constexpr int kSelSmall = 32;                 // a bin this small is ranked by one warp
constexpr int kSelMaxWarps = 32;

// Shared scratch of one CTA's selections. hist and n_cand are zero between selections
// (sel_init before the first one; every selection leaves them zero).
struct SelectShared {
  unsigned hist[kSelBins];
  int wsum[kSelMaxWarps];                  // per-warp totals
  int mn[kSelMaxWarps], mx[kSelMaxWarps];  // per-warp min / max of the valid values
  int w_a[kSelMaxWarps], w_b[kSelMaxWarps];  // per-warp counts of the collect
  int cand[kSelSmall];                     // the values of a small bin
  int n_cand;
  int res[3];                              // located bin or value; keys above it; its count
  unsigned fhist[512];                     // the fast path's histogram (kFastBins), zero
  int cand_i[kSelSmall];                   // the fast path: indices of the small bin's values
};

__device__ __forceinline__ unsigned sel_lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Shared-memory atomics by the shared-window address: the helpers below reach their
// scratch through references, which the compiler sees as generic addresses.
// (No memory clobber: loads may be scheduled across it; every later read of the counters
// comes after a barrier.)
__device__ __forceinline__ void sel_red_add(unsigned* p, unsigned v) {
  asm volatile("red.shared.add.u32 [%0], %1;" ::"r"(smem_addr(p)), "r"(v));
}

__device__ __forceinline__ int sel_atom_add(int* p, int v) {
  int old;
  asm volatile("atom.shared.add.s32 %0, [%1], %2;" : "=r"(old) : "r"(smem_addr(p)), "r"(v)
               : "memory");
  return old;
}

// All NT threads; a CTA barrier must follow before the first selection.
template <int NT>
__device__ __forceinline__ void sel_init(SelectShared& ss) {
  for (int i = threadIdx.x; i < kSelBins; i += NT) ss.hist[i] = 0u;
  for (int i = threadIdx.x; i < 512; i += NT) ss.fhist[i] = 0u;
  if (threadIdx.x == 0) ss.n_cand = 0;
}

// (min, max) of the valid (not INT_MIN) entries of vals[0, n), for every thread; an empty
// set gives (INT_MAX, INT_MIN). One CTA barrier.
template <int NT>
__device__ HSA_SEL_NOINLINE int2 sel_min_max(const int* vals, int n, SelectShared& ss) {
  constexpr int kWarps = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int mn = INT_MAX, mx = INT_MIN;
  for (int i0 = threadIdx.x; i0 < n; i0 += 4 * NT) {
    int v[4];
#pragma unroll
    for (int u = 0; u < 4; u++) {
      const int i = i0 + u * NT;
      v[u] = i < n ? vals[i] : INT_MIN;
    }
#pragma unroll
    for (int u = 0; u < 4; u++) {
      if (v[u] != INT_MIN) {
        mn = min(mn, v[u]);
        mx = max(mx, v[u]);
      }
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, off));
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  }
  if (lane == 0) {
    ss.mn[warp] = mn;
    ss.mx[warp] = mx;
  }
  __syncthreads();
  mn = ss.mn[0];
  mx = ss.mx[0];
#pragma unroll
  for (int w = 1; w < kWarps; w++) {
    mn = min(mn, ss.mn[w]);
    mx = max(mx, ss.mx[w]);
  }
  return make_int2(mn, mx);
}

// Returns (T, need_eq, eq_total): the K-th largest value T of the valid entries of
// vals[0, n) (0 < K <= their number), need_eq = K - #(values > T) (how many of the entries
// equal to T are kept: the lowest-index ones) and eq_total = #(values == T). The valid
// values' min and max are computed here unless the caller has them (have_range).
//
// Keys are the values' offsets from the minimum (unsigned, order-preserving). Level 0 counts
// the top 11 bits of the keys' range; threads 0..255 own 8 bins each, sum them, scan the sums
// (in-warp suffix sums by shuffles, warp totals through shared memory) and the one thread
// whose bins hold the K-th key walks them. A bin of width one gives T; a bin with at most 32
// keys is gathered and ranked by one warp; otherwise the next level counts the next 11 bits
// of the keys in that bin. Per level: 3 CTA barriers (4 when the small bin is ranked).
template <int NT>
__device__ HSA_SEL_NOINLINE int3 sel_kth_largest(const int* vals, int n, int K, SelectShared& ss,
                                             bool have_range, int vmin, int vmax) {
  static_assert(NT >= kSelScan && NT % 32 == 0 && NT <= 32 * kSelMaxWarps, "thread count");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (!have_range) {
    const int2 r = sel_min_max<NT>(vals, n, ss);
    vmin = r.x;
    vmax = r.y;
  }
  const unsigned umin = (unsigned)vmin;
  const unsigned range = (unsigned)vmax - umin;  // exact: vmin <= vmax
  int shift = max(0, (32 - __clz(range)) - kSelDigitBits);
  int match_shift = 32;  // keys taking part agree with `prefix` in bits >= match_shift
  unsigned prefix = 0;
  int above = 0;  // keys known to lie above T
  for (;;) {
    for (int i0 = tid; i0 < n; i0 += 4 * NT) {
      int v[4];
#pragma unroll
      for (int u = 0; u < 4; u++) {
        const int i = i0 + u * NT;
        v[u] = i < n ? vals[i] : INT_MIN;
      }
#pragma unroll
      for (int u = 0; u < 4; u++) {
        const unsigned key = (unsigned)v[u] - umin;
        const bool m = v[u] != INT_MIN &&
                       (match_shift >= 32 || (key >> match_shift) == (prefix >> match_shift));
        if (m) sel_red_add(&ss.hist[(key >> shift) & (kSelBins - 1)], 1u);
      }
    }
    __syncthreads();
    int cnt[8], sum = 0, s = 0;
    if (tid < kSelScan) {
      uint4* hp = reinterpret_cast<uint4*>(&ss.hist[8 * tid]);
      const uint4 c0 = hp[0], c1 = hp[1];
      hp[0] = make_uint4(0u, 0u, 0u, 0u);  // zero for the next level or selection
      hp[1] = make_uint4(0u, 0u, 0u, 0u);
      cnt[0] = (int)c0.x; cnt[1] = (int)c0.y; cnt[2] = (int)c0.z; cnt[3] = (int)c0.w;
      cnt[4] = (int)c1.x; cnt[5] = (int)c1.y; cnt[6] = (int)c1.z; cnt[7] = (int)c1.w;
#pragma unroll
      for (int b = 0; b < 8; b++) sum += cnt[b];
      s = sum;  // keys in this thread's bins or those of the higher lanes of its warp
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_down_sync(0xffffffffu, s, off);
        if (lane + off < 32) s += y;
      }
      if (lane == 0) ss.wsum[warp] = s;
    }
    __syncthreads();
    if (tid < kSelScan) {
      int higher = 0;
#pragma unroll
      for (int w = 0; w < kSelScan / 32; w++) higher += w > warp ? ss.wsum[w] : 0;
      const int incl = above + higher + s;  // keys with digit >= 8 tid, and those above
      const int excl = incl - sum;          // keys with digit >= 8 tid + 8, and those above
      if (excl < K && K <= incl) {
        int acc = excl, d = 8 * tid, c = 0;
#pragma unroll
        for (int b = 7; b >= 0; b--) {
          if (c == 0 && acc + cnt[b] >= K) {
            d = 8 * tid + b;
            c = cnt[b];
          } else if (c == 0) {
            acc += cnt[b];
          }
        }
        ss.res[0] = d;
        ss.res[1] = acc;  // keys in higher bins
        ss.res[2] = c;
      }
    }
    __syncthreads();
    const int d = ss.res[0], cnt_d = ss.res[2];
    above = ss.res[1];
    prefix |= (unsigned)d << shift;
    if (shift == 0) return make_int3((int)(umin + prefix), K - above, cnt_d);
    match_shift = shift;
    if (cnt_d <= kSelSmall) {
      // gather the bin's values; one warp ranks them
      for (int i0 = tid; i0 < n; i0 += 4 * NT) {
        int v[4];
#pragma unroll
        for (int u = 0; u < 4; u++) {
          const int i = i0 + u * NT;
          v[u] = i < n ? vals[i] : INT_MIN;
        }
#pragma unroll
        for (int u = 0; u < 4; u++) {
          const unsigned key = (unsigned)v[u] - umin;
          if (v[u] != INT_MIN && (key >> match_shift) == (prefix >> match_shift))
            ss.cand[sel_atom_add(&ss.n_cand, 1)] = v[u];
        }
      }
      __syncthreads();
      if (warp == 0) {
        const int c = lane < cnt_d ? ss.cand[lane] : INT_MIN;
        int gt = 0, ge = 0;
        for (int j = 0; j < cnt_d; j++) {
          const int cj = ss.cand[j];
          gt += cj > c ? 1 : 0;
          ge += cj >= c ? 1 : 0;
        }
        const int need = K - above;
        const unsigned hit = __ballot_sync(0xffffffffu, lane < cnt_d && gt < need && need <= ge);
        if (lane == __ffs(hit) - 1) {
          ss.res[0] = c;
          ss.res[1] = above + gt;
          ss.res[2] = ge - gt;
        }
        if (lane == 0) ss.n_cand = 0;
      }
      __syncthreads();
      return make_int3(ss.res[0], K - ss.res[1], ss.res[2]);
    }
    shift = max(0, shift - kSelDigitBits);
  }
}

// Emits, in ascending index order, every i with vals[i] > T plus the first need_eq indices
// with vals[i] == T, writing out[position] = add + i; returns how many. Warp w owns a
// contiguous range, read 4 x 32 entries at a time; positions come from ballots (one CTA
// barrier for the per-warp counts). When all entries equal to T are kept (need_eq ==
// eq_total), or none are, the test is a plain threshold and no tie ranks are needed.
template <int NT>
__device__ HSA_SEL_NOINLINE int sel_collect(const int* vals, int n, int T, int need_eq, int eq_total,
                                        SelectShared& ss, int* out, int add) {
  constexpr int kWarps = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int per = ((n + kWarps * 32 - 1) / (kWarps * 32)) * 32;
  const int w0 = min(n, warp * per), w1 = min(n, w0 + per);
  const unsigned lt = sel_lanemask_lt();
  const bool ties_split = need_eq > 0 && need_eq < eq_total;
  // threshold form: keep v > t_lo (placeholders INT_MIN are never kept: t_lo >= INT_MIN)
  const int t_lo = (need_eq > 0 && !ties_split) ? T - 1 : T;
  if (!ties_split) {
    int cnt = 0;
    for (int i0 = w0; i0 < w1; i0 += 128) {
#pragma unroll
      for (int u = 0; u < 4; u++) {
        const int i = i0 + 32 * u + lane;
        cnt += (i < w1 && vals[i] > t_lo) ? 1 : 0;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, off);
    if (lane == 0) ss.w_a[warp] = cnt;
    __syncthreads();
    int pos = 0, total = 0;
#pragma unroll
    for (int w = 0; w < kWarps; w++) {
      const int c = ss.w_a[w];
      pos += w < warp ? c : 0;
      total += c;
    }
    for (int i0 = w0; i0 < w1; i0 += 128) {
      bool take[4];
#pragma unroll
      for (int u = 0; u < 4; u++) {
        const int i = i0 + 32 * u + lane;
        take[u] = i < w1 && vals[i] > t_lo;
      }
#pragma unroll
      for (int u = 0; u < 4; u++) {
        const unsigned tm = __ballot_sync(0xffffffffu, take[u]);
        if (take[u]) out[pos + __popc(tm & lt)] = add + i0 + 32 * u + lane;
        pos += __popc(tm);
      }
    }
    __syncthreads();
    return total;
  }
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
  for (int w = 0; w < kWarps; w++) {
    const int kept_w = ss.w_a[w] + min(max(need_eq - eq_acc, 0), ss.w_b[w]);
    if (w == warp) {
      pos = total;
      eq_base = eq_acc;
    }
    total += kept_w;
    eq_acc += ss.w_b[w];
  }
  for (int i0 = w0; i0 < w1; i0 += 32) {
    const int i = i0 + lane;
    const int v = i < w1 ? vals[i] : INT_MIN;
    const bool gt = i < w1 && v > T, eq = i < w1 && v == T;
    const unsigned eqm = __ballot_sync(0xffffffffu, eq);
    const bool take = gt || (eq && eq_base + __popc(eqm & lt) < need_eq);
    const unsigned tm = __ballot_sync(0xffffffffu, take);
    if (take) out[pos + __popc(tm & lt)] = add + i;
    eq_base += __popc(eqm);
    pos += __popc(tm);
  }
  __syncthreads();
  return total;
}

// ------------------------------------------------ fast path: range known, three barriers
//
// When the values' range [vmin, vmax] is known before the selection (the scorer records each
// row's range of maxima) and every thread can hold its share of the row in registers, a
// 512-bin histogram of the keys' top 9 bits above vmin is built in the pass that reads the
// values. Every warp then finds the bin d holding the K-th largest key from the histogram by
// itself (no scan barrier). When d holds at most 32 values (the usual case: the tile maxima
// of a 128K-token row put a few values in that bin) one pass gathers them with their indices
// and counts, per thread, the values in higher bins; every warp ranks the gathered values by
// itself, which gives T and which equal values are kept; the thread's values, still in
// registers, are then written in ascending order. Three CTA barriers in all. A larger bin
// returns -1 and the caller takes the general path (sel_kth_largest, sel_collect).
constexpr int kFastBinBits = 9;
constexpr int kFastBins = 1 << kFastBinBits;

__device__ __forceinline__ int fast_shift(int vmin, int vmax) {
  const unsigned range = (unsigned)vmax - (unsigned)vmin;
  return max(0, (32 - __clz(range)) - kFastBinBits);
}

// Bin of v (a value inside the range; clamped, so that a value outside it cannot index past
// the histogram).
__device__ __forceinline__ int fast_bin(int v, unsigned umin, int shift) {
  return (int)min(((unsigned)v - umin) >> shift, (unsigned)(kFastBins - 1));
}

// Every warp: (d, keys in higher bins, keys in d) for the K-th largest key (0 < K <= the
// histogram's total). Lane l reads bins 4l..4l+3 of each group of 128 (conflict-free 16-byte
// reads); warp sums give the groups' totals.
__device__ __forceinline__ int3 fast_locate(const unsigned* fhist, int K) {
  const int lane = threadIdx.x & 31;
  const uint32_t hb = smem_addr(fhist);
  int part[kFastBins / 128], tot[kFastBins / 128];
  uint4 c[kFastBins / 128];
#pragma unroll
  for (int g = 0; g < kFastBins / 128; g++) c[g] = lds128(hb + (128 * g + 4 * lane) * 4);
#pragma unroll
  for (int g = 0; g < kFastBins / 128; g++) {
    part[g] = (int)(c[g].x + c[g].y + c[g].z + c[g].w);
    tot[g] = __reduce_add_sync(0xffffffffu, part[g]);
  }
  int acc = 0, mine = 0, gsel = 0;
  uint4 cm = make_uint4(0u, 0u, 0u, 0u);
  bool found = false;
#pragma unroll
  for (int g = kFastBins / 128 - 1; g >= 0; g--) {
    if (!found && acc + tot[g] >= K) {
      found = true;
      gsel = g;
      mine = part[g];
      cm = c[g];
    } else if (!found) {
      acc += tot[g];
    }
  }
  int incl = mine;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_down_sync(0xffffffffu, incl, off);
    if (lane + off < 32) incl += y;
  }
  const int excl = incl - mine;
  const int L = __ffs(__ballot_sync(0xffffffffu, acc + excl < K && K <= acc + incl)) - 1;
  int d = 0, above = 0, cnt = 0;
  if (lane == L) {
    const int cb[4] = {(int)cm.x, (int)cm.y, (int)cm.z, (int)cm.w};
    int a2 = acc + excl;
    bool f2 = false;
#pragma unroll
    for (int b = 3; b >= 0; b--) {
      if (!f2 && a2 + cb[b] >= K) {
        f2 = true;
        d = 128 * gsel + 4 * lane + b;
        cnt = cb[b];
      } else if (!f2) {
        a2 += cb[b];
      }
    }
    above = a2;
  }
  return make_int3(__shfl_sync(0xffffffffu, d, L), __shfl_sync(0xffffffffu, above, L),
                   __shfl_sync(0xffffffffu, cnt, L));
}

// The fast path for rows of at most R values a thread: each thread keeps its contiguous
// span of values in registers across the three passes (histogram, gather, write), so a
// pass is a few instructions a value; the ranking loops run over the bin's count. get(x)
// returns (value, id) of entry x (value INT_MIN: no candidate); out receives the kept
// entries' ids in ascending order of x. Returns min(K, valid entries), or -1 (nothing
// written) when the K-th key's bin holds more than kSelSmall values; K <= 0 writes nothing
// and returns 0. Expects fhist and n_cand zero and leaves them zero; three CTA barriers (two
// when everything is kept, none when K <= 0).
// The entries of a row for sel_fast_reg: value vals[x] and id ids[x] (ids nullable: id =
// add + x). One type for every caller, so that the selection's code exists once.
struct SelRow {
  const int* vals;
  const int* ids;
  int add;
  __device__ __forceinline__ int2 operator()(int x) const {
    return make_int2(vals[x], ids != nullptr ? ids[x] : add + x);
  }
};

template <int NT, int R, typename Get>
__device__ __forceinline__ int sel_fast_reg(Get get, int n, int K, int vmin, int vmax,
                                            SelectShared& ss, int* out) {
  constexpr int kWarps = NT / 32;
  if (K <= 0) return 0;  // keeps nothing (the same in every thread: no barrier is skipped)
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned umin = (unsigned)vmin;
  const int shift = fast_shift(vmin, vmax);
  const int per = (n + NT - 1) / NT;  // <= R (the caller checks n <= R * NT)
  const int x0 = min(n, tid * per), nv = min(n, x0 + per) - x0;
  int v[R], id[R];
  unsigned kb[R];
  int valid = 0;
#pragma unroll
  for (int r = 0; r < R; r++) {  // all loads first
    const int2 e = r < nv ? get(x0 + r) : make_int2(INT_MIN, -1);
    v[r] = e.x;
    id[r] = e.y;
  }
#pragma unroll
  for (int r = 0; r < R; r++) {
    kb[r] = min(((unsigned)v[r] - umin) >> shift, (unsigned)(kFastBins - 1));
    if (v[r] != INT_MIN) {
      valid++;
      sel_red_add(&ss.fhist[kb[r]], 1u);
    }
  }
  const int valid_w = __reduce_add_sync(0xffffffffu, valid);
  if (lane == 0) ss.wsum[warp] = valid_w;
  __syncthreads();
  int n_valid = 0, vbase = 0;
#pragma unroll
  for (int w = 0; w < kWarps; w++) {
    const int c = ss.wsum[w];
    n_valid += c;
    vbase += w < warp ? c : 0;
  }
  const int keep_n = min(K, n_valid);
  if (keep_n == n_valid) {  // everything valid is kept (also keep_n == 0)
    int incl = valid;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += y;
    }
    int pos = vbase + incl - valid;
#pragma unroll
    for (int r = 0; r < R; r++)
      if (v[r] != INT_MIN) out[pos++] = id[r];
    for (int i = tid; i < kFastBins; i += NT) ss.fhist[i] = 0u;
    __syncthreads();
    return keep_n;
  }
  const int3 loc = fast_locate(ss.fhist, keep_n);
  const unsigned d = (unsigned)loc.x;
  const int above = loc.y, cnt = loc.z;
  if (cnt > kSelSmall) {
    __syncthreads();  // every warp has read the histogram and the per-warp counts
    for (int i = tid; i < kFastBins; i += NT) ss.fhist[i] = 0u;
    __syncthreads();
    return -1;
  }
  int gt = 0;
#pragma unroll
  for (int r = 0; r < R; r++) {
    if (v[r] == INT_MIN) continue;
    if (kb[r] > d) {
      gt++;
    } else if (kb[r] == d) {
      const int slot = sel_atom_add(&ss.n_cand, 1);
      if (slot < kSelSmall) {  // (the histogram counted exactly these)
        ss.cand[slot] = v[r];
        ss.cand_i[slot] = x0 + r;
      }
    }
  }
  const int gt_w = __reduce_add_sync(0xffffffffu, gt);
  if (lane == 0) ss.w_b[warp] = gt_w;
  __syncthreads();
  // every warp ranks the bin's values
  const int c = lane < cnt ? ss.cand[lane] : INT_MIN;
  const int ci = lane < cnt ? ss.cand_i[lane] : INT_MAX;
  int gtc = 0, gec = 0;
  for (int j = 0; j < cnt; j++) {
    const int cj = __shfl_sync(0xffffffffu, c, j);
    gtc += cj > c ? 1 : 0;
    gec += cj >= c ? 1 : 0;
  }
  const int need = keep_n - above;
  const int L = __ffs(__ballot_sync(0xffffffffu, lane < cnt && gtc < need && need <= gec)) - 1;
  const int T = __shfl_sync(0xffffffffu, c, L);
  const int need_eq = need - __shfl_sync(0xffffffffu, gtc, L);
  const int eq_total = __popc(__ballot_sync(0xffffffffu, lane < cnt && c == T));
  const bool split = need_eq < eq_total;  // only some of the values equal to T are kept
  bool kp = lane < cnt && c >= T;
  if (split) {  // rare: ties at the threshold, ranked by index
    int eq_before = 0;
    for (int j = 0; j < cnt; j++) {
      const int cj = __shfl_sync(0xffffffffu, c, j);
      const int cij = __shfl_sync(0xffffffffu, ci, j);
      eq_before += (cj == T && cij < ci) ? 1 : 0;
    }
    kp = lane < cnt && (c > T || (c == T && eq_before < need_eq));
  }
  const unsigned keep = __ballot_sync(0xffffffffu, kp);
  const int w_first = min(n, warp * 32 * per);
  int base = __popc(__ballot_sync(0xffffffffu, kp && ci < w_first));
#pragma unroll
  for (int w = 0; w < kWarps; w++) base += w < warp ? ss.w_b[w] : 0;
  bool tk[R];
  int mine = 0;
#pragma unroll
  for (int r = 0; r < R; r++) {
    bool t = v[r] != INT_MIN && (kb[r] > d || (kb[r] == d && v[r] >= T));
    if (split && v[r] == T) {
      int k = 0;
      for (unsigned m = keep; m != 0u; m &= m - 1)
        k += ss.cand_i[__ffs(m) - 1] == x0 + r ? 1 : 0;
      t = k > 0;
    }
    tk[r] = t;
    mine += t ? 1 : 0;
  }
  int incl = mine;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  int pos = base + incl - mine;
#pragma unroll
  for (int r = 0; r < R; r++)
    if (tk[r]) out[pos++] = id[r];
  for (int i = tid; i < kFastBins; i += NT) ss.fhist[i] = 0u;
  if (tid == 0) ss.n_cand = 0;
  __syncthreads();
  return keep_n;
}

// One warp (all its lanes): the `drop` lowest-ranked entries of vals[0, n) (the smallest
// value, the higher index first among equal values) into out[0, drop), in that order; each
// is marked taken by INT_MAX in vals (the values must lie below it). A round is a warp-wide
// minimum over every lane's smallest entry, the lane scanning its entries four at a time
// with independent partial minima.
__device__ __forceinline__ void sel_peel_lowest(int* vals, int n, int drop, int* out) {
  const int lane = threadIdx.x & 31;
  auto better = [](int v, int i, int bv, int bi) { return v < bv || (v == bv && i > bi); };
  for (int e = 0; e < drop; e++) {
    int bv[4] = {INT_MAX, INT_MAX, INT_MAX, INT_MAX}, bi[4] = {-1, -1, -1, -1};
    int i = lane;
    for (; i + 96 < n; i += 128) {
#pragma unroll
      for (int u = 0; u < 4; u++) {
        const int v = vals[i + 32 * u];
        if (better(v, i + 32 * u, bv[u], bi[u])) {
          bv[u] = v;
          bi[u] = i + 32 * u;
        }
      }
    }
    for (; i < n; i += 32) {
      const int v = vals[i];
      if (better(v, i, bv[0], bi[0])) {
        bv[0] = v;
        bi[0] = i;
      }
    }
#pragma unroll
    for (int u = 1; u < 4; u++)
      if (better(bv[u], bi[u], bv[0], bi[0])) {
        bv[0] = bv[u];
        bi[0] = bi[u];
      }
    const int mv = __reduce_min_sync(0xffffffffu, bv[0]);
    const int mi = __reduce_max_sync(0xffffffffu, bv[0] == mv ? bi[0] : -1);
    if (lane == 0) {
      out[e] = mi;
      vals[mi] = INT_MAX;
    }
    __syncwarp();
  }
}

// sel_fast_reg on a SelRow, out of line (one copy of the code for every call site).
template <int NT, int R>
__device__ __noinline__ int sel_fast_row(SelRow row, int n, int K, int vmin, int vmax,
                                         SelectShared& ss, int* out) {
  return sel_fast_reg<NT, R>(row, n, K, vmin, vmax, ss, out);
}

// A row src[0, n) of ints in global memory (in an array whose base is 16-byte aligned) to be
// staged in shared memory at dst_base (16-byte aligned, room for n + 3 ints): the copy of
// src[i] lands at dst_base[o + i]. The 16-byte-aligned span [src - o, src - o + body) is
// copied in bulk, the ragged tail with plain loads.
struct StagedRow {
  const int32_t* s0;  // src - o, 16-byte aligned, inside the array
  int* dst_base;
  int o, body, n;
  __device__ int* dst() const { return dst_base + o; }
  __device__ uint32_t bytes() const { return (uint32_t)body * 4u; }
};

__device__ __forceinline__ StagedRow plan_row(int* dst_base, const int32_t* src, int n) {
  StagedRow r;
  r.o = (int)((reinterpret_cast<uintptr_t>(src) >> 2) & 3);
  r.s0 = src - r.o;
  r.body = ((n + r.o) / 4) * 4;
  r.dst_base = dst_base;
  r.n = n;
  return r;
}

// One thread: the bulk copies of a planned row (at most 64 KiB each), completing on `bar`.
__device__ __forceinline__ void issue_row(const StagedRow& r, uint64_t* bar) {
  for (int off = 0; off < r.body; off += 16384)
    bulk_load(r.dst_base + off, r.s0 + off, (uint32_t)min(16384, r.body - off) * 4u, bar);
}

// NT threads: the ragged tail of a planned row.
template <int NT>
__device__ __forceinline__ void tail_row(const StagedRow& r) {
  for (int i = r.body + threadIdx.x; i < r.n + r.o; i += NT) r.dst_base[i] = __ldg(r.s0 + i);
}

}  // namespace hsa
