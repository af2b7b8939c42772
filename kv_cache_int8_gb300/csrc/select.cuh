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
};

__device__ __forceinline__ unsigned sel_lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// All NT threads; a CTA barrier must follow before the first selection.
template <int NT>
__device__ __forceinline__ void sel_init(SelectShared& ss) {
  for (int i = threadIdx.x; i < kSelBins; i += NT) ss.hist[i] = 0u;
  if (threadIdx.x == 0) ss.n_cand = 0;
}

// (min, max) of the valid (not INT_MIN) entries of vals[0, n), for every thread; an empty
// set gives (INT_MAX, INT_MIN). One CTA barrier.
template <int NT>
__device__ __noinline__ int2 sel_min_max(const int* vals, int n, SelectShared& ss) {
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
__device__ __noinline__ int3 sel_kth_largest(const int* vals, int n, int K, SelectShared& ss,
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
        if (m) atomicAdd(&ss.hist[(key >> shift) & (kSelBins - 1)], 1u);
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
            ss.cand[atomicAdd(&ss.n_cand, 1)] = v[u];
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
__device__ __noinline__ int sel_collect(const int* vals, int n, int T, int need_eq, int eq_total,
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
