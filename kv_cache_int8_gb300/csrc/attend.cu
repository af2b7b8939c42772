// attend.cu -- exact split-K decode attention over a block list, merged by log-sum-exp.
//
// Sources: "KV Cache 与长上下文推理", section "KV Cache 回顾" (decode attention
// softmax(q_t K^T / sqrt(d_k)) V over the cached keys and values), section "Token Eviction
// 与 Sparse Attention" (StreamingLLM: attention sinks + sliding window) and section
// "Flash Attention" (tiled attention that never materialises the score row); InfiniteHiP
// article (163.com), section "实现 7.24 倍的端到端解码加速" (attention over the block-sparse
// mask the pruning modules produce) and its latency section (the attention kernel reads CPU
// memory while it runs); HCAttention abstract (values stay in CPU memory and are fetched
// late, for the final aggregation only).
//
// Work: the attended set of (sequence b, kv head h) is a list of segments, each a
// 16-token page clipped to a token range: the sink pages, the kept blocks (clipped to the
// candidate region), the window pages. Dense decode uses every page of [0, N). A CTA takes
// a share of the list (sparse attend: every nsplit-th segment; dense decode: a contiguous
// range) for all G query heads of the group, so every K/V byte is read once per group.
// Scores of a token: 8 lanes (16 channels each) form G partial dot products and reduce them
// with a transposing butterfly; softmax in the log2 domain with a running max and sum per
// head; CTAs of one (b, h) are merged by the last one to finish (atomic counter, no
// waiting).
//
// HBM path: a producer lane fills a ring of 8 KiB slots (K page then V page of one head,
// 4 KiB each) with cp.async.bulk copies tracked by mbarriers; each compute warp owns fixed
// slots and processes whole segments on its own (see the HBM-path section).
// Host path: K/V live in pinned host memory; the compute warps copy each segment into
// shared memory with 16-byte loads through the mapped alias, one segment ahead, and
// process it together (scores: warp w takes tokens 4w..4w+3; softmax: warp j owns head j;
// values: warp w owns channels [64 (w & 1) + 2 lane, +2) of tokens 8 (w >> 1) .. +8).
#include <algorithm>
#include <cfloat>

#include "common.cuh"
#include "internal.h"
#include "select.cuh"

// Split-K grid sizing (CTAs per SM); overridable at build time for tuning.
#ifndef HSA_SPARSE_CTAS_PER_SM
#define HSA_SPARSE_CTAS_PER_SM 1
#endif
#ifndef HSA_DENSE_CTAS_PER_SM
#define HSA_DENSE_CTAS_PER_SM 3
#endif
#ifndef HSA_HOST_CTAS_PER_SM
#define HSA_HOST_CTAS_PER_SM 3
#endif
#ifndef HSA_SPARSE_WARPS
#define HSA_SPARSE_WARPS 12
#endif
// Sparse attend: leave one SM per (sequence, kv head) to the prune kernel that is still
// running when the attend starts, when that costs at most a quarter of the splits.
#ifndef HSA_SPARSE_RESERVE
#define HSA_SPARSE_RESERVE 1
#endif
// The whole decode step runs the pruning modules inside the sparse attention (0: a pruning
// kernel, then the sparse attention, as hsa_select + hsa_attend).
// 1: with K1 >= K2 the selecting attention ranks only the blocks at or above the K2-th
// largest chunk maximum (sel_blocks_over_threshold), else the two modules' fast paths
#ifndef HSA_SEL_THRESHOLD
#define HSA_SEL_THRESHOLD 1
#endif
// 1: the selecting attention's CTAs of a row prefetch the candidate blocks' K/V pages into L2
// (each CTA a 1/nsplit share) as soon as the candidates are known
#ifndef HSA_SEL_PREFETCH
#define HSA_SEL_PREFETCH 1
#endif
#ifndef HSA_FUSED_SELECT
#define HSA_FUSED_SELECT 1
#endif

namespace hsa {
namespace {

constexpr int kWarps = 4;                        // compute warps of the host path
constexpr int kCompute = kWarps * 32;
constexpr int kStages = 8;
// HBM path, sparse attend: for CTAs with many segments 12 compute warps + the producer, two
// ring slots each (measured on GB300 at 1M tokens, about 22 segments a CTA: the attention
// 12.9 against 15.6 us with 8 warps, the step 188.0 against 189.5 us; 10 warps 189.4), for
// fewer segments 8 (the batched case's pruning-form attention, about 19 a CTA, measured
// faster with 8). A CTA of it does not fit beside a prune CTA (registers), so the prune
// keeps its SMs to itself; an attention launched early beside it leaves those SMs free
// (HSA_SPARSE_RESERVE).
constexpr int kSparseWarps = HSA_SPARSE_WARPS;  // ring: two slots per compute warp
constexpr int kSparseManySegs = 20;
// CTAs with at most this many segments take as many compute warps with one slot each, so
// that no warp takes a second segment (a 128K row's attention called alone, 11 a CTA: the
// reuse step 16.6 against 17.2 us with 8 warps and two slots)
#ifndef HSA_SPARSE_FEW_WARPS
#define HSA_SPARSE_FEW_WARPS 11
#endif
constexpr int kSparseFewWarps = HSA_SPARSE_FEW_WARPS;
constexpr int kDenseWarps = 4, kDenseStages = 8;     // HBM path, dense decode
constexpr int kSlotBytes = 2 * kBlockBytesBf16;  // K page + V page of one head
constexpr int kHostThreads = kCompute;
static_assert(kHostThreads * 16 * 2 == kBlockBytesBf16, "a host-path segment copy: 2 x 16 B a thread");
constexpr int kMaxSplits = 64;
constexpr int kTileBlocksSel = 4;              // blocks per 64-token chunk (a scorer tile)
constexpr int kSelRegVals = 8;  // values a thread of the selecting attention keeps in registers
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kNeg = -FLT_MAX;                 // "no token" score

// Per-head slots of the shared scratch areas: 4 for groups of up to 4 query heads, else 8.
__host__ __device__ constexpr int head_slots(int G) { return G <= 4 ? 4 : 8; }

struct AttArgs {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const int32_t* page_table;
  const int32_t* seq_lens;
  const int32_t* block_idx;
  const int32_t* n_blocks;
  const int32_t* sel_pages;  // nullable: page of each kept block, beside block_idx
  const int32_t* seg_slots;  // nullable: block-cache slot of every segment (then k / v point
                             // at the cache's K and V halves and num_pages is its capacity)
  int seg_stride;
  // nullable, with seg_slots (block cache, cumulative-mass policy): seg_l2 [B][Hkv][seg_stride]
  // [G] gets each segment's log-sum-exp (log2 domain) per query head; the last CTA of (b, h)
  // adds each segment's attention mass to mass[slot_key[slot] - 1]
  float* seg_l2;
  float* mass;
  const int32_t* slot_key;
  float* out;
  float* lse;
  float* part_ml;
  float* part_o;
  int* counters;
  int* err;
  int hkv, max_pages, num_pages, k2, sink, window, nsplit;
  int kv_heads, kv_div;  // K/V heads of the cache; attention rows per kv head (row h reads
                         // kv head h / kv_div: hq / hkv with per-head selection, else 1)
  float qscale;  // sm_scale * log2(e)
  int early;     // K/V, q, page table are ready before the selection (whole decode step)
  unsigned* row_range;  // nullable: [rows][4] words that the last CTA of a row clears
};

struct Segments {
  int n;  // context length
  int n_sink, n_win, n_sel_max, n_sel;
  int sink_end, cand_hi, w0, win_k0;
  const int32_t* sel;
  int total;  // n_sink + n_win + n_sel_max: the split ranges are known before the selection
};

// The attended set as a list of segments: the sink pages, the window pages, then up to K2
// kept blocks. Everything but the number of kept blocks (n_sel: read_selection, or the HBM
// path's producer with the kept ids) is known from the sequence length alone.
template <bool DENSE>
__device__ __forceinline__ Segments make_segments(const AttArgs& a, int b, int h) {
  Segments s;
  int n = a.seq_lens[b];
  if (n < 0 || n > a.max_pages * kPage) n = 0;  // reported by the caller's check
  s.n = n;
  s.sel = nullptr;
  s.n_sel = 0;
  if (DENSE) {
    s.n_sink = 0;
    s.n_sel_max = 0;
    s.n_win = (n + kPage - 1) / kPage;
    s.sink_end = 0;
    s.cand_hi = 0;
    s.w0 = 0;
    s.win_k0 = 0;
  } else {
    s.sink_end = min(a.sink, n);
    s.n_sink = (s.sink_end + kPage - 1) / kPage;
    s.cand_hi = n - a.window;
    s.n_sel_max = s.cand_hi > a.sink ? a.k2 : 0;
    s.w0 = max(n - a.window, s.sink_end);
    s.win_k0 = s.w0 / kPage;
    s.n_win = s.w0 < n ? (n + kPage - 1) / kPage - s.win_k0 : 0;
  }
  s.total = s.n_sink + s.n_win + s.n_sel_max;
  return s;
}

// The kept blocks of (b, h), written by the previous kernel: read after grid_dep_wait().
__device__ __forceinline__ void read_selection(Segments& s, const AttArgs& a, int b, int h) {
  if (s.n_sel_max == 0) return;
  s.sel = a.block_idx + ((size_t)b * a.hkv + h) * a.k2;
  s.n_sel = max(0, min(a.n_blocks[(size_t)b * a.hkv + h], s.n_sel_max));
}

// Kept block r of the list, whose id kk was read from it: its page index k and token range
// [t0, t1) inside the candidate region (empty past the count of kept blocks or for an id
// outside the sequence).
__device__ __forceinline__ void kept_segment(const Segments& s, int r, int kk, int sink, int& k,
                                             int& t0, int& t1) {
  k = 0;
  t0 = t1 = 0;
  if (r >= s.n_sel) return;
  const int kmax = (s.n + kPage - 1) / kPage;
  if (kk < 0 || kk >= kmax) return;
  k = kk;
  t0 = max(k * kPage, sink);
  t1 = min(k * kPage + kPage, s.cand_hi);
}

// Segment i: page index k (token block) and the attended token range [t0, t1) (empty when
// t0 >= t1).
__device__ __forceinline__ void segment_at(const Segments& s, int i, int sink, int& k, int& t0,
                                           int& t1) {
  if (i < s.n_sink) {
    k = i;
    t0 = i * kPage;
    t1 = min(t0 + kPage, s.sink_end);
  } else if (i < s.n_sink + s.n_win) {
    k = s.win_k0 + (i - s.n_sink);
    t0 = max(k * kPage, s.w0);
    t1 = min(k * kPage + kPage, s.n);
  } else {
    kept_segment(s, i - s.n_sink - s.n_win, s.sel[i - s.n_sink - s.n_win], sink, k, t0, t1);
  }
}

__device__ __forceinline__ void unpack16(const uint4& a, const uint4& b, float f[16]) {
  f[0] = bf16_lo(a.x); f[1] = bf16_hi(a.x); f[2] = bf16_lo(a.y); f[3] = bf16_hi(a.y);
  f[4] = bf16_lo(a.z); f[5] = bf16_hi(a.z); f[6] = bf16_lo(a.w); f[7] = bf16_hi(a.w);
  f[8] = bf16_lo(b.x); f[9] = bf16_hi(b.x); f[10] = bf16_lo(b.y); f[11] = bf16_hi(b.y);
  f[12] = bf16_lo(b.z); f[13] = bf16_hi(b.z); f[14] = bf16_lo(b.w); f[15] = bf16_hi(b.w);
}

__device__ __forceinline__ void compute_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(kCompute) : "memory");
}

// Shared memory of the compute warps besides the K/V slots (H = head_slots(G)).
template <int H>
struct Scratch {
  float score[kPage][H];  // per token, per head (log2-scaled logits)
  float prob[kPage][H];   // softmax weights of the segment
  float rescale[H];       // factor applied to the running state of each head
  float m[H], l[H];       // final running max / sum per head
};

// Running state of one lane.
template <int G>
struct State {
  static constexpr int kOwn = (G + kWarps - 1) / kWarps;  // heads owned by one warp
  float acc[G][2];  // weighted value sums, 2 channels x G heads
  float m[kOwn], l[kOwn];  // running max / sum of heads warp + kWarps i (lane 0 meaningful)
};

// The G dot products of a token, reduced over its 8 lanes: afterwards lane `sl` holds the
// full score of head hidx(sl). Partner lanes exchange halves of their vectors at each step.
template <int G>
__device__ __forceinline__ float reduce_scores(float (&v)[G], int sl, int& hidx) {
  if constexpr (G == 8) {
    const bool b2 = sl & 4, b1 = sl & 2, b0 = sl & 1;
    float u[4];
#pragma unroll
    for (int i = 0; i < 4; i++) {
      const float r = __shfl_xor_sync(0xffffffffu, b2 ? v[i] : v[4 + i], 4);
      u[i] = (b2 ? v[4 + i] : v[i]) + r;  // head (b2 ? 4 : 0) + i
    }
    float w2[2];
#pragma unroll
    for (int i = 0; i < 2; i++) {
      const float r = __shfl_xor_sync(0xffffffffu, b1 ? u[i] : u[2 + i], 2);
      w2[i] = (b1 ? u[2 + i] : u[i]) + r;  // head (b2 ? 4 : 0) + (b1 ? 2 : 0) + i
    }
    const float r = __shfl_xor_sync(0xffffffffu, b0 ? w2[0] : w2[1], 1);
    hidx = sl;
    return (b0 ? w2[1] : w2[0]) + r;
  } else if constexpr (G == 4) {
    const bool b2 = sl & 4, b1 = sl & 2;
    const float s0 = b2 ? v[0] : v[2], s1 = b2 ? v[1] : v[3];
    const float r0 = __shfl_xor_sync(0xffffffffu, s0, 4);
    const float r1 = __shfl_xor_sync(0xffffffffu, s1, 4);
    const float u0 = (b2 ? v[2] : v[0]) + r0, u1 = (b2 ? v[3] : v[1]) + r1;
    const float r = __shfl_xor_sync(0xffffffffu, b1 ? u0 : u1, 2);
    float w = (b1 ? u1 : u0) + r;
    w += __shfl_xor_sync(0xffffffffu, w, 1);
    hidx = (b2 ? 2 : 0) + (b1 ? 1 : 0);
    return w;
  } else if constexpr (G == 2) {
    const bool b2 = sl & 4;
    const float r = __shfl_xor_sync(0xffffffffu, b2 ? v[0] : v[1], 4);
    float w = (b2 ? v[1] : v[0]) + r;
    w += __shfl_xor_sync(0xffffffffu, w, 2);
    w += __shfl_xor_sync(0xffffffffu, w, 1);
    hidx = b2 ? 1 : 0;
    return w;
  } else {
    float w = v[0];
    w += __shfl_xor_sync(0xffffffffu, w, 4);
    w += __shfl_xor_sync(0xffffffffu, w, 2);
    w += __shfl_xor_sync(0xffffffffu, w, 1);
    hidx = 0;
    return w;
  }
}

template <int G>
__device__ __forceinline__ void load_query(float (&qf)[G][16], const AttArgs& a, int b, int h,
                                           int sl) {
#pragma unroll
  for (int j = 0; j < G; j++) {
    const __nv_bfloat16* qp = a.q + ((size_t)b * a.hkv * G + (size_t)h * G + j) * kHeadDim;
    const uint4 u0 = *reinterpret_cast<const uint4*>(qp + 8 * sl);
    const uint4 u1 = *reinterpret_cast<const uint4*>(qp + 64 + 8 * sl);
    float f[16];
    unpack16(u0, u1, f);
#pragma unroll
    for (int e = 0; e < 16; e++) qf[j][e] = f[e] * a.qscale;
  }
}

// One segment held in shared memory at `slot` (K page, then V page): scores, softmax and
// value accumulation. Called by the 128 compute threads together.
template <int G>
__device__ __forceinline__ void process_segment(State<G>& st, const float (&qf)[G][16],
                                                Scratch<head_slots(G)>& sc, uint32_t slot,
                                                int k, int t0, int t1) {
  constexpr int H = head_slots(G);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // scores
  {
    const int grp = lane >> 3, sl = lane & 7;
    const int r = warp * 4 + grp;
    const uint32_t kb = slot + r * (kHeadDim * 2);
    const uint4 k0 = lds128(kb + sl * 16), k1 = lds128(kb + (sl + 8) * 16);
    float kf[16];
    unpack16(k0, k1, kf);
    float v[G];
#pragma unroll
    for (int j = 0; j < G; j++) {
      float acc = 0.0f;
#pragma unroll
      for (int e = 0; e < 16; e++) acc = fmaf(qf[j][e], kf[e], acc);
      v[j] = acc;
    }
    int hidx;
    const float s = reduce_scores<G>(v, sl, hidx);
    const int t = k * kPage + r;
    constexpr int kOwners = 8 / G;  // lanes holding the same head; the first one writes
    if ((sl & (kOwners - 1)) == 0) sc.score[r][hidx] = (t >= t0 && t < t1) ? s : kNeg;
  }
  compute_bar();
  // softmax of the segment, one warp per head (warp w owns heads w, w + 4; lanes 0..15
  // carry the 16 tokens)
#pragma unroll
  for (int i = 0; i < State<G>::kOwn; i++) {
    const int hh = warp + kWarps * i;
    if (hh >= G) continue;
    const float s = lane < kPage ? sc.score[lane][hh] : kNeg;
    float mx = s;
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    const float m_new = fmaxf(st.m[i], mx);
    const float c = exp2f(st.m[i] - m_new);
    const float p = s == kNeg ? 0.0f : exp2f(s - m_new);
    float ps = p;
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
    st.l[i] = st.l[i] * c + ps;
    st.m[i] = m_new;
    if (lane < kPage) sc.prob[lane][hh] = p;
    if (lane == 0) sc.rescale[hh] = c;
  }
  compute_bar();
  // values
  {
    const int d = (warp & 1) * 64 + 2 * lane;
    const int th = warp >> 1;
#pragma unroll
    for (int j = 0; j < G; j++) {
      const float c = sc.rescale[j];
      st.acc[j][0] *= c;
      st.acc[j][1] *= c;
    }
    const uint32_t vb = slot + kBlockBytesBf16 + d * 2;
    const int tb = k * kPage + th * 8;
#pragma unroll
    for (int tt = 0; tt < 8; tt++) {
      const int t = tb + tt;
      if (t < t0 || t >= t1) continue;  // warp-uniform; skipped slots may hold any bits
      uint32_t w;
      asm volatile("ld.shared.u32 %0, [%1];" : "=r"(w) : "r"(vb + (th * 8 + tt) * kHeadDim * 2));
      const float lo = bf16_lo(w), hi = bf16_hi(w);
      float p[H];
#pragma unroll
      for (int q4 = 0; q4 < H / 4; q4++) {
        const float4 p4 = *reinterpret_cast<const float4*>(&sc.prob[th * 8 + tt][4 * q4]);
        p[4 * q4] = p4.x;
        p[4 * q4 + 1] = p4.y;
        p[4 * q4 + 2] = p4.z;
        p[4 * q4 + 3] = p4.w;
      }
#pragma unroll
      for (int j = 0; j < G; j++) {
        st.acc[j][0] = fmaf(p[j], lo, st.acc[j][0]);
        st.acc[j][1] = fmaf(p[j], hi, st.acc[j][1]);
      }
    }
  }
  // the next segment's score writes are ordered after these reads by its first barrier
}

// Output of a CTA from its merged state in shared memory (o[G][128], m[G], l[G]): either the
// final result (one split) or a partial, and then the combine over all splits by the last
// CTA of (b, h) to finish. `red` (shared, at least G * kMaxSplits + 8 floats) may alias
// `o`. Called by all threads of the CTA after the merged state is complete. NB: splits a
// thread of the combine loads per round trip.
// Cumulative-mass cache policy: adds each attended segment's attention mass, summed over the
// G query heads (p = 2^(seg_l2 - lse2) per head), to the cumulative mass of the block that its
// cache slot holds. One CTA per (b, h), once the final log-sum-exp lse2[j] of every head is
// known. A block can be two segments of one call: the sink's last page or the window's first
// page when either is partial, and a kept block or the other of the two (same slot). Such a
// block's masses are summed, in segment order, by the boundary segment that holds it, so that
// every entry is written by one thread and the result does not depend on timing. scratch:
// 2 * seg_stride words of shared memory.
template <int G>
__device__ void add_segment_mass(const AttArgs& a, int b, int h, const float* lse2,
                                 float* scratch) {
  const Segments S = make_segments<false>(a, b, h);
  const int n = a.seg_stride;
  int* slot_s = reinterpret_cast<int*>(scratch);
  float* w_s = scratch + n;
  const size_t sbase = ((size_t)b * a.hkv + h) * n;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    int slot = a.seg_slots[sbase + i];
    if (slot >= a.num_pages) slot = -1;  // num_pages: the cache's capacity here
    float w = 0.0f;
    if (slot >= 0) {
      const float* l2 = a.seg_l2 + (sbase + i) * G;
#pragma unroll
      for (int j = 0; j < G; j++) {
        const float v = __ldcg(l2 + j);
        if (v > kNeg) w += exp2f(v - lse2[j]);
      }
    }
    slot_s[i] = slot;
    w_s[i] = w;
  }
  __syncthreads();
  const int bs = S.n_sink - 1;                  // the sink's last segment, or -1
  const int bw = S.n_win > 0 ? S.n_sink : -1;   // the window's first segment, or -1
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int slot = slot_s[i];
    if (slot < 0) continue;
    const int owner = (bs >= 0 && slot_s[bs] == slot) ? bs
                      : (bw >= 0 && slot_s[bw] == slot) ? bw : i;
    if (owner != i) continue;
    float w = w_s[i];
    if (i == bs || i == bw) {
      w = 0.0f;
      for (int j = 0; j < n; j++)
        if (slot_s[j] == slot) w += w_s[j];
    }
    const int key = a.slot_key[slot] - 1;
    if (key >= 0) a.mass[key] += w;
  }
}

template <int G, int NB, bool MASS = false>
__device__ void finish_common(const AttArgs& a, int b, int h, int split, const float* o,
                              const float* m, const float* l, float* red, int nthreads) {
  const int tid = threadIdx.x;
  __shared__ int is_last;
  __shared__ float lse2[8];  // final log-sum-exp per head, log2 domain (cumulative-mass policy)
  const int hq = a.hkv * G;
  if (tid < nthreads) {
    for (int x = tid; x < G * kHeadDim; x += nthreads) {
      const int j = x / kHeadDim, d = x % kHeadDim;
      const size_t row = (size_t)b * hq + (size_t)h * G + j;
      const float L = l[j];
      if (a.nsplit == 1) {
        a.out[row * kHeadDim + d] = L > 0.0f ? o[x] / L : 0.0f;
        if (d == 0 && a.lse) a.lse[row] = L > 0.0f ? (m[j] + log2f(L)) * kLn2 : -INFINITY;
        if (MASS && d == 0) lse2[j] = L > 0.0f ? m[j] + log2f(L) : kNeg;
      } else {
        const size_t p = row * a.nsplit + split;
        a.part_o[p * kHeadDim + d] = o[x];
        if (d == 0) *reinterpret_cast<float2*>(a.part_ml + 2 * p) = make_float2(m[j], L);
      }
    }
  }
  if (a.nsplit == 1) {
    if (a.row_range != nullptr && tid == 0)
      *reinterpret_cast<uint4*>(a.row_range + ((size_t)b * a.hkv + h) * 4) = make_uint4(0, 0, 0, 0);
    if constexpr (MASS) {
      __syncthreads();
      add_segment_mass<G>(a, b, h, lse2, red);
    }
    return;
  }
  // One acquire-release increment by thread 0 between two CTA barriers: the first barrier
  // orders every thread's partial writes before the release, the second orders the last
  // CTA's reads of the other partials after the acquire (the pattern of a grid barrier).
  __syncthreads();
  if (tid == 0) {
    const int prev = atomic_add_acq_rel_gpu(&a.counters[(size_t)b * a.hkv + h], 1);
    is_last = prev == a.nsplit - 1;
  }
  __syncthreads();
  if (!is_last) return;
  // Two threads per (head, 4 channels), each taking one half of the splits: a thread loads
  // the (m, l) pairs and partial outputs of up to NB splits before it uses any (one round
  // trip per NB splits) and merges them online, keeping its state relative to the largest m
  // seen so far; then the two threads of a pair (adjacent lanes) merge their states. Both
  // 2 * G * 32 and the block size are multiples of 32, so every warp takes part in an
  // iteration with all its lanes or not at all.
  const int per = (a.nsplit + 1) >> 1;
  for (int x = tid; x < 2 * G * 32; x += blockDim.x) {
    const int it = x >> 1, half = x & 1;
    const int j = it >> 5, d4 = (it & 31) * 4;
    const size_t row = (size_t)b * hq + (size_t)h * G + j;
    const float2* ml = reinterpret_cast<const float2*>(a.part_ml) + row * a.nsplit;
    const float4* po = reinterpret_cast<const float4*>(a.part_o + row * a.nsplit * kHeadDim + d4);
    const int s_lo = half * per, s_hi = min(a.nsplit, s_lo + per);
    float M = kNeg, L = 0.0f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int sp0 = s_lo; sp0 < s_hi; sp0 += NB) {
      float2 mlv[NB];
      float4 ov[NB];
#pragma unroll
      for (int u = 0; u < NB; u++) {
        if (sp0 + u < s_hi) {
          mlv[u] = __ldcg(ml + sp0 + u);
          ov[u] = __ldcg(po + (size_t)(sp0 + u) * (kHeadDim / 4));
        } else {
          mlv[u] = make_float2(kNeg, 0.0f);
          ov[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int u = 0; u < NB; u++) {
        if (!(mlv[u].y > 0.0f)) continue;
        const float m_new = fmaxf(M, mlv[u].x);
        const float c = exp2f(M - m_new), w = exp2f(mlv[u].x - m_new);
        L = L * c + mlv[u].y * w;
        acc.x = acc.x * c + ov[u].x * w;
        acc.y = acc.y * c + ov[u].y * w;
        acc.z = acc.z * c + ov[u].z * w;
        acc.w = acc.w * c + ov[u].w * w;
        M = m_new;
      }
    }
    // the pair: a state with l = 0 has m = kNeg and contributes nothing
    const float Mo = __shfl_xor_sync(0xffffffffu, M, 1);
    const float Lo = __shfl_xor_sync(0xffffffffu, L, 1);
    float4 ao;
    ao.x = __shfl_xor_sync(0xffffffffu, acc.x, 1);
    ao.y = __shfl_xor_sync(0xffffffffu, acc.y, 1);
    ao.z = __shfl_xor_sync(0xffffffffu, acc.z, 1);
    ao.w = __shfl_xor_sync(0xffffffffu, acc.w, 1);
    if (half == 0) {
      const float Mn = fmaxf(M, Mo);
      const float c = L > 0.0f ? exp2f(M - Mn) : 0.0f;
      const float co = Lo > 0.0f ? exp2f(Mo - Mn) : 0.0f;
      L = L * c + Lo * co;
      acc.x = acc.x * c + ao.x * co;
      acc.y = acc.y * c + ao.y * co;
      acc.z = acc.z * c + ao.z * co;
      acc.w = acc.w * c + ao.w * co;
      const float inv = L > 0.0f ? 1.0f / L : 0.0f;
      *reinterpret_cast<float4*>(a.out + row * kHeadDim + d4) =
          make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
      if (d4 == 0 && a.lse) a.lse[row] = L > 0.0f ? (Mn + log2f(L)) * kLn2 : -INFINITY;
      if (MASS && d4 == 0) lse2[j] = L > 0.0f ? Mn + log2f(L) : kNeg;
    }
  }
  if constexpr (MASS) {
    __syncthreads();
    add_segment_mass<G>(a, b, h, lse2, red);
  }
  if (tid == 0) a.counters[(size_t)b * a.hkv + h] = 0;
  if (a.row_range != nullptr && tid == 0)
    *reinterpret_cast<uint4*>(a.row_range + ((size_t)b * a.hkv + h) * 4) = make_uint4(0, 0, 0, 0);
}

// Block-level state (host path): the two token halves merged into o[G][128]; m, l from the
// softmax warps. `red` holds at least G * 128 + 8 floats.
template <int G>
__device__ void finish(const AttArgs& a, State<G>& st, Scratch<head_slots(G)>& sc, int b, int h,
                       int split, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int d = (warp & 1) * 64 + 2 * lane;
  if (warp < kWarps && (warp >> 1) == 1) {
#pragma unroll
    for (int j = 0; j < G; j++) {
      red[j * kHeadDim + d] = st.acc[j][0];
      red[j * kHeadDim + d + 1] = st.acc[j][1];
    }
  }
#pragma unroll
  for (int i = 0; i < State<G>::kOwn; i++) {
    const int hh = warp + kWarps * i;
    if (hh < G && lane == 0) {
      sc.m[hh] = st.m[i];
      sc.l[hh] = st.l[i];
    }
  }
  __syncthreads();
  if (warp < kWarps && (warp >> 1) == 0) {
#pragma unroll
    for (int j = 0; j < G; j++) {
      red[j * kHeadDim + d] += st.acc[j][0];
      red[j * kHeadDim + d + 1] += st.acc[j][1];
    }
  }
  __syncthreads();
  finish_common<G, 8>(a, b, h, split, red, sc.m, sc.l, red, kCompute);
}

template <int G>
__device__ __forceinline__ void init_state(State<G>& st) {
#pragma unroll
  for (int j = 0; j < G; j++) st.acc[j][0] = st.acc[j][1] = 0.0f;
#pragma unroll
  for (int i = 0; i < State<G>::kOwn; i++) {
    st.m[i] = kNeg;
    st.l[i] = 0.0f;
  }
}

size_t red_floats(int G) {
  return std::max<size_t>((size_t)G * kHeadDim, (size_t)G * kMaxSplits + 8);
}

// ------------------------------------------------------------------ HBM path
//
// Warp-per-segment: compute warp w owns ring slots w, w + 4 and processes its segments
// start to finish on its own (no CTA barrier per segment), so four segments are in
// flight per CTA. Per segment: 4 rounds of (4 tokens x 8 lanes) give each lane the scores
// of tokens 4r + lane / 8 for head hidx(lane % 8); the per-head running max and sum are
// kept by every lane of that head; the weights go through the warp's own shared scratch
// to the value phase, where lane l owns channels 4l .. 4l + 3 of all G heads.

template <int H>
struct WarpScratch {
  float prob[kPage][H];  // weights of the segment's tokens, per head
  float rescale[H];      // factor applied to the running sums of each head
  float pad[4];
};

template <int G>
struct WarpState {
  float acc[G][4];  // weighted value sums: channels 4 lane .. 4 lane + 3, per head
  float m, l;       // running max / sum of head hidx (this lane's head)
};

// seg_out (nullable): receives the segment's log-sum-exp of the scaled scores (log2 domain)
// of each query head, m + log2(sum 2^(s - m)).
template <int G>
__device__ __forceinline__ void warp_segment(WarpState<G>& st, const float (&qf)[G][16],
                                             WarpScratch<head_slots(G)>& ws, uint32_t slot,
                                             int k, int t0, int t1, float* seg_out) {
  constexpr int H = head_slots(G);
  const int lane = threadIdx.x & 31;
  const int g = lane >> 3, sl = lane & 7;
  float sc[4];
  int hidx = 0;
#pragma unroll
  for (int it = 0; it < 4; it++) {
    const int r = 4 * it + g;
    const uint32_t kb = slot + r * (kHeadDim * 2);
    const uint4 k0 = lds128(kb + sl * 16), k1 = lds128(kb + (sl + 8) * 16);
    float kf[16];
    unpack16(k0, k1, kf);
    float v[G];
#pragma unroll
    for (int j = 0; j < G; j++) {
      float acc = 0.0f;
#pragma unroll
      for (int e = 0; e < 16; e++) acc = fmaf(qf[j][e], kf[e], acc);
      v[j] = acc;
    }
    const float s = reduce_scores<G>(v, sl, hidx);
    const int t = k * kPage + r;
    sc[it] = (t >= t0 && t < t1) ? s : kNeg;
  }
  // softmax of the segment for head hidx: max and sum over the 4 token groups
  float bm = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
  bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 8));
  bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 16));
  const float m_new = fmaxf(st.m, bm);
  const float c = exp2f(st.m - m_new);
  float p[4], ps = 0.0f;
#pragma unroll
  for (int it = 0; it < 4; it++) {
    p[it] = sc[it] == kNeg ? 0.0f : exp2f(sc[it] - m_new);
    ps += p[it];
  }
  ps += __shfl_xor_sync(0xffffffffu, ps, 8);
  ps += __shfl_xor_sync(0xffffffffu, ps, 16);
  st.l = st.l * c + ps;
  st.m = m_new;
  constexpr int kOwners = 8 / G;  // lanes of a group holding the same head; the first writes
  if (seg_out != nullptr && g == 0 && (sl & (kOwners - 1)) == 0)
    seg_out[hidx] = ps > 0.0f ? m_new + log2f(ps) : kNeg;
  if ((sl & (kOwners - 1)) == 0) {
#pragma unroll
    for (int it = 0; it < 4; it++) ws.prob[4 * it + g][hidx] = p[it];
    if (g == 0) ws.rescale[hidx] = c;
  }
  __syncwarp();
  // values: lane owns channels 4 lane .. 4 lane + 3
  float cj[H];
#pragma unroll
  for (int q4 = 0; q4 < H / 4; q4++) {
    const float4 c4 = *reinterpret_cast<const float4*>(&ws.rescale[4 * q4]);
    cj[4 * q4] = c4.x;
    cj[4 * q4 + 1] = c4.y;
    cj[4 * q4 + 2] = c4.z;
    cj[4 * q4 + 3] = c4.w;
  }
#pragma unroll
  for (int j = 0; j < G; j++)
#pragma unroll
    for (int e = 0; e < 4; e++) st.acc[j][e] *= cj[j];
  const uint32_t vb = slot + kBlockBytesBf16 + lane * 8;
#pragma unroll 4
  for (int r = 0; r < kPage; r++) {
    const int t = k * kPage + r;
    if (t < t0 || t >= t1) continue;  // warp-uniform; skipped slots may hold any bits
    uint32_t w0, w1;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(w0), "=r"(w1) : "r"(vb + r * kHeadDim * 2));
    const float vf[4] = {bf16_lo(w0), bf16_hi(w0), bf16_lo(w1), bf16_hi(w1)};
    float pj[H];
#pragma unroll
    for (int q4 = 0; q4 < H / 4; q4++) {
      const float4 p4 = *reinterpret_cast<const float4*>(&ws.prob[r][4 * q4]);
      pj[4 * q4] = p4.x;
      pj[4 * q4 + 1] = p4.y;
      pj[4 * q4 + 2] = p4.z;
      pj[4 * q4 + 3] = p4.w;
    }
#pragma unroll
    for (int j = 0; j < G; j++)
#pragma unroll
      for (int e = 0; e < 4; e++) st.acc[j][e] = fmaf(pj[j], vf[e], st.acc[j][e]);
  }
  __syncwarp();  // the next segment rewrites the scratch
}

// The W compute warps' running states merged into one per head (o[j][d] = sum over warps of
// acc_w * 2^(m_w - M_j), l likewise), then the CTA's output or split partial and the combine
// (finish_common). Called by all threads after a CTA barrier; `ring` (the K/V ring, no
// longer in use) holds the merge area, `mstate` [2][W][H] floats.
template <int G, int W, int NB, bool MASS>
__device__ __forceinline__ void merge_warps(const AttArgs& a, const WarpState<G>& st,
                                            uint8_t* ring, float* mstate, int b, int h,
                                            int split) {
  constexpr int H = head_slots(G);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // merge the warps: o[j][d] = sum_w acc_w * 2^(m_w - M_j), l likewise
  float* o = reinterpret_cast<float*>(ring);  // [W][G][128], then the merged [G][128]
  float* mw = mstate;                          // [W][H] max, then [W][H] sum
  float* lw = mstate + W * H;
  if (warp < W) {
    const int sl = lane & 7;
    constexpr int kOwners = 8 / G;
    int hidx = 0;
    if constexpr (G == 8) hidx = sl;
    if constexpr (G == 4) hidx = ((sl & 4) ? 2 : 0) + ((sl & 2) ? 1 : 0);
    if constexpr (G == 2) hidx = (sl & 4) ? 1 : 0;
    if (lane < 8 && (sl & (kOwners - 1)) == 0) {
      mw[warp * H + hidx] = st.m;
      lw[warp * H + hidx] = st.l;
    }
#pragma unroll
    for (int j = 0; j < G; j++)
      *reinterpret_cast<float4*>(o + (warp * G + j) * kHeadDim + 4 * lane) =
          make_float4(st.acc[j][0], st.acc[j][1], st.acc[j][2], st.acc[j][3]);
  }
  __syncthreads();
  float* mo = o + W * G * kHeadDim;  // merged [G][128]
  float* mm = mo + G * kHeadDim;          // [H]
  float* ml = mm + H;                     // [H]
  if (tid < W * 32) {
    for (int x = tid; x < G * kHeadDim; x += W * 32) {
      const int j = x / kHeadDim, d = x % kHeadDim;
      float M = kNeg;
#pragma unroll
      for (int w = 0; w < W; w++) M = fmaxf(M, mw[w * H + j]);
      float O = 0.0f, L = 0.0f;
#pragma unroll
      for (int w = 0; w < W; w++) {
        const float lv = lw[w * H + j];
        const float wt = lv > 0.0f ? exp2f(mw[w * H + j] - M) : 0.0f;
        O = fmaf(o[(w * G + j) * kHeadDim + d], wt, O);
        L = fmaf(lv, wt, L);
      }
      mo[x] = O;
      if (d == 0) {
        mm[j] = M;
        ml[j] = L;
      }
    }
  }
  __syncthreads();
  finish_common<G, NB, MASS>(a, b, h, split, mo, mm, ml, o, W * 32);
}

// W compute warps and NS ring slots (NS a multiple of W): the sparse path uses 8 warps and 16
// slots, enough for every segment of a CTA to be in flight at once; dense decode uses 4 and 8
// with three CTAs per SM.
// MASS: the block cache's cumulative-mass policy (a.seg_l2 set): every segment's log-sum-exp
// per head is written out for the combine, which adds the segments' attention mass.
template <int G, bool DENSE, int W, int NS, bool MASS>
__global__ void __launch_bounds__((W + 1) * 32, (W == 4 && G <= 4 ? 3 : 1))
    attend_tma_kernel(const AttArgs a) {
  static_assert(NS % W == 0, "each compute warp owns fixed ring slots");
  constexpr int H = head_slots(G);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + NS * kSlotBytes);
  uint64_t* empty = full + NS;
  WarpScratch<H>* wscr = reinterpret_cast<WarpScratch<H>*>(empty + NS);  // [W]
  float* mstate = reinterpret_cast<float*>(wscr + W);                    // [W][2][H]
  int4* meta = reinterpret_cast<int4*>(mstate + 2 * W * H);              // [NS] (k, t0, t1)

  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // Early mode: only the kept blocks come from the previous kernel; the producer waits for
  // it just before its first kept block. Otherwise every input may, so wait first.
  if (!a.early) grid_dep_wait();
  grid_dep_launch();
  const int n_raw = a.seq_lens[b];
  if (tid == 0 && split == 0 && h == 0 && (n_raw < 0 || n_raw > a.max_pages * kPage))
    set_error(a.err, kDevErrCheck);
  Segments S = make_segments<DENSE>(a, b, h);
  // The CTA's segments, local index j -> segment first + j * stride. Sparse attend deals the
  // list out round-robin, so that the kept blocks (known last) are spread over every CTA of
  // (b, h); dense decode takes a contiguous range of pages.
  int first, stride, cnt;
  if (DENSE) {
    first = (int)((long long)S.total * split / a.nsplit);
    cnt = (int)((long long)S.total * (split + 1) / a.nsplit) - first;
    stride = 1;
  } else {
    first = split;
    stride = a.nsplit;
    cnt = S.total > split ? (S.total - split + a.nsplit - 1) / a.nsplit : 0;
  }
  // local segments [0, n_pre) are sink or window pages: they need no selection
  const int n_sw = S.n_sink + S.n_win;
  const int n_pre = n_sw <= first ? 0 : min(cnt, (n_sw - first + stride - 1) / stride);

  if (tid == 0) {
    for (int s = 0; s < NS; s++) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);  // the slot's owning warp
    }
    fence_barrier_init();
  }
  __syncthreads();

  WarpState<G> st;
#pragma unroll
  for (int j = 0; j < G; j++)
#pragma unroll
    for (int e = 0; e < 4; e++) st.acc[j][e] = 0.0f;
  st.m = kNeg;
  st.l = 0.0f;
  if (warp == W) {
    // producer warp: the lanes resolve the block and page ids of 32 segments at once; lane 0
    // then publishes each segment's (block, t0, t1) with its slot and issues the copies
    bool ok = true, have_sel = false;
    const uint64_t policy = l2_evict_first_policy();  // each K/V page is read once
    for (int jb = 0; ok && jb < cnt;) {
      // batches of up to 32 segments, none straddling n_pre: the sink and window pages are
      // fetched before the wait for the selection
      const int jend = jb < n_pre ? min(n_pre, jb + 32) : min(cnt, jb + 32);
      if (!have_sel && jb >= n_pre) {
        grid_dep_wait();  // the kept blocks come from the previous kernel
        have_sel = true;
      }
      int k = 0, t0 = 0, t1 = 0, page = -1;
      if (jb + lane < jend) {
        const int i = first + (jb + lane) * stride;
        const size_t sbase = ((size_t)b * a.hkv + h) * a.seg_stride;
        if (i < n_sw) {
          segment_at(S, i, a.sink, k, t0, t1);
          if (t0 < t1)
            page = a.seg_slots ? a.seg_slots[sbase + i] : a.page_table[(size_t)b * a.max_pages + k];
        } else {
          // a kept block: the count of kept blocks, its id and (when given) its page, all in
          // one round trip (both lists hold K2 entries; r < K2)
          const int r = i - n_sw;
          const size_t at = ((size_t)b * a.hkv + h) * a.k2 + r;
          const int nb = a.n_blocks[(size_t)b * a.hkv + h];
          const int kk = a.block_idx[at];
          const int pp = a.seg_slots ? a.seg_slots[sbase + i] : (a.sel_pages ? a.sel_pages[at] : -1);
          S.n_sel = max(0, min(nb, S.n_sel_max));
          kept_segment(S, r, kk, a.sink, k, t0, t1);
          if (t0 < t1)
            page = (a.seg_slots || a.sel_pages) ? pp : a.page_table[(size_t)b * a.max_pages + k];
        }
        if (t0 < t1 && (page < 0 || page >= a.num_pages)) {
          set_error(a.err, kDevErrCheck);
          page = -1;
        }
        if (page < 0) t0 = t1 = 0;
      }
      const int n = jend - jb;
      // A copy of segment j goes to ring slot j % NS once that slot's previous segment is
      // done. While a sparse batch uses every slot for the first time (no waits), each lane
      // issues its own segment's copies, all lanes at once; otherwise lane 0 issues them in
      // order, waiting for slots as they free up (dense decode always: its long contiguous
      // ranges never fit the ring, and the extra path measurably slowed it).
      if (!DENSE && jend <= NS) {
        if (lane < n) {
          const int s = jb + lane;
          meta[s] = make_int4(k, t0, t1, 0);
          if (page >= 0) {
            const size_t off = a.seg_slots ? (size_t)page * (2 * kPage * kHeadDim)
                                           : ((size_t)page * a.kv_heads + h / a.kv_div) *
                                                 kPage * kHeadDim;
            mbar_arrive_expect_tx(&full[s], kSlotBytes);
            bulk_load_hint(ring + s * kSlotBytes, a.k + off, kBlockBytesBf16, &full[s], policy);
            bulk_load_hint(ring + s * kSlotBytes + kBlockBytesBf16, a.v + off, kBlockBytesBf16,
                           &full[s], policy);
          } else {
            mbar_arrive(&full[s]);
          }
        }
        jb = jend;
        continue;
      }
      for (int q = 0; q < n; q++) {
        const int kq = __shfl_sync(0xffffffffu, k, q);
        const int t0q = __shfl_sync(0xffffffffu, t0, q);
        const int t1q = __shfl_sync(0xffffffffu, t1, q);
        const int pq = __shfl_sync(0xffffffffu, page, q);
        if (lane == 0) {
          const int j = jb + q, s = j % NS;
          if (j >= NS && !mbar_wait(&empty[s], ((j / NS) - 1) & 1)) {
            set_error(a.err, kDevErrTimeout);
            ok = false;
          } else {
            meta[s] = make_int4(kq, t0q, t1q, 0);
            if (pq >= 0) {
              // a page of the cache, or one slot (K block then V block) of the block cache
              const size_t off = a.seg_slots ? (size_t)pq * (2 * kPage * kHeadDim)
                                             : ((size_t)pq * a.kv_heads + h / a.kv_div) *
                                                   kPage * kHeadDim;
              mbar_arrive_expect_tx(&full[s], kSlotBytes);
              bulk_load_hint(ring + s * kSlotBytes, a.k + off, kBlockBytesBf16, &full[s], policy);
              bulk_load_hint(ring + s * kSlotBytes + kBlockBytesBf16, a.v + off, kBlockBytesBf16,
                             &full[s], policy);
            } else {
              mbar_arrive(&full[s]);
            }
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
      }
      jb = jend;
    }
    if (!ok && lane == 0) {
      const int issued = cnt;
      for (int j = max(0, issued - NS); j < issued; j++) mbar_wait(&full[j % NS], (j / NS) & 1);
    }
  } else {
    float qf[G][16];
    load_query<G>(qf, a, b, h, lane & 7);
    for (int j = warp; j < cnt; j += W) {
      const int s = j % NS;
      if (!mbar_wait(&full[s], (j / NS) & 1)) {
        set_error(a.err, kDevErrTimeout);
        break;
      }
      const int4 m4 = meta[s];  // written before the producer's arrive on full[s]
      float* seg_out = nullptr;
      if constexpr (MASS)
        seg_out = a.seg_l2 + (((size_t)b * a.hkv + h) * a.seg_stride + first + j * stride) * G;
      if (m4.y < m4.z)
        warp_segment<G>(st, qf, wscr[warp], smem_addr(ring + s * kSlotBytes), m4.x, m4.y, m4.z,
                        seg_out);
      else if (MASS && lane < G)
        seg_out[lane] = kNeg;  // no token: no mass
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
  }
  grid_dep_wait();  // completion of this grid implies completion of the previous one
  __syncthreads();
  merge_warps<G, W, DENSE ? 8 : 16, MASS>(a, st, ring, mstate, b, h, split);
}

// ------------------------------------ sparse attention that runs the pruning modules itself
//
// The whole decode step's sparse attention for 64-token chunks: every CTA of (sequence b,
// row h) runs both pruning modules on the scorer's tile maxima (the chunk scores) and block
// maxima itself, so neither a pruning kernel nor a round trip for its kept-block list stands
// between the scorer and the attention. The CTAs of a row take the same deterministic steps
// on the same data and agree on the selection; split 0 writes it out for the caller.
//
// Order inside a CTA: the sink and window pages (inputs of the step, except the page that
// holds the newest token, which the append beside the scorer writes) are copied before the
// wait for the scorer, and so is the row of page ids when it fits; after the wait the tile
// maxima (and the row of block maxima when it fits) are staged, all warps select (module 1:
// top-K1 chunks; module 2: top-K2 blocks of those chunks; select.cuh's three-barrier path
// on the value range the scorer recorded, its general path otherwise), the producer issues
// the kept blocks' copies, and the compute warps process the CTA's segments as in the HBM
// path above. The last CTA of a row clears the row's range words for the next step.
struct SelArgs {
  const int32_t* block_max;  // [rows][max_pages]
  const int32_t* tile_max;   // [rows][max_tiles]
  int32_t* block_idx;        // [rows][k2] out (split 0): kept blocks ascending, -1 padded
  int32_t* n_blocks;         // [rows] out (split 0)
  const unsigned* row_range;  // [rows][4] the scorer's range of each row's maxima
  int max_tiles, k1;
  int a_cap;   // ints of area A: the tile maxima, then module 2's values and block ids
  int n2_cap;  // module 2's candidates (4 blocks per kept chunk)
  int k1_cap, k2_cap;
  int row_cap;   // > 0: the row of block maxima is staged (ints)
  int prow_cap;  // > 0: the row of page ids is staged (ints)
};

// Byte offsets of the kernel's dynamic shared memory (after 128-byte alignment).
struct SelSmem {
  size_t full, sbar, wscr, mstate, meta, ss, area, kept1, selb, selp, brow, prow, end;
};

template <int G, int W, int NS>
__host__ __device__ SelSmem sel_smem_layout(const SelArgs& sa) {
  constexpr int H = head_slots(G);
  SelSmem l;
  size_t o = (size_t)NS * kSlotBytes;  // the K/V ring
  l.full = o;                          // full [NS], empty [NS]
  o += 2 * NS * sizeof(uint64_t);
  l.sbar = o;  // staging barriers: tile maxima, block-maxima row, page row
  o += 4 * sizeof(uint64_t);
  l.wscr = o;
  o += W * sizeof(WarpScratch<H>);
  l.mstate = o;
  o += 2 * W * H * sizeof(float);
  o = (o + 15) / 16 * 16;
  l.meta = o;
  o += NS * sizeof(int4);
  l.ss = o;
  o += (sizeof(SelectShared) + 15) / 16 * 16;
  l.area = o;
  o += (size_t)sa.a_cap * 4;
  l.kept1 = o;
  o += (size_t)sa.k1_cap * 4;
  l.selb = o;
  o += (size_t)sa.k2_cap * 4;
  l.selp = o;
  o += (size_t)sa.k2_cap * 4;
  l.brow = o;
  o += sa.row_cap > 0 ? ((size_t)sa.row_cap + 4) * 4 : 0;
  l.prow = o;
  o += sa.prow_cap > 0 ? ((size_t)sa.prow_cap + 4) * 4 : 0;
  l.end = o;
  return l;
}

// The kept blocks of a row when K1 >= K2, by NT threads (all of the CTA). The two modules
// then keep the top K2 blocks of the candidate region (ranked by maximum, the lower index
// first among equals), and T1, the K2-th largest chunk maximum, bounds them from below: the
// top K2 chunks each hold a block equal to their maximum, so at least K2 blocks reach T1.
// Steps: T1 by the register histogram of the chunk maxima (values in [t_min, t_max]; two CTA
// barriers); the blocks >= T1 (only chunks >= T1 hold one) written in ascending order to
// cv / ci (values / ids; cap entries); the n_c - K2 lowest ranked of them (usually a few)
// taken one a round by warp 0, every kept block then written to its place in selb
// (ascending: its index among the candidates minus the dropped ones before it); with more
// than kPeel to drop, the selection of select.cuh over the candidates (values in
// [T1, vmax]). The kept blocks' pages go to selp (prow staged, else -1). Returns K2, or -1
// with nothing written (fhist and n_cand left zero) when the row needs the general modules:
// K2 or fewer valid chunks, a bin of the K2-th value wider than kSelSmall, or more than cap
// candidates. The same value in every thread.
template <int NT, int R, int P>
__device__ __forceinline__ int sel_blocks_over_threshold(const int* tiles, int n1, int c_lo,
                                                         const int* brow, int k_lo, int k_hi,
                                                         int K2, int t_min, int t_max, int vmax,
                                                         const int* prow, int* cv, int* ci,
                                                         int cap, SelectShared& ss, int* selb,
                                                         int* selp, const __nv_bfloat16* k_head,
                                                         const __nv_bfloat16* v_head,
                                                         size_t page_elems, int num_pages,
                                                         int split, int nsplit) {
  constexpr int kW = NT / 32;
  constexpr int kPeel = 8;  // at most this many dropped candidates are taken one a round
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned umin = (unsigned)t_min;
  const int shift = fast_shift(t_min, t_max);
  const int per = (n1 + NT - 1) / NT;  // <= R (checked by the caller)
  const int x0 = min(n1, tid * per), nv = min(n1, x0 + per) - x0;
  int v[R];
#pragma unroll
  for (int r = 0; r < R; r++) v[r] = r < nv ? tiles[x0 + r] : INT_MIN;
  int valid = 0;
#pragma unroll
  for (int r = 0; r < R; r++)
    if (v[r] != INT_MIN) {
      valid++;
      sel_red_add(&ss.fhist[fast_bin(v[r], umin, shift)], 1u);
    }
  const int vw = __reduce_add_sync(0xffffffffu, valid);
  if (lane == 0) ss.wsum[warp] = vw;
  __syncthreads();
  int n_valid = 0;
#pragma unroll
  for (int w = 0; w < kW; w++) n_valid += ss.wsum[w];
  int3 loc = make_int3(0, 0, 0);
  if (n_valid > K2) loc = fast_locate(ss.fhist, K2);
  if (n_valid <= K2 || loc.z > kSelSmall) {
    __syncthreads();  // every warp has read the histogram
    for (int i = tid; i < kFastBins; i += NT) ss.fhist[i] = 0u;
    __syncthreads();
    return -1;
  }
  // T1: the (K2 - above)-th largest value of the located bin, ranked by every warp
  const int d = loc.x, above = loc.y, cnt = loc.z;
#pragma unroll
  for (int r = 0; r < R; r++)
    if (v[r] != INT_MIN && fast_bin(v[r], umin, shift) == d) {
      const int slot = sel_atom_add(&ss.n_cand, 1);
      if (slot < kSelSmall) ss.cand[slot] = v[r];
    }
  __syncthreads();
  int T1;
  {
    const int c = lane < cnt ? ss.cand[lane] : INT_MIN;
    int gtc = 0, gec = 0;
    for (int j = 0; j < cnt; j++) {
      const int cj = __shfl_sync(0xffffffffu, c, j);
      gtc += cj > c ? 1 : 0;
      gec += cj >= c ? 1 : 0;
    }
    const int need = K2 - above;
    const int L = __ffs(__ballot_sync(0xffffffffu, lane < cnt && gtc < need && need <= gec)) - 1;
    T1 = __shfl_sync(0xffffffffu, c, L);
  }
  // the candidates: blocks >= T1 of the thread's chunks, counted, then placed in order
  int nc = 0;
#pragma unroll
  for (int r = 0; r < R; r++)
    if (v[r] >= T1 && v[r] != INT_MIN) {
#pragma unroll
      for (int q = 0; q < P; q++) {
        const int kk = (c_lo + x0 + r) * P + q;
        if (kk >= k_lo && kk < k_hi && brow[kk - k_lo] >= T1) nc++;
      }
    }
  int incl = nc;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  if (lane == 31) ss.w_a[warp] = incl;
  for (int i = tid; i < kFastBins; i += NT) ss.fhist[i] = 0u;  // read by every warp above
  if (tid == 0) ss.n_cand = 0;
  __syncthreads();
  int n_c = 0, base = 0;
#pragma unroll
  for (int w = 0; w < kW; w++) {
    n_c += ss.w_a[w];
    base += w < warp ? ss.w_a[w] : 0;
  }
  const int drop = n_c - K2;  // >= 0: the K2 chunks above T1 each hold one
  if (n_c > cap) return -1;  // nothing written; fhist and n_cand zero
  int pos = base + incl - nc;
#pragma unroll
  for (int r = 0; r < R; r++)
    if (v[r] >= T1 && v[r] != INT_MIN) {
#pragma unroll
      for (int q = 0; q < P; q++) {
        const int kk = (c_lo + x0 + r) * P + q;
        if (kk >= k_lo && kk < k_hi) {
          const int bv = brow[kk - k_lo];
          if (bv >= T1) {
            cv[pos] = bv;
            ci[pos] = kk;
            pos++;
          }
        }
      }
    }
  __syncthreads();
  // the kept blocks are among the candidates: warm L2 with their K and V pages now (the row's
  // CTAs split them by index), so that the copies issued after the selection hit L2
  if (HSA_SEL_PREFETCH && prow != nullptr) {
    for (int i = split + tid * nsplit; i < n_c; i += NT * nsplit) {
      const int page = prow[ci[i] - k_lo];
      if (page < 0 || page >= num_pages) continue;  // reported when the copy is resolved
      const size_t off = (size_t)page * page_elems;
      bulk_prefetch_l2(k_head + off, kBlockBytesBf16);
      bulk_prefetch_l2(v_head + off, kBlockBytesBf16);
    }
  }
  if (drop > kPeel) {
    // many to drop: the register selection over the candidates (ids written in order), else
    // the radix select and ordered collect (positions among the candidates)
    int got = sel_fast_row<NT, R>(SelRow{cv, ci, 0}, n_c, K2, T1, vmax, ss, selb);
    if (got < 0) {
      const int3 r3 = sel_kth_largest<NT>(cv, n_c, K2, ss, true, T1, vmax);
      got = sel_collect<NT>(cv, n_c, r3.x, r3.y, r3.z, ss, selb, 0);
      for (int i = tid; i < got; i += NT) selb[i] = ci[selb[i]];
    }
    for (int i = tid; i < K2; i += NT) selp[i] = prow != nullptr ? prow[selb[i] - k_lo] : -1;
    __syncthreads();
    return K2;
  }
  // a few to drop: the lowest ranked, taken one a round by warp 0
  if (drop > 0 && warp == 0) sel_peel_lowest(cv, n_c, drop, ss.cand_i);
  if (drop > 0) __syncthreads();
  // every kept candidate's place: its index minus the dropped ones before it
  for (int i = tid; i < n_c; i += NT) {
    int before = 0;
    bool dropped = false;
    for (int e = 0; e < drop; e++) {
      const int de = ss.cand_i[e];
      before += de < i ? 1 : 0;
      dropped = dropped || de == i;
    }
    if (!dropped) {
      const int kk = ci[i];
      selb[i - before] = kk;
      selp[i - before] = prow != nullptr ? prow[kk - k_lo] : -1;
    }
  }
  __syncthreads();  // every thread has read the dropped list
  if (tid == 0) ss.n_cand = 0;
  return K2;
}

template <int G, int W, int NS>
__global__ void __launch_bounds__((W + 1) * 32, 1)
    attend_select_kernel(const AttArgs a, const SelArgs sa) {
  static_assert(NS % W == 0 && NS <= 32, "each compute warp owns fixed ring slots; one batch");
  constexpr int NT = (W + 1) * 32;
  constexpr int P = kTileBlocksSel;  // blocks per 64-token chunk
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  const SelSmem L = sel_smem_layout<G, W, NS>(sa);
  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.full);
  uint64_t* empty = full + NS;
  uint64_t* sbar = reinterpret_cast<uint64_t*>(smem + L.sbar);
  WarpScratch<head_slots(G)>* wscr = reinterpret_cast<WarpScratch<head_slots(G)>*>(smem + L.wscr);
  float* mstate = reinterpret_cast<float*>(smem + L.mstate);
  int4* meta = reinterpret_cast<int4*>(smem + L.meta);
  SelectShared& ss = *reinterpret_cast<SelectShared*>(smem + L.ss);
  int* area = reinterpret_cast<int*>(smem + L.area);
  int* kept1 = reinterpret_cast<int*>(smem + L.kept1);
  int* selb = reinterpret_cast<int*>(smem + L.selb);
  int* selp = reinterpret_cast<int*>(smem + L.selp);

  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  grid_dep_launch();
  const int n_raw = a.seq_lens[b];
  const bool bad_len = n_raw < 0 || n_raw > a.max_pages * kPage;
  if (tid == 0 && split == 0 && h == 0 && bad_len) set_error(a.err, kDevErrCheck);
  Segments S = make_segments<false>(a, b, h);
  const int first = split, stride = a.nsplit;
  const int cnt = S.total > split ? (S.total - split + stride - 1) / stride : 0;
  const int n_sw = S.n_sink + S.n_win;
  const int n_pre = n_sw <= first ? 0 : min(cnt, (n_sw - first + stride - 1) / stride);
  // the page of the newest token is written by the append running beside the scorer: its
  // copy waits for the scorer (whose completion the append's waits for)
  const int i_last = S.n_win > 0 ? n_sw - 1 : (S.n_sink > 0 && S.sink_end == S.n ? S.n_sink - 1 : -1);
  const int j_def = (i_last >= first && (i_last - first) % stride == 0) ? (i_last - first) / stride : -1;
  const int jA = min(n_pre, NS);  // local segments [0, jA) but j_def go out before the wait

  // candidate region in blocks and chunks
  int k_lo = 0, k_hi = 0, c_lo = 0, n1 = 0;
  if (S.cand_hi > a.sink && !bad_len) {
    k_lo = a.sink / kPage;
    k_hi = (S.cand_hi + kPage - 1) / kPage;
    c_lo = k_lo / P;
    n1 = (k_hi + P - 1) / P - c_lo;
  }
  const size_t row = (size_t)b * a.hkv + h;
  const bool use_row = sa.row_cap > 0;
  const bool use_prow = sa.prow_cap > 0;
  const StagedRow t_plan = plan_row(area, sa.tile_max + row * sa.max_tiles + c_lo, n1);
  const StagedRow r_plan =
      plan_row(reinterpret_cast<int*>(smem + L.brow), sa.block_max + row * a.max_pages + k_lo,
               use_row ? k_hi - k_lo : 0);
  const StagedRow p_plan =
      plan_row(reinterpret_cast<int*>(smem + L.prow), a.page_table + (size_t)b * a.max_pages + k_lo,
               use_prow ? k_hi - k_lo : 0);

  if (tid == 0) {
    for (int s = 0; s < NS; s++) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < 3; s++) mbar_init(&sbar[s], 1);
    fence_barrier_init();
  }
  sel_init<NT>(ss);
  __syncthreads();

  const uint64_t policy = l2_evict_first_policy();  // each K/V page is read once
  auto issue = [&](int s, int page) {  // the K and V pages of one segment into ring slot s
    if (page >= 0) {
      const size_t off = ((size_t)page * a.kv_heads + h / a.kv_div) * kPage * kHeadDim;
      mbar_arrive_expect_tx(&full[s], kSlotBytes);
      bulk_load_hint(ring + s * kSlotBytes, a.k + off, kBlockBytesBf16, &full[s], policy);
      bulk_load_hint(ring + s * kSlotBytes + kBlockBytesBf16, a.v + off, kBlockBytesBf16, &full[s],
                     policy);
    } else {
      mbar_arrive(&full[s]);
    }
  };
  // segment i of the CTA's rows: (k, t0, t1) and its page (-1: nothing to read)
  auto resolve = [&](int i, int& k, int& t0, int& t1) -> int {
    int page = -1;
    if (i < n_sw) {
      segment_at(S, i, a.sink, k, t0, t1);
      if (t0 < t1) page = __ldg(a.page_table + (size_t)b * a.max_pages + k);
    } else {
      kept_segment(S, i - n_sw, i - n_sw < S.n_sel ? selb[i - n_sw] : -1, a.sink, k, t0, t1);
      if (t0 < t1)
        page = use_prow ? selp[i - n_sw] : __ldg(a.page_table + (size_t)b * a.max_pages + k);
    }
    if (t0 < t1 && (page < 0 || page >= a.num_pages)) {
      set_error(a.err, kDevErrCheck);
      page = -1;
    }
    if (page < 0) t0 = t1 = 0;
    return page;
  };

  // ---- before the wait: the page row (an input) and the sink / window copies
  // the deferred segment is resolved here too (only its copy waits), by lane j_def
  int def_k = 0, def_t0 = 0, def_t1 = 0, def_page = -1;
  if (warp == W) {
    if (lane == 0 && use_prow && p_plan.bytes() > 0) {
      mbar_arrive_expect_tx(&sbar[2], p_plan.bytes());
      issue_row(p_plan, &sbar[2]);
    }
    if (lane < jA) {
      int k = 0, t0 = 0, t1 = 0;
      const int page = resolve(first + lane * stride, k, t0, t1);
      if (lane != j_def) {
        meta[lane] = make_int4(k, t0, t1, 0);
        issue(lane, page);
      } else {
        def_k = k;
        def_t0 = t0;
        def_t1 = t1;
        def_page = page;
      }
    }
  }
  if (use_prow) tail_row<NT>(p_plan);

  grid_dep_wait();  // the scorer's maxima and the appended token are complete

  // ---- stage the chunk scores (and the row of block maxima)
  if (tid == 0) {
    if (t_plan.bytes() > 0) {
      mbar_arrive_expect_tx(&sbar[0], t_plan.bytes());
      issue_row(t_plan, &sbar[0]);
    }
    if (use_row && r_plan.bytes() > 0) {
      mbar_arrive_expect_tx(&sbar[1], r_plan.bytes());
      issue_row(r_plan, &sbar[1]);
    }
  }
  // the row's range of tile and block maxima, recorded by the scorer (zero: none)
  const uint4 rr = __ldcg(reinterpret_cast<const uint4*>(sa.row_range) + row);
  const int t_max = (int)(rr.x ^ 0x80000000u), t_min = (int)(~rr.y ^ 0x80000000u);
  const int b_max = (int)(rr.z ^ 0x80000000u), b_min = (int)(~rr.w ^ 0x80000000u);
  tail_row<NT>(t_plan);
  if (use_row) tail_row<NT>(r_plan);
  if (t_plan.bytes() > 0 && !mbar_wait(&sbar[0], 0)) set_error(a.err, kDevErrTimeout);
  __syncthreads();  // the plain-load tails are visible

  const int* tiles = t_plan.dst();
  const int* brow = r_plan.dst();
  const int* prow = p_plan.dst();
  constexpr int kRegVals = kSelRegVals;
  // ---- K1 >= K2 (module 1 keeps K2 chunks): the blocks at or above the K2-th chunk maximum
  int got2 = -1;
  bool ids = false;  // selb holds block ids (fast path) rather than positions in cand2
  bool mapped = false;  // selb / selp hold the kept blocks' ids and pages
  if (HSA_SEL_THRESHOLD && sa.k1 >= a.k2 && a.k2 > 0 && use_row && n1 > 0 &&
      n1 <= kRegVals * NT && rr.x != 0u && rr.y != 0u && rr.z != 0u && rr.w != 0u) {
    bool ok = true;
    if (r_plan.bytes() > 0 && !mbar_wait(&sbar[1], 0)) ok = false;
    if (use_prow && p_plan.bytes() > 0 && !mbar_wait(&sbar[2], 0)) ok = false;
    if (!ok) set_error(a.err, kDevErrTimeout);
    got2 = sel_blocks_over_threshold<NT, kRegVals, P>(
        tiles, n1, c_lo, brow, k_lo, k_hi, a.k2, t_min, t_max, b_max, use_prow ? prow : nullptr,
        area, area + sa.n2_cap, sa.n2_cap, ss, selb, selp,
        a.k + (size_t)(h / a.kv_div) * kPage * kHeadDim,
        a.v + (size_t)(h / a.kv_div) * kPage * kHeadDim, (size_t)a.kv_heads * kPage * kHeadDim,
        a.num_pages, split, a.nsplit);
    mapped = got2 >= 0;
  }
  if (!mapped) {
  // ---- module 1: top-K1 chunks (ascending); the fast path when the scorer's range is known
  int got1 = -1;
  const int keep1 = min(sa.k1, n1);
  if (n1 > 0 && n1 <= kRegVals * NT && rr.x != 0u && rr.y != 0u)
    got1 = sel_fast_row<NT, kRegVals>(SelRow{tiles, nullptr, c_lo}, n1, sa.k1, t_min, t_max, ss,
                                      kept1);
  if (got1 < 0) {
    got1 = 0;
    if (keep1 > 0) {
      int T = INT_MIN, need_eq = 0, eq_total = 0;
      if (keep1 < n1) {
        const int3 r = sel_kth_largest<NT>(tiles, n1, keep1, ss, false, 0, 0);
        T = r.x;
        need_eq = r.y;
        eq_total = r.z;
      }
      got1 = sel_collect<NT>(tiles, n1, T, need_eq, eq_total, ss, kept1, c_lo);
    }
  }

  // ---- module 2: the kept chunks' blocks (outside the candidate region: placeholders never
  // kept), top-K2, ascending
  if (use_row && r_plan.bytes() > 0 && !mbar_wait(&sbar[1], 0)) set_error(a.err, kDevErrTimeout);
  const int32_t* bm = sa.block_max + row * a.max_pages;
  int* vals2 = area;  // the tile maxima are no longer read (the collect ended on a barrier)
  int* cand2 = area + sa.n2_cap;
  // the candidates laid out as (vals2, cand2); the fast path writes the kept block ids, the
  // general path positions in cand2
  const int n2 = got1 * P;
  const bool range2 = rr.z != 0u && rr.w != 0u;
  int valid = 0, mn2 = INT_MAX, mx2 = INT_MIN;
  for (int x0 = tid; x0 < n2; x0 += 4 * NT) {
    int v[4], kk[4];
#pragma unroll
    for (int u = 0; u < 4; u++) {
      const int x = x0 + u * NT;
      kk[u] = x < n2 ? kept1[x / P] * P + x % P : -1;
      const bool in = kk[u] >= k_lo && kk[u] < k_hi;
      v[u] = in ? (use_row ? brow[kk[u] - k_lo] : __ldcg(bm + kk[u])) : INT_MIN;
    }
#pragma unroll
    for (int u = 0; u < 4; u++) {
      const int x = x0 + u * NT;
      if (x < n2) {
        cand2[x] = kk[u];
        vals2[x] = v[u];
        if (v[u] != INT_MIN) {
          valid++;
          mn2 = min(mn2, v[u]);
          mx2 = max(mx2, v[u]);
        }
      }
    }
  }
  if (range2 && n2 > 0 && n2 <= kRegVals * NT) {
    __syncthreads();  // the candidates are laid out
    got2 = sel_fast_row<NT, kRegVals>(SelRow{vals2, cand2, 0}, n2, a.k2, b_min, b_max, ss, selb);
    ids = got2 >= 0;
  }
  if (got2 < 0) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      valid += __shfl_xor_sync(0xffffffffu, valid, off);
      mn2 = min(mn2, __shfl_xor_sync(0xffffffffu, mn2, off));
      mx2 = max(mx2, __shfl_xor_sync(0xffffffffu, mx2, off));
    }
    if (lane == 0) {
      ss.wsum[warp] = valid;
      ss.mn[warp] = mn2;
      ss.mx[warp] = mx2;
    }
    __syncthreads();
    int n2_valid = 0;
#pragma unroll
    for (int w = 0; w < NT / 32; w++) {
      n2_valid += ss.wsum[w];
      mn2 = min(mn2, ss.mn[w]);
      mx2 = max(mx2, ss.mx[w]);
    }
    const int keep2 = min(a.k2, n2_valid);
    got2 = 0;
    if (keep2 > 0) {
      int T = INT_MIN, need_eq = 0, eq_total = 0;
      if (keep2 < n2_valid) {
        const int3 r = sel_kth_largest<NT>(vals2, n2, keep2, ss, true, mn2, mx2);
        T = r.x;
        need_eq = r.y;
        eq_total = r.z;
      }
      got2 = sel_collect<NT>(vals2, n2, T, need_eq, eq_total, ss, selb, 0);  // positions
    } else {
      __syncthreads();  // every thread has read the per-warp totals
    }
  }
  if (use_prow && p_plan.bytes() > 0 && !mbar_wait(&sbar[2], 0)) set_error(a.err, kDevErrTimeout);
  for (int i = tid; i < got2; i += NT) {
    const int kk = ids ? selb[i] : cand2[selb[i]];
    selb[i] = kk;
    selp[i] = use_prow ? prow[kk - k_lo] : -1;
  }
  __syncthreads();
  }
  if (split == 0) {
    for (int i = tid; i < a.k2; i += NT) sa.block_idx[row * a.k2 + i] = i < got2 ? selb[i] : -1;
    if (tid == 0) sa.n_blocks[row] = got2;
  }
  S.n_sel = min(got2, S.n_sel_max);

  WarpState<G> st;
#pragma unroll
  for (int j = 0; j < G; j++)
#pragma unroll
    for (int e = 0; e < 4; e++) st.acc[j][e] = 0.0f;
  st.m = kNeg;
  st.l = 0.0f;
  if (warp == W) {
    // ---- producer, after the selection: the deferred page, then the remaining segments
    // (kept blocks, and sink / window pages beyond the first NS), 32 at a time: the lanes
    // resolve them together; first uses of a ring slot go out from every lane at once, the
    // others from lane 0 in order as the slots free up
    if (j_def >= 0 && j_def < jA) {  // resolved before the wait by lane j_def
      const int kd = __shfl_sync(0xffffffffu, def_k, j_def);
      const int t0d = __shfl_sync(0xffffffffu, def_t0, j_def);
      const int t1d = __shfl_sync(0xffffffffu, def_t1, j_def);
      const int pd = __shfl_sync(0xffffffffu, def_page, j_def);
      if (lane == 0) {
        meta[j_def] = make_int4(kd, t0d, t1d, 0);
        issue(j_def, pd);
      }
    }
    const int n_post = cnt - jA;
    bool ok = true;
    for (int eb = 0; ok && eb < n_post; eb += 32) {
      const int j = eb + lane < n_post ? jA + eb + lane : -1;
      int k = 0, t0 = 0, t1 = 0, page = -1;
      if (j >= 0) page = resolve(first + j * stride, k, t0, t1);
      if (j >= 0 && j < NS) {
        meta[j] = make_int4(k, t0, t1, 0);
        issue(j, page);
      }
      const int n = min(32, n_post - eb);
      for (int q = 0; q < n; q++) {
        const int jq = __shfl_sync(0xffffffffu, j, q);
        const int kq = __shfl_sync(0xffffffffu, k, q);
        const int t0q = __shfl_sync(0xffffffffu, t0, q);
        const int t1q = __shfl_sync(0xffffffffu, t1, q);
        const int pq = __shfl_sync(0xffffffffu, page, q);
        if (jq < NS) continue;  // issued above
        if (lane == 0) {
          const int s = jq % NS;
          if (!mbar_wait(&empty[s], ((jq / NS) - 1) & 1)) {
            set_error(a.err, kDevErrTimeout);
            ok = false;
          } else {
            meta[s] = make_int4(kq, t0q, t1q, 0);
            issue(s, pq);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
      }
    }
    if (!ok && lane == 0) {
      for (int j = max(0, cnt - NS); j < cnt; j++) mbar_wait(&full[j % NS], (j / NS) & 1);
    }
  } else {
    float qf[G][16];
    load_query<G>(qf, a, b, h, lane & 7);
    for (int j = warp; j < cnt; j += W) {
      const int s = j % NS;
      if (!mbar_wait(&full[s], (j / NS) & 1)) {
        set_error(a.err, kDevErrTimeout);
        break;
      }
      const int4 m4 = meta[s];  // written before the producer's arrive on full[s]
      if (m4.y < m4.z)
        warp_segment<G>(st, qf, wscr[warp], smem_addr(ring + s * kSlotBytes), m4.x, m4.y, m4.z,
                        nullptr);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
  }
  __syncthreads();
  merge_warps<G, W, 16, false>(a, st, ring, mstate, b, h, split);
}

// ---------------------------------------------------------- mapped-host path

template <int G, bool DENSE>
__global__ void __launch_bounds__(kHostThreads, G <= 4 ? 3 : 2) attend_host_kernel(const AttArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  uint8_t* slots = smem;  // two slots: the segment in use and the next one
  using Sc = Scratch<head_slots(G)>;
  Sc& sc = *reinterpret_cast<Sc*>(smem + 2 * kSlotBytes);
  float* red = reinterpret_cast<float*>(smem + 2 * kSlotBytes + sizeof(Sc));

  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31;
  grid_dep_wait();
  grid_dep_launch();
  const int n_raw = a.seq_lens[b];
  if (tid == 0 && split == 0 && h == 0 && (n_raw < 0 || n_raw > a.max_pages * kPage))
    set_error(a.err, kDevErrCheck);
  Segments S = make_segments<DENSE>(a, b, h);
  read_selection(S, a, b, h);
  const int i0 = (int)((long long)S.total * split / a.nsplit);
  const int i1 = (int)((long long)S.total * (split + 1) / a.nsplit);
  State<G> st;
  init_state<G>(st);
  float qf[G][16];
  load_query<G>(qf, a, b, h, lane & 7);

  // each thread copies 64 of the segment's 8192 bytes: 16 bytes at 16 tid and at 2048 + 16 tid
  // of K, then of V, so that every warp load reads a contiguous, fully used 512-byte span
  // (each sector crosses the host link once)
  auto fetch = [&](int i, uint4 (&buf)[4], int& k, int& t0, int& t1) {
    segment_at(S, i, a.sink, k, t0, t1);
    if (t0 >= t1) return;
    const int page = a.page_table[(size_t)b * a.max_pages + k];
    if (page < 0 || page >= a.num_pages) {
      set_error(a.err, kDevErrCheck);
      t0 = t1 = 0;
      return;
    }
    const size_t off = ((size_t)page * a.kv_heads + h / a.kv_div) * kPage * kHeadDim;
    const uint8_t* kp = reinterpret_cast<const uint8_t*>(a.k + off);
    const uint8_t* vp = reinterpret_cast<const uint8_t*>(a.v + off);
    buf[0] = ldg128_nc(kp + tid * 16);
    buf[1] = ldg128_nc(kp + kBlockBytesBf16 / 2 + tid * 16);
    buf[2] = ldg128_nc(vp + tid * 16);
    buf[3] = ldg128_nc(vp + kBlockBytesBf16 / 2 + tid * 16);
  };
  auto store = [&](int slot, const uint4 (&buf)[4]) {
    uint8_t* kd = slots + slot * kSlotBytes + tid * 16;
    uint8_t* vd = kd + kBlockBytesBf16;
    *reinterpret_cast<uint4*>(kd) = buf[0];
    *reinterpret_cast<uint4*>(kd + kBlockBytesBf16 / 2) = buf[1];
    *reinterpret_cast<uint4*>(vd) = buf[2];
    *reinterpret_cast<uint4*>(vd + kBlockBytesBf16 / 2) = buf[3];
  };
  uint4 nxt[4];
  int kn = 0, t0n = 0, t1n = 0;
  if (i0 < i1) fetch(i0, nxt, kn, t0n, t1n);
  for (int i = i0; i < i1; i++) {
    const int slot = (i - i0) & 1;
    const int k = kn, t0 = t0n, t1 = t1n;
    if (t0 < t1) store(slot, nxt);
    if (i + 1 < i1) fetch(i + 1, nxt, kn, t0n, t1n);  // in flight while this one computes
    compute_bar();
    if (t0 < t1) process_segment<G>(st, qf, sc, smem_addr(slots + slot * kSlotBytes), k, t0, t1);
  }
  __syncthreads();
  finish<G>(a, st, sc, b, h, split, red);
}

// ---------------------------------------------------------- block-cache fill

// One warp per fill entry (slot, page, head): the 4 KiB K block and the 4 KiB V block are
// read from host memory (each warp load a contiguous 512-byte span) into the slot.
__global__ void __launch_bounds__(256) cache_fill_kernel(const int4* fill, const int32_t* n_fill,
                                                         const uint8_t* k_host,
                                                         const uint8_t* v_host, uint8_t* data,
                                                         int hkv, int num_pages, int capacity,
                                                         int* err) {
  grid_dep_wait();  // the plan comes from the previous kernel
  grid_dep_launch();
  const int n = *n_fill;
  const int lane = threadIdx.x & 31;
  const int nwarps = gridDim.x * (blockDim.x >> 5);
  for (int j = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); j < n; j += nwarps) {
    const int4 e = fill[j];
    if (e.x < 0 || e.x >= capacity || e.y < 0 || e.y >= num_pages || e.z < 0 || e.z >= hkv) {
      if (lane == 0) set_error(err, kDevErrCheck);
      continue;
    }
    const size_t src = ((size_t)e.y * hkv + e.z) * kBlockBytesBf16;
    uint8_t* dst = data + (size_t)e.x * kSlotBytes;
    uint4 r[8];
#pragma unroll
    for (int u = 0; u < 8; u++) r[u] = ldg128_nc(k_host + src + u * 512 + lane * 16);
#pragma unroll
    for (int u = 0; u < 8; u++) *reinterpret_cast<uint4*>(dst + u * 512 + lane * 16) = r[u];
#pragma unroll
    for (int u = 0; u < 8; u++) r[u] = ldg128_nc(v_host + src + u * 512 + lane * 16);
#pragma unroll
    for (int u = 0; u < 8; u++)
      *reinterpret_cast<uint4*>(dst + kBlockBytesBf16 + u * 512 + lane * 16) = r[u];
  }
}

template <int G, int W, int NS>
constexpr size_t tma_smem() {
  constexpr int H = head_slots(G);
  // the merge area ((W + 1) * G * 128 + 2 * H floats) fits in the ring
  static_assert(((W + 1) * G * kHeadDim + 2 * H) * sizeof(float) <= (size_t)NS * kSlotBytes,
                "merge area");
  return 128 + (size_t)NS * kSlotBytes + 2 * NS * sizeof(uint64_t) +
         W * sizeof(WarpScratch<H>) + 2 * W * H * sizeof(float) + NS * sizeof(int4);
}

template <int G>
size_t host_smem() {
  return 128 + 2 * kSlotBytes + sizeof(Scratch<head_slots(G)>) + red_floats(G) * sizeof(float);
}
static_assert(kStages % kWarps == 0, "each compute warp owns fixed ring slots");

template <int G, bool DENSE, int W, int NS>
cudaError_t launch_tma(const AttArgs& a, dim3 grid, cudaStream_t st) {
  constexpr size_t smem = tma_smem<G, W, NS>();
  auto kern = attend_tma_kernel<G, DENSE, W, NS, false>;
  if constexpr (!DENSE)
    if (a.seg_l2 != nullptr) kern = attend_tma_kernel<G, false, W, NS, true>;
  cudaError_t e = set_kernel_smem(kern, smem);
  if (e != cudaSuccess) return e;
  return launch_kernel(kern, grid, dim3((W + 1) * 32), smem, st, true, a);
}

template <int G, bool DENSE>
cudaError_t launch_g(AttArgs a, dim3 grid, bool host, cudaStream_t st) {
  if (host) {
    const size_t smem = host_smem<G>();
    cudaError_t e = set_kernel_smem(attend_host_kernel<G, DENSE>, smem);
    if (e != cudaSuccess) return e;
    return launch_kernel(attend_host_kernel<G, DENSE>, grid, dim3(kHostThreads), smem, st, true, a);
  }
  if constexpr (DENSE) {
    return launch_tma<G, true, kDenseWarps, kDenseStages>(a, grid, st);
  } else if constexpr (G > 4) {
    // groups of 8 hold 8 x 16 query floats per lane: at most two warps per SM sub-partition
    // (registers), so the sparse attend takes 7 compute warps there
    return launch_tma<G, false, 7, 14>(a, grid, st);
  } else {
    // a CTA's share of a row's segments (sink pages, kept blocks, window pages) decides the
    // shape: kSparseWarps compute warps from kSparseManySegs on, else 8
    const long long segs =
        (a.sink + kPage - 1) / kPage + a.k2 + (a.window + kPage - 1) / kPage + 1;
    const long long per_cta = (segs + a.nsplit - 1) / a.nsplit;
    if (per_cta >= kSparseManySegs)
      return launch_tma<G, false, kSparseWarps, 2 * kSparseWarps>(a, grid, st);
    if constexpr (kSparseFewWarps > 0) {
      if (per_cta <= kSparseFewWarps)
        return launch_tma<G, false, kSparseFewWarps, kSparseFewWarps>(a, grid, st);
    }
    return launch_tma<G, false, 8, 16>(a, grid, st);
  }
}

constexpr size_t kSelSmemLimit = 227 * 1024 - 256;  // room for the static shared memory

template <int G, int W, int NS>
size_t sel_smem_bytes(const SelArgs& sa) {
  return 128 + sel_smem_layout<G, W, NS>(sa).end;
}

// Shared-memory capacities of attend_select_kernel for a shape; false when the selection
// does not fit (then the step runs the pruning kernel and the plain sparse attention). The
// rows of block maxima and of page ids are staged when they fit too.
template <int G, int W, int NS>
bool plan_select(const Shape& s, SelArgs& sa, bool stage_pages) {
  constexpr int P = kTileBlocksSel;
  if (!HSA_FUSED_SELECT || s.chunk != P * kPage || s.k0 > 0) return false;
  auto up4 = [](long long x) { return (int)((x + 3) / 4 * 4); };
  const long long n1max = ((long long)s.max_pages + P - 1) / P;
  // Measured on GB300: the kernel beats the pruning kernel + plain attention when every
  // thread holds its share of a row's chunk scores in registers (rows of up to 8 x threads
  // chunks: the 128K-token configurations); longer rows go to the pruning kernel, whose
  // 512 threads select them faster (1M tokens: 196.4 against 198.0 us a step).
  if (n1max > (long long)kSelRegVals * (W + 1) * 32) return false;
  const long long keep1 = std::min<long long>(module1_keep(s), n1max);
  const long long n2max = keep1 * P;
  sa.n2_cap = up4(std::max<long long>(n2max, 1));
  sa.a_cap = std::max(up4(n1max + 4), 2 * sa.n2_cap);
  sa.k1_cap = up4(std::max<long long>(keep1, 1));
  sa.k2_cap = up4(std::max<long long>(std::min<long long>(s.k2, n2max), 1));
  sa.row_cap = 0;
  sa.prow_cap = 0;
  if (sel_smem_bytes<G, W, NS>(sa) > kSelSmemLimit) return false;
  sa.row_cap = up4(s.max_pages);
  if (sel_smem_bytes<G, W, NS>(sa) > kSelSmemLimit) sa.row_cap = 0;
  if (stage_pages) {
    sa.prow_cap = up4(s.max_pages);
    if (sel_smem_bytes<G, W, NS>(sa) > kSelSmemLimit) sa.prow_cap = 0;
  }
  return true;
}

// The attention's warps and ring slots for a group size (as launch_g's sparse path).
// Launch shapes of the selecting attention: 8 compute warps with two ring slots each (7 for
// groups of 8 query heads), or, for groups of up to 4 when a CTA's share of a row is at most
// kSelFewWarps segments, that many compute warps with one slot each, so that no warp takes a
// second segment: measured on GB300, a 128K step (about 11 segments a CTA) 41.6 against
// 42.9 us (10 warps: 43.1; 12: 41.7), the batched case of 8 sequences (about 19 a CTA) 120.5
// against 119.4 us with 11, so it keeps 8.
#ifndef HSA_SEL_FEW_WARPS
#define HSA_SEL_FEW_WARPS 11
#endif
constexpr int kSelFewWarps = HSA_SEL_FEW_WARPS;
template <int G, bool FEW = false>
struct SelShape {
  static constexpr int W = G > 4 ? 7 : (FEW ? kSelFewWarps : 8);
  static constexpr int NS = FEW && G <= 4 ? kSelFewWarps : 2 * W;
};

// The capacities are planned for the 8-warp shape, whose shared memory is the larger.
template <int G>
bool plan_select_g(const Shape& s, SelArgs& sa, bool stage_pages) {
  return plan_select<G, SelShape<G>::W, SelShape<G>::NS>(s, sa, stage_pages);
}

template <int G, bool FEW>
cudaError_t launch_select_shape(const AttArgs& a, const SelArgs& sa, dim3 grid,
                                cudaStream_t st) {
  constexpr int W = SelShape<G, FEW>::W, NS = SelShape<G, FEW>::NS;
  const size_t smem = sel_smem_bytes<G, W, NS>(sa);
  auto kern = attend_select_kernel<G, W, NS>;
  cudaError_t e = set_kernel_smem(kern, smem);
  if (e != cudaSuccess) return e;
  return launch_kernel(kern, grid, dim3((W + 1) * 32), smem, st, true, a, sa);
}

template <int G>
cudaError_t launch_select_g(const AttArgs& a, const SelArgs& sa, dim3 grid, cudaStream_t st,
                            bool few) {
  if constexpr (G <= 4 && kSelFewWarps > 0) {  // (0: the 8-warp shape only)
    if (few) return launch_select_shape<G, true>(a, sa, grid, st);
  }
  return launch_select_shape<G, false>(a, sa, grid, st);
}

bool plan_select_any(const Shape& s, SelArgs& sa, bool stage_pages) {
  switch (s.group) {
    case 1: return plan_select_g<1>(s, sa, stage_pages);
    case 2: return plan_select_g<2>(s, sa, stage_pages);
    case 4: return plan_select_g<4>(s, sa, stage_pages);
    case 8: return plan_select_g<8>(s, sa, stage_pages);
    default: return false;
  }
}

}  // namespace

int attend_splits(const Shape& s, bool dense, bool host, int num_sms, bool reserve) {
  const long long units = (long long)s.batch * s.hkv;
  long long segs;
  if (dense) {
    segs = s.max_pages;
  } else {
    segs = (s.sink + kPage - 1) / kPage + s.k2 + (s.window + kPage - 1) / kPage + 1;
  }
  // dense: about three CTAs per SM; sparse: fewer, each with several segments
  const int per_sm =
      host ? HSA_HOST_CTAS_PER_SM : (dense ? HSA_DENSE_CTAS_PER_SM : HSA_SPARSE_CTAS_PER_SM);
  long long want = ((long long)num_sms * per_sm + units - 1) / units;
  // without a pruning kernel beside it: one wave of CTAs, at most one per SM each
  if (!dense && !host && !reserve) want = std::max<long long>(1, (long long)num_sms * per_sm / units);
  if (!dense && !host && reserve && HSA_SPARSE_RESERVE && num_sms > units) {
    const long long reserved = std::max<long long>(1, (num_sms - units) / units);
    if (4 * reserved >= 3 * want) want = reserved;
  }
  want = std::min<long long>(want, std::max<long long>(1, segs / 4));
  return (int)std::max<long long>(1, std::min<long long>(want, kMaxSplits));
}

cudaError_t launch_cache_fill(const Shape& s, const BlockCache& c, const void* fill,
                              const int32_t* n_fill, const void* k_host, const void* v_host,
                              int* err, int num_sms, cudaStream_t st) {
  const cudaError_t e = set_kernel_smem(cache_fill_kernel, 0);
  if (e != cudaSuccess) return e;
  return launch_kernel(cache_fill_kernel, dim3(2 * num_sms), dim3(256), 0, st, true,
                       static_cast<const int4*>(fill), n_fill,
                       static_cast<const uint8_t*>(k_host), static_cast<const uint8_t*>(v_host),
                       static_cast<uint8_t*>(c.data), s.hkv, s.num_pages, c.capacity, err);
}

cudaError_t launch_attend(const Shape& s, bool dense, bool host, const void* q,
                          const void* k_cache, const void* v_cache, const int32_t* page_table,
                          const int32_t* seq_lens, const int32_t* block_idx,
                          const int32_t* n_blocks, float* out, float* lse,
                          const AttendBuffers& buf, int* err, cudaStream_t st, bool early) {
  if (buf.nsplit < 1 || buf.nsplit > kMaxSplits) return cudaErrorInvalidValue;
  AttArgs a;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.k = static_cast<const __nv_bfloat16*>(k_cache);
  a.v = static_cast<const __nv_bfloat16*>(v_cache);
  a.page_table = page_table;
  a.seq_lens = seq_lens;
  a.block_idx = block_idx;
  a.n_blocks = n_blocks;
  a.sel_pages = buf.sel_pages;
  a.seg_slots = buf.seg_slots;
  a.seg_stride = buf.seg_stride;
  a.seg_l2 = buf.seg_slots ? buf.seg_l2 : nullptr;
  a.mass = buf.mass;
  a.slot_key = buf.slot_key;
  a.out = out;
  a.lse = lse;
  a.part_ml = buf.part_ml;
  a.part_o = buf.part_o;
  a.counters = buf.counters;
  a.err = err;
  a.hkv = s.hkv;
  a.kv_div = s.kv_div;
  a.kv_heads = s.hkv / s.kv_div;
  a.max_pages = s.max_pages;
  a.num_pages = buf.seg_slots ? buf.cache_capacity : s.num_pages;
  a.k2 = s.k2;
  a.sink = s.sink;
  a.window = s.window;
  a.nsplit = buf.nsplit;
  a.qscale = s.sm_scale * kLog2e;
  a.early = (early && !host) ? 1 : 0;
  a.row_range = nullptr;
  dim3 grid(buf.nsplit, s.hkv, s.batch);
  switch (s.group) {
    case 1:
      return dense ? launch_g<1, true>(a, grid, host, st) : launch_g<1, false>(a, grid, host, st);
    case 2:
      return dense ? launch_g<2, true>(a, grid, host, st) : launch_g<2, false>(a, grid, host, st);
    case 4:
      return dense ? launch_g<4, true>(a, grid, host, st) : launch_g<4, false>(a, grid, host, st);
    case 8:
      return dense ? launch_g<8, true>(a, grid, host, st) : launch_g<8, false>(a, grid, host, st);
    default:
      return cudaErrorInvalidValue;
  }
}

bool attend_select_supported(const Shape& s, bool page_table_aligned) {
  SelArgs sa;
  return plan_select_any(s, sa, page_table_aligned);
}

cudaError_t launch_attend_select(const Shape& s, const void* q, const void* k_cache,
                                 const void* v_cache, const int32_t* page_table,
                                 const int32_t* seq_lens, const int32_t* block_max,
                                 const int32_t* tile_max, unsigned* row_range,
                                 int32_t* block_idx, int32_t* n_blocks, float* out, float* lse,
                                 const AttendBuffers& buf, int* err, cudaStream_t st) {
  if (buf.nsplit < 1 || buf.nsplit > kMaxSplits) return cudaErrorInvalidValue;
  const bool stage_pages = (reinterpret_cast<uintptr_t>(page_table) & 15) == 0;
  SelArgs sa;
  if (!plan_select_any(s, sa, stage_pages)) return cudaErrorInvalidValue;
  // the staging copies start from the 16-byte boundary at or below a row's first entry
  if ((reinterpret_cast<uintptr_t>(block_max) & 15) != 0 ||
      (reinterpret_cast<uintptr_t>(tile_max) & 15) != 0)
    return cudaErrorInvalidValue;
  if (row_range == nullptr || (reinterpret_cast<uintptr_t>(row_range) & 15) != 0)
    return cudaErrorInvalidValue;
  sa.block_max = block_max;
  sa.tile_max = tile_max;
  sa.row_range = row_range;
  sa.block_idx = block_idx;
  sa.n_blocks = n_blocks;
  sa.max_tiles = (s.max_pages + kTileBlocksSel - 1) / kTileBlocksSel;
  sa.k1 = module1_keep(s);
  AttArgs a = {};
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.k = static_cast<const __nv_bfloat16*>(k_cache);
  a.v = static_cast<const __nv_bfloat16*>(v_cache);
  a.page_table = page_table;
  a.seq_lens = seq_lens;
  a.out = out;
  a.lse = lse;
  a.part_ml = buf.part_ml;
  a.part_o = buf.part_o;
  a.counters = buf.counters;
  a.err = err;
  a.hkv = s.hkv;
  a.kv_div = s.kv_div;
  a.kv_heads = s.hkv / s.kv_div;
  a.max_pages = s.max_pages;
  a.num_pages = s.num_pages;
  a.k2 = s.k2;
  a.sink = s.sink;
  a.window = s.window;
  a.nsplit = buf.nsplit;
  a.qscale = s.sm_scale * kLog2e;
  a.early = 1;
  a.row_range = row_range;
  dim3 grid(buf.nsplit, s.hkv, s.batch);
  // segments of a row at most (sink pages, kept blocks, window pages with a partial one) and
  // a CTA's share of them
  const long long segs =
      (s.sink + kPage - 1) / kPage + s.k2 + (s.window + kPage - 1) / kPage + 1;
  const bool few = (segs + buf.nsplit - 1) / buf.nsplit <= kSelFewWarps;
  switch (s.group) {
    case 1: return launch_select_g<1>(a, sa, grid, st, few);
    case 2: return launch_select_g<2>(a, sa, grid, st, few);
    case 4: return launch_select_g<4>(a, sa, grid, st, few);
    case 8: return launch_select_g<8>(a, sa, grid, st, few);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace hsa
