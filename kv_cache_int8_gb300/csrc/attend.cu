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
// candidate region), the window pages. Dense decode uses every page of [0, N). A CTA
// takes a contiguous share of the list for all G query heads of the group, so every K/V
// byte is read once per group. Within a segment, warp w handles tokens 4w..4w+3 and 8
// lanes share a token (16 channels each); each 8-lane group keeps its own online-softmax
// state (log2 domain), merged across the CTA at the end; CTAs of one (b, h) are merged by
// the last one to finish (atomic counter, no waiting).
//
// HBM path: a producer lane fills a ring of 8 KiB slots (K page then V page of one head,
// 4 KiB each) with cp.async.bulk copies tracked by mbarriers. Host path: K/V live in
// pinned host memory; each lane issues its own 16-byte loads through the mapped alias.
#include <algorithm>
#include <cfloat>

#include "common.cuh"
#include "internal.h"

namespace hsa {
namespace {

constexpr int kWarps = 4;                              // compute warps: 16 tokens per segment
constexpr int kStages = 8;
constexpr int kSlotBytes = 2 * kBlockBytesBf16;        // K page + V page of one head
constexpr int kTmaThreads = (kWarps + 1) * 32;
constexpr int kHostThreads = kWarps * 32;
constexpr int kMaxSplits = 64;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct AttArgs {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const int32_t* page_table;
  const int32_t* seq_lens;
  const int32_t* block_idx;
  const int32_t* n_blocks;
  float* out;
  float* lse;
  float* part_ml;
  float* part_o;
  int* counters;
  int* err;
  int hkv, max_pages, num_pages, k2, sink, window, nsplit;
  float qscale;  // sm_scale * log2(e)
};

struct Segments {
  int n;                 // context length
  int n_sink, n_sel, n_win;
  int sink_end, cand_hi, w0, win_k0;
  const int32_t* sel;
  int total;
};

template <bool DENSE>
__device__ __forceinline__ Segments make_segments(const AttArgs& a, int b, int h) {
  Segments s;
  int n = a.seq_lens[b];
  if (n < 0 || n > a.max_pages * kPage) n = 0;  // reported by the caller's check
  s.n = n;
  if (DENSE) {
    s.n_sink = 0;
    s.n_sel = 0;
    s.n_win = (n + kPage - 1) / kPage;
    s.sink_end = 0;
    s.cand_hi = 0;
    s.w0 = 0;
    s.win_k0 = 0;
    s.sel = nullptr;
  } else {
    s.sink_end = min(a.sink, n);
    s.n_sink = (s.sink_end + kPage - 1) / kPage;
    s.cand_hi = n - a.window;
    s.sel = a.block_idx + ((size_t)b * a.hkv + h) * a.k2;
    s.n_sel = s.cand_hi > a.sink ? max(0, min(a.n_blocks[(size_t)b * a.hkv + h], a.k2)) : 0;
    s.w0 = max(n - a.window, s.sink_end);
    s.win_k0 = s.w0 / kPage;
    s.n_win = s.w0 < n ? (n + kPage - 1) / kPage - s.win_k0 : 0;
  }
  s.total = s.n_sink + s.n_sel + s.n_win;
  return s;
}

// Segment i: page index k (token block) and the attended token range [t0, t1).
__device__ __forceinline__ void segment_at(const Segments& s, int i, int sink, int& k, int& t0,
                                           int& t1) {
  if (i < s.n_sink) {
    k = i;
    t0 = i * kPage;
    t1 = min(t0 + kPage, s.sink_end);
  } else if (i < s.n_sink + s.n_sel) {
    k = s.sel[i - s.n_sink];
    const int kmax = (s.n + kPage - 1) / kPage;
    if (k < 0 || k >= kmax) {
      k = 0;
      t0 = t1 = 0;
      return;
    }
    t0 = max(k * kPage, sink);
    t1 = min(k * kPage + kPage, s.cand_hi);
  } else {
    k = s.win_k0 + (i - s.n_sink - s.n_sel);
    t0 = max(k * kPage, s.w0);
    t1 = min(k * kPage + kPage, s.n);
  }
}

// Per-lane online-softmax state for the G heads over 16 channels.
template <int G>
struct State {
  float m[G], l[G], o[G][16];
};

template <int G>
__device__ __forceinline__ void unpack16(const uint4& a, const uint4& b, float f[16]) {
  f[0] = bf16_lo(a.x); f[1] = bf16_hi(a.x); f[2] = bf16_lo(a.y); f[3] = bf16_hi(a.y);
  f[4] = bf16_lo(a.z); f[5] = bf16_hi(a.z); f[6] = bf16_lo(a.w); f[7] = bf16_hi(a.w);
  f[8] = bf16_lo(b.x); f[9] = bf16_hi(b.x); f[10] = bf16_lo(b.y); f[11] = bf16_hi(b.y);
  f[12] = bf16_lo(b.z); f[13] = bf16_hi(b.z); f[14] = bf16_lo(b.w); f[15] = bf16_hi(b.w);
}

// One token: scores of the G heads (8-lane butterfly), online update, value accumulation.
// Every lane of the warp must call (the shuffles span the warp); `valid` is per 8-lane group.
template <int G>
__device__ __forceinline__ void attend_token(State<G>& st, const float (&qf)[G][16],
                                             const uint4& k0, const uint4& k1, const uint4& v0,
                                             const uint4& v1, bool valid) {
  float kf[16];
  unpack16<G>(k0, k1, kf);
  float s[G];
#pragma unroll
  for (int j = 0; j < G; j++) {
    float acc = 0.0f;
#pragma unroll
    for (int e = 0; e < 16; e++) acc = fmaf(qf[j][e], kf[e], acc);
    s[j] = acc;
  }
#pragma unroll
  for (int off = 1; off < 8; off <<= 1)
#pragma unroll
    for (int j = 0; j < G; j++) s[j] += __shfl_xor_sync(0xffffffffu, s[j], off);
  if (!valid) return;
  float vf[16];
  unpack16<G>(v0, v1, vf);
#pragma unroll
  for (int j = 0; j < G; j++) {
    if (s[j] > st.m[j]) {
      const float c = exp2f(st.m[j] - s[j]);
      st.m[j] = s[j];
      st.l[j] *= c;
#pragma unroll
      for (int e = 0; e < 16; e++) st.o[j][e] *= c;
    }
    const float p = exp2f(s[j] - st.m[j]);
    st.l[j] += p;
#pragma unroll
    for (int e = 0; e < 16; e++) st.o[j][e] = fmaf(p, vf[e], st.o[j][e]);
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
    unpack16<G>(u0, u1, f);
#pragma unroll
    for (int e = 0; e < 16; e++) qf[j][e] = f[e] * a.qscale;
  }
}

// Merge of the 16 per-group states of a CTA, then either the final output (one split) or
// a partial plus the last-CTA combine. `red` is shared memory of at least
// 16 * G * (2 + 128) floats. Called by all threads of the CTA.
template <int G>
__device__ void finish(const AttArgs& a, const State<G>& st, int b, int h, int split,
                       float* red, int nthreads) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int grp = lane >> 3, sl = lane & 7;
  float* rm = red;                       // [16][G]
  float* rl = rm + 16 * G;               // [16][G]
  float* ro = rl + 16 * G;               // [16][G][128]
  __shared__ int is_last;
  if (warp < kWarps) {
    const int r = warp * 4 + grp;
#pragma unroll
    for (int j = 0; j < G; j++) {
      if (sl == 0) {
        rm[r * G + j] = st.m[j];
        rl[r * G + j] = st.l[j];
      }
#pragma unroll
      for (int e = 0; e < 8; e++) {
        ro[(r * G + j) * kHeadDim + 8 * sl + e] = st.o[j][e];
        ro[(r * G + j) * kHeadDim + 64 + 8 * sl + e] = st.o[j][8 + e];
      }
    }
  }
  __syncthreads();
  const int hq = a.hkv * G;
  if (tid < kHeadDim) {
    const int d = tid;
#pragma unroll
    for (int j = 0; j < G; j++) {
      float M = -FLT_MAX;
      for (int r = 0; r < 16; r++) M = fmaxf(M, rm[r * G + j]);
      float L = 0.0f, O = 0.0f;
      for (int r = 0; r < 16; r++) {
        const float w = rl[r * G + j] > 0.0f ? exp2f(rm[r * G + j] - M) : 0.0f;
        L = fmaf(rl[r * G + j], w, L);
        O = fmaf(ro[(r * G + j) * kHeadDim + d], w, O);
      }
      const size_t row = (size_t)b * hq + (size_t)h * G + j;
      if (a.nsplit == 1) {
        a.out[row * kHeadDim + d] = L > 0.0f ? O / L : 0.0f;
        if (d == 0 && a.lse) a.lse[row] = L > 0.0f ? (M + log2f(L)) * kLn2 : -INFINITY;
      } else {
        const size_t p = row * a.nsplit + split;
        a.part_o[p * kHeadDim + d] = O;
        if (d == 0) {
          a.part_ml[2 * p] = M;
          a.part_ml[2 * p + 1] = L;
        }
      }
    }
  }
  if (a.nsplit == 1) return;
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const int prev = atomicAdd(&a.counters[(size_t)b * a.hkv + h], 1);
    is_last = prev == a.nsplit - 1;
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  if (tid < kHeadDim) {
    const int d = tid;
#pragma unroll
    for (int j = 0; j < G; j++) {
      const size_t row = (size_t)b * hq + (size_t)h * G + j;
      const float* ml = a.part_ml + 2 * row * a.nsplit;
      const float* po = a.part_o + row * a.nsplit * kHeadDim;
      float M = -FLT_MAX;
      for (int sp = 0; sp < a.nsplit; sp++) M = fmaxf(M, __ldcg(ml + 2 * sp));
      float L = 0.0f, O = 0.0f;
      for (int sp = 0; sp < a.nsplit; sp++) {
        const float l = __ldcg(ml + 2 * sp + 1);
        const float w = l > 0.0f ? exp2f(__ldcg(ml + 2 * sp) - M) : 0.0f;
        L = fmaf(l, w, L);
        O = fmaf(__ldcg(po + (size_t)sp * kHeadDim + d), w, O);
      }
      a.out[row * kHeadDim + d] = L > 0.0f ? O / L : 0.0f;
      if (d == 0 && a.lse) a.lse[row] = L > 0.0f ? (M + log2f(L)) * kLn2 : -INFINITY;
    }
  }
  if (tid == 0) a.counters[(size_t)b * a.hkv + h] = 0;
}

template <int G>
__device__ __forceinline__ void init_state(State<G>& st) {
#pragma unroll
  for (int j = 0; j < G; j++) {
    st.m[j] = -FLT_MAX;
    st.l[j] = 0.0f;
#pragma unroll
    for (int e = 0; e < 16; e++) st.o[j][e] = 0.0f;
  }
}

// ------------------------------------------------------------------ HBM path

template <int G, bool DENSE>
__global__ void __launch_bounds__(kTmaThreads, 2) attend_tma_kernel(const AttArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kSlotBytes);
  uint64_t* empty = full + kStages;

  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n_raw = a.seq_lens[b];
  if (tid == 0 && split == 0 && h == 0 && (n_raw < 0 || n_raw > a.max_pages * kPage))
    set_error(a.err, kDevErrCheck);
  const Segments S = make_segments<DENSE>(a, b, h);
  const int i0 = (int)((long long)S.total * split / a.nsplit);
  const int i1 = (int)((long long)S.total * (split + 1) / a.nsplit);

  if (tid == 0) {
    for (int s = 0; s < kStages; s++) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kWarps);
    }
    fence_barrier_init();
  }
  __syncthreads();

  State<G> st;
  init_state<G>(st);
  if (warp == kWarps) {
    if (lane == 0) {
      bool ok = true;
      for (int i = i0; i < i1; i++) {
        const int j = i - i0, s = j % kStages;
        if (j >= kStages && !mbar_wait(&empty[s], ((j / kStages) - 1) & 1)) {
          set_error(a.err, kDevErrTimeout);
          ok = false;
          break;
        }
        int k, t0, t1;
        segment_at(S, i, a.sink, k, t0, t1);
        int page = -1;
        if (t0 < t1) {
          page = a.page_table[(size_t)b * a.max_pages + k];
          if (page < 0 || page >= a.num_pages) {
            set_error(a.err, kDevErrCheck);
            page = -1;
          }
        }
        if (page >= 0) {
          const size_t off = ((size_t)page * a.hkv + h) * kPage * kHeadDim;
          mbar_arrive_expect_tx(&full[s], kSlotBytes);
          bulk_load(ring + s * kSlotBytes, a.k + off, kBlockBytesBf16, &full[s]);
          bulk_load(ring + s * kSlotBytes + kBlockBytesBf16, a.v + off, kBlockBytesBf16, &full[s]);
        } else {
          mbar_arrive(&full[s]);
        }
      }
      if (!ok) {
        const int issued = i1 - i0;
        for (int j = max(0, issued - kStages); j < issued; j++)
          mbar_wait(&full[j % kStages], (j / kStages) & 1);
      }
    }
  } else {
    const int grp = lane >> 3, sl = lane & 7;
    const int r = warp * 4 + grp;  // token slot within the page
    float qf[G][16];
    load_query<G>(qf, a, b, h, sl);
    for (int i = i0; i < i1; i++) {
      const int j = i - i0, s = j % kStages;
      if (!mbar_wait(&full[s], (j / kStages) & 1)) {
        set_error(a.err, kDevErrTimeout);
        break;
      }
      int k, t0, t1;
      segment_at(S, i, a.sink, k, t0, t1);
      if (t0 < t1) {
        const int t = k * kPage + r;
        const uint32_t kb = smem_addr(ring + s * kSlotBytes) + r * (kHeadDim * 2);
        const uint32_t vb = kb + kBlockBytesBf16;
        const uint4 k0 = lds128(kb + sl * 16), k1 = lds128(kb + (sl + 8) * 16);
        const uint4 v0 = lds128(vb + sl * 16), v1 = lds128(vb + (sl + 8) * 16);
        attend_token<G>(st, qf, k0, k1, v0, v1, t >= t0 && t < t1);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
  }
  __syncthreads();
  finish<G>(a, st, b, h, split, reinterpret_cast<float*>(ring), kTmaThreads);
}

// ---------------------------------------------------------- mapped-host path

template <int G, bool DENSE>
__global__ void __launch_bounds__(kHostThreads, 2) attend_host_kernel(const AttArgs a) {
  extern __shared__ uint8_t smem_raw[];
  float* red = reinterpret_cast<float*>(smem_raw);
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int grp = lane >> 3, sl = lane & 7;
  const int r = warp * 4 + grp;
  const int n_raw = a.seq_lens[b];
  if (tid == 0 && split == 0 && h == 0 && (n_raw < 0 || n_raw > a.max_pages * kPage))
    set_error(a.err, kDevErrCheck);
  const Segments S = make_segments<DENSE>(a, b, h);
  const int i0 = (int)((long long)S.total * split / a.nsplit);
  const int i1 = (int)((long long)S.total * (split + 1) / a.nsplit);
  State<G> st;
  init_state<G>(st);
  float qf[G][16];
  load_query<G>(qf, a, b, h, sl);
  // two segments per round, all eight 16-byte loads of a lane in flight together
  for (int i = i0; i < i1; i += 2) {
    uint4 kk[2][2], vv[2][2];
    int k[2], t0[2], t1[2];
    bool live[2];
#pragma unroll
    for (int u = 0; u < 2; u++) {
      live[u] = false;
      if (i + u < i1) {
        segment_at(S, i + u, a.sink, k[u], t0[u], t1[u]);
        if (t0[u] < t1[u]) {
          const int page = a.page_table[(size_t)b * a.max_pages + k[u]];
          if (page >= 0 && page < a.num_pages) {
            live[u] = true;
            const size_t off = (((size_t)page * a.hkv + h) * kPage + r) * kHeadDim;
            kk[u][0] = ldg128_nc(a.k + off + 8 * sl);
            kk[u][1] = ldg128_nc(a.k + off + 64 + 8 * sl);
            vv[u][0] = ldg128_nc(a.v + off + 8 * sl);
            vv[u][1] = ldg128_nc(a.v + off + 64 + 8 * sl);
          } else {
            set_error(a.err, kDevErrCheck);
          }
        }
      }
    }
#pragma unroll
    for (int u = 0; u < 2; u++) {
      if (!live[u]) continue;  // uniform across the warp: same segment for all lanes
      const int t = k[u] * kPage + r;
      attend_token<G>(st, qf, kk[u][0], kk[u][1], vv[u][0], vv[u][1], t >= t0[u] && t < t1[u]);
    }
  }
  __syncthreads();
  finish<G>(a, st, b, h, split, red, kHostThreads);
}

size_t red_bytes(int G) { return sizeof(float) * 16 * G * (2 + kHeadDim); }

template <int G, bool DENSE>
cudaError_t launch_g(const AttArgs& a, dim3 grid, bool host, cudaStream_t st) {
  if (host) {
    const size_t smem = red_bytes(G);
    cudaError_t e = cudaFuncSetAttribute(attend_host_kernel<G, DENSE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attend_host_kernel<G, DENSE><<<grid, kHostThreads, smem, st>>>(a);
  } else {
    const size_t ring = (size_t)kStages * kSlotBytes + 2 * kStages * sizeof(uint64_t);
    const size_t smem = 128 + std::max(ring, red_bytes(G));
    cudaError_t e = cudaFuncSetAttribute(attend_tma_kernel<G, DENSE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attend_tma_kernel<G, DENSE><<<grid, kTmaThreads, smem, st>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace

int attend_splits(const Shape& s, bool dense, bool host, int num_sms) {
  const long long units = (long long)s.batch * s.hkv;
  const int per_sm = host ? 4 : 2;
  long long segs;
  if (dense) {
    segs = s.max_pages;
  } else {
    segs = (s.sink + kPage - 1) / kPage + 1 + s.k2 + (s.window + kPage - 1) / kPage + 1;
  }
  long long want = ((long long)num_sms * per_sm + units - 1) / units;
  // at least two segments per CTA so that loads and compute overlap
  want = std::min<long long>(want, std::max<long long>(1, segs / 2));
  return (int)std::max<long long>(1, std::min<long long>(want, kMaxSplits));
}

cudaError_t launch_attend(const Shape& s, bool dense, bool host, const void* q,
                          const void* k_cache, const void* v_cache, const int32_t* page_table,
                          const int32_t* seq_lens, const int32_t* block_idx,
                          const int32_t* n_blocks, float* out, float* lse,
                          const AttendBuffers& buf, int* err, cudaStream_t st) {
  if (buf.nsplit < 1 || buf.nsplit > kMaxSplits) return cudaErrorInvalidValue;
  AttArgs a;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.k = static_cast<const __nv_bfloat16*>(k_cache);
  a.v = static_cast<const __nv_bfloat16*>(v_cache);
  a.page_table = page_table;
  a.seq_lens = seq_lens;
  a.block_idx = block_idx;
  a.n_blocks = n_blocks;
  a.out = out;
  a.lse = lse;
  a.part_ml = buf.part_ml;
  a.part_o = buf.part_o;
  a.counters = buf.counters;
  a.err = err;
  a.hkv = s.hkv;
  a.max_pages = s.max_pages;
  a.num_pages = s.num_pages;
  a.k2 = s.k2;
  a.sink = s.sink;
  a.window = s.window;
  a.nsplit = buf.nsplit;
  a.qscale = s.sm_scale * kLog2e;
  dim3 grid(buf.nsplit, s.hkv, s.batch);
  switch (s.group) {
    case 1:
      return dense ? launch_g<1, true>(a, grid, host, st) : launch_g<1, false>(a, grid, host, st);
    case 2:
      return dense ? launch_g<2, true>(a, grid, host, st) : launch_g<2, false>(a, grid, host, st);
    case 4:
      return dense ? launch_g<4, true>(a, grid, host, st) : launch_g<4, false>(a, grid, host, st);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace hsa
