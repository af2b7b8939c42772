// quantize.cu -- int8 per-channel key codes: full-context scales, codes, decode-step append.
//
// Source: "HCAttention: Extreme KV cache compression via heterogeneous attention computing
// for LLMs", abstract and contribution list (keys are quantised and kept on the GPU for
// global scoring); "KV Cache 与长上下文推理", section "KV Cache 量化" (INT8 keys) and
// section "KV Cache 回顾" (each decode step appends the new token's k, v).
//
// Reading: one scale per (sequence, kv head, channel) over the whole context,
// s = f32(amax / 127); code = clamp(rint_half_even(f32(k / s)), -127, 127); s = 0 -> 0.
// All decisions are taken in IEEE fp32 (__fdiv_rn, no fast math).
//
// Data: a CTA owns one (sequence, kv head) and a run of pages; thread t owns token slot
// t / 16 and the 8 channels [8 (t % 16), 8 (t % 16) + 8) of every page it visits, so each
// warp reads 512 contiguous bytes of bf16 per page with 16-byte loads.
#include "append.cuh"
#include "common.cuh"
#include "internal.h"

namespace hsa {
namespace {

using namespace append_detail;

constexpr int kThreads = 256;        // 16 slots x 16 channel groups of 8
constexpr int kPagesPerCta = 32;

__device__ __forceinline__ bool seq_ok(int n, int max_pages) {
  return n >= 0 && n <= max_pages * kPage;
}

// Divisor of amax giving the key scale: the largest code magnitude of the format.
__device__ __forceinline__ float scale_divisor(int fmt) {
  return fmt == kFmtFp8 ? 448.0f : (float)key_levels(fmt);
}

// Pass 1 of full quantisation: amax per (b, h, channel) over tokens t < N_b, as the bit
// pattern of a non-negative float (ordered like the value), merged with atomicMax.
__global__ void __launch_bounds__(kThreads) key_amax_kernel(
    const __nv_bfloat16* __restrict__ k_cache, const int32_t* __restrict__ page_table,
    const int32_t* __restrict__ seq_lens, unsigned* __restrict__ amax_bits, int hkv,
    int max_pages, int num_pages, int* err) {
  const int b = blockIdx.z, h = blockIdx.y;
  const int slot = threadIdx.x >> 4, grp = threadIdx.x & 15;
  const int n = seq_lens[b];
  __shared__ unsigned am[kHeadDim];
  if (threadIdx.x < kHeadDim) am[threadIdx.x] = 0u;
  __syncthreads();
  float mx[8];
#pragma unroll
  for (int i = 0; i < 8; i++) mx[i] = 0.0f;
  if (seq_ok(n, max_pages)) {
    const int p0 = blockIdx.x * kPagesPerCta;
    const int p1 = min(p0 + kPagesPerCta, (n + kPage - 1) / kPage);
    for (int p = p0; p < p1; p++) {
      const int t = p * kPage + slot;
      if (t >= n) continue;
      const int page = page_table[(size_t)b * max_pages + p];
      if (page < 0 || page >= num_pages) {
        set_error(err, kDevErrCheck);
        continue;
      }
      const size_t off = (((size_t)page * hkv + h) * kPage + slot) * kHeadDim + grp * 8;
      float f[8];
      unpack8(ldg128_nc(k_cache + off), f);
#pragma unroll
      for (int i = 0; i < 8; i++) mx[i] = fmaxf(mx[i], fabsf(f[i]));
    }
  }
#pragma unroll
  for (int i = 0; i < 8; i++) mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 16));
  if ((threadIdx.x & 31) < 16) {
#pragma unroll
    for (int i = 0; i < 8; i++) atomicMax(&am[grp * 8 + i], __float_as_uint(mx[i]));
  }
  __syncthreads();
  if (threadIdx.x < kHeadDim && am[threadIdx.x] != 0u)
    atomicMax(&amax_bits[((size_t)b * hkv + h) * kHeadDim + threadIdx.x], am[threadIdx.x]);
}

// Pass 2 (full) or append: codes of tokens [t_begin, N_b) with per-channel scales
// (full: s = f32(amax / levels), also stored, levels 127 for 8-bit and 7 for 4-bit codes;
// append: the stored scales). Full mode zeroes the codes of last-page slots past N_b.
__global__ void __launch_bounds__(kThreads) key_codes_kernel(
    const __nv_bfloat16* __restrict__ k_cache, const int32_t* __restrict__ page_table,
    const int32_t* __restrict__ seq_lens, const unsigned* __restrict__ amax_bits,
    const float* __restrict__ k_scale_in, float* __restrict__ k_scale_out, int append_from,
    int full, int8_t* __restrict__ kq, int hkv, int max_pages, int num_pages, int* err,
    int bits) {
  const int b = blockIdx.z, h = blockIdx.y;
  const int slot = threadIdx.x >> 4, grp = threadIdx.x & 15;
  const int n = seq_lens[b];
  if (!seq_ok(n, max_pages)) {
    if (threadIdx.x == 0) set_error(err, kDevErrCheck);
    return;
  }
  const size_t sbase = ((size_t)b * hkv + h) * kHeadDim + grp * 8;
  float s[8];
#pragma unroll
  for (int i = 0; i < 8; i++)
    s[i] = full ? __fdiv_rn(__uint_as_float(amax_bits[sbase + i]), scale_divisor(bits))
                : k_scale_in[sbase + i];
  if (full && blockIdx.x == 0 && slot == 0) {
#pragma unroll
    for (int i = 0; i < 8; i++) k_scale_out[sbase + i] = s[i];
  }
  int t_begin = 0;
  if (!full) t_begin = append_from < 0 ? n - 1 : append_from;
  t_begin = max(t_begin, 0);
  const int p_begin = t_begin / kPage;
  const int p0 = p_begin + blockIdx.x * kPagesPerCta;
  const int p1 = min(p0 + kPagesPerCta, (n + kPage - 1) / kPage);
  for (int p = p0; p < p1; p++) {
    const int t = p * kPage + slot;
    if (t < t_begin) continue;
    const int page = page_table[(size_t)b * max_pages + p];
    if (page < 0 || page >= num_pages) {
      set_error(err, kDevErrCheck);
      continue;
    }
    const size_t off = (((size_t)page * hkv + h) * kPage + slot) * kHeadDim + grp * 8;
    if (t < n) {
      float f[8];
      unpack8(ldg128_nc(k_cache + off), f);
      store_key_codes(kq, off, f, s, bits);
    } else if (full) {
      const int c[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      store_codes(kq, off, c, bits == kFmtFp8 ? 8 : bits);
    }
  }
}

// Decode-step append: slot N_b - 1 of every sequence receives k_new, v_new and the codes
// of k_new under the stored scales. One CTA per sequence, thread = (head, channel group).
// With `beside` (whole decode step only, where the predecessor is the scorer, which neither
// writes this kernel's inputs nor reads the slot it writes) the kernel runs concurrently
// with its predecessor and waits for it only before exiting; otherwise it waits first.

__global__ void append_kv_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                                 __nv_bfloat16* k_cache, __nv_bfloat16* v_cache, int8_t* kq,
                                 const float* __restrict__ k_scale,
                                 const int32_t* __restrict__ page_table,
                                 const int32_t* __restrict__ seq_lens, int hkv, int max_pages,
                                 int num_pages, int* err, int beside, int bits) {
  if (!beside) grid_dep_wait();
  grid_dep_launch();
  append_token(blockIdx.x, threadIdx.x, k_new, v_new, k_cache, v_cache, kq, k_scale, page_table,
               seq_lens, hkv, max_pages, num_pages, err, bits);
  grid_dep_wait();
}


// The kernels' key-format code of a shape.
int key_format(const Shape& s) { return s.key_fp8 ? kFmtFp8 : s.key_bits; }

}  // namespace

cudaError_t launch_key_amax(const Shape& s, const void* k_cache, const int32_t* page_table,
                            const int32_t* seq_lens, unsigned* amax_bits, int* err,
                            cudaStream_t st) {
  dim3 grid((s.max_pages + kPagesPerCta - 1) / kPagesPerCta, s.hkv, s.batch);
  key_amax_kernel<<<grid, kThreads, 0, st>>>(static_cast<const __nv_bfloat16*>(k_cache),
                                             page_table, seq_lens, amax_bits, s.hkv, s.max_pages,
                                             s.num_pages, err);
  return cudaGetLastError();
}

cudaError_t launch_key_codes(const Shape& s, const void* k_cache, const int32_t* page_table,
                             const int32_t* seq_lens, const unsigned* amax_bits,
                             const float* k_scale_in, float* k_scale_out, int append_from,
                             bool full, int8_t* kq, int* err, cudaStream_t st) {
  int pages = s.max_pages;
  if (!full) pages = append_from < 0 ? 1 : s.max_pages - append_from / kPage;
  if (pages <= 0) return cudaSuccess;
  dim3 grid((pages + kPagesPerCta - 1) / kPagesPerCta, s.hkv, s.batch);
  key_codes_kernel<<<grid, kThreads, 0, st>>>(static_cast<const __nv_bfloat16*>(k_cache),
                                              page_table, seq_lens, amax_bits, k_scale_in,
                                              k_scale_out, append_from, full ? 1 : 0, kq, s.hkv,
                                              s.max_pages, s.num_pages, err, key_format(s));
  return cudaGetLastError();
}

// The decode step's inputs (q, k_new, v_new), staged from mapped pinned host memory into
// device buffers by 16-byte loads over the host link, four in flight per thread: one small
// kernel instead of three copy-engine transfers.
__global__ void __launch_bounds__(256) stage_io_kernel(const uint4* q, const uint4* kn,
                                                       const uint4* vn, uint4* dq, uint4* dkn,
                                                       uint4* dvn, int nq, int nkv) {
  grid_dep_wait();  // the previous step's kernels may still read the staged copies
  grid_dep_launch();
  const int total = nq + 2 * nkv;
  const int stride = gridDim.x * blockDim.x;
  for (int i0 = blockIdx.x * blockDim.x + threadIdx.x; i0 < total; i0 += 4 * stride) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; u++) {
      const int i = i0 + u * stride;
      if (i < nq) v[u] = q[i];
      else if (i < nq + nkv) v[u] = kn[i - nq];
      else if (i < total) v[u] = vn[i - nq - nkv];
    }
#pragma unroll
    for (int u = 0; u < 4; u++) {
      const int i = i0 + u * stride;
      if (i < nq) dq[i] = v[u];
      else if (i < nq + nkv) dkn[i - nq] = v[u];
      else if (i < total) dvn[i - nq - nkv] = v[u];
    }
  }
}

cudaError_t launch_stage_io(const Shape& s, const void* q, const void* k_new, const void* v_new,
                            void* dq, void* dk_new, void* dv_new, int num_sms, cudaStream_t st) {
  const int nq = s.batch * s.hq * kHeadDim * 2 / 16;
  const int nkv = s.batch * s.hkv * kHeadDim * 2 / 16;
  const int total = nq + 2 * nkv;
  const int grid = std::max(1, std::min(num_sms, (total + 4 * 256 - 1) / (4 * 256)));
  const cudaError_t e = set_kernel_smem(stage_io_kernel, 0);
  if (e != cudaSuccess) return e;
  return launch_kernel(stage_io_kernel, dim3(grid), dim3(256), 0, st, true,
                       static_cast<const uint4*>(q), static_cast<const uint4*>(k_new),
                       static_cast<const uint4*>(v_new), static_cast<uint4*>(dq),
                       static_cast<uint4*>(dk_new), static_cast<uint4*>(dv_new), nq, nkv);
}

cudaError_t launch_append_kv(const Shape& s, const void* k_new, const void* v_new,
                             void* k_cache, void* v_cache, int8_t* kq, const float* k_scale,
                             const int32_t* page_table, const int32_t* seq_lens, int* err,
                             cudaStream_t st, bool beside) {
  const int threads = ((s.hkv * 16 + 31) / 32) * 32;
  const cudaError_t e = set_kernel_smem(append_kv_kernel, 0);
  if (e != cudaSuccess) return e;
  return launch_kernel(append_kv_kernel, dim3(s.batch), dim3(threads), 0, st, beside,
                       static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new),
                       static_cast<__nv_bfloat16*>(k_cache), static_cast<__nv_bfloat16*>(v_cache),
                       kq, k_scale, page_table, seq_lens, s.hkv, s.max_pages, s.num_pages, err,
                       beside ? 1 : 0, key_format(s));
}

}  // namespace hsa
