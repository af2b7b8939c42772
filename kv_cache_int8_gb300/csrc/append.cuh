// append.cuh -- the decode step's append of the new token: its bf16 K and V into slot N - 1
// of the paged caches and its key codes with the stored scales. Shared by the append kernel
// (quantize.cu) and the scorer (score.cu), which does it beside its scan in the whole step.
//
// Source: "KV Cache 与长上下文推理", section "KV Cache 回顾" (each decode step appends the new
// token's k and v) and section "KV Cache 量化" (INT8, INT4 and FP8 key formats).
#pragma once

#include "common.cuh"

namespace hsa {
namespace append_detail {

__device__ __forceinline__ void unpack8(const uint4& u, float f[8]) {
  f[0] = bf16_lo(u.x); f[1] = bf16_hi(u.x);
  f[2] = bf16_lo(u.y); f[3] = bf16_hi(u.y);
  f[4] = bf16_lo(u.z); f[5] = bf16_hi(u.z);
  f[6] = bf16_lo(u.w); f[7] = bf16_hi(u.w);
}

// Eight 4-bit codes in one word: code 2i in the low nibble of byte i, code 2i + 1 in the high.
__device__ __forceinline__ uint32_t pack_codes4(const int c[8]) {
  uint32_t r = 0;
#pragma unroll
  for (int i = 0; i < 4; i++)
    r |= (uint32_t)((c[2 * i] & 0xF) | ((c[2 * i + 1] & 0xF) << 4)) << (8 * i);
  return r;
}

__device__ __forceinline__ uint2 pack_codes(const int c[8]) {
  uint2 r;
  r.x = (c[0] & 0xFF) | ((c[1] & 0xFF) << 8) | ((c[2] & 0xFF) << 16) | ((uint32_t)(c[3] & 0xFF) << 24);
  r.y = (c[4] & 0xFF) | ((c[5] & 0xFF) << 8) | ((c[6] & 0xFF) << 16) | ((uint32_t)(c[7] & 0xFF) << 24);
  return r;
}

// The codes of 8 consecutive channels at element offset `off` of the key-code cache:
// 8 bytes of 8-bit codes, or 4 bytes of 4-bit codes at half the offset.
__device__ __forceinline__ void store_codes(int8_t* kq, size_t off, const int c[8], int bits) {
  if (bits == 4)
    *reinterpret_cast<uint32_t*>(kq + off / 2) = pack_codes4(c);
  else
    *reinterpret_cast<uint2*>(kq + off) = pack_codes(c);
}

// Key formats: the integer code widths 8 and 4, and FP8 E4M3 codes (8-bit layout).
constexpr int kFmtFp8 = 0xF8;

// E4M3 codes of four f32 values (byte i of the result <- x[i]): round to nearest even,
// saturating at +-448.
__device__ __forceinline__ uint32_t e4m3x4(const float x[4]) {
  unsigned short lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(x[1]), "f"(x[0]));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(x[3]), "f"(x[2]));
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

// The codes of the 8 values f (channel scales s) at element offset `off`, in format fmt:
// integer codes clamp(rint_even(f32(f / s)), +-levels), or E4M3 codes of f32(f / s); a zero
// scale gives code 0.
__device__ __forceinline__ void store_key_codes(int8_t* kq, size_t off, const float f[8],
                                                const float s[8], int fmt) {
  if (fmt == kFmtFp8) {
    float x[8];
#pragma unroll
    for (int i = 0; i < 8; i++) x[i] = s[i] == 0.0f ? 0.0f : __fdiv_rn(f[i], s[i]);
    *reinterpret_cast<uint2*>(kq + off) = make_uint2(e4m3x4(x), e4m3x4(x + 4));
    return;
  }
  const int levels = key_levels(fmt);
  int c[8];
#pragma unroll
  for (int i = 0; i < 8; i++) c[i] = key_code(f[i], s[i], levels);
  store_codes(kq, off, c, fmt);
}

}  // namespace append_detail

// Thread slot t (of hkv * 16) of sequence b: kv head t / 16, channels [8 (t % 16), +8) of the
// token at slot N_b - 1. Bad lengths or pages set the error word and write nothing.
__device__ __forceinline__ void append_token(int b, int t, const uint4* __restrict__ k_new,
                                             const uint4* __restrict__ v_new,
                                             __nv_bfloat16* k_cache, __nv_bfloat16* v_cache,
                                             int8_t* kq, const float* __restrict__ k_scale,
                                             const int32_t* __restrict__ page_table,
                                             const int32_t* __restrict__ seq_lens, int hkv,
                                             int max_pages, int num_pages, int* err, int bits) {
  const int h = t >> 4, grp = t & 15;
  if (h >= hkv) return;
  const int n = seq_lens[b];
  if (n < 1 || n > max_pages * kPage) {
    set_error(err, kDevErrCheck);
    return;
  }
  const int tok = n - 1;
  const int page = page_table[(size_t)b * max_pages + tok / kPage];
  if (page < 0 || page >= num_pages) {
    set_error(err, kDevErrCheck);
    return;
  }
  const size_t off = (((size_t)page * hkv + h) * kPage + tok % kPage) * kHeadDim + grp * 8;
  const size_t src = ((size_t)b * hkv + h) * (kHeadDim / 8) + grp;
  const uint4 kv = k_new[src];
  *reinterpret_cast<uint4*>(k_cache + off) = kv;
  *reinterpret_cast<uint4*>(v_cache + off) = v_new[src];
  float f[8];
  append_detail::unpack8(kv, f);
  const float* s = k_scale + ((size_t)b * hkv + h) * kHeadDim + grp * 8;
  append_detail::store_key_codes(kq, off, f, s, bits);
}

}  // namespace hsa
