// internal.h -- launch interface between the C-ABI layer (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace hsa {

// Problem sizes copied out of the public descriptor after validation.
struct Shape {
  int batch, hq, hkv, group, max_pages, num_pages;
  int chunk, k1, k2, sink, window;
  int chunk0, k0;  // module 0 (k0 > 0): coarse chunks of chunk0 tokens, top k0
  int key_bits;    // 8: 8-bit key codes [page][hkv][16][128]; 4: 4-bit, [page][hkv][16][64] bytes
  int per_head;    // 1: every query head selects its own blocks (rows = hq, not hkv)
  int key_fp8;     // 1: FP8 E4M3 key codes (8-bit layout), fp32 scores
  int cache_policy;  // block cache victims: 0 least recently used, 1 least cumulative mass
  int kv_div = 1;  // attention rows per kv head (hq / hkv for a per-head attention launch)
  float sm_scale;  // resolved (> 0)
  // rows of the selection (block and tile maxima, kept chunks and blocks) per sequence
  int sel_rows() const { return per_head ? hq : hkv; }
};

// Chunks that module 1 keeps where only the kept blocks are output (the whole decode step):
// min(K1, K2). With K1 >= K2 the two modules keep the top K2 blocks of their candidates
// (ranked by maximum, the lower index first among equals): every chunk ranked above the chunk
// of such a block holds a block ranked above that block (its maximum is at least as large,
// and among equal maxima its blocks have the lower indices), so that chunk has fewer than K2
// chunks above it. The top K2 chunks therefore already hold all K2 blocks, and module 2 then
// ranks half as many candidates at K1 = 2 K2. Measured on GB300: 128K step 43.74 -> 43.41 us,
// 1M 194.5 -> 191.7 us; with a module 0 in front (1M, three modules) 191.5 -> 194.7 us, so
// that stack keeps K1.
#ifndef HSA_SEL_K1_MIN
#define HSA_SEL_K1_MIN 1
#endif
inline int module1_keep(const Shape& s) {
  return HSA_SEL_K1_MIN && s.k0 == 0 && s.k2 < s.k1 ? s.k2 : s.k1;
}

// ---- quantize.cu
cudaError_t launch_key_amax(const Shape& s, const void* k_cache, const int32_t* page_table,
                            const int32_t* seq_lens, unsigned* amax_bits, int* err,
                            cudaStream_t st);
cudaError_t launch_key_codes(const Shape& s, const void* k_cache, const int32_t* page_table,
                             const int32_t* seq_lens, const unsigned* amax_bits,
                             const float* k_scale_in, float* k_scale_out, int append_from,
                             bool full, int8_t* kq, int* err, cudaStream_t st);
// beside: launched to run concurrently with the scorer of the same decode step (see
// hsa_decode_step); false for a standalone append.
cudaError_t launch_append_kv(const Shape& s, const void* k_new, const void* v_new,
                             void* k_cache, void* v_cache, int8_t* kq, const float* k_scale,
                             const int32_t* page_table, const int32_t* seq_lens, int* err,
                             cudaStream_t st, bool beside);

// Copies q [B][Hq][128], k_new and v_new [B][Hkv][128] (bf16, 16-byte aligned, readable by
// the device: mapped pinned host memory) into the device buffers dq, dk_new, dv_new.
cudaError_t launch_stage_io(const Shape& s, const void* q, const void* k_new, const void* v_new,
                            void* dq, void* dk_new, void* dv_new, int num_sms, cudaStream_t st);

// ---- score.cu
// block_max: [B][Hkv][max_pages]; tile_max (nullable): [B][Hkv][score_max_tiles], the max of
// each 64-token tile, which the prune kernel uses as the chunk score when chunks are 64.
// row_range (nullable): [rows][4] words raised by atomicMax to the row's range of maxima,
// (max tile, ~min tile, max block, ~min block) as order-preserving unsigned images
// ((unsigned)v ^ 0x80000000); zero before the scorer runs (a word left from an earlier call
// only widens the range); launch_attend_select reads and clears them.
// app (nullable): the decode step's append of the new token (k_new, v_new [B][Hkv][128] bf16
// into slot N_b - 1 of k_cache / v_cache, its codes into kq), done by the scorer's last CTA
// beside its scan; only valid when that slot is not a candidate (a window of >= 1 token).
struct AppendArgs {
  const void* k_new;
  const void* v_new;
  void* k_cache;
  void* v_cache;
  int8_t* kq;
};
int score_max_tiles(const Shape& s);
cudaError_t launch_score_blocks(const Shape& s, const CUtensorMap& kq_map,
                                const CUtensorMap& kq_map4, const void* q,
                                const float* k_scale, const int32_t* page_table,
                                const int32_t* seq_lens, int32_t* block_max, int32_t* tile_max,
                                unsigned* row_range, const AppendArgs* app, int* err,
                                int num_sms, cudaStream_t st);

// ---- prune.cu
// page_table / sel_pages (both nullable): also write the page of every kept block into
// sel_pages [B][Hkv][K2], entries [0, n_blocks) (for launch_attend's sel_pages).
// row_range (nullable): the scorer's range of each row's maxima (launch_score_blocks);
// module 1 then skips its min/max pass, and the prune clears the words for the next step.
cudaError_t launch_prune(const Shape& s, const int32_t* seq_lens, const int32_t* block_max,
                         const int32_t* tile_max, int32_t* chunk_idx, int32_t* n_chunks,
                         int32_t* block_idx, int32_t* n_blocks, const int32_t* page_table,
                         int32_t* sel_pages, int* err, cudaStream_t st,
                         unsigned* row_range = nullptr);
int prune_max_chunks();
size_t prune_smem_bytes(const Shape& s);

// The GPU block cache: device arrays in one caller-owned, zero-initialised buffer.
struct BlockCache {
  int32_t* header;      // [0]: step counter
  int32_t* slot_of;     // [num_pages * hkv]: slot + 1, 0 when absent
  int32_t* slot_key;    // [capacity]: page * hkv + head + 1, 0 when free
  int32_t* slot_stamp;  // [capacity]: last step that used the slot
  float* mass;          // [num_pages * hkv]: cumulative attention mass of every block
  void* data;           // [capacity][2][16][128] bf16: K block then V block of each slot
  int capacity;
};
// Segments per (sequence, kv head) in the plan's seg_slot and fill arrays.
int block_cache_seg_stride(const Shape& s);
size_t block_cache_plan_smem(const Shape& s, int capacity);
// One CTA: looks up the attention's segments, picks the victims for the misses (least
// recently used, or least cumulative mass with s.cache_policy 1), writes seg_slot
// [B][Hkv][stride] and the fill list (int4 [B * Hkv * stride], count in n_fill).
cudaError_t launch_cache_plan(const Shape& s, const int32_t* seq_lens, const int32_t* page_table,
                              const int32_t* block_idx, const int32_t* n_blocks,
                              const BlockCache& c, int32_t* seg_slot, void* fill,
                              int32_t* n_fill, int* err, cudaStream_t st);

// ---- attend.cu
// early: the caller guarantees that K/V, q, the page table and the lengths are complete when
// the kernel starts (only the selection comes from the previous kernel), as in the whole
// decode step; the sink and window pages are then fetched before waiting for the selection.
struct AttendBuffers {
  float* part_ml;   // [B][Hq][nsplit] (m, l) pairs
  float* part_o;    // [B][Hq][nsplit][128]
  int* counters;    // [B][Hkv]
  int nsplit;
  const int32_t* sel_pages = nullptr;  // optional: the kept blocks' pages, from launch_prune
  const int32_t* seg_slots = nullptr;  // optional: block-cache slots of the segments (then
  int seg_stride = 0;                  // k / v are the cache's K and V halves)
  int cache_capacity = 0;
  // optional, with seg_slots (cache policy 1): seg_l2 [B][Hkv][seg_stride][G] scratch for
  // each segment's log2-domain log-sum-exp per query head; the last CTA of (b, h) adds each
  // segment's attention mass to mass[slot_key[slot] - 1]
  float* seg_l2 = nullptr;
  float* mass = nullptr;
  const int32_t* slot_key = nullptr;
};
// Copies the block cache's fill list (from launch_cache_plan) in from host memory:
// k_host / v_host are device aliases of the pinned host K/V.
cudaError_t launch_cache_fill(const Shape& s, const BlockCache& c, const void* fill,
                              const int32_t* n_fill, const void* k_host, const void* v_host,
                              int* err, int num_sms, cudaStream_t st);
// reserve: leave SMs to a pruning kernel that runs beside the sparse attention
int attend_splits(const Shape& s, bool dense, bool host, int num_sms, bool reserve = true);
cudaError_t launch_attend(const Shape& s, bool dense, bool host, const void* q,
                          const void* k_cache, const void* v_cache, const int32_t* page_table,
                          const int32_t* seq_lens, const int32_t* block_idx,
                          const int32_t* n_blocks, float* out, float* lse,
                          const AttendBuffers& buf, int* err, cudaStream_t st, bool early);

// The whole decode step's sparse attention that runs both pruning modules itself (64-token
// chunks, two modules): s is the attention's shape (rows = selection rows). Reads the
// scorer's block_max / tile_max, writes the kept blocks to block_idx [rows][k2] and their
// count to n_blocks [rows] as launch_prune would, and the attention output. Supported when
// the selection fits the kernel's shared memory (else the pruning kernel and launch_attend).
bool attend_select_supported(const Shape& s, bool page_table_aligned);
cudaError_t launch_attend_select(const Shape& s, const void* q, const void* k_cache,
                                 const void* v_cache, const int32_t* page_table,
                                 const int32_t* seq_lens, const int32_t* block_max,
                                 const int32_t* tile_max, unsigned* row_range,
                                 int32_t* block_idx, int32_t* n_blocks, float* out, float* lse,
                                 const AttendBuffers& buf, int* err, cudaStream_t st);

}  // namespace hsa
