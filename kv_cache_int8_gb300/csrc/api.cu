// api.cu -- the C ABI of libhsa (declared in include/hsa.h): argument checks, workspace
// layout, TMA descriptor encoding and kernel launches. No allocation, no synchronisation
// (hsa_read_device_error excepted), no abort.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/hsa.h"
#include "common.cuh"
#include "internal.h"

namespace {

using hsa::Shape;

constexpr size_t kAlign = 256;
constexpr size_t kErrBytes = 256;   // the error word sits at offset 0 of every workspace
constexpr int kMaxSplits = 64;      // split-K partial buffers are sized for this many
constexpr int kMaxBatch = 1024;
constexpr int kMaxHkv = 64;

inline size_t up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

inline bool aligned(const void* p, size_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

// Structural checks of the descriptor; fills `s`. `need_prune` adds the module fields.
int32_t check_dims(const hsa_dims* d, Shape& s, bool need_prune) {
  if (d == nullptr) return HSA_ERR_INVALID_ARG;
  if (d->batch < 1 || d->hq < 1 || d->hkv < 1 || d->max_pages_per_seq < 1 || d->num_pages < 1)
    return HSA_ERR_INVALID_ARG;
  if (d->hq % d->hkv != 0) return HSA_ERR_INVALID_ARG;
  if (d->head_dim != hsa::kHeadDim || d->page_size != hsa::kPage) return HSA_ERR_UNSUPPORTED;
  const int g = d->hq / d->hkv;
  if (g != 1 && g != 2 && g != 4 && g != 8) return HSA_ERR_UNSUPPORTED;
  if (d->batch > kMaxBatch || d->hkv > kMaxHkv) return HSA_ERR_UNSUPPORTED;
  if ((long long)d->num_pages * d->hkv * hsa::kPage > INT32_MAX ||
      (long long)d->max_pages_per_seq * hsa::kPage > INT32_MAX / 2)
    return HSA_ERR_UNSUPPORTED;
  if (d->sink < 0 || d->window < 0 || d->k1 < 0 || d->k2 < 0 || d->k0 < 0)
    return HSA_ERR_INVALID_ARG;
  if (need_prune) {
    if (d->block != hsa::kPage) return HSA_ERR_UNSUPPORTED;
    if (d->chunk <= 0 || d->chunk % d->block != 0) return HSA_ERR_INVALID_ARG;
    if (d->k0 > 0 && (d->chunk0 < d->chunk || d->chunk0 % d->chunk != 0))
      return HSA_ERR_INVALID_ARG;
  }
  if (!(d->sm_scale == d->sm_scale)) return HSA_ERR_INVALID_ARG;  // NaN
  if (d->key_bits != 0 && d->key_bits != 4 && d->key_bits != 8) return HSA_ERR_UNSUPPORTED;
  if (d->per_head != 0 && d->per_head != 1) return HSA_ERR_INVALID_ARG;
  if (d->key_fp8 != 0 && d->key_fp8 != 1) return HSA_ERR_INVALID_ARG;
  if (d->key_fp8 && d->key_bits == 4) return HSA_ERR_UNSUPPORTED;
  if (d->cache_policy != 0 && d->cache_policy != 1) return HSA_ERR_INVALID_ARG;
  s.batch = d->batch;
  s.hq = d->hq;
  s.hkv = d->hkv;
  s.group = g;
  s.max_pages = d->max_pages_per_seq;
  s.num_pages = d->num_pages;
  s.chunk = d->chunk;
  s.k1 = d->k1;
  s.k2 = d->k2;
  s.sink = d->sink;
  s.window = d->window;
  s.chunk0 = d->k0 > 0 ? d->chunk0 : 0;
  s.k0 = d->k0;
  s.key_bits = d->key_bits == 4 ? 4 : 8;
  s.per_head = d->per_head;
  s.key_fp8 = d->key_fp8;
  s.cache_policy = d->cache_policy;
  s.kv_div = 1;
  s.sm_scale = d->sm_scale > 0.0f ? d->sm_scale : 1.0f / std::sqrt((float)hsa::kHeadDim);
  return HSA_OK;
}

// ---- workspace layouts
size_t quantize_ws(const Shape& s) { return kErrBytes + up((size_t)s.batch * s.hkv * hsa::kHeadDim * 4); }
size_t select_bm_bytes(const Shape& s) {
  return up((size_t)s.batch * s.sel_rows() * s.max_pages * 4);
}
size_t select_tm_bytes(const Shape& s) {
  return up((size_t)s.batch * s.sel_rows() * hsa::score_max_tiles(s) * 4);
}
// The prune works on selection rows: one per kv head, or one per query head.
Shape prune_shape(const Shape& s) {
  Shape p = s;
  p.hkv = s.sel_rows();
  return p;
}
// The sparse attention with per-head selection: one attention row per query head (group of
// one), reading K/V of kv head row / kv_div.
Shape attend_shape(const Shape& s, bool dense) {
  Shape a = s;
  if (s.per_head && !dense) {
    a.hkv = s.hq;
    a.group = 1;
    a.kv_div = s.group;
  }
  return a;
}
size_t select_ws(const Shape& s) { return kErrBytes + select_bm_bytes(s) + select_tm_bytes(s); }
struct AttendLayout {
  size_t counters, part_ml, part_o, end;
};
AttendLayout attend_layout(const Shape& s, size_t base) {
  AttendLayout l;
  l.counters = base;
  l.part_ml = l.counters + up((size_t)s.batch * s.sel_rows() * 4);
  l.part_o = l.part_ml + up((size_t)s.batch * s.hq * kMaxSplits * 2 * 4);
  l.end = l.part_o + up((size_t)s.batch * s.hq * kMaxSplits * hsa::kHeadDim * 4);
  return l;
}
size_t attend_ws(const Shape& s) { return attend_layout(s, kErrBytes).end; }

// Per-call scratch of the block cache: seg_slot [B][Hkv][stride], the fill list, its count,
// and with cache policy 1 each segment's log-sum-exp per query head, seg_l2 [..][stride][G].
struct CacheScratch {
  size_t seg_slot, fill, n_fill, seg_l2, end;
};
CacheScratch cache_scratch(const Shape& s, size_t base) {
  const size_t F = (size_t)s.batch * s.hkv * hsa::block_cache_seg_stride(s);
  CacheScratch c;
  c.seg_slot = base;
  c.fill = c.seg_slot + up(F * 4);
  c.n_fill = c.fill + up(F * 16);
  c.seg_l2 = c.n_fill + kAlign;
  c.end = c.seg_l2 + (s.cache_policy == 1 ? up(F * s.group * 4) : 0);
  return c;
}
size_t cached_ws(const Shape& s) {
  return cache_scratch(s, attend_layout(s, kErrBytes).end).end;
}

// The block cache buffer: header, slot_of [num_pages * hkv], slot_key / slot_stamp
// [capacity], mass [num_pages * hkv] (fp32 cumulative attention mass), data [capacity][8 KiB].
constexpr int kMaxCacheSlots = 32768;
constexpr int kMaxMassSegments = 8192;  // segments per (sequence, kv head), cache policy 1
struct CacheLayout {
  size_t slot_of, slot_key, slot_stamp, mass, data, end;
};
CacheLayout cache_layout(const Shape& s, int capacity) {
  CacheLayout l;
  l.slot_of = kAlign;
  l.slot_key = l.slot_of + up((size_t)s.num_pages * s.hkv * 4);
  l.slot_stamp = l.slot_key + up((size_t)capacity * 4);
  l.mass = l.slot_stamp + up((size_t)capacity * 4);
  l.data = l.mass + up((size_t)s.num_pages * s.hkv * 4);
  l.end = l.data + (size_t)capacity * 2 * hsa::kBlockBytesBf16;
  return l;
}
// The capacity must hold one call's working set (every segment of every (sequence, kv
// head)) and fit the plan's shared memory.
int32_t check_cache_capacity(const Shape& s, int capacity) {
  if (capacity < s.batch * s.hkv * hsa::block_cache_seg_stride(s)) return HSA_ERR_INVALID_ARG;
  if (capacity > kMaxCacheSlots) return HSA_ERR_UNSUPPORTED;
  // the mass policy's combine stages two words a segment in the attention's ring
  if (s.cache_policy == 1 && hsa::block_cache_seg_stride(s) > kMaxMassSegments)
    return HSA_ERR_UNSUPPORTED;
  if (hsa::block_cache_plan_smem(s, capacity) > 227 * 1024) return HSA_ERR_UNSUPPORTED;
  return HSA_OK;
}
hsa::BlockCache block_cache_at(const Shape& s, void* buf, int capacity) {
  const CacheLayout l = cache_layout(s, capacity);
  char* p = static_cast<char*>(buf);
  hsa::BlockCache c;
  c.header = reinterpret_cast<int32_t*>(p);
  c.slot_of = reinterpret_cast<int32_t*>(p + l.slot_of);
  c.slot_key = reinterpret_cast<int32_t*>(p + l.slot_key);
  c.slot_stamp = reinterpret_cast<int32_t*>(p + l.slot_stamp);
  c.mass = reinterpret_cast<float*>(p + l.mass);
  c.data = p + l.data;
  c.capacity = capacity;
  return c;
}

struct StepLayout {
  size_t block_max, tile_max, row_range, block_idx, n_blocks, sel_pages, q, k_new, v_new, out,
      lse;
  AttendLayout att;
  CacheScratch cache;
  size_t end;
};
StepLayout step_layout(const Shape& s) {
  StepLayout l;
  l.block_max = kErrBytes;
  l.tile_max = l.block_max + select_bm_bytes(s);
  l.row_range = l.tile_max + select_tm_bytes(s);  // [B][rows][4] words
  l.block_idx = l.row_range + up((size_t)s.batch * s.sel_rows() * 16);
  l.n_blocks = l.block_idx + up((size_t)s.batch * s.sel_rows() * std::max(s.k2, 1) * 4);
  l.sel_pages = l.n_blocks + up((size_t)s.batch * s.sel_rows() * 4);
  l.q = l.sel_pages + up((size_t)s.batch * s.sel_rows() * std::max(s.k2, 1) * 4);
  l.k_new = l.q + up((size_t)s.batch * s.hq * hsa::kHeadDim * 2);
  l.v_new = l.k_new + up((size_t)s.batch * s.hkv * hsa::kHeadDim * 2);
  l.out = l.v_new + up((size_t)s.batch * s.hkv * hsa::kHeadDim * 2);
  l.lse = l.out + up((size_t)s.batch * s.hq * hsa::kHeadDim * 4);
  l.att = attend_layout(s, l.lse + up((size_t)s.batch * s.hq * 4));
  l.cache = cache_scratch(s, l.att.end);
  l.end = l.cache.end;
  return l;
}

int32_t check_ws(const Shape& s, void* ws, size_t bytes, size_t need) {
  if (ws == nullptr || !aligned(ws, kAlign)) return HSA_ERR_INVALID_ARG;
  if (bytes < need) return HSA_ERR_WORKSPACE_TOO_SMALL;
  (void)s;
  return HSA_OK;
}

// ---- device facts (cached per device)
int num_sms() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  int v = cache[dev].load();
  if (v == 0) {
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
      v = 148;
    cache[dev].store(v);
  }
  return v;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Two views of the key-code cache, both stored with the 128-byte swizzle. map: 2-D, rows of
// 128 bytes (one token of 8-bit codes, two of 4-bit codes), a box is one (page, head) block.
// map4: 4-D [page][head][row][128 B], a box is the blocks of one head in 4 consecutive pages
// (one copy instead of four where the page table is contiguous).
int32_t encode_kq_map(const Shape& s, const int8_t* kq, CUtensorMap* map, CUtensorMap* map4) {
  // the maps depend only on the base pointer and the shape: this thread keeps the pairs of
  // the last kKeep code caches it saw (a model's layers each have their own), replaced in turn
  struct Entry {
    const int8_t* kq = nullptr;
    long long pages = -1;
    int hkv = -1, rows_per_block = -1;
    CUtensorMap map, map4;
  };
  constexpr int kKeep = 64;
  thread_local Entry kept[kKeep];
  thread_local int next = 0;
  // 8-bit codes: one 128-byte row per token, 16 rows a block; 4-bit: two tokens a row
  const int rows_per_block = s.key_bits == 4 ? hsa::kPage / 2 : hsa::kPage;
  const long long rows = (long long)s.num_pages * s.hkv * rows_per_block;
  for (int i = 0; i < kKeep; i++) {
    const Entry& e = kept[i];
    if (e.kq == kq && e.pages == s.num_pages && e.hkv == s.hkv &&
        e.rows_per_block == rows_per_block) {
      *map = e.map;
      *map4 = e.map4;
      return HSA_OK;
    }
  }
  auto fn = encode_fn();
  if (fn == nullptr) return HSA_ERR_CUDA;
  cuuint64_t dims[2] = {(cuuint64_t)hsa::kHeadDim, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)hsa::kHeadDim};
  cuuint32_t box[2] = {(cuuint32_t)hsa::kHeadDim, (cuuint32_t)rows_per_block};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<int8_t*>(kq), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return HSA_ERR_CUDA;
  const cuuint64_t blk = (cuuint64_t)rows_per_block * hsa::kHeadDim;  // bytes per block
  cuuint64_t dims4[4] = {(cuuint64_t)hsa::kHeadDim, (cuuint64_t)rows_per_block,
                         (cuuint64_t)s.hkv, (cuuint64_t)s.num_pages};
  cuuint64_t strides4[3] = {(cuuint64_t)hsa::kHeadDim, blk, blk * s.hkv};
  cuuint32_t box4[4] = {(cuuint32_t)hsa::kHeadDim, (cuuint32_t)rows_per_block, 1, 4};
  r = fn(map4, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<int8_t*>(kq), dims4, strides4, box4,
         estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return HSA_ERR_CUDA;
  Entry& e = kept[next];
  next = (next + 1) % kKeep;
  e.kq = kq;
  e.pages = s.num_pages;
  e.hkv = s.hkv;
  e.rows_per_block = rows_per_block;
  e.map = *map;
  e.map4 = *map4;
  return HSA_OK;
}

// Whether kernels of the current device address host memory by its host pointers: the GPU
// reaches pageable memory through the host's own page tables (address translation services
// over a coherent link), so a host buffer, pinned or not, needs no alias lookup. Queried once
// per device; the lookups it saves cost a few microseconds each per call.
bool host_pointers_direct() {
  static std::atomic<int> cache[64];  // 0 unknown, 1 direct, 2 aliases needed
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  int v = cache[dev].load();
  if (v == 0) {
    int pageable = 0, host_tables = 0;
    if (cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccess, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&host_tables, cudaDevAttrPageableMemoryAccessUsesHostPageTables,
                               dev) != cudaSuccess) {
      cudaGetLastError();
      pageable = 0;
    }
    v = (pageable && host_tables) ? 1 : 2;
    cache[dev].store(v);
  }
  return v == 1;
}

// Device alias of a host buffer the GPU can address (mapped pinned memory, or any host
// memory with host_pointers_direct); false (error state cleared) if it has none.
bool host_alias(const void* p, void** out) {
  if (host_pointers_direct()) {
    *out = const_cast<void*>(p);
    return true;
  }
  void* dp = nullptr;
  if (cudaHostGetDevicePointer(&dp, const_cast<void*>(p), 0) != cudaSuccess || dp == nullptr) {
    cudaGetLastError();
    return false;
  }
  *out = dp;
  return true;
}

// Device alias of a pinned host buffer (kv_on_host) or the pointer itself.
int32_t kv_pointer(const hsa_dims* d, const void* p, const void** out) {
  if (!d->kv_on_host || host_pointers_direct()) {
    *out = p;
    return HSA_OK;
  }
  void* dp = nullptr;
  if (cudaHostGetDevicePointer(&dp, const_cast<void*>(p), 0) != cudaSuccess || dp == nullptr) {
    cudaGetLastError();
    return HSA_ERR_INVALID_ARG;
  }
  *out = dp;
  return HSA_OK;
}

// The scratch of hsa_select_noalloc: one fixed 4 MiB array of device memory that every GPU
// loading the library holds until the process exits (word 0: its device error word).
constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;
__device__ __align__(256) static unsigned char g_select_scratch[kNoAllocScratchBytes];

// Device address of g_select_scratch in the current device's context. Host code sees only a
// stand-in for the array, never its device address; the lookup is a host-side table lookup
// once the library's device code is loaded (the first lookup on a device loads it), and is
// made on every call so that it always matches the current context.
int32_t noalloc_scratch(char** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_select_scratch) != cudaSuccess || p == nullptr) {
    cudaGetLastError();
    return HSA_ERR_CUDA;
  }
  *out = static_cast<char*>(p);
  return HSA_OK;
}

inline int32_t cuda_status(cudaError_t e) { return e == cudaSuccess ? HSA_OK : HSA_ERR_CUDA; }

inline cudaStream_t as_stream(void* p) { return reinterpret_cast<cudaStream_t>(p); }

int32_t do_score(const Shape& s, const void* q, const int8_t* kq, const float* k_scale,
                 const int32_t* page_table, const int32_t* seq_lens, int32_t* block_max,
                 int32_t* tile_max, int* err, cudaStream_t st, unsigned* row_range = nullptr,
                 const hsa::AppendArgs* app = nullptr) {
  CUtensorMap map, map4;
  int32_t rc = encode_kq_map(s, kq, &map, &map4);
  if (rc != HSA_OK) return rc;
  return cuda_status(hsa::launch_score_blocks(s, map, map4, q, k_scale, page_table, seq_lens,
                                              block_max, tile_max, row_range, app, err,
                                              num_sms(), st));
}

int32_t check_prune_fits(const Shape& s0) {
  const Shape s = prune_shape(s0);
  const long long n1max = ((long long)s.max_pages * hsa::kPage + s.chunk - 1) / s.chunk;
  if (n1max > hsa::prune_max_chunks()) return HSA_ERR_UNSUPPORTED;
  if (hsa::prune_smem_bytes(s) > 227 * 1024) return HSA_ERR_UNSUPPORTED;
  return HSA_OK;
}

int32_t do_attend(const hsa_dims* d, const Shape& s, bool dense, const void* q, const void* k,
                  const void* v, const int32_t* pt, const int32_t* lens, const int32_t* bidx,
                  const int32_t* nb, float* out, float* lse, char* ws, const AttendLayout& l,
                  cudaStream_t st, bool early, const int32_t* sel_pages = nullptr) {
  const void* kd = nullptr;
  const void* vd = nullptr;
  int32_t rc = kv_pointer(d, k, &kd);
  if (rc != HSA_OK) return rc;
  rc = kv_pointer(d, v, &vd);
  if (rc != HSA_OK) return rc;
  const bool host = d->kv_on_host != 0;
  hsa::AttendBuffers buf;
  buf.counters = reinterpret_cast<int*>(ws + l.counters);
  buf.part_ml = reinterpret_cast<float*>(ws + l.part_ml);
  buf.part_o = reinterpret_cast<float*>(ws + l.part_o);
  buf.sel_pages = sel_pages;
  const Shape sa = attend_shape(s, dense);
  // SMs are left free only for a pruning kernel that runs beside an early attention
  buf.nsplit = std::min(kMaxSplits, hsa::attend_splits(sa, dense, host, num_sms(), early));
  return cuda_status(hsa::launch_attend(sa, dense, host, q, kd, vd, pt, lens, bidx, nb, out, lse,
                                        buf, reinterpret_cast<int*>(ws), st, early));
}

// The attention over K/V in host memory through the block cache: plan (lookups, victims),
// fill (the misses copied in over the host link), then the HBM attention reading the slots.
// kd / vd: device aliases of the host K/V.
int32_t do_attend_cached(const Shape& s, const void* q, const void* kd, const void* vd,
                         const int32_t* pt, const int32_t* lens, const int32_t* bidx,
                         const int32_t* nb, float* out, float* lse, char* ws,
                         const AttendLayout& l, const CacheScratch& cs, void* cache,
                         int capacity, cudaStream_t st) {
  int* err = reinterpret_cast<int*>(ws);
  const hsa::BlockCache c = block_cache_at(s, cache, capacity);
  int32_t* seg_slot = reinterpret_cast<int32_t*>(ws + cs.seg_slot);
  void* fill = ws + cs.fill;
  int32_t* n_fill = reinterpret_cast<int32_t*>(ws + cs.n_fill);
  if (hsa::launch_cache_plan(s, lens, pt, bidx, nb, c, seg_slot, fill, n_fill, err, st) !=
      cudaSuccess)
    return HSA_ERR_CUDA;
  if (hsa::launch_cache_fill(s, c, fill, n_fill, kd, vd, err, num_sms(), st) != cudaSuccess)
    return HSA_ERR_CUDA;
  hsa::AttendBuffers buf;
  buf.counters = reinterpret_cast<int*>(ws + l.counters);
  buf.part_ml = reinterpret_cast<float*>(ws + l.part_ml);
  buf.part_o = reinterpret_cast<float*>(ws + l.part_o);
  buf.nsplit = std::min(kMaxSplits, hsa::attend_splits(s, false, false, num_sms()));
  buf.seg_slots = seg_slot;
  buf.seg_stride = hsa::block_cache_seg_stride(s);
  buf.cache_capacity = capacity;
  if (s.cache_policy == 1) {
    buf.seg_l2 = reinterpret_cast<float*>(ws + cs.seg_l2);
    buf.mass = c.mass;
    buf.slot_key = c.slot_key;
  }
  const char* data = static_cast<const char*>(c.data);
  return cuda_status(hsa::launch_attend(s, false, false, q, data, data + hsa::kBlockBytesBf16, pt,
                                        lens, bidx, nb, out, lse, buf, err, st, false));
}

// The outputs of a host-I/O step that were computed into the workspace: copied back.
int32_t copy_outputs_back(const Shape& s, const hsa_step_io* io, const float* out,
                          const float* lse, bool direct_out, cudaStream_t st) {
  if (!io->io_on_host || direct_out) return HSA_OK;
  cudaError_t e = cudaMemcpyAsync(io->out, out, (size_t)s.batch * s.hq * hsa::kHeadDim * 4,
                                  cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess && io->lse)
    e = cudaMemcpyAsync(io->lse, lse, (size_t)s.batch * s.hq * 4, cudaMemcpyDeviceToHost, st);
  return e == cudaSuccess ? HSA_OK : HSA_ERR_CUDA;
}

}  // namespace

extern "C" {

size_t hsa_workspace_bytes(const hsa_dims* d, int32_t op) {
  Shape s;
  const bool prune = op == HSA_OP_SELECT || op == HSA_OP_STEP;
  if (check_dims(d, s, prune) != HSA_OK) return 0;
  switch (op) {
    case HSA_OP_QUANTIZE: return quantize_ws(s);
    case HSA_OP_SELECT: return select_ws(s);
    case HSA_OP_ATTEND:
    case HSA_OP_DENSE: return attend_ws(s);
    case HSA_OP_STEP: return step_layout(s).end;
    case HSA_OP_CACHED: return cached_ws(s);
    default: return 0;
  }
}

const char* hsa_status_string(int32_t status) {
  switch (status) {
    case HSA_OK: return "ok";
    case HSA_ERR_INVALID_ARG: return "invalid argument";
    case HSA_ERR_UNSUPPORTED: return "unsupported shape";
    case HSA_ERR_CUDA: return "CUDA error";
    case HSA_ERR_TIMEOUT: return "device wait timed out";
    case HSA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case HSA_ERR_DEVICE_CHECK: return "device bounds check failed";
    default: return "unknown status";
  }
}

int32_t hsa_quantize_keys(const hsa_dims* d, const void* k_cache, const int32_t* page_table,
                          const int32_t* seq_lens, int32_t mode, int32_t append_from,
                          int8_t* kq, float* k_scale, void* workspace, size_t workspace_bytes,
                          void* stream) {
  Shape s;
  int32_t rc = check_dims(d, s, false);
  if (rc != HSA_OK) return rc;
  if (!k_cache || !page_table || !seq_lens || !kq || !k_scale) return HSA_ERR_INVALID_ARG;
  if (!aligned(k_cache, 16) || !aligned(kq, 16) || !aligned(k_scale, 16)) return HSA_ERR_INVALID_ARG;
  if (mode != 0 && mode != 1) return HSA_ERR_INVALID_ARG;
  const void* kd = nullptr;
  rc = kv_pointer(d, k_cache, &kd);
  if (rc != HSA_OK) return rc;
  cudaStream_t st = as_stream(stream);
  if (mode == 0) {
    rc = check_ws(s, workspace, workspace_bytes, quantize_ws(s));
    if (rc != HSA_OK) return rc;
    char* ws = static_cast<char*>(workspace);
    unsigned* amax = reinterpret_cast<unsigned*>(ws + kErrBytes);
    int* err = reinterpret_cast<int*>(ws);
    cudaError_t e = cudaMemsetAsync(amax, 0, (size_t)s.batch * s.hkv * hsa::kHeadDim * 4, st);
    if (e == cudaSuccess) e = hsa::launch_key_amax(s, kd, page_table, seq_lens, amax, err, st);
    if (e == cudaSuccess)
      e = hsa::launch_key_codes(s, kd, page_table, seq_lens, amax, nullptr, k_scale, 0, true, kq,
                                err, st);
    return cuda_status(e);
  }
  if (append_from >= s.max_pages * hsa::kPage) return HSA_ERR_INVALID_ARG;
  int* err = nullptr;
  if (workspace != nullptr) {
    if (!aligned(workspace, kAlign) || workspace_bytes < kErrBytes) return HSA_ERR_INVALID_ARG;
    err = static_cast<int*>(workspace);
  }
  return cuda_status(hsa::launch_key_codes(s, kd, page_table, seq_lens, nullptr, k_scale, nullptr,
                                           append_from, false, kq, err, st));
}

int32_t hsa_append_kv(const hsa_dims* d, const void* k_new, const void* v_new, void* k_cache,
                      void* v_cache, int8_t* kq, const float* k_scale,
                      const int32_t* page_table, const int32_t* seq_lens, void* stream) {
  Shape s;
  int32_t rc = check_dims(d, s, false);
  if (rc != HSA_OK) return rc;
  if (!k_new || !v_new || !k_cache || !v_cache || !kq || !k_scale || !page_table || !seq_lens)
    return HSA_ERR_INVALID_ARG;
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) ||
      !aligned(v_cache, 16) || !aligned(kq, 16))
    return HSA_ERR_INVALID_ARG;
  const void* kd = nullptr;
  const void* vd = nullptr;
  rc = kv_pointer(d, k_cache, &kd);
  if (rc != HSA_OK) return rc;
  rc = kv_pointer(d, v_cache, &vd);
  if (rc != HSA_OK) return rc;
  return cuda_status(hsa::launch_append_kv(s, k_new, v_new, const_cast<void*>(kd),
                                           const_cast<void*>(vd), kq, k_scale, page_table,
                                           seq_lens, nullptr, as_stream(stream), false));
}

int32_t hsa_score_blocks(const hsa_dims* d, const void* q, const int8_t* kq,
                         const float* k_scale, const int32_t* page_table,
                         const int32_t* seq_lens, int32_t* block_max, int32_t* tile_max,
                         void* stream) {
  Shape s;
  int32_t rc = check_dims(d, s, false);
  if (rc != HSA_OK) return rc;
  if (!q || !kq || !k_scale || !page_table || !seq_lens || !block_max) return HSA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(kq, 16) || !aligned(k_scale, 16)) return HSA_ERR_INVALID_ARG;
  return do_score(s, q, kq, k_scale, page_table, seq_lens, block_max, tile_max, nullptr,
                  as_stream(stream));
}

int32_t hsa_prune(const hsa_dims* d, const int32_t* seq_lens, const int32_t* block_max,
                  const int32_t* tile_max, int32_t* chunk_idx, int32_t* n_chunks,
                  int32_t* block_idx, int32_t* n_blocks, void* stream) {
  Shape s;
  int32_t rc = check_dims(d, s, true);
  if (rc != HSA_OK) return rc;
  if (!seq_lens || !block_max || !n_blocks || (!block_idx && s.k2 > 0)) return HSA_ERR_INVALID_ARG;
  if (!aligned(block_max, 16) || !aligned(tile_max, 16)) return HSA_ERR_INVALID_ARG;
  rc = check_prune_fits(s);
  if (rc != HSA_OK) return rc;
  return cuda_status(hsa::launch_prune(prune_shape(s), seq_lens, block_max, tile_max, chunk_idx,
                                       n_chunks, block_idx, n_blocks, nullptr, nullptr, nullptr,
                                       as_stream(stream)));
}

int32_t hsa_select(const hsa_dims* d, const void* q, const int8_t* kq, const float* k_scale,
                   const int32_t* page_table, const int32_t* seq_lens, int32_t* chunk_idx,
                   int32_t* n_chunks, int32_t* block_idx, int32_t* n_blocks, void* workspace,
                   size_t workspace_bytes, void* stream) {
  Shape s;
  int32_t rc = check_dims(d, s, true);
  if (rc != HSA_OK) return rc;
  if (!q || !kq || !k_scale || !page_table || !seq_lens || !n_blocks || (!block_idx && s.k2 > 0))
    return HSA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(kq, 16) || !aligned(k_scale, 16)) return HSA_ERR_INVALID_ARG;
  rc = check_prune_fits(s);
  if (rc != HSA_OK) return rc;
  rc = check_ws(s, workspace, workspace_bytes, select_ws(s));
  if (rc != HSA_OK) return rc;
  char* ws = static_cast<char*>(workspace);
  int* err = reinterpret_cast<int*>(ws);
  int32_t* bm = reinterpret_cast<int32_t*>(ws + kErrBytes);
  int32_t* tm = reinterpret_cast<int32_t*>(ws + kErrBytes + select_bm_bytes(s));
  cudaStream_t st = as_stream(stream);
  rc = do_score(s, q, kq, k_scale, page_table, seq_lens, bm, tm, err, st);
  if (rc != HSA_OK) return rc;
  return cuda_status(hsa::launch_prune(prune_shape(s), seq_lens, bm, tm, chunk_idx, n_chunks,
                                       block_idx, n_blocks, nullptr, nullptr, err, st));
}

int32_t hsa_attend(const hsa_dims* d, const void* q, const void* k_cache, const void* v_cache,
                   const int32_t* page_table, const int32_t* seq_lens, const int32_t* block_idx,
                   const int32_t* n_blocks, float* out, float* lse, void* workspace,
                   size_t workspace_bytes, void* stream) {
  Shape s;
  int32_t rc = check_dims(d, s, false);
  if (rc != HSA_OK) return rc;
  if (!q || !k_cache || !v_cache || !page_table || !seq_lens || !n_blocks || !out ||
      (!block_idx && s.k2 > 0))
    return HSA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16))
    return HSA_ERR_INVALID_ARG;
  rc = check_ws(s, workspace, workspace_bytes, attend_ws(s));
  if (rc != HSA_OK) return rc;
  char* ws = static_cast<char*>(workspace);
  return do_attend(d, s, false, q, k_cache, v_cache, page_table, seq_lens, block_idx, n_blocks,
                   out, lse, ws, attend_layout(s, kErrBytes), as_stream(stream), false);
}

int32_t dense_decode(const hsa_dims* d, const void* q, const void* k_cache, const void* v_cache,
                     const int32_t* page_table, const int32_t* seq_lens, float* out, float* lse,
                     void* workspace, size_t workspace_bytes, void* stream) {
  Shape s;
  int32_t rc = check_dims(d, s, false);
  if (rc != HSA_OK) return rc;
  if (!q || !k_cache || !v_cache || !page_table || !seq_lens || !out) return HSA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16))
    return HSA_ERR_INVALID_ARG;
  rc = check_ws(s, workspace, workspace_bytes, attend_ws(s));
  if (rc != HSA_OK) return rc;
  char* ws = static_cast<char*>(workspace);
  return do_attend(d, s, true, q, k_cache, v_cache, page_table, seq_lens, nullptr, nullptr, out,
                   lse, ws, attend_layout(s, kErrBytes), as_stream(stream), false);
}

// The whole step (reuse = false) or its append + attend with a selection given by the
// caller (reuse = true: block_idx / n_blocks are inputs).
static int32_t decode_step_impl(const hsa_dims* d, const hsa_step_io* io, void* k_cache,
                                void* v_cache, int8_t* kq, const float* k_scale,
                                const int32_t* page_table, const int32_t* seq_lens,
                                int32_t* block_idx, int32_t* n_blocks, void* workspace,
                                size_t workspace_bytes, void* stream, bool reuse,
                                void* block_cache = nullptr, int32_t capacity = 0) {
  Shape s;
  int32_t rc = check_dims(d, s, !reuse);
  if (rc != HSA_OK) return rc;
  if (block_cache != nullptr) {
    if (s.per_head) return HSA_ERR_UNSUPPORTED;  // the cache plan works per kv head
    if (!d->kv_on_host || !aligned(block_cache, kAlign)) return HSA_ERR_INVALID_ARG;
    rc = check_cache_capacity(s, capacity);
    if (rc != HSA_OK) return rc;
  }
  if (!io || !io->q || !io->k_new || !io->v_new || !io->out || !k_cache || !v_cache || !kq ||
      !k_scale || !page_table || !seq_lens)
    return HSA_ERR_INVALID_ARG;
  if (reuse && s.k2 > 0 && (!block_idx || !n_blocks)) return HSA_ERR_INVALID_ARG;
  if (!aligned(io->q, 16) || !aligned(io->k_new, 16) || !aligned(io->v_new, 16) ||
      !aligned(io->out, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(kq, 16) || !aligned(k_scale, 16))
    return HSA_ERR_INVALID_ARG;
  if (!reuse) {
    rc = check_prune_fits(s);
    if (rc != HSA_OK) return rc;
  }
  const StepLayout l = step_layout(s);
  rc = check_ws(s, workspace, workspace_bytes, l.end);
  if (rc != HSA_OK) return rc;
  char* ws = static_cast<char*>(workspace);
  int* err = reinterpret_cast<int*>(ws);
  cudaStream_t st = as_stream(stream);
  const void* q = io->q;
  const void* kn = io->k_new;
  const void* vn = io->v_new;
  float* out = io->out;
  float* lse = io->lse;
  const size_t qb = (size_t)s.batch * s.hq * hsa::kHeadDim * 2;
  const size_t kvb = (size_t)s.batch * s.hkv * hsa::kHeadDim * 2;
  // Host I/O: with mapped pinned buffers (the default for pinned memory on this platform) a
  // small kernel stages the inputs and the attend writes the outputs straight to host
  // memory; otherwise copy-engine transfers through the workspace.
  bool direct_out = false;
  if (io->io_on_host) {
    void *hq = nullptr, *hkn = nullptr, *hvn = nullptr, *hout = nullptr, *hlse = nullptr;
    const bool mapped = host_alias(io->q, &hq) && host_alias(io->k_new, &hkn) &&
                        host_alias(io->v_new, &hvn) && host_alias(io->out, &hout) &&
                        (io->lse == nullptr || host_alias(io->lse, &hlse));
    if (mapped) {
      if (hsa::launch_stage_io(s, hq, hkn, hvn, ws + l.q, ws + l.k_new, ws + l.v_new, num_sms(),
                               st) != cudaSuccess)
        return HSA_ERR_CUDA;
      out = static_cast<float*>(hout);
      lse = static_cast<float*>(hlse);
      direct_out = true;
    } else {
      cudaError_t e = cudaMemcpyAsync(ws + l.q, io->q, qb, cudaMemcpyHostToDevice, st);
      if (e == cudaSuccess)
        e = cudaMemcpyAsync(ws + l.k_new, io->k_new, kvb, cudaMemcpyHostToDevice, st);
      if (e == cudaSuccess)
        e = cudaMemcpyAsync(ws + l.v_new, io->v_new, kvb, cudaMemcpyHostToDevice, st);
      if (e != cudaSuccess) return HSA_ERR_CUDA;
      out = reinterpret_cast<float*>(ws + l.out);
      lse = io->lse ? reinterpret_cast<float*>(ws + l.lse) : nullptr;
    }
    q = ws + l.q;
    kn = ws + l.k_new;
    vn = ws + l.v_new;
  }
  const void* kd = nullptr;
  const void* vd = nullptr;
  rc = kv_pointer(d, k_cache, &kd);
  if (rc != HSA_OK) return rc;
  rc = kv_pointer(d, v_cache, &vd);
  if (rc != HSA_OK) return rc;
  int32_t* bm = reinterpret_cast<int32_t*>(ws + l.block_max);
  int32_t* tm = reinterpret_cast<int32_t*>(ws + l.tile_max);
  int32_t* bidx = block_idx ? block_idx : reinterpret_cast<int32_t*>(ws + l.block_idx);
  int32_t* nb = n_blocks ? n_blocks : reinterpret_cast<int32_t*>(ws + l.n_blocks);
  cudaError_t e;
  if (reuse) {
    // the new token first (the attend reads it among the window's tokens), then the attend
    // over sink + window + the given kept blocks, clipped to the current candidate region
    e = hsa::launch_append_kv(s, kn, vn, const_cast<void*>(kd), const_cast<void*>(vd), kq,
                              k_scale, page_table, seq_lens, err, st, false);
    if (e != cudaSuccess) return HSA_ERR_CUDA;
    rc = block_cache ? do_attend_cached(s, q, kd, vd, page_table, seq_lens, block_idx, n_blocks,
                                        out, lse, ws, l.att, l.cache, block_cache, capacity, st)
                     : do_attend(d, s, false, q, k_cache, v_cache, page_table, seq_lens,
                                 block_idx, n_blocks, out, lse, ws, l.att, st, false);
    if (rc != HSA_OK) return rc;
    return copy_outputs_back(s, io, out, lse, direct_out, st);
  }
  // With a window of at least one token the new token (slot N - 1) is never a scored
  // candidate, so the append runs beside the scorer; with no window it goes first.
  const bool beside = s.window >= 1;
  if (!beside) {
    e = hsa::launch_append_kv(s, kn, vn, const_cast<void*>(kd), const_cast<void*>(vd), kq,
                              k_scale, page_table, seq_lens, err, st, false);
    if (e != cudaSuccess) return HSA_ERR_CUDA;
  }
  // K/V in device memory: the sparse attention runs both pruning modules itself when they
  // fit its shared memory (no pruning kernel, no kept-block list round trip in between); the
  // scorer then, with a window, appends the new token itself (one kernel fewer between the
  // two). Either way the scorer records each row's range of maxima for the selection, and
  // whichever kernel selects clears them.
  const Shape sa = attend_shape(s, false);
  const bool fused = block_cache == nullptr && !d->kv_on_host &&
                     hsa::attend_select_supported(sa, aligned(page_table, 16));
  unsigned* row_range = reinterpret_cast<unsigned*>(ws + l.row_range);
  const hsa::AppendArgs app = {kn, vn, const_cast<void*>(kd), const_cast<void*>(vd), kq};
  rc = do_score(s, q, kq, k_scale, page_table, seq_lens, bm, tm, err, st, row_range,
                (fused && beside) ? &app : nullptr);
  if (rc != HSA_OK) return rc;
  if (beside && !fused) {
    e = hsa::launch_append_kv(s, kn, vn, const_cast<void*>(kd), const_cast<void*>(vd), kq,
                              k_scale, page_table, seq_lens, err, st, true);
    if (e != cudaSuccess) return HSA_ERR_CUDA;
  }
  if (fused) {
    hsa::AttendBuffers buf;
    buf.counters = reinterpret_cast<int*>(ws + l.att.counters);
    buf.part_ml = reinterpret_cast<float*>(ws + l.att.part_ml);
    buf.part_o = reinterpret_cast<float*>(ws + l.att.part_o);
    buf.nsplit = std::min(kMaxSplits, hsa::attend_splits(sa, false, false, num_sms(), false));
    e = hsa::launch_attend_select(sa, q, kd, vd, page_table, seq_lens, bm, tm, row_range,
                                  bidx, nb, out, lse, buf, err, st);
    if (e != cudaSuccess) return HSA_ERR_CUDA;
    return copy_outputs_back(s, io, out, lse, direct_out, st);
  }
  // the prune also resolves the kept blocks' pages, so the attend needs one round trip for them
  int32_t* sel_pages = reinterpret_cast<int32_t*>(ws + l.sel_pages);
  Shape ps = prune_shape(s);
  ps.k1 = module1_keep(ps);  // no chunk ids are output: the same kept blocks
  e = hsa::launch_prune(ps, seq_lens, bm, tm, nullptr, nullptr, bidx, nb, page_table, sel_pages,
                        err, st, row_range);
  if (e != cudaSuccess) return HSA_ERR_CUDA;
  rc = block_cache ? do_attend_cached(s, q, kd, vd, page_table, seq_lens, bidx, nb, out, lse, ws,
                                      l.att, l.cache, block_cache, capacity, st)
                   : do_attend(d, s, false, q, k_cache, v_cache, page_table, seq_lens, bidx, nb,
                               out, lse, ws, l.att, st, true, sel_pages);
  if (rc != HSA_OK) return rc;
  return copy_outputs_back(s, io, out, lse, direct_out, st);
}

int32_t hsa_decode_step_kernels(const hsa_dims* d) {
  Shape s;
  if (check_dims(d, s, true) != HSA_OK) return -1;
  const bool fused = !d->kv_on_host &&
                     hsa::attend_select_supported(attend_shape(s, false), true);
  if (fused) return s.window >= 1 ? 2 : 3;  // (append,) scorer with its ranges, selecting attend
  return 4;                                 // scorer, append, pruning kernel, attend
}

int32_t hsa_decode_step_cached(const hsa_dims* d, const hsa_step_io* io, void* k_cache,
                               void* v_cache, int8_t* kq, const float* k_scale,
                               const int32_t* page_table, const int32_t* seq_lens,
                               int32_t* block_idx, int32_t* n_blocks, void* block_cache,
                               int32_t capacity, void* workspace, size_t workspace_bytes,
                               void* stream) {
  if (block_cache == nullptr) return HSA_ERR_INVALID_ARG;
  return decode_step_impl(d, io, k_cache, v_cache, kq, k_scale, page_table, seq_lens, block_idx,
                          n_blocks, workspace, workspace_bytes, stream, false, block_cache,
                          capacity);
}

size_t hsa_block_cache_bytes(const hsa_dims* d, int32_t capacity) {
  Shape s;
  if (check_dims(d, s, false) != HSA_OK || s.per_head) return 0;
  if (check_cache_capacity(s, capacity) != HSA_OK) return 0;
  return cache_layout(s, capacity).end;
}

float* hsa_block_cache_mass(const hsa_dims* d, void* block_cache, int32_t capacity) {
  Shape s;
  if (!block_cache || check_dims(d, s, false) != HSA_OK || s.per_head) return nullptr;
  if (check_cache_capacity(s, capacity) != HSA_OK) return nullptr;
  return block_cache_at(s, block_cache, capacity).mass;
}

int32_t hsa_attend_cached(const hsa_dims* d, const void* q, const void* k_cache,
                          const void* v_cache, const int32_t* page_table,
                          const int32_t* seq_lens, const int32_t* block_idx,
                          const int32_t* n_blocks, void* block_cache, int32_t capacity,
                          float* out, float* lse, void* workspace, size_t workspace_bytes,
                          void* stream) {
  Shape s;
  int32_t rc = check_dims(d, s, false);
  if (rc != HSA_OK) return rc;
  if (!q || !k_cache || !v_cache || !page_table || !seq_lens || !out || !block_cache ||
      (s.k2 > 0 && (!block_idx || !n_blocks)))
    return HSA_ERR_INVALID_ARG;
  if (!d->kv_on_host || !aligned(q, 16) || !aligned(out, 16) || !aligned(block_cache, kAlign))
    return HSA_ERR_INVALID_ARG;
  if (s.per_head) return HSA_ERR_UNSUPPORTED;  // the cache plan works per kv head
  rc = check_cache_capacity(s, capacity);
  if (rc != HSA_OK) return rc;
  rc = check_ws(s, workspace, workspace_bytes, cached_ws(s));
  if (rc != HSA_OK) return rc;
  const void* kd = nullptr;
  const void* vd = nullptr;
  rc = kv_pointer(d, k_cache, &kd);
  if (rc != HSA_OK) return rc;
  rc = kv_pointer(d, v_cache, &vd);
  if (rc != HSA_OK) return rc;
  char* ws = static_cast<char*>(workspace);
  const AttendLayout l = attend_layout(s, kErrBytes);
  return do_attend_cached(s, q, kd, vd, page_table, seq_lens, block_idx, n_blocks, out, lse, ws,
                          l, cache_scratch(s, l.end), block_cache, capacity, as_stream(stream));
}

// ---- recorded steps
// A decode loop calls hsa_decode_step with the same arguments every step: new contents, the
// same buffers. The kernels read every input from its buffer when they run, so the launches
// of one argument set are recorded once into a CUDA graph and replayed: one graph launch per
// call instead of one launch per kernel (host time that the GPU otherwise waits through).
// Keyed by every argument value and the device; the most recently used kStepGraphs sets are
// kept. Not used while the caller's stream is being captured (the caller's graph then
// records the kernels themselves), nor with HSA_STEP_GRAPHS=0 in the environment.
struct StepKey {
  hsa_dims d;
  hsa_step_io io;
  const void* ptr[9];
  size_t ws_bytes;
  int device;
};

struct StepGraph {
  StepKey key;
  cudaGraphExec_t exec;
  unsigned long long used;
};

constexpr size_t kStepGraphs = 64;

bool step_graphs_enabled() {
  static const bool on = [] {
    const char* e = std::getenv("HSA_STEP_GRAPHS");
    return e == nullptr || std::strcmp(e, "0") != 0;
  }();
  return on;
}

// This thread's stream for recording on `device` (created once, never destroyed: the
// recorded graphs are launched on the caller's stream).
cudaStream_t record_stream(int device) {
  thread_local cudaStream_t streams[64] = {};
  if (device < 0 || device >= 64) return nullptr;
  if (streams[device] == nullptr &&
      cudaStreamCreateWithFlags(&streams[device], cudaStreamNonBlocking) != cudaSuccess)
    streams[device] = nullptr;
  return streams[device];
}

int32_t hsa_decode_step(const hsa_dims* d, const hsa_step_io* io, void* k_cache, void* v_cache,
                        int8_t* kq, const float* k_scale, const int32_t* page_table,
                        const int32_t* seq_lens, int32_t* block_idx, int32_t* n_blocks,
                        void* workspace, size_t workspace_bytes, void* stream) {
  auto direct = [&](void* s) {
    return decode_step_impl(d, io, k_cache, v_cache, kq, k_scale, page_table, seq_lens,
                            block_idx, n_blocks, workspace, workspace_bytes, s, false);
  };
  cudaStream_t st = as_stream(stream);
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  int dev = -1;
  if (!step_graphs_enabled() || d == nullptr || io == nullptr ||
      cudaStreamIsCapturing(st, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone ||
      cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return direct(stream);
  }
  StepKey key;
  std::memset(&key, 0, sizeof(key));  // padding included: keys compare as bytes
  key.d = *d;
  key.io = *io;
  const void* ptr[9] = {k_cache, v_cache, kq, k_scale, page_table, seq_lens, block_idx,
                        n_blocks, workspace};
  std::memcpy(key.ptr, ptr, sizeof(ptr));
  key.ws_bytes = workspace_bytes;
  key.device = dev;
  static std::mutex mu;
  static std::vector<StepGraph>* graphs = new std::vector<StepGraph>();  // kept to exit
  static unsigned long long clock = 0;
  {
    std::lock_guard<std::mutex> g(mu);
    for (StepGraph& e : *graphs) {
      if (std::memcmp(&e.key, &key, sizeof(key)) == 0) {
        e.used = ++clock;
        return cudaGraphLaunch(e.exec, st) == cudaSuccess ? HSA_OK : HSA_ERR_CUDA;
      }
    }
  }
  // record the step's launches on this thread's stream, then launch the graph on `stream`
  cudaStream_t rec = record_stream(dev);
  if (rec == nullptr || cudaStreamBeginCapture(rec, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
    cudaGetLastError();
    return direct(stream);
  }
  const int32_t rc = direct(rec);
  cudaGraph_t graph = nullptr;
  const cudaError_t ec = cudaStreamEndCapture(rec, &graph);
  cudaGraphExec_t exec = nullptr;
  if (rc == HSA_OK && ec == cudaSuccess && graph != nullptr &&
      cudaGraphInstantiate(&exec, graph, 0) != cudaSuccess)
    exec = nullptr;
  if (graph != nullptr) cudaGraphDestroy(graph);
  cudaGetLastError();
  if (rc != HSA_OK && rc != HSA_ERR_CUDA) return rc;  // rejected arguments: nothing launched
  if (exec == nullptr) return direct(stream);         // something could not be recorded
  {
    std::lock_guard<std::mutex> g(mu);
    if (graphs->size() >= kStepGraphs) {
      auto old = std::min_element(graphs->begin(), graphs->end(),
                                  [](const StepGraph& a, const StepGraph& b) { return a.used < b.used; });
      cudaGraphExecDestroy(old->exec);
      graphs->erase(old);
    }
    graphs->push_back(StepGraph{key, exec, ++clock});
  }
  return cudaGraphLaunch(exec, st) == cudaSuccess ? HSA_OK : HSA_ERR_CUDA;
}

int32_t hsa_decode_step_reuse(const hsa_dims* d, const hsa_step_io* io, void* k_cache,
                              void* v_cache, int8_t* kq, const float* k_scale,
                              const int32_t* page_table, const int32_t* seq_lens,
                              const int32_t* block_idx, const int32_t* n_blocks, void* workspace,
                              size_t workspace_bytes, void* stream) {
  return decode_step_impl(d, io, k_cache, v_cache, kq, k_scale, page_table, seq_lens,
                          const_cast<int32_t*>(block_idx), const_cast<int32_t*>(n_blocks),
                          workspace, workspace_bytes, stream, true);
}

int32_t hsa_read_device_error(void* workspace, void* stream, int32_t* code) {
  if (code == nullptr) return HSA_ERR_INVALID_ARG;
  if (workspace == nullptr) {  // the error word of hsa_select_noalloc
    char* scratch = nullptr;
    const int32_t rc = noalloc_scratch(&scratch);
    if (rc != HSA_OK) return rc;
    workspace = scratch;
  }
  if (!aligned(workspace, kAlign)) return HSA_ERR_INVALID_ARG;
  cudaStream_t st = as_stream(stream);
  int v = 0;
  if (cudaStreamSynchronize(st) != cudaSuccess) return HSA_ERR_CUDA;
  if (cudaMemcpy(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return HSA_ERR_CUDA;
  if (cudaMemset(workspace, 0, sizeof(int)) != cudaSuccess) return HSA_ERR_CUDA;
  *code = v;
  return HSA_OK;
}

// ---------------------------------------------------------------------------------------
// hsa_select_noalloc: hsa_select for callers that cannot allocate device memory. Its
// scratch (an error word, then the per-block and per-tile score maxima) lives in one fixed
// array that every GPU loading this library holds until the process exits.

int32_t hsa_select_noalloc(const hsa_dims* d, const void* q, const int8_t* kq,
                           const float* k_scale, const int32_t* page_table,
                           const int32_t* seq_lens, int32_t* chunk_idx, int32_t* n_chunks,
                           int32_t* block_idx, int32_t* n_blocks, void* stream) {
  Shape s;
  int32_t rc = check_dims(d, s, true);
  if (rc != HSA_OK) return rc;
  if (!q || !kq || !k_scale || !page_table || !seq_lens || !n_blocks || (!block_idx && s.k2 > 0))
    return HSA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(kq, 16) || !aligned(k_scale, 16)) return HSA_ERR_INVALID_ARG;
  rc = check_prune_fits(s);
  if (rc != HSA_OK) return rc;
  // the select workspace's layout: error word, block maxima, tile maxima
  if (select_ws(s) > kNoAllocScratchBytes) return HSA_ERR_WORKSPACE_TOO_SMALL;
  char* scratch = nullptr;
  rc = noalloc_scratch(&scratch);
  if (rc != HSA_OK) return rc;
  int* err = reinterpret_cast<int*>(scratch);
  int32_t* bm = reinterpret_cast<int32_t*>(scratch + kErrBytes);
  int32_t* tm = reinterpret_cast<int32_t*>(scratch + kErrBytes + select_bm_bytes(s));
  cudaStream_t st = as_stream(stream);
  // Every entry of the maxima that the prune kernel reads is written by the scorer in the
  // same call, so only the error word has to start at zero: it does (static device memory
  // starts zeroed) and hsa_read_device_error(NULL, ...) clears it after reading it.
  rc = do_score(s, q, kq, k_scale, page_table, seq_lens, bm, tm, err, st);
  if (rc != HSA_OK) return rc;
  return cuda_status(hsa::launch_prune(prune_shape(s), seq_lens, bm, tm, chunk_idx, n_chunks,
                                       block_idx, n_blocks, nullptr, nullptr, err, st));
}

}  // extern "C"
