// common.cuh -- shared constants and inline-PTX helpers of libhsa (sm_103a).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <utility>

namespace hsa {

constexpr int kHeadDim = 128;   // channels per head
constexpr int kPage = 16;       // tokens per page == tokens per block
constexpr int kBlockBytesI8 = kPage * kHeadDim;        // 2 KiB of int8 codes per (page, head)
constexpr int kBlockBytesBf16 = kPage * kHeadDim * 2;  // 4 KiB of bf16 per (page, head)

// Codes written to the workspace error word (same values as the public status codes).
constexpr int kDevErrTimeout = 4;
constexpr int kDevErrCheck = 6;

// Upper bound of every spin-wait, in SM clock cycles (about two seconds).
constexpr long long kWaitLimitCycles = 4000000000LL;

__device__ __forceinline__ void set_error(int* err, int code) {
  if (err != nullptr) atomicCAS(err, 0, code);
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// Makes the initialised barriers visible to the asynchronous (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase of parity `parity` to complete; false after kWaitLimitCycles.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitLimitCycles) return false;
  }
  return true;
}

// ------------------------------------------------------------- TMA copies

// 2-D tiled tensor copy global -> shared, completing on `bar` (tx bytes = box bytes).
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

// An L2 policy under which the lines a copy brings in are the first to be evicted. Data read
// once (the int8 key codes of the scan, the K/V pages of the attend) then does not push the
// small arrays that the next kernels read again (page table, block maxima) out of L2.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// tma_load_2d with an L2 cache policy (see l2_evict_first_policy).
__device__ __forceinline__ void tma_load_2d_hint(void* dst, const CUtensorMap* map, int x, int y,
                                                 uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// 4-D tiled tensor copy global -> shared with an L2 cache policy.
__device__ __forceinline__ void tma_load_4d_hint(void* dst, const CUtensorMap* map, int x, int y,
                                                 int z, int w, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_addr(bar)),
      "l"(policy)
      : "memory");
}

// Bulk prefetch of [src, src + bytes) into L2 (bytes a multiple of 16, src 16-byte aligned);
// no completion to wait for.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(src)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void tma_prefetch_descriptor(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 1-D bulk copy global -> shared (16-byte aligned addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// bulk_load with an L2 cache policy (see l2_evict_first_policy).
__device__ __forceinline__ void bulk_load_hint(void* dst, const void* src, uint32_t bytes,
                                               uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// Atomic add at GPU scope with acquire and release semantics; returns the old value.
__device__ __forceinline__ int atomic_add_acq_rel_gpu(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v)
               : "memory");
  return old;
}

// ----------------------------------------------- programmatic dependent launch
//
// Kernels of one step are launched with programmatic stream serialisation: a kernel may
// start while its predecessor in the stream still runs. grid_dep_wait() returns once the
// predecessor grid has completed and its writes are visible (at once when the kernel was
// launched without the attribute); grid_dep_launch() lets the successor start launching.
// Every kernel that is launched this way calls grid_dep_wait() on every path before it
// exits, so that its own completion implies its predecessor's.

__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void grid_dep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Dynamic shared memory of a kernel, and the largest shared-memory carveout: kernels of one
// step overlap on an SM (the next one is launched while the previous one runs), and an SM
// configured for a kernel with little shared memory could not take the next kernel's CTAs
// until it drains.
// The attributes are set once per (kernel, device) and raised when a launch needs more (a
// cudaDeviceReset would drop them; the library never calls it).
struct SmemAttrCache {
  std::mutex mu;
  std::map<std::pair<const void*, int>, size_t> bytes;  // dynamic bytes already allowed
};
inline SmemAttrCache& smem_attr_cache() {
  static SmemAttrCache c;
  return c;
}

template <typename Kernel>
cudaError_t set_kernel_smem(Kernel kernel, size_t dynamic_bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const auto key = std::make_pair(reinterpret_cast<const void*>(kernel), dev);
  SmemAttrCache& c = smem_attr_cache();
  // under the lock, so that concurrent callers never lower a limit another one relies on
  std::lock_guard<std::mutex> g(c.mu);
  const auto it = c.bytes.find(key);
  if (it != c.bytes.end() && it->second >= dynamic_bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)dynamic_bytes);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                           (int)cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  c.bytes[key] = dynamic_bytes;
  return cudaSuccess;
}

// Launch with (pdl) or without programmatic stream serialisation.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t st, bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ------------------------------------------------------------------ loads

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

// Read-only, L1-bypassing 16-byte load (also used on mapped host memory).
__device__ __forceinline__ uint4 ldg128_nc(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// bf16 pair (packed in a 32-bit word) to two floats, exactly.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// ----------------------------------------------------- int8 code (fp32 RN)

// clamp(rint_half_even(f32(x / s)), -levels, levels); s == 0 gives 0.
__device__ __forceinline__ int key_code(float x, float s, int levels) {
  if (s == 0.0f) return 0;
  int r = __float2int_rn(__fdiv_rn(x, s));
  return max(-levels, min(levels, r));
}

// clamp(rint_half_even(f32(x / s)), -127, 127); s == 0 gives 0.
__device__ __forceinline__ int int8_code(float x, float s) { return key_code(x, s, 127); }

// Largest key code of a key format: 127 for 8-bit codes, 7 for 4-bit codes.
__host__ __device__ __forceinline__ int key_levels(int bits) { return bits == 4 ? 7 : 127; }

}  // namespace hsa
