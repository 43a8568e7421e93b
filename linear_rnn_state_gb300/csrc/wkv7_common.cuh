// Shared device helpers for the WKV7 kernels: TMA tensor loads, mbarriers
// with bounded waits, element conversion and the device status word.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "wkv7_launch.h"

namespace wkv7 {

// Bits of the device status word the kernels report through (a pointer in
// their arguments). Host code reads and clears it in wkv7_status().
enum : unsigned { STATUS_TIMEOUT = 1u, STATUS_BOUNDS = 2u };

// Check of a plain global load or store in the debug build (WKV7_DEBUG):
// true when the n objects at p lie inside the buffer x; otherwise the status
// word records STATUS_BOUNDS and the caller skips the access (a skipped load
// reads as zero). Other builds return true without looking.
template <typename T>
__device__ __forceinline__ bool in_extent(unsigned* status, const Extent& x, const T* p, int n = 1) {
#ifdef WKV7_DEBUG
  const uintptr_t a = reinterpret_cast<uintptr_t>(p), lo = reinterpret_cast<uintptr_t>(x.lo);
  if (a >= lo && a + (size_t)n * sizeof(T) <= lo + x.bytes) return true;
  if (status) atomicOr(status, STATUS_BOUNDS);
  return false;
#else
  (void)status, (void)x, (void)p, (void)n;
  return true;
#endif
}

// ---------------------------------------------------------------- types ---

template <typename T> struct Elem;
template <> struct Elem<float> {
  static constexpr int bytes = 4;
};
template <> struct Elem<__nv_bfloat16> {
  static constexpr int bytes = 2;
};

// Load 4 consecutive elements (16 B of fp32 or 8 B of bf16) from shared
// memory as float4.
__device__ __forceinline__ float4 lds4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 lds4(const __nv_bfloat16* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  float4 f;
  f.x = __uint_as_float(u.x << 16);
  f.y = __uint_as_float(u.x & 0xFFFF0000u);
  f.z = __uint_as_float(u.y << 16);
  f.w = __uint_as_float(u.y & 0xFFFF0000u);
  return f;
}
__device__ __forceinline__ float ld1(const float* p) { return *p; }
__device__ __forceinline__ float ld1(const __nv_bfloat16* p) { return __bfloat162float(*p); }

__device__ __forceinline__ void st1(float* p, float x) { *p = x; }
__device__ __forceinline__ void st1(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

// ------------------------------------------------------------- mbarrier ---

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// How long a kernel waits on an mbarrier before it gives up: about 2 s, or
// 1 ms in the debug build (WKV7_DEBUG), whose tests make a wait run out.
#ifdef WKV7_DEBUG
constexpr uint64_t kWaitLimitNs = 1000000ull;
#else
constexpr uint64_t kWaitLimitNs = 2000000000ull;
#endif

// Wait for the phase with the given parity to complete, giving up after
// about `limit_ns` nanoseconds. On timeout the status word records it and the
// function returns false; the caller then leaves the kernel.
__device__ __forceinline__ bool mbar_wait_bounded(unsigned* status, uint64_t* bar, uint32_t parity,
                                                  uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t start = globaltimer_ns();
  for (uint32_t spin = 1;; ++spin) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((spin & 255u) == 0 && globaltimer_ns() - start > limit_ns) {
      if (status) atomicOr(status, STATUS_TIMEOUT);
      return false;
    }
  }
}

// ------------------------------------------------------------------ TMA ---

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 4-D tiled tensor load global -> shared, completion counted on `bar`.
// Coordinates are (x = element in the row, head, time step, batch).
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int h,
                                            int t, int b) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(h), "r"(t), "r"(b), "r"(smem_addr(bar))
      : "memory");
}

// 3-D tiled tensor load global -> shared (checkpoint states).
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ----------------------------------------------------------- reductions ---

// Sum over groups of G consecutive lanes (G a power of two <= 32); every
// lane of the group receives the total.
template <int G>
__device__ __forceinline__ float group_allreduce(float x) {
#pragma unroll
  for (int o = 1; o < G; o <<= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

}  // namespace wkv7
