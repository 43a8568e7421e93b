// Warp-level tf32 tensor-core helpers for the chunked WKV7 kernels.
//
// Every product uses mma.sync m16n8k8 (tf32 inputs, fp32 accumulation) with
// one fixed fragment convention. Operands in shared memory use row strides
// of 72 or 24 floats (= 8 mod 32): the float2 loads along k of each
// half-warp then touch every bank once. A matrix read only transposed
// (scalar loads down a column pair) uses 68 (= 4 mod 16) instead, which keeps
// those loads conflict-free. Within each 8-wide k block the hardware
// k slot q of lane (g = lane/4, t = lane%4) is bound to physical column
//   slot t -> 2t,  slot t+4 -> 2t+1,
// in both operands (the sum over k is order-free). Then
//   A fragment: (a0, a2) = A[g][k0+2t .. +1],  (a1, a3) = A[g+8][k0+2t .. +1]
//   B fragment: (b0, b1) = B^T[n0+g][k0+2t .. +1]
//   C fragment: (c0, c1) = C[g][n0+2t .. +1],  (c2, c3) = C[g+8][n0+2t .. +1]
// so an accumulator tile is, register for register, the A fragment of the
// next product over the same index (c2a), and every shared-memory operand is
// read as float2 from a row-major matrix whose rows run along k ("A" as
// A[m][k], "B" stored transposed as BT[n][k]).
#pragma once

#include <stdint.h>

namespace wkv7 {

// Round to the nearest tf32 value (10 explicit mantissa bits), kept in an
// fp32 bit pattern.
__device__ __forceinline__ uint32_t tf32_bits(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ float tf32r(float x) { return __uint_as_float(tf32_bits(x)); }

// d += a * b for one 16x8x8 tile.
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// A fragment of rows r0..r0+15, k block k0..k0+7 of a row-major matrix whose
// entries are already tf32 values.
__device__ __forceinline__ void frag_a(uint32_t (&a)[4], const float* m, int ld, int r0, int k0, int g, int t) {
  const float2 lo = *reinterpret_cast<const float2*>(m + (r0 + g) * ld + k0 + 2 * t);
  const float2 hi = *reinterpret_cast<const float2*>(m + (r0 + g + 8) * ld + k0 + 2 * t);
  a[0] = __float_as_uint(lo.x);
  a[2] = __float_as_uint(lo.y);
  a[1] = __float_as_uint(hi.x);
  a[3] = __float_as_uint(hi.y);
}

// B fragment of columns n0..n0+7, k block k0..k0+7, read from the transposed
// operand BT[n][k] (tf32 values).
__device__ __forceinline__ void frag_b(uint32_t& b0, uint32_t& b1, const float* bt, int ld, int n0, int k0, int g,
                                       int t) {
  const float2 v = *reinterpret_cast<const float2*>(bt + (n0 + g) * ld + k0 + 2 * t);
  b0 = __float_as_uint(v.x);
  b1 = __float_as_uint(v.y);
}

// A fragment as frag_a, from fp32 values that still need rounding to tf32.
__device__ __forceinline__ void frag_a_r(uint32_t (&a)[4], const float* m, int ld, int r0, int k0, int g, int t) {
  const float2 lo = *reinterpret_cast<const float2*>(m + (r0 + g) * ld + k0 + 2 * t);
  const float2 hi = *reinterpret_cast<const float2*>(m + (r0 + g + 8) * ld + k0 + 2 * t);
  a[0] = tf32_bits(lo.x);
  a[2] = tf32_bits(lo.y);
  a[1] = tf32_bits(hi.x);
  a[3] = tf32_bits(hi.y);
}

// A fragment of A[m][k] read from storage laid out [k][m] (scalar loads;
// tf32 values).
__device__ __forceinline__ void frag_a_t(uint32_t (&a)[4], const float* m, int ld, int m0, int k0, int g, int t) {
  const float* p = m + (k0 + 2 * t) * ld + m0 + g;
  a[0] = __float_as_uint(p[0]);
  a[2] = __float_as_uint(p[ld]);
  a[1] = __float_as_uint(p[8]);
  a[3] = __float_as_uint(p[ld + 8]);
}

// B fragment of B[k][n] read from storage laid out [k][n] (scalar loads;
// tf32 values).
__device__ __forceinline__ void frag_b_t(uint32_t& b0, uint32_t& b1, const float* m, int ld, int n0, int k0, int g,
                                         int t) {
  const float* p = m + (k0 + 2 * t) * ld + n0 + g;
  b0 = __float_as_uint(p[0]);
  b1 = __float_as_uint(p[ld]);
}

// frag_b_t from fp32 values that still need rounding to tf32.
__device__ __forceinline__ void frag_b_t_r(uint32_t& b0, uint32_t& b1, const float* m, int ld, int n0, int k0, int g,
                                           int t) {
  const float* p = m + (k0 + 2 * t) * ld + n0 + g;
  b0 = tf32_bits(p[0]);
  b1 = tf32_bits(p[ld]);
}

// Fragments in the hardware's own k order (slot t -> column t, slot t+4 ->
// column t+4), for products whose two operands are both read transposed:
// A[m][k] from storage [k][m] and B[k][n] from storage [k][n]. With a row
// stride of 8 mod 32 (or 24 for 16-wide blocks) every such load is
// conflict-free.
__device__ __forceinline__ void frag_a_ts(uint32_t (&a)[4], const float* m, int ld, int m0, int k0, int g, int t) {
  const float* p = m + (k0 + t) * ld + m0 + g;
  a[0] = __float_as_uint(p[0]);
  a[1] = __float_as_uint(p[8]);
  a[2] = __float_as_uint(p[4 * ld]);
  a[3] = __float_as_uint(p[4 * ld + 8]);
}
__device__ __forceinline__ void frag_b_ts(uint32_t& b0, uint32_t& b1, const float* m, int ld, int n0, int k0, int g,
                                          int t) {
  const float* p = m + (k0 + t) * ld + n0 + g;
  b0 = __float_as_uint(p[0]);
  b1 = __float_as_uint(p[4 * ld]);
}

// Accumulator tile -> A fragment over the same columns (rounded to tf32).
__device__ __forceinline__ void c2a(uint32_t (&a)[4], const float (&c)[4]) {
  a[0] = tf32_bits(c[0]);
  a[1] = tf32_bits(c[2]);
  a[2] = tf32_bits(c[1]);
  a[3] = tf32_bits(c[3]);
}

__device__ __forceinline__ void zero4(float (&c)[4]) { c[0] = c[1] = c[2] = c[3] = 0.f; }

// 16-byte asynchronous copy global -> shared (both addresses 16-byte aligned).
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src)
               : "memory");
}
// 16-byte asynchronous copy that writes zeros instead when `valid` is false.
__device__ __forceinline__ void cp_async16_zfill(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src), "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Named barrier over `count` threads (a multiple of 32).
__device__ __forceinline__ void named_bar(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Arrival at a named barrier without waiting (the producer side of bar.sync on the same
// barrier and count).
__device__ __forceinline__ void named_arrive(int id, int count) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Named barrier that also returns whether any participating thread passed a
// true predicate.
__device__ __forceinline__ bool named_bar_or(int id, int count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n bar.red.or.pred p, %2, %3, q;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

}  // namespace wkv7
