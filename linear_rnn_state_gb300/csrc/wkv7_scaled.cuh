// Column-scaled form of the WKV7 recurrence, shared by the fast kernels.
//
// Within a chunk of steps starting after t0-1, write the state as
// S(t) = S~(t) diag(c(t)) with c(t) = w(t0) * ... * w(t) (c(t0-1) = 1). The
// step S <- S diag(w) + v k^T + sa b^T then becomes a pure rank-2 update
//     S~(t) = S~(t-1) + v(t) k~(t)^T + sa(t) b~(t)^T,   k~ = k / c(t), b~ = b / c(t)
// and the products the scan needs read
//     sa(t) = S~(t-1) a^(t),  a^(t) = c(t-1) * a(t)
//     y(t)  = S~(t) r^(t),    r^(t) = c(t) * r(t).
// Four multiply-adds per state element and step instead of five. The decay
// is folded into per-step column vectors computed once per chunk ("the
// prologue"), and the state is renormalised (S = S~ diag(c)) at chunk ends.
//
// sa(t+1) = S~(t) a^(t+1) = X(t) + sa(t) beta(t) with X(t) = u~(t) a^(t+1),
// u~(t) = S~(t-1) + v k~^T and beta(t) = b(t) . a(t+1): the row sum X(t) can
// start before sa(t) is known, which takes the cross-lane reduction off the
// serial path.
//
// The form needs every c and 1/c of a chunk to stay well inside fp32 range;
// the kernels use it only when every decay lies in [kWMin, kWMax] (see
// decay_is_safe) and hand any other head to the direct-form kernels.
#pragma once

#include "wkv7_common.cuh"

namespace wkv7 {

// Decays outside this range (or NaN) send a head to the direct-form path.
// With chunks of at most 16 steps the running products stay within
// [2^-64, 2^64].
constexpr float kWMin = 0.0625f;
constexpr float kWMax = 16.0f;

__device__ __forceinline__ bool decay_is_safe(float w) { return w >= kWMin && w <= kWMax; }

__device__ __forceinline__ float2 f2(float s) { return make_float2(s, s); }

// Element-pair arithmetic: packed fp32x2 FMA (fma.rn.f32x2), one
// instruction for two multiply-adds; the kernels are issue-bound, so fewer
// instructions beat the packed form's longer issue interval.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float hsum(float2 a) { return a.x + a.y; }

// Hardware reciprocal approximation (PTX rcp.approx.f32, at most 1 ulp off).
// Used for 1/c: a scale factor whose exact rounding does not matter, since
// the state is multiplied back by c itself.
__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// Sum each of R per-row values over the G lanes of a row group
// (reduce-scatter: the set halves on each of the high lane bits, then the
// last value is summed over the remaining bits). Returns the total of row
// row_of_lane<G, R>(cg) of the caller's row group.
template <int G, int R>
__device__ __forceinline__ float rowsum_scatter(float (&v)[R], int cg) {
  int n = R;
#pragma unroll
  for (int mask = G / 2; mask >= 1; mask >>= 1) {
    if (n > 1) {
      const int h = n / 2;
      const bool upper = (cg & mask) != 0;
#pragma unroll
      for (int i = 0; i < R / 2; ++i) {
        if (i < h) {
          const float send = upper ? v[i] : v[h + i];
          const float keep = upper ? v[h + i] : v[i];
          v[i] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
        }
      }
      n = h;
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], mask);
    }
  }
  return v[0];
}

// Row (within the row group) whose total rowsum_scatter leaves in lane cg,
// and whether this lane is the first of the copies holding it.
template <int G, int R>
__device__ __forceinline__ int row_of_lane(int cg) {
  constexpr int copies = G / R;
  return cg / copies;
}
template <int G, int R>
__device__ __forceinline__ bool row_writer(int cg) {
  constexpr int copies = G / R;
  return (cg % copies) == 0;
}

__device__ __forceinline__ float4 ld_f4(const float* p) { return *reinterpret_cast<const float4*>(p); }

// One 32-bit shared-memory load, kept separate (not merged into a vector
// load): on GB300 a warp issues a broadcast 32-bit shared load about every
// cycle, while a 64- or 128-bit one costs about twelve.
__device__ __forceinline__ float lds32(const float* p) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))));
  return v;
}
// Four consecutive floats as four 32-bit loads.
__device__ __forceinline__ float4 lds32x4(const float* p) {
  return make_float4(lds32(p), lds32(p + 1), lds32(p + 2), lds32(p + 3));
}

// Element load from a raw staged vector (fp32 or bf16) as float.
__device__ __forceinline__ float raw1(const float* p) { return *p; }
__device__ __forceinline__ float raw1(const __nv_bfloat16* p) { return __bfloat162float(*p); }

}  // namespace wkv7
