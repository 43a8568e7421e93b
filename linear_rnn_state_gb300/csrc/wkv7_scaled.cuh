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

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) { return __fmul2_rn(a, b); }

__device__ __forceinline__ float4 ld_f4(const float* p) { return *reinterpret_cast<const float4*>(p); }

// Element load from a raw staged vector (fp32 or bf16) as float.
__device__ __forceinline__ float raw1(const float* p) { return *p; }
__device__ __forceinline__ float raw1(const __nv_bfloat16* p) { return __bfloat162float(*p); }

}  // namespace wkv7
