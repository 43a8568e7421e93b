// The decay as the chunked kernels read it from an input tile: the value w
// itself, or, for a decay given as logits z, w = exp(-0.606531 sigmoid(z))
// (the time-mix of "rx_pretrain.c", tm_pre_forward, with RX_WDECAY_COEFF),
// formed in fp32 where the tile is read, so no separate pass over HBM makes w.
#pragma once

namespace wkv7 {

constexpr float kWDecayCoeff = 0.606531f;

__device__ __forceinline__ float sigmoid_fast(float z) { return __fdividef(1.f, 1.f + __expf(-z)); }

// w from z in two special-function operations: sigmoid(z) = 1/2 + tanh(z/2)/2
// and exp(-c s) = 2^(-c log2(e) s). tanh.approx is within about 2^-11 of
// tanh, so w is within about 1.5e-4 of exp(-0.606531 sigmoid(z)) (relative),
// finer than the bf16 rounding a decay passed as w carries.
__device__ __forceinline__ float decay_from_logit(float z) {
  float th, w;
  asm("tanh.approx.f32 %0, %1;" : "=f"(th) : "f"(0.5f * z));
  const float s = fmaf(0.5f, th, 0.5f);
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(w) : "f"(-kWDecayCoeff * 1.4426950408889634f * s));
  return w;
}

template <bool kLogit>
__device__ __forceinline__ float decay_value(float x) {
  if constexpr (kLogit)
    return decay_from_logit(x);
  else
    return x;
}

template <bool kLogit>
__device__ __forceinline__ float2 decay_value2(float2 x) {
  return make_float2(decay_value<kLogit>(x.x), decay_value<kLogit>(x.y));
}

// Gradient w.r.t. the logit z from w dw: the time-mix backward's
// dsig = dw w (-RX_WDECAY_COEFF), dz = dsig sigmoid(z) (1 - sigmoid(z)).
__device__ __forceinline__ float logit_grad_from_wdw(float wdw, float z) {
  const float s = sigmoid_fast(z);
  return wdw * (-kWDecayCoeff) * s * (1.f - s);
}

}  // namespace wkv7
