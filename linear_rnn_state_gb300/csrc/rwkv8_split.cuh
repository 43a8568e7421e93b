// Split of an fp32 value into two tf32 values for the tensor cores, with
// integer arithmetic only (no conversion instructions).
//
// tf32 keeps the sign, the 8 exponent bits and the top 10 mantissa bits of
// an fp32 pattern (the 13 bits below are zero). Adding half a tf32 unit
// (bit 12) to the pattern and clearing the 13 low bits rounds the
// magnitude to the nearest tf32 value (ties away from zero; a carry out of
// the mantissa moves correctly into the exponent). Then
//     hi = round(x),  lo = x - hi   (exact in fp32, |lo| <= 2^-11 |hi|),
// and lo rounded the same way, so a x b is a_hi b_hi + a_hi b_lo + a_lo b_hi
// up to terms near 2^-21 |a b|. Finite inputs of normal magnitude only
// (inf and NaN are not split meaningfully).
#pragma once

#include <stdint.h>

#include "wkv7_mma.cuh"

namespace rwkv8 {

__device__ __forceinline__ uint32_t tf32_round_bits(uint32_t bits) { return (bits + 0x1000u) & 0xffffe000u; }

__device__ __forceinline__ void split_tf32(float x, uint32_t& hi, uint32_t& lo) {
  hi = tf32_round_bits(__float_as_uint(x));
  lo = tf32_round_bits(__float_as_uint(x - __uint_as_float(hi)));
}

// d += a b for one m16n8k8 tile in split tf32, from fp32 fragment values
// (a in A-fragment order, b0 / b1 the B fragment): the two small cross terms
// first, then the main product.
__device__ __forceinline__ void mma_split(float (&d)[4], const float (&a)[4], float b0, float b1) {
  uint32_t ah[4], al[4], bh0, bl0, bh1, bl1;
#pragma unroll
  for (int i = 0; i < 4; ++i) split_tf32(a[i], ah[i], al[i]);
  split_tf32(b0, bh0, bl0);
  split_tf32(b1, bh1, bl1);
  wkv7::mma_tf32(d, al, bh0, bh1);
  wkv7::mma_tf32(d, ah, bl0, bl1);
  wkv7::mma_tf32(d, ah, bh0, bh1);
}

}  // namespace rwkv8
