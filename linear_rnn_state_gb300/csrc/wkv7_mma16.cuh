// Warp-level bf16 tensor-core helpers (mma.sync m16n8k16, fp32 accumulation)
// for the chunked WKV7 kernels: fragment loads by ldmatrix from row-major
// shared-memory tiles, accumulator-to-operand packing, masked stores.
//
// Fragment convention (the instruction's own): with g = lane / 4, t = lane % 4,
//   A (16 x 16): a0 = A[g][2t .. 2t+1], a1 = A[g+8][2t ..], a2 = A[g][2t+8 ..], a3 = A[g+8][2t+8 ..]
//   B (16 x 8):  b0 = B[2t .. 2t+1][g], b1 = B[2t+8 .. 2t+9][g]
//   C (16 x 8):  c0, c1 = C[g][2t .. 2t+1], c2, c3 = C[g+8][2t ..]
// so two accumulator tiles over adjacent 8-column blocks are, packed to bf16
// pairs, the A fragment of a product over those 16 columns (c2a16).
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "wkv7_common.cuh"

namespace wkv7 {

constexpr int kB64 = 72;  // row stride (bf16 elements) of 64-wide tiles
constexpr int kB16 = 24;  // row stride of 16-wide tiles
typedef __nv_bfloat16 bf16_t;

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ float2 unpack_bf16(uint32_t u) {
  return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
}
__device__ __forceinline__ void st_pair(bf16_t* p, float2 x) { *reinterpret_cast<uint32_t*>(p) = pack_bf16(x.x, x.y); }

// d += a * b for one 16 x 8 x 16 tile (bf16 inputs, fp32 accumulation).
__device__ __forceinline__ void mma16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm4(uint32_t (&r)[4], const bf16_t* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_addr(p)));
}
__device__ __forceinline__ void ldsm4t(uint32_t (&r)[4], const bf16_t* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_addr(p)));
}
__device__ __forceinline__ void stsm4t(bf16_t* p, const uint32_t (&r)[4]) {
  asm volatile("stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1,%2,%3,%4};" ::"r"(smem_addr(p)), "r"(r[0]),
               "r"(r[1]), "r"(r[2]), "r"(r[3])
               : "memory");
}

// Fragment loads for one k16 block. "A" is 16 rows (m) x 16 k, "B" two n8
// tiles x 16 k (r[0], r[1] for columns n0 .. n0+7, r[2], r[3] for n0+8 ..).
// Storage is row-major with stride ld; the suffix says how it is laid out:
//   a_mk: A[m][k] stored [m][k];  a_km: stored [k][m] (transposed load)
//   b_nk: B^T[n][k] stored [n][k]; b_kn: B[k][n] stored [k][n] (transposed load)
__device__ __forceinline__ void a_mk(uint32_t (&r)[4], const bf16_t* s, int ld, int m0, int k0, int lane) {
  ldsm4(r, s + (m0 + (lane & 7) + ((lane >> 3) & 1) * 8) * ld + k0 + (lane >> 4) * 8);
}
__device__ __forceinline__ void a_km(uint32_t (&r)[4], const bf16_t* s, int ld, int m0, int k0, int lane) {
  ldsm4t(r, s + (k0 + (lane & 7) + (lane >> 4) * 8) * ld + m0 + ((lane >> 3) & 1) * 8);
}
__device__ __forceinline__ void b_nk(uint32_t (&r)[4], const bf16_t* s, int ld, int n0, int k0, int lane) {
  ldsm4(r, s + (n0 + (lane & 7) + (lane >> 4) * 8) * ld + k0 + ((lane >> 3) & 1) * 8);
}
__device__ __forceinline__ void b_kn(uint32_t (&r)[4], const bf16_t* s, int ld, int n0, int k0, int lane) {
  ldsm4t(r, s + (k0 + (lane & 7) + ((lane >> 3) & 1) * 8) * ld + n0 + (lane >> 4) * 8);
}
// Two accumulator tiles (columns k0 .. k0+7 and k0+8 .. k0+15 of 16 rows) as
// the A fragment of a product over those 16 columns.
__device__ __forceinline__ void c2a16(uint32_t (&a)[4], const float (&lo)[4], const float (&hi)[4]) {
  a[0] = pack_bf16(lo[0], lo[1]);
  a[1] = pack_bf16(lo[2], lo[3]);
  a[2] = pack_bf16(hi[0], hi[1]);
  a[3] = pack_bf16(hi[2], hi[3]);
}
// acc[nt] += A B over K = 16 * KB for two n8 tiles, A from [m][k], B from [n][k].
template <int KB>
__device__ __forceinline__ void mm_mk_nk(float (&acc)[2][4], const bf16_t* A, int lda, int m0, const bf16_t* Bt, int ldb,
                                         int n0, int lane) {
#pragma unroll
  for (int kb = 0; kb < KB; ++kb) {
    uint32_t a[4], b[4];
    a_mk(a, A, lda, m0, 16 * kb, lane);
    b_nk(b, Bt, ldb, n0, 16 * kb, lane);
    mma16(acc[0], a, b[0], b[1]);
    mma16(acc[1], a, b[2], b[3]);
  }
}
// Store a 16 x 16 fp32 accumulator (tiles acc[0], acc[1]) as bf16 [t][s] (row stride kB16),
// keeping lower: s < t (+ diagonal if incl), upper: s > t (+ diagonal if incl).
__device__ __forceinline__ void store_masked16(const float (&acc)[2][4], bf16_t* dst, bool lower, bool incl, int g,
                                               int t4) {
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int t = g + 8 * h, s = 8 * nt + 2 * t4;
      float x[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int se = s + e;
        const bool keep = lower ? (se < t || (incl && se == t)) : (se > t || (incl && se == t));
        x[e] = keep ? acc[nt][2 * h + e] : 0.f;
      }
      st_pair(dst + t * kB16 + s, make_float2(x[0], x[1]));
    }
}

// ------------------------------------------------- operands in one or two parts ---
//
// An operand in kP bf16 parts: kP = 1, one bf16 value; kP = 2, a pair hi + lo (hi = the
// value rounded to bf16, lo = the remainder rounded to bf16, about 16 bits in all), and a
// product a b is then taken as a_lo b_hi + a_hi b_lo + a_hi b_hi.

// A fragment (A or two n8 tiles of B) of an operand in kP bf16 parts: h, and for kP = 2 l.
template <int kP>
struct FragP {
  uint32_t h[4];
  uint32_t l[kP == 2 ? 4 : 1];
};

// Two accumulator tiles as the A fragment of a product over their 16 columns, and for kP
// = 2 the remainder after rounding to bf16 as the lo part.
template <int kP>
__device__ __forceinline__ void c2a_p(FragP<kP>& a, const float (&lo)[4], const float (&hi)[4]) {
  c2a16(a.h, lo, hi);
  if constexpr (kP == 2) {
    const float2 u0 = unpack_bf16(a.h[0]), u1 = unpack_bf16(a.h[1]), u2 = unpack_bf16(a.h[2]),
                 u3 = unpack_bf16(a.h[3]);
    const float rl[4] = {lo[0] - u0.x, lo[1] - u0.y, lo[2] - u1.x, lo[3] - u1.y};
    const float rh[4] = {hi[0] - u2.x, hi[1] - u2.y, hi[2] - u3.x, hi[3] - u3.y};
    c2a16(a.l, rl, rh);
  }
}
// Fragments of a row-major tile stored in kP parts: hi, and lo (read only for kP = 2).
template <int kP>
__device__ __forceinline__ void a_mk_p(FragP<kP>& a, const bf16_t* hi, const bf16_t* lo, int ld, int m0, int k0,
                                       int lane) {
  a_mk(a.h, hi, ld, m0, k0, lane);
  if constexpr (kP == 2) a_mk(a.l, lo, ld, m0, k0, lane);
}
template <int kP>
__device__ __forceinline__ void b_nk_p(FragP<kP>& b, const bf16_t* hi, const bf16_t* lo, int ld, int n0, int k0,
                                       int lane) {
  b_nk(b.h, hi, ld, n0, k0, lane);
  if constexpr (kP == 2) b_nk(b.l, lo, ld, n0, k0, lane);
}
// acc (two n8 tiles) += a b with the parts each side has: the small terms first.
__device__ __forceinline__ void mma2(float (&acc)[2][4], const uint32_t (&a)[4], const uint32_t (&b)[4]) {
  mma16(acc[0], a, b[0], b[1]);
  mma16(acc[1], a, b[2], b[3]);
}
template <int kPa, int kPb>
__device__ __forceinline__ void mma_pp(float (&acc)[2][4], const FragP<kPa>& a, const FragP<kPb>& b) {
  if constexpr (kPa == 2) mma2(acc, a.l, b.h);
  if constexpr (kPb == 2) mma2(acc, a.h, b.l);
  mma2(acc, a.h, b.h);
}
// An fp32 value stored as kP bf16 parts: hi, and lo (written only for kP = 2).
template <int kP>
__device__ __forceinline__ void put_p(bf16_t* hi, bf16_t* lo, float x) {
  const bf16_t h = __float2bfloat16_rn(x);
  *hi = h;
  if constexpr (kP == 2) *lo = __float2bfloat16_rn(x - __bfloat162float(h));
}
// Eight fp32 values as one 16-byte piece per part.
__device__ __forceinline__ uint4 pack8(const float (&x)[8]) {
  return make_uint4(pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]), pack_bf16(x[4], x[5]), pack_bf16(x[6], x[7]));
}
__device__ __forceinline__ void lo8(float (&x)[8]) {  // x <- x - bf16(x), exact in fp32
#pragma unroll
  for (int e = 0; e < 8; ++e) x[e] -= __bfloat162float(__float2bfloat16_rn(x[e]));
}
template <int kP>
__device__ __forceinline__ void put8_p(bf16_t* hi, bf16_t* lo, float (&x)[8]) {
  *reinterpret_cast<uint4*>(hi) = pack8(x);
  if constexpr (kP == 2) {
    lo8(x);
    *reinterpret_cast<uint4*>(lo) = pack8(x);
  }
}

template <int kP>
__device__ __forceinline__ void a_km_p(FragP<kP>& a, const bf16_t* hi, const bf16_t* lo, int ld, int m0, int k0,
                                       int lane) {
  a_km(a.h, hi, ld, m0, k0, lane);
  if constexpr (kP == 2) a_km(a.l, lo, ld, m0, k0, lane);
}
template <int kP>
__device__ __forceinline__ void b_kn_p(FragP<kP>& b, const bf16_t* hi, const bf16_t* lo, int ld, int n0, int k0,
                                       int lane) {
  b_kn(b.h, hi, ld, n0, k0, lane);
  if constexpr (kP == 2) b_kn(b.l, lo, ld, n0, k0, lane);
}
// A pair of fp32 values stored as kP bf16 pairs: hi, and lo (written only for kP = 2).
template <int kP>
__device__ __forceinline__ void st_pair_p(bf16_t* hi, bf16_t* lo, float2 x) {
  const uint32_t h = pack_bf16(x.x, x.y);
  *reinterpret_cast<uint32_t*>(hi) = h;
  if constexpr (kP == 2) {
    const float2 u = unpack_bf16(h);
    *reinterpret_cast<uint32_t*>(lo) = pack_bf16(x.x - u.x, x.y - u.y);
  }
}

// A 16 x 16 fp32 accumulator (tiles acc[0], acc[1]) as kP bf16 parts [t][s] (row stride
// kB16), keeping lower: s < t (+ diagonal if incl), upper: s > t (+ diagonal if incl).
template <int kP>
__device__ __forceinline__ void store_masked16_p(const float (&acc)[2][4], bf16_t* hi, bf16_t* lo, bool lower,
                                                 bool incl, int g, int t4) {
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int t = g + 8 * h, s = 8 * nt + 2 * t4;
      float x[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int se = s + e;
        const bool keep = lower ? (se < t || (incl && se == t)) : (se > t || (incl && se == t));
        x[e] = keep ? acc[nt][2 * h + e] : 0.f;
      }
      st_pair_p<kP>(hi + t * kB16 + s, lo + t * kB16 + s, make_float2(x[0], x[1]));
    }
}
// acc[nt] += A B over K = 16 * KB for two n8 tiles, A from [m][k], B from [n][k], both in kP parts.
template <int KB, int kP>
__device__ __forceinline__ void mm_mk_nk_p(float (&acc)[2][4], const bf16_t* A, const bf16_t* Al, int lda, int m0,
                                           const bf16_t* Bt, const bf16_t* Btl, int ldb, int n0, int lane) {
#pragma unroll
  for (int kb = 0; kb < KB; ++kb) {
    FragP<kP> a, b;
    a_mk_p<kP>(a, A, Al, lda, m0, 16 * kb, lane);
    b_nk_p<kP>(b, Bt, Btl, ldb, n0, 16 * kb, lane);
    mma_pp<kP, kP>(acc, a, b);
  }
}

// Column s of T = (I - M)^-1 for a strictly lower 16 x 16 fp32 M (row stride kLD floats,
// rows 16-byte aligned): forward substitution, col[t] = [t == s] + sum_{u < t} M[t][u] col[u]
// summed in ascending u, each row of M read four entries per load.
template <int kLD>
__device__ __forceinline__ void unit_lower_inverse_col16(const float* M, int s, float (&col)[16]) {
#pragma unroll
  for (int t = 0; t < 16; ++t) {
    float x = t == s ? 1.f : 0.f;
#pragma unroll
    for (int u4 = 0; u4 < t; u4 += 4) {
      const float4 m = *reinterpret_cast<const float4*>(M + t * kLD + u4);
      x = fmaf(m.x, col[u4], x);
      if (u4 + 1 < t) x = fmaf(m.y, col[u4 + 1], x);
      if (u4 + 2 < t) x = fmaf(m.z, col[u4 + 2], x);
      if (u4 + 3 < t) x = fmaf(m.w, col[u4 + 3], x);
    }
    col[t] = x;
  }
}

}  // namespace wkv7
