// WKV7 forward scan on tensor cores (sm_103a): chunked form, bf16 or fp32 inputs, N = 64.
//
// Same result as "rx_pretrain.c", rx_wkv7_forward_seq, per (b, h):
//   sa = S a ;  S <- S diag(w) + v k^T + sa b^T ;  y = S r.
// Over a chunk of L = 16 steps with start state S0 and c(t) = w(1)...w(t)
// (chunk-relative, c(0) = 1), the column-scaled state S~ = S diag(1/c) turns
// every step into a rank-2 update, and the chunk unrolls into small dense
// products (time-major L x N matrices, rows = steps):
//   A^ = a * c(t-1), R^ = r * c(t), K~ = k / c(t), B~ = b / c(t),
//   Kb = k * c(L)/c(t), Bb = b * c(L)/c(t)
//   Mka = A^ K~^T, Mba = A^ B~^T (strictly lower), Mkr = R^ K~^T, Mbr = R^ B~^T (lower)
//   SA  = (I - Mba)^-1 (A^ S0^T + Mka V)            rows: sa(t)
//   Y   = R^ S0^T + Mkr V + Mbr SA                   rows: y(t)
//   S(L) = S0 diag(c(L)) + V^T Kb + SA^T Bb
// (exact up to rounding; the reverse scan uses the same algebra). The
// products run on tensor cores with bf16 operands (mma.sync m16n8k16,
// wkv7_mma16.cuh) and fp32 accumulation; the state stays fp32 in registers.
// With bf16 inputs each operand is one bf16 value (the inputs' own precision;
// the scaled operands and the state rounded to bf16 as they enter a product).
// With fp32 inputs each operand is a pair hi + lo of bf16 values (hi = x
// rounded to bf16, lo = the remainder rounded to bf16) and a product a b is
// taken as a_lo b_hi + a_hi b_lo + a_hi b_hi, about 16 bits of each operand.
// The state update takes Kb and Bb as such pairs for either input type.
//
// One CTA per (b, h), twelve warps in three groups working one chunk apart:
//  - forming warps (4..7) turn chunk n+2's r, w, k, v, a, b (TMA tensor loads
//    into a ring of stages) into the scaled operands;
//  - products warps (8..11) make chunk n+1's four L x L products and
//    T = (I - Mba)^-1 (forward substitution, one warp), and store the y rows
//    and checkpoint the state warps staged a round before;
//  - state warps (0..3) each own 16 rows i of S as mma accumulator tiles
//    and compute S0 [A^ R^]^T, SA, Y and S(L) for chunk n, staging y and the
//    checkpoints (fp32 inputs: the state warps store the checkpoints).
// Operand blocks rotate over three buffers. The input ring has four stages
// for bf16 inputs and three for fp32 (twice the bytes); with fp32 inputs the
// state warps store the checkpoints themselves instead of staging them.
// A chunk whose decays leave [1/16, 16] (or hold a NaN) is run step by step
// in the direct form by the state warps, in fp32.
#include "wkv7_decay.cuh"
#include "wkv7_launch.h"
#include "wkv7_mma.cuh"
#include "wkv7_mma16.cuh"
#include "wkv7_scaled.cuh"

namespace wkv7 {
namespace {

constexpr int kN = 64, kL = 16;
constexpr int kLD64 = 72;  // row stride (floats) of 64-wide operands: conflict-free fragment loads
constexpr int kLD16 = 24;  // row stride of 16-wide operands

// Operand block of one chunk: bf16 tiles (row strides of 72 and 24 elements put the eight
// 16-byte rows of every ldmatrix on distinct banks). kP = 1 (bf16 inputs): each operand is
// one bf16 value, the inputs' own precision. kP = 2 (fp32 inputs): each operand is a pair
// hi + lo ([0] = the value rounded to bf16, [1] = the remainder rounded to bf16), about 16
// bits, and a product a b is taken as a_lo b_hi + a_hi b_lo + a_hi b_hi. Kb and Bb are
// pairs either way: the state update keeps them to about 16 bits.
template <int kP>
struct alignas(16) Prep16 {
  bf16_t X1[kP][2 * kL * kB64];  // rows 0..15: a^(t); rows 16..31: r^(t)   [t][j]
  bf16_t V[kP][kL * kB64];       // v(s)[i]                                   [s][i]
  bf16_t Kb[2][kL * kB64];       // k(s)[j] c(L)[j] / c(s)[j]                 [s][j]
  bf16_t Bb[2][kL * kB64];       // b(s)[j] c(L)[j] / c(s)[j]                 [s][j]
  bf16_t M[kP][3][kL * kB16];    // Mka (strictly lower), Mkr, Mbr (lower)    [t][s]
  bf16_t Tinv[kP][kL * kB16];    // (I - Mba)^-1                              [t][s]
  float Mba[kL * kLD16];         // Mba (strictly lower, fp32: T is formed from it)
  float cL[kN];                  // c(L) (fp32)
  int unsafe;
  int pad_[31];
};
static_assert(offsetof(Prep16<1>, Mba) % 16 == 0 && offsetof(Prep16<2>, Mba) % 16 == 0,
              "Mba rows are read 16 bytes at a time");

// Per input type: input ring depth and refill point, checkpoint staging, operand parts and
// the row stride of the staged y rows. With fp32 inputs (three stages of twice the bytes) the
// stage of chunk n is refilled once the chunk is formed (round n - 2), two rounds before the
// next chunk in it is formed, and a chunk in the direct form reads its rows from global
// memory; refilled after round n the forming group waited for its copy every round. With
// bf16 inputs (four stages) the stage is refilled after round n, a round to spare, and the
// direct form reads the stage.
template <typename TIn>
struct Fwd3Io;
template <>
struct Fwd3Io<__nv_bfloat16> {
  static constexpr int kStages = 4;
  static constexpr int kRefillAhead = 0;  // the stage of chunk n + kRefillAhead is refilled after round n
  static constexpr bool kStageCk = true;
  static constexpr int kP = 1;
  static constexpr int kYS = kB64;  // padded: the transposed matrix stores of y hit distinct banks
};
template <>
struct Fwd3Io<float> {
  static constexpr int kStages = 3;
  static constexpr int kRefillAhead = 2;
  static constexpr bool kStageCk = false;
  static constexpr int kP = 2;
  static constexpr int kYS = kN;
};

template <typename TIn>
struct Fwd3Smem {
  using Io = Fwd3Io<TIn>;
  static constexpr int kStages = Io::kStages;
  static constexpr bool kStageCk = Io::kStageCk;
  TIn raw[kStages][6][kL * kN];  // TMA ring: r, w, k, v, a, b of one chunk per stage
  Prep16<Io::kP> prep[3];
  bf16_t X2[2][Io::kP][2 * kL * kB64];  // per chunk in flight: rows 0..15: k~(s); rows 16..31: b~(s)   [s][j]
  TIn ys[2][kL * Io::kYS];  // y of the chunk [t][i], on its way out (state warps write, products warps store)
  // epilogue: the head's ln_w, ln_b, r_k; per chunk (ring of 4, written by the forming
  // group two rounds before the state warps run the chunk, read by the products group the
  // round after) the bonus partials of the two 32-column halves and the v rows
  float epi[3][kN];
  float epi_sp[4][kL];
  __nv_bfloat16 epi_v[4][kL * kN];
  // checkpoints on their way out (state warps write, products warps store); bf16 inputs only
  float ck[kStageCk ? 2 : 1][kStageCk ? kN * kLD64 : 4];
  float pq[4][kN];  // forming group: the product of each quarter's four decays, per column
  uint64_t full[kStages];
  int abort_flag;
};

constexpr int kThreads = 384;  // warps 0-3: state; 4-7: forming; 8-11: products
enum { V_R = 0, V_W = 1, V_K = 2, V_V = 3, V_A = 4, V_B = 5 };

__device__ __forceinline__ float bf(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ float bf(const float* p) { return *p; }
__device__ __forceinline__ float2 bf2(const __nv_bfloat16* p) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
}
__device__ __forceinline__ float2 bf2(const float* p) { return *reinterpret_cast<const float2*>(p); }

// ---------------------------------------------------------- forming group ---
// 128 threads; thread (lane, q = ptid / 32) forms columns 2 lane, 2 lane + 1 of steps
// 4 q .. 4 q + 3: pairs of row elements, so every load and store moves two columns. The
// running products c(t) are taken per quarter of four steps and the quarters' products
// chained in step order through shared memory; the same group barrier votes on whether the
// chunk leaves the scaled form's range.
template <typename TIn, bool kLogit, bool kEpi>
__device__ void form_chunk(Fwd3Smem<TIn>& sm, Prep16<Fwd3Io<TIn>::kP>& P, bf16_t (*X2)[2 * kL * kB64], int stage,
                           int len, int ptid, int eslot) {
  constexpr int kP = Fwd3Io<TIn>::kP, kLo = kP - 1;  // index of the lo part (the hi part for kP = 1)
  const TIn* rs = sm.raw[stage][0];
  const int lane = ptid & 31, q = ptid >> 5, j = 2 * lane, t0 = 4 * q;
  // decays of this thread's four steps; padding steps past the end of the sequence decay by 1
  float2 wv[4], av[4], rv[4], kv[4], bv[4], vv[4];
  bool unsafe = false;
  float2 pq = make_float2(1.f, 1.f);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int o = (t0 + e) * kN + j;
    wv[e] = t0 + e < len ? decay_value2<kLogit>(bf2(rs + V_W * kL * kN + o)) : make_float2(1.f, 1.f);
    unsafe |= !decay_is_safe(wv[e].x) || !decay_is_safe(wv[e].y);
    pq = fmul2(pq, wv[e]);
  }
  *reinterpret_cast<float2*>(&sm.pq[q][j]) = pq;
  // the other rows are read before the group barrier, so their loads overlap it
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int o = (t0 + e) * kN + j;
    av[e] = bf2(rs + V_A * kL * kN + o);
    rv[e] = bf2(rs + V_R * kL * kN + o);
    kv[e] = bf2(rs + V_K * kL * kN + o);
    bv[e] = bf2(rs + V_B * kL * kN + o);
    vv[e] = bf2(rs + V_V * kL * kN + o);
  }
  unsafe = named_bar_or(1, 128, unsafe);
  if (ptid == 0) P.unsafe = unsafe;
  if constexpr (kEpi) {
    // the epilogue's bonus sum_j r_j k_j r_k[j] of each step over the 64 columns,
    // reduce-scattered over the lanes (lane bits 4, 3 pick the step), and the v rows
    const float2 rk = *reinterpret_cast<const float2*>(&sm.epi[2][j]);
    float p[4], q2[2];
#pragma unroll
    for (int e = 0; e < 4; ++e) p[e] = fmaf(rv[e].x * kv[e].x, rk.x, rv[e].y * kv[e].y * rk.y);
    const bool b4 = lane & 16, b3 = lane & 8;
#pragma unroll
    for (int u = 0; u < 2; ++u)
      q2[u] = (b4 ? p[2 + u] : p[u]) + __shfl_xor_sync(0xffffffffu, b4 ? p[u] : p[2 + u], 16);
    float sum = (b3 ? q2[1] : q2[0]) + __shfl_xor_sync(0xffffffffu, b3 ? q2[0] : q2[1], 8);
    sum += __shfl_xor_sync(0xffffffffu, sum, 4);
    sum += __shfl_xor_sync(0xffffffffu, sum, 2);
    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
    if ((lane & 7) == 0) sm.epi_sp[eslot][t0 + 2 * (b4 ? 1 : 0) + (b3 ? 1 : 0)] = sum;
#pragma unroll
    for (int e = 0; e < 4; ++e)
      *reinterpret_cast<uint32_t*>(&sm.epi_v[eslot][(t0 + e) * kN + j]) =
          *reinterpret_cast<const uint32_t*>(rs + V_V * kL * kN + (t0 + e) * kN + j);
  }
  if (unsafe) return;  // the state warps run the chunk step by step
  float2 cL = make_float2(1.f, 1.f), c = cL;  // c = c(t0 - 1) after the loop
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    cL = fmul2(cL, *reinterpret_cast<const float2*>(&sm.pq[u][j]));
    if (u < q) c = cL;
  }
  if (q == 0) *reinterpret_cast<float2*>(&P.cL[j]) = cL;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int t = t0 + e;
    const float2 cprev = c;
    c = fmul2(c, wv[e]);
    const float2 ic = make_float2(rcp_approx(c.x), rcp_approx(c.y)), s = fmul2(cL, ic);
    const int o0 = t * kB64 + j, o1 = (kL + t) * kB64 + j;
    st_pair_p<kP>(X2[0] + o0, X2[kLo] + o0, fmul2(kv[e], ic));
    st_pair_p<kP>(X2[0] + o1, X2[kLo] + o1, fmul2(bv[e], ic));
    st_pair_p<kP>(P.X1[0] + o0, P.X1[kLo] + o0, fmul2(av[e], cprev));
    st_pair_p<kP>(P.X1[0] + o1, P.X1[kLo] + o1, fmul2(rv[e], c));
    // v in kP parts (exact for bf16 inputs); kb and bb as hi and lo parts
    st_pair_p<kP>(P.V[0] + o0, P.V[kLo] + o0, vv[e]);
    st_pair_p<2>(P.Kb[0] + o0, P.Kb[1] + o0, fmul2(kv[e], s));
    st_pair_p<2>(P.Bb[0] + o0, P.Bb[1] + o0, fmul2(bv[e], s));
  }
}

// --------------------------------------------------------- products group ---
// The four L x L products and T of a formed chunk (128 threads; skipped by the caller for
// a chunk in the direct form). Warp pw computes the Gram block [A^ | R^](rows 16 (pw / 2))
// x [K~ | B~](rows 16 (pw % 2))^T (K = 64 in four k16 steps); Mka, Mkr, Mbr are stored in
// kP bf16 parts, Mba in fp32, from which one warp forms T by fp32 forward substitution
// and stores it in kP parts.
template <int kP>
__device__ void gram_chunk16(Prep16<kP>& P, const bf16_t (*X2)[2 * kL * kB64], int gtid) {
  constexpr int kLo = kP - 1;
  const int pw = gtid >> 5, lane = gtid & 31, g = lane >> 2, t4 = lane & 3;
  const int mt = pw >> 1, nb = pw & 1;
  float acc[2][4];
  zero4(acc[0]);
  zero4(acc[1]);
#pragma unroll
  for (int kb = 0; kb < 4; ++kb) {
    FragP<kP> a, b;
    a_mk_p<kP>(a, P.X1[0], P.X1[kLo], kB64, 16 * mt, 16 * kb, lane);
    b_nk_p<kP>(b, X2[0], X2[kLo], kB64, 16 * nb, 16 * kb, lane);
    mma_pp<kP, kP>(acc, a, b);
  }
  if (pw != 1) {
    // pw 0: Mka (s < t); 2: Mkr, 3: Mbr (s <= t)
    const int m = pw == 0 ? 0 : pw - 1;
    store_masked16(acc, P.M[0][m], true, pw >= 2, g, t4);
    if constexpr (kP == 2) {  // the remainders after rounding to bf16
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[nt][e] -= __bfloat162float(__float2bfloat16_rn(acc[nt][e]));
      store_masked16(acc, P.M[kLo][m], true, pw >= 2, g, t4);
    }
    return;
  }
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int tt = g + 8 * h, s = 8 * nt + 2 * t4;
      *reinterpret_cast<float2*>(P.Mba + tt * kLD16 + s) =
          make_float2(s < tt ? acc[nt][2 * h] : 0.f, s + 1 < tt ? acc[nt][2 * h + 1] : 0.f);
    }
  __syncwarp();
  // T = (I - Mba)^-1 by forward substitution in fp32; lane s (< 16) owns column s
  const int s = lane & 15;
  float col[kL];
  unit_lower_inverse_col16<kLD16>(P.Mba, s, col);
  if (lane < 16) {
#pragma unroll
    for (int tt = 0; tt < kL; ++tt) put_p<kP>(P.Tinv[0] + tt * kB16 + s, P.Tinv[kLo] + tt * kB16 + s, col[tt]);
  }
}

// ----------------------------------------------------------- state warps ---

struct StateCtx {
  float S[8][4];  // rows i0+g, i0+g+8; columns 8*nt + 2*t4 + {0, 1}
  int i0, g, t4;
  int yb;  // which y staging buffer this round writes
};

// The state into a staging tile (rows of kLD64 floats).
__device__ __forceinline__ void stage_state(const StateCtx& c, float* dst) {
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) {
    const int col = 8 * nt + 2 * c.t4;
    *reinterpret_cast<float2*>(dst + (c.i0 + c.g) * kLD64 + col) = make_float2(c.S[nt][0], c.S[nt][1]);
    *reinterpret_cast<float2*>(dst + (c.i0 + c.g + 8) * kLD64 + col) = make_float2(c.S[nt][2], c.S[nt][3]);
  }
}

// A staged 64 x 64 state to global memory (kT threads, whole rows per instruction);
// dst lies in the buffer x (checked in the debug build).
template <int kT>
__device__ __forceinline__ void flush_state(const float* src, float* dst, int ptid, const Extent& x, unsigned* status) {
#pragma unroll
  for (int q = 0; q < (kN * kN / 4 + kT - 1) / kT; ++q) {
    const int idx = ptid + kT * q;  // row idx / 16, columns 4 (idx % 16) ..
    if (kT * (q + 1) > kN * kN / 4 && idx >= kN * kN / 4) break;
    float4* p = reinterpret_cast<float4*>(dst + 4 * idx);
    if (in_extent(status, x, p)) *p = *reinterpret_cast<const float4*>(src + (idx >> 4) * kLD64 + 4 * (idx & 15));
  }
}

// A chunk's staged y rows ([t][i] bf16, row stride kB64) to global memory: kT threads, 16
// rows x 8 pieces of 16 bytes, rows past the end of the sequence skipped.
template <int kT>
__device__ __forceinline__ void flush_y(const __nv_bfloat16* src, __nv_bfloat16* dst, size_t vstep, int len, int ptid,
                                        const Extent& x, unsigned* status) {
#pragma unroll
  for (int q = 0; q < (kL * 8 + kT - 1) / kT; ++q) {
    const int idx = ptid + kT * q;
    if (kT * (q + 1) > kL * 8 && idx >= kL * 8) break;
    const int row = idx >> 3, piece = idx & 7;
    uint4* p = reinterpret_cast<uint4*>(dst + (size_t)row * vstep + 8 * piece);
    if (row < len && in_extent(status, x, p)) *p = *reinterpret_cast<const uint4*>(src + row * kB64 + 8 * piece);
  }
}

// The same for fp32 rows: 16 rows x 8 pieces of 32 bytes.
template <int kT>
__device__ __forceinline__ void flush_y(const float* src, float* dst, size_t vstep, int len, int ptid, const Extent& x,
                                        unsigned* status) {
#pragma unroll
  for (int q = 0; q < (kL * 8 + kT - 1) / kT; ++q) {
    const int idx = ptid + kT * q;
    if (kT * (q + 1) > kL * 8 && idx >= kL * 8) break;
    const int row = idx >> 3, piece = idx & 7;
    uint4* p = reinterpret_cast<uint4*>(dst + (size_t)row * vstep + 8 * piece);
    if (row < len && in_extent(status, x, p, 2)) {
      p[0] = *reinterpret_cast<const uint4*>(src + row * kN + 8 * piece);
      p[1] = *reinterpret_cast<const uint4*>(src + row * kN + 8 * piece + 4);
    }
  }
}

__device__ __forceinline__ void store_state(const StateCtx& c, float* dst, const Extent& x, unsigned* status) {
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) {
    const int col = 8 * nt + 2 * c.t4;
    float2* p0 = reinterpret_cast<float2*>(dst + (c.i0 + c.g) * kN + col);
    float2* p1 = reinterpret_cast<float2*>(dst + (c.i0 + c.g + 8) * kN + col);
    if (in_extent(status, x, p0)) *p0 = make_float2(c.S[nt][0], c.S[nt][1]);
    if (in_extent(status, x, p1)) *p1 = make_float2(c.S[nt][2], c.S[nt][3]);
  }
}

// Chunk on tensor cores with bf16 operands in kP parts (bf16 inputs: one; fp32 inputs: hi
// + lo). Four k16 steps over j for S0 [A^ R^]^T, one k16 step over s for every product
// with V, T, Mbr; Kb and Bb enter the state update as hi + lo pairs, so the carried state
// keeps them to about 16 bits. The state, P and SA enter the next product in kP parts.
// Writes the chunk's y into ys: bf16 rows of stride kB64 by transposed matrix stores, or
// fp32 rows of stride kN.
template <typename TIn>
__device__ void state_chunk16(StateCtx& c, Fwd3Smem<TIn>& sm, const Prep16<Fwd3Io<TIn>::kP>& P, int lane) {
  constexpr int kP = Fwd3Io<TIn>::kP, kLo = kP - 1;
  const int i0 = c.i0;
  using Acc2 = float[2][4];
  // PA = S0 A^^T (later + V^T Mka^T), PR = S0 R^^T (later + ...): [i][t]
  float PA[2][4], PR[2][4];
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    zero4(PA[q]);
    zero4(PR[q]);
  }
  FragP<kP> b;
#pragma unroll
  for (int kb = 0; kb < 4; ++kb) {
    FragP<kP> a;
    c2a_p<kP>(a, c.S[2 * kb], c.S[2 * kb + 1]);
    b_nk_p<kP>(b, P.X1[0], P.X1[kLo], kB64, 0, 16 * kb, lane);  // A^, steps 0..15 as two n8 tiles
    mma_pp<kP, kP>(PA, a, b);
    b_nk_p<kP>(b, P.X1[0], P.X1[kLo], kB64, kL, 16 * kb, lane);  // R^
    mma_pp<kP, kP>(PR, a, b);
  }
  FragP<kP> av;  // V^T rows i0.., k = s
  a_km_p<kP>(av, P.V[0], P.V[kLo], kB64, i0, 0, lane);
  b_nk_p<kP>(b, P.M[0][0], P.M[kLo][0], kB16, 0, 0, lane);  // Mka
  mma_pp<kP, kP>(PA, av, b);
  b_nk_p<kP>(b, P.M[0][1], P.M[kLo][1], kB16, 0, 0, lane);  // Mkr
  mma_pp<kP, kP>(PR, av, b);
  // S(L) = S0 diag(c(L)) + V^T Kb + SA^T Bb; the first two terms need no SA, so they are
  // issued here, while SA is under way
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) {
    const float2 cl = *reinterpret_cast<const float2*>(P.cL + 8 * nt + 2 * c.t4);
    c.S[nt][0] *= cl.x;
    c.S[nt][1] *= cl.y;
    c.S[nt][2] *= cl.x;
    c.S[nt][3] *= cl.y;
  }
  FragP<2> bk;
#pragma unroll
  for (int np = 0; np < 4; ++np) {
    b_kn_p<2>(bk, P.Kb[0], P.Kb[1], kB64, 16 * np, 0, lane);
    mma_pp<kP, 2>(reinterpret_cast<Acc2&>(c.S[2 * np]), av, bk);
  }
  // SA^T = PA T^T  [i][t]
  float SA[2][4];
  zero4(SA[0]);
  zero4(SA[1]);
  {
    FragP<kP> a;
    c2a_p<kP>(a, PA[0], PA[1]);
    b_nk_p<kP>(b, P.Tinv[0], P.Tinv[kLo], kB16, 0, 0, lane);
    mma_pp<kP, kP>(SA, a, b);
  }
  FragP<kP> asa;
  c2a_p<kP>(asa, SA[0], SA[1]);
  // Y^T = PR + SA^T Mbr^T, stored as the chunk's y rows [t][i]
  b_nk_p<kP>(b, P.M[0][2], P.M[kLo][2], kB16, 0, 0, lane);
  mma_pp<kP, kP>(PR, asa, b);
  if constexpr (kP == 1) {
    uint32_t yv[4];
    c2a16(yv, PR[0], PR[1]);
    stsm4t(&sm.ys[c.yb][((lane & 7) + (lane >> 4) * 8) * kB64 + i0 + ((lane >> 3) & 1) * 8], yv);
  } else {
#pragma unroll
    for (int q = 0; q < 2; ++q)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int i = i0 + c.g + 8 * h, tt = 8 * q + 2 * c.t4;
        st1(&sm.ys[c.yb][tt * kN + i], PR[q][2 * h]);
        st1(&sm.ys[c.yb][(tt + 1) * kN + i], PR[q][2 * h + 1]);
      }
  }
  // + SA^T Bb
#pragma unroll
  for (int np = 0; np < 4; ++np) {
    b_kn_p<2>(bk, P.Bb[0], P.Bb[1], kB64, 16 * np, 0, lane);
    mma_pp<kP, 2>(reinterpret_cast<Acc2&>(c.S[2 * np]), asa, bk);
  }
}

// Chunk in the direct form (any decay), fp32 on the CUDA cores, from its input stage.
template <typename TIn, bool kLogit>
__device__ void state_chunk_direct(StateCtx& c, Fwd3Smem<TIn>& sm, int stage, int len) {
  const int g = c.g, t4 = c.t4, i0 = c.i0;
  const TIn* rs = sm.raw[stage][0];
  for (int t = 0; t < len; ++t) {
    const TIn* row = rs + t * kN;
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const float2 a = bf2(row + V_A * kL * kN + 8 * nt + 2 * t4);
      s0 = fmaf(c.S[nt][0], a.x, fmaf(c.S[nt][1], a.y, s0));
      s1 = fmaf(c.S[nt][2], a.x, fmaf(c.S[nt][3], a.y, s1));
    }
    s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
    s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
    s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
    s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
    const float v0 = bf(row + V_V * kL * kN + i0 + g), v1 = bf(row + V_V * kL * kN + i0 + g + 8);
    float y0 = 0.f, y1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const int col = 8 * nt + 2 * t4;
      const float2 w = decay_value2<kLogit>(bf2(row + V_W * kL * kN + col)), k = bf2(row + V_K * kL * kN + col);
      const float2 b = bf2(row + V_B * kL * kN + col), r = bf2(row + V_R * kL * kN + col);
      c.S[nt][0] = fmaf(s0, b.x, fmaf(c.S[nt][0], w.x, v0 * k.x));
      c.S[nt][1] = fmaf(s0, b.y, fmaf(c.S[nt][1], w.y, v0 * k.y));
      c.S[nt][2] = fmaf(s1, b.x, fmaf(c.S[nt][2], w.x, v1 * k.x));
      c.S[nt][3] = fmaf(s1, b.y, fmaf(c.S[nt][3], w.y, v1 * k.y));
      y0 = fmaf(c.S[nt][0], r.x, fmaf(c.S[nt][1], r.y, y0));
      y1 = fmaf(c.S[nt][2], r.x, fmaf(c.S[nt][3], r.y, y1));
    }
    y0 += __shfl_xor_sync(0xffffffffu, y0, 1);
    y0 += __shfl_xor_sync(0xffffffffu, y0, 2);
    y1 += __shfl_xor_sync(0xffffffffu, y1, 1);
    y1 += __shfl_xor_sync(0xffffffffu, y1, 2);
    if (t4 == 0) {
      constexpr int kYS = Fwd3Io<TIn>::kYS;
      st1(&sm.ys[c.yb][t * kYS + i0 + g], y0);
      st1(&sm.ys[c.yb][t * kYS + i0 + g + 8], y1);
    }
  }
}

// The same from the chunk's rows in global memory (row0 = the offset of its first row, vstep
// between steps), for an input stage refilled as soon as its chunk was formed.
template <typename TIn, bool kLogit>
__device__ void state_chunk_direct_global(StateCtx& c, Fwd3Smem<TIn>& sm, const FwdArgs& args, size_t row0,
                                          size_t vstep, int len) {
  const int g = c.g, t4 = c.t4, i0 = c.i0;
  auto ld2 = [&](int v, int t, int col) {
    const TIn* p = static_cast<const TIn*>(args.in[v]) + row0 + (size_t)t * vstep + col;
    return in_extent(args.status, args.ext.in[v], p, 2) ? bf2(p) : make_float2(0.f, 0.f);
  };
  auto ld1 = [&](int v, int t, int col) {
    const TIn* p = static_cast<const TIn*>(args.in[v]) + row0 + (size_t)t * vstep + col;
    return in_extent(args.status, args.ext.in[v], p) ? bf(p) : 0.f;
  };
  for (int t = 0; t < len; ++t) {
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const float2 a = ld2(V_A, t, 8 * nt + 2 * t4);
      s0 = fmaf(c.S[nt][0], a.x, fmaf(c.S[nt][1], a.y, s0));
      s1 = fmaf(c.S[nt][2], a.x, fmaf(c.S[nt][3], a.y, s1));
    }
    s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
    s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
    s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
    s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
    const float v0 = ld1(V_V, t, i0 + g), v1 = ld1(V_V, t, i0 + g + 8);
    float y0 = 0.f, y1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const int col = 8 * nt + 2 * t4;
      const float2 w = decay_value2<kLogit>(ld2(V_W, t, col)), k = ld2(V_K, t, col);
      const float2 b = ld2(V_B, t, col), r = ld2(V_R, t, col);
      c.S[nt][0] = fmaf(s0, b.x, fmaf(c.S[nt][0], w.x, v0 * k.x));
      c.S[nt][1] = fmaf(s0, b.y, fmaf(c.S[nt][1], w.y, v0 * k.y));
      c.S[nt][2] = fmaf(s1, b.x, fmaf(c.S[nt][2], w.x, v1 * k.x));
      c.S[nt][3] = fmaf(s1, b.y, fmaf(c.S[nt][3], w.y, v1 * k.y));
      y0 = fmaf(c.S[nt][0], r.x, fmaf(c.S[nt][1], r.y, y0));
      y1 = fmaf(c.S[nt][2], r.x, fmaf(c.S[nt][3], r.y, y1));
    }
    y0 += __shfl_xor_sync(0xffffffffu, y0, 1);
    y0 += __shfl_xor_sync(0xffffffffu, y0, 2);
    y1 += __shfl_xor_sync(0xffffffffu, y1, 1);
    y1 += __shfl_xor_sync(0xffffffffu, y1, 2);
    if (t4 == 0) {
      constexpr int kYS = Fwd3Io<TIn>::kYS;
      st1(&sm.ys[c.yb][t * kYS + i0 + g], y0);
      st1(&sm.ys[c.yb][t * kYS + i0 + g + 8], y1);
    }
  }
}

// The chunk's staged y rows through the time-mix epilogue ("rx_pretrain.c":
// gn_forward and the bonus) to global memory: for every step t and head, with
// mean and var over the N channels and rstd = 1 / sqrt(var + 64e-5),
//   out = (y - mean) rstd ln_w + ln_b + (sum_j r_j k_j r_k[j]) v,
// plus (y - mean) rstd to args.nv and (rstd, bonus) to args.stats when given.
// The products group, eight threads per row (eight channels each); the bonus
// partials and v rows were staged by the forming group.
__device__ void flush_epilogue(const Fwd3Smem<__nv_bfloat16>& sm, const FwdArgs& args, int m, size_t vbase, size_t vstep,
                               int len, int ptid) {
  const int t = ptid >> 3, i0 = 8 * (ptid & 7), es = m % 4;
  auto load8 = [](const __nv_bfloat16* p, float (&x)[8]) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wv[q]));
      x[2 * q] = f.x;
      x[2 * q + 1] = f.y;
    }
  };
  float y[8], v[8];
  load8(&sm.ys[m & 1][t * kB64 + i0], y);
  load8(&sm.epi_v[es][t * kN + i0], v);
  float sum = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) sum += y[e];
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  const float mean = sum * (1.f / kN);
  float sq = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    y[e] -= mean;
    sq = fmaf(y[e], y[e], sq);
  }
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
  const float rstd = rsqrtf(sq * (1.f / kN) + 64e-5f);
  const float bon = sm.epi_sp[es][t];
  uint32_t po[4], pn[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    float o2[2], n2[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int e = 2 * q + h;
      n2[h] = y[e] * rstd;
      o2[h] = fmaf(n2[h], sm.epi[0][i0 + e], fmaf(bon, v[e], sm.epi[1][i0 + e]));
    }
    const __nv_bfloat162 bo = __floats2bfloat162_rn(o2[0], o2[1]), bn = __floats2bfloat162_rn(n2[0], n2[1]);
    po[q] = *reinterpret_cast<const uint32_t*>(&bo);
    pn[q] = *reinterpret_cast<const uint32_t*>(&bn);
  }
  if (t < len) {
    const size_t off = vbase + ((size_t)m * kL + t) * vstep + i0;
    uint4* py = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(args.y) + off);
    if (in_extent(args.status, args.ext.y, py)) *py = make_uint4(po[0], po[1], po[2], po[3]);
    if (args.nv) {
      uint4* pv = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(args.nv) + off);
      if (in_extent(args.status, args.ext.nv, pv)) *pv = make_uint4(pn[0], pn[1], pn[2], pn[3]);
    }
    if (args.stats && (ptid & 7) == 0) {
      float2* ps = reinterpret_cast<float2*>(args.stats + 2 * (off / kN));
      if (in_extent(args.status, args.ext.stats, ps)) *ps = make_float2(rstd, bon);
    }
  }
}

template <typename TIn, bool kLogit, bool kEpi>
__global__ void __launch_bounds__(kThreads, 1) wkv7_fwd3_kernel(const __grid_constant__ FwdArgs args) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  using Smem = Fwd3Smem<TIn>;
  constexpr int kStages = Smem::kStages;
  constexpr bool kStageCk = Smem::kStageCk;
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
  const int T = args.T, H = args.H;
  const int head = blockIdx.x, bi = head / H, hi = head % H;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int role = warp < 4 ? 0 : warp < 8 ? 1 : 2;  // state, forming, products
  const int ftid = tid - 128, gtid = tid - 256;
  const int nchunks = (T + kL - 1) / kL;
  constexpr int kStageBytes = 6 * kL * kN * (int)sizeof(TIn);

  // Chunk n: the state warps run it in round n, the products group makes its
  // L x L products and T in round n-1, the forming group forms it in round
  // n-2. Its inputs arrive by TMA in a ring of kStages stages; after round n
  // the stage of chunk n + kRefillAhead is refilled.
  constexpr int kRefillAhead = Smem::Io::kRefillAhead;
  auto issue = [&](int chunk) {
    const int st = chunk % kStages;
    mbar_arrive_expect_tx(&sm.full[st], kStageBytes);
    for (int v = 0; v < 6; ++v) tma_load_4d(sm.raw[st][v], &args.map[v], &sm.full[st], 0, hi, chunk * kL, bi);
  };
  // TMA copies are issued by the first thread of products warp 10: the products group has
  // the shortest round, and its warp 9 (T) the longest work in it
  constexpr int kIssuer = 320;
  if (tid == kIssuer) {
    for (int s = 0; s < kStages; ++s) mbar_init(&sm.full[s], 1);
    fence_mbar_init();
    for (int v = 0; v < 6; ++v) prefetch_tensormap(&args.map[v]);
    for (int ch = 0; ch < kStages && ch < nchunks; ++ch) issue(ch);
  }
  if (tid == 0) sm.abort_flag = 0;
  if constexpr (kEpi) {
    for (int i = tid; i < 3 * kN; i += kThreads) {
      const float* src = (i < kN ? args.ln_w : i < 2 * kN ? args.ln_b : args.r_k) + (size_t)hi * kN + i % kN;
      const Extent& x = i < kN ? args.ext.ln_w : i < 2 * kN ? args.ext.ln_b : args.ext.r_k;
      sm.epi[i / kN][i % kN] = in_extent(args.status, x, src) ? *src : 0.f;
    }
  }

  StateCtx c;
  c.g = lane >> 2;
  c.t4 = lane & 3;
  c.i0 = 16 * warp;
  if (role == 0) {
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) c.S[nt][e] = 0.f;
    if (args.s_init) {
      const float* src = args.s_init + (size_t)head * kN * kN;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const int col = 8 * nt + 2 * c.t4;
        const float2* p0 = reinterpret_cast<const float2*>(src + (c.i0 + c.g) * kN + col);
        const float2* p1 = reinterpret_cast<const float2*>(src + (c.i0 + c.g + 8) * kN + col);
        const float2 lo = in_extent(args.status, args.ext.s_init, p0) ? *p0 : make_float2(0.f, 0.f);
        const float2 hi2 = in_extent(args.status, args.ext.s_init, p1) ? *p1 : make_float2(0.f, 0.f);
        c.S[nt][0] = lo.x;
        c.S[nt][1] = lo.y;
        c.S[nt][2] = hi2.x;
        c.S[nt][3] = hi2.y;
      }
    }
  }
  __syncthreads();

  // Each forming thread waits for the stage itself. A timeout raises the CTA's
  // abort flag and the thread forms the chunk all the same (from whatever the
  // stage holds), so the group's named barriers stay matched; every thread
  // reads the flag after the round's barrier and leaves the loop.
  int waited = 0;  // chunks whose stage has landed (forming group)
  int issued = min(kStages, nchunks);  // chunks whose copy was started (every thread keeps count)
  auto chunk_len = [&](int chunk) { return min(kL, T - chunk * kL); };
  auto form = [&](int chunk) {
    const bool ok = mbar_wait_bounded(args.status, &sm.full[chunk % kStages], (chunk / kStages) & 1);
    if (ok)
      waited = chunk + 1;
    else
      *reinterpret_cast<volatile int*>(&sm.abort_flag) = 1;
    form_chunk<TIn, kLogit, kEpi>(sm, sm.prep[chunk % 3], sm.X2[chunk & 1], chunk % kStages, chunk_len(chunk), ftid,
                                  chunk % 4);
  };
  auto grams = [&](int chunk) {
    auto& P = sm.prep[chunk % 3];
    if (!P.unsafe) gram_chunk16<Fwd3Io<TIn>::kP>(P, sm.X2[chunk & 1], gtid);
  };

  // refill the stage of a chunk just formed (every thread calls it after a barrier)
  auto refill = [&](int formed) {
    if (tid == kIssuer && formed + kStages < nchunks) {
      fence_proxy_async_smem();
      issue(formed + kStages);
    }
    issued = min(formed + 1 + kStages, nchunks);
  };
  // pipeline fill: form chunks 0 and 1, products of chunk 0
  if (role == 1) form(0);
  bool aborted = __syncthreads_or(sm.abort_flag) != 0;
  if (!aborted) {
    if constexpr (kRefillAhead == 2) refill(0);
    if (role == 1 && nchunks > 1) form(1);
    if (role == 2) grams(0);
    aborted = __syncthreads_or(sm.abort_flag) != 0;
    if constexpr (kRefillAhead == 2) {
      if (!aborted) refill(1);
    }
  }
  TIn* y = static_cast<TIn*>(args.y);
  const size_t vstep = (size_t)H * kN;
  const size_t vbase = ((size_t)bi * T * H + hi) * kN;
  float* ck_head = args.ckpt ? args.ckpt + (size_t)head * args.nck * kN * kN : nullptr;

  for (int n = 0; n < nchunks && !aborted; ++n) {
    if (role == 1) {
      if (n + 2 < nchunks) form(n + 2);
    } else if (role == 2) {
      if (n + 1 < nchunks) grams(n + 1);
      // the checkpoint and the y rows the state warps staged in the previous round, stored by
      // the products warps other than the one forming T (the longest products work)
      if (n > 0 && gtid >> 5 != 1) {
        const int fl = gtid < 32 ? gtid : gtid - 32;
        if (kStageCk && ck_head && ((n - 1) * kL) % args.C == 0)
          flush_state<96>(sm.ck[(n - 1) & 1], ck_head + (size_t)((n - 1) * kL / args.C) * kN * kN, fl, args.ext.ckpt,
                          args.status);
        if constexpr (!kEpi) {
          if (y)
            flush_y<96>(sm.ys[(n - 1) & 1], y + vbase + (size_t)(n - 1) * kL * vstep, vstep, chunk_len(n - 1), fl,
                        args.ext.y, args.status);
        }
      }
      if constexpr (kEpi) {
        if (n > 0) flush_epilogue(sm, args, n - 1, vbase, vstep, chunk_len(n - 1), gtid);
      }
    } else {
      const auto& P = sm.prep[n % 3];
      const int t0 = n * kL, len = chunk_len(n);
      if (ck_head && t0 % args.C == 0) {
        if constexpr (kStageCk)
          stage_state(c, sm.ck[n & 1]);
        else
          store_state(c, ck_head + (size_t)(t0 / args.C) * kN * kN, args.ext.ckpt, args.status);
      }
      c.yb = n & 1;
      if (P.unsafe) {
        if constexpr (kRefillAhead > 0)
          state_chunk_direct_global<TIn, kLogit>(c, sm, args, vbase + (size_t)t0 * vstep, vstep, len);
        else
          state_chunk_direct<TIn, kLogit>(c, sm, n % kStages, len);
      }
      else
        state_chunk16<TIn>(c, sm, P, lane);
    }
    __syncthreads();
    aborted = *reinterpret_cast<volatile int*>(&sm.abort_flag) != 0;
    if constexpr (kRefillAhead == 0) {
      // the stage of chunk n is free (formed two rounds ago, direct steps done); refill it
      if (!aborted && tid == kIssuer && n + kStages < nchunks) {
        fence_proxy_async_smem();
        issue(n + kStages);
      }
      if (!aborted) issued = min(n + 1 + kStages, nchunks);
    } else {
      if (!aborted) refill(n + kRefillAhead);  // the stage of chunk n + 2, formed in this round
    }
  }
  if (aborted) {
    // let the copies still in flight land before the CTA's shared memory is released
    if (tid == 128)
      for (int ch = waited; ch < issued; ++ch)
        mbar_wait_bounded(nullptr, &sm.full[ch % kStages], (ch / kStages) & 1, 200000000ull);
    __syncthreads();
    return;
  }
  // the last staged checkpoint and y rows
  if (role == 2 && nchunks > 0) {
    const int n = nchunks - 1;
    if (kStageCk && ck_head && (n * kL) % args.C == 0)
      flush_state<128>(sm.ck[n & 1], ck_head + (size_t)(n * kL / args.C) * kN * kN, gtid, args.ext.ckpt, args.status);
    if constexpr (kEpi)
      flush_epilogue(sm, args, n, vbase, vstep, chunk_len(n), gtid);
    else if (y)
      flush_y<128>(sm.ys[n & 1], y + vbase + (size_t)n * kL * vstep, vstep, chunk_len(n), gtid, args.ext.y,
                   args.status);
  }
  if (role == 0 && args.s_final) store_state(c, args.s_final + (size_t)head * kN * kN, args.ext.s_final, args.status);
}

}  // namespace

template <typename TIn, bool kLogit, bool kEpi>
cudaError_t launch_fwd3_impl(const FwdArgs& args, cudaStream_t stream) {
  const size_t smem = sizeof(Fwd3Smem<TIn>);
  static_assert(sizeof(Fwd3Smem<TIn>) <= 227 * 1024, "shared memory over budget");
  cudaError_t e = cudaFuncSetAttribute(wkv7_fwd3_kernel<TIn, kLogit, kEpi>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  wkv7_fwd3_kernel<TIn, kLogit, kEpi><<<(unsigned)(args.B * args.H), kThreads, smem, stream>>>(args);
  return cudaGetLastError();
}

cudaError_t launch_fwd3(const FwdArgs& args, bool bf16, cudaStream_t stream) {
  using bf16_t = __nv_bfloat16;
  if (!bf16) {  // the decay as w, no epilogue (the API allows nothing else for fp32 inputs)
    if (args.w_logit || args.epilogue) return cudaErrorInvalidValue;
    return launch_fwd3_impl<float, false, false>(args, stream);
  }
  if (args.epilogue)
    return args.w_logit ? launch_fwd3_impl<bf16_t, true, true>(args, stream)
                        : launch_fwd3_impl<bf16_t, false, true>(args, stream);
  return args.w_logit ? launch_fwd3_impl<bf16_t, true, false>(args, stream)
                      : launch_fwd3_impl<bf16_t, false, false>(args, stream);
}

}  // namespace wkv7
