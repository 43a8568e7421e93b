// WKV7 backward-through-time on tensor cores (sm_103a), split into a carry
// chain and a parallel output pass: bf16 inputs, N = 64, checkpoints every
// 16 steps.
//
// Same result as "rx_pretrain.c", rx_wkv7_backward (the reverse scan of its
// equations (1)-(3)): per (b, h), with G = dL/dS carried from the last step
// back to the first,
//   dr = S_t^T dy ; G += dy r^T ; dk = G^T v ; db = G^T sa ;
//   dw = colsum(G o S_prev) ; dv = G k ; dsa = G b ; da = S_prev^T dsa ;
//   G <- G diag(w) + dsa a^T ;  dS_init = G after the first step.
// Chunk algebra (L = 16 steps, checkpoint S0 = state before the chunk, Gc =
// gradient w.r.t. the state after it, scaled operands A^, R^, K~, B~, Kb, Bb
// and T = (I - Mba)^-1 as in the forward kernel):
//   SA  = T (A^ S0^T + Mka V)                 rows sa(t) (recomputed)
//   DSA = T^T (Bb Gc^T + Mbr^T DY)            rows dsa(t)
//   DV  = Kb Gc^T + Mkr^T DY + Mka^T DSA
//   DK~ = (V Gc) diag(c(L)) + triu(V DY^T) R^ + triu(V DSA^T, 1) A^,  dk = DK~ / c
//   DB~ = (SA Gc) diag(c(L)) + triu(SA DY^T) R^ + triu(SA DSA^T, 1) A^, db = DB~ / c
//   DR^ = DY S0 + tril(DY V^T) K~ + tril(DY SA^T) B~,                  dr = DR^ c
//   DA^ = DSA S0 + tril(DSA V^T, -1) K~ + tril(DSA SA^T, -1) B~,       da = DA^ c(t-1)
//   carry: Gc' = Gc diag(c(L)) + DY^T R^ + DSA^T A^
//   w(t) dw(t) = colsum(Gc' o S0) - sum_{u<t} x(u) - a(t) da(t)        (first 8 steps)
//              = sum_{u>=t} x(u) - a(t) da(t) + colsum(Gc o S(L))      (last 8 steps)
// with x = r dr - k dk - b db + a da per step and column.
//
// Only the carry Gc is sequential over chunks, and it needs neither k, v
// nor the state: DSA^T = Gc (T^T Bb)^T + DY^T (Mbr T). So the backward runs
// as two kernels:
//  * wkv7_bwd4_carry_kernel - one CTA per (b, h), chunks in reverse, a
//    three-stage pipeline of warp groups: four "state" warps (16 rows of Gc
//    each, as accumulator tiles) advance the carry through chunk n with three
//    small products, four warps finish chunk n-1's T^T Bb and Mbr T, four
//    form chunk n-2's scaled R^, A^, B~, Bb and DY. It stores Gc for every
//    chunk (as bf16) and dS_init.
//  * wkv7_bwd4_out_kernel - one CTA per (b, h, chunk), all independent: from
//    the chunk's inputs, checkpoint and stored carry it forms every gradient
//    of the chunk. Three CTAs share an SM. The dw anchors come from the
//    chunk's own column products: with S(L) = S0 diag(c(L)) + V^T Kb + SA^T Bb,
//      colsum(Gc o S(L)) = c(L) colsum(Gc o S0) + sum_t (Kb o V Gc + Bb o SA Gc)
//      colsum(Gc' o S0)  = c(L) colsum(Gc o S0) + sum_t (R^ o DY S0 + A^ o DSA S0).
// Arithmetic: every product accumulates in fp32. The carry kernel's products
// take bf16 operands (mma.sync m16n8k16): one bf16 value per operand for bf16
// inputs, a pair hi + lo (three products per product) for fp32 inputs; it
// carries Gc in fp32 and stores it as bf16 (fp32 for fp32 inputs) for the
// output kernel. The output kernel's products take bf16 operands
// (mma.sync m16n8k16): the chunk's inputs, the stored bf16 carry, and the fp32
// checkpoint rounded once to bf16; its scaling, triangular solve and dw sums
// are fp32. A chunk whose decays leave [1/16, 16] (or hold a NaN) is run step
// by step in fp32 by both kernels.
#include "wkv7_decay.cuh"
#include "wkv7_launch.h"
#include "wkv7_mma.cuh"
#include "wkv7_mma16.cuh"
#include "wkv7_scaled.cuh"
#include "wkv7_tmem.cuh"

namespace wkv7 {
namespace {

constexpr int kN = 64, kL = 16;
constexpr int kLD64 = 72;  // row stride (floats) of 64-wide operands read along k
constexpr int kLD16 = 24;  // row stride of 16-wide operands
constexpr int kTile = kL * kN;
constexpr int kThreads = 256;
enum { V_R = 0, V_W = 1, V_K = 2, V_V = 3, V_A = 4, V_B = 5, V_DY = 6 };

__device__ __forceinline__ float bf(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ float bf(const float* p) { return *p; }
__device__ __forceinline__ float2 bf2(const __nv_bfloat16* p) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
}
__device__ __forceinline__ float2 bf2(const float* p) { return *reinterpret_cast<const float2*>(p); }

__device__ __forceinline__ float quad_sum(float x) {
  x += __shfl_xor_sync(0xffffffffu, x, 1);
  return x + __shfl_xor_sync(0xffffffffu, x, 2);
}
__device__ __forceinline__ float col_sum(float x) {  // over the 8 row groups g of the warp
  x += __shfl_xor_sync(0xffffffffu, x, 4);
  x += __shfl_xor_sync(0xffffffffu, x, 8);
  return x + __shfl_xor_sync(0xffffffffu, x, 16);
}

// ================================================================ carry ===

enum { C_R = 0, C_W = 1, C_A = 2, C_B = 3, C_DY = 4, C_NV = 5 };  // vectors staged for the carry (nv: epilogue)
constexpr int kCarryStages = 4;
constexpr int kCarryThreads = 384;  // warps 0-3: state; 4-7: forming (F); 8-11: products (P)

// Operands of one chunk for the carry update: bf16 tiles (rows of kB64 / kB16 elements,
// read by ldmatrix) in kP parts, one for bf16 inputs and hi + lo for fp32 inputs. The
// forming group writes the vectors and the two Gram blocks, the products group adds T a
// round later, the state warps read them all a round after that.
template <int kP>
struct alignas(16) OpC16 {
  bf16_t Rh[kP][kL * kB64];   // R^ [t][j]
  bf16_t DYs[kP][kL * kB64];  // DY [t][i]
  bf16_t Ah[kP][kL * kB64];   // A^ [t][j]
  bf16_t Bb[kP][kL * kB64];   // Bb [s][j]
  bf16_t Mbr[kP][kL * kB16];  // R^ B~^T (with diagonal) [t][s]
  bf16_t Tm[kP][kL * kB16];   // T = (I - Mba)^-1 [t][s]
  float cL[kN];               // c(L), fp32
  int unsafe;
  int pad_[3];
};
template <int kP>
struct alignas(16) ScratchC16 {
  bf16_t Bt[kP][kL * kB64];  // B~ [t][j]
  float Mba[kL * kLD16];     // A^ B~^T (strictly lower) [t][s], fp32: T is formed from it
};
static_assert(offsetof(ScratchC16<1>, Mba) % 16 == 0 && offsetof(ScratchC16<2>, Mba) % 16 == 0,
              "Mba rows are read 16 bytes at a time");
template <typename TIn>
constexpr int kCarryParts = sizeof(TIn) == 2 ? 1 : 2;

// Shared memory of the carry kernel for bf16 (TIn = bf16_t: six vectors per stage, the
// epilogue's nv the sixth; carries stored as bf16) or fp32 inputs (five vectors; carries
// stored as fp32).
template <typename TIn>
struct CarrySmemT {
  static constexpr int kVecs = sizeof(TIn) == 2 ? 6 : 5;
  static constexpr int kP = kCarryParts<TIn>;
  typedef TIn CarryT;
  TIn raw[kCarryStages][kVecs][kTile];  // r, w, a, b, dy (or dout), nv (epilogue) of one chunk per stage
  OpC16<kP> op[3];
  ScratchC16<kP> sc[2];
  float Pc[4][kN];       // products of the decays of four-step blocks
  TIn gst[2][kN * 72];   // carries on their way out (state warps write, products warps store)
  uint64_t full[kCarryStages];
  int abort_flag;
};
typedef CarrySmemT<bf16_t> CarrySmem;

// Sum over the 32 lanes (xor 16, 8, 4, 2, 1).
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// The time-mix epilogue's group-norm backward for one row (step) of one head, as the 32
// lanes of a warp hold it (lane l: channels 2 l, 2 l + 1): from the gradient of the
// epilogue's output d and the normalized output nv, the scan's upstream gradient
//     dn = d ln_w ;  dy = rstd (dn - mean(dn) - nv mean(dn nv)),
// rounded to bf16 (the scan's dy is bf16).
__device__ __forceinline__ __nv_bfloat162 gn_backward_row(float2 d, float2 nv, float2 lw, float rstd) {
  const float dn0 = d.x * lw.x, dn1 = d.y * lw.y;
  const float s1 = warp_sum(dn0 + dn1);
  const float s2 = warp_sum(fmaf(dn0, nv.x, dn1 * nv.y));
  const float m1 = s1 * (1.f / kN), m2 = s2 * (1.f / kN);
  return __floats2bfloat162_rn(rstd * (dn0 - m1 - nv.x * m2), rstd * (dn1 - m1 - nv.y * m2));
}

// Forming group (128 threads): the scaled operands of a chunk. Thread
// (lane, pf) forms columns 2 lane, 2 lane + 1 of steps 4 pf .. 4 pf + 3. The
// running products c(t) are taken per block of four steps and the blocks'
// products chained in step order. Returns (uniformly over the group) whether
// some decay leaves the range of the scaled form.
template <typename TIn, bool kLogit, bool kEpi>
__device__ bool form_carry(ScratchC16<kCarryParts<TIn>>& sc, float (&Pc)[4][kN], TIn* rs,
                           OpC16<kCarryParts<TIn>>& op, int len, int ftid, const float* epi_rstd, float2 epi_lw) {
  constexpr int kP = kCarryParts<TIn>, kLo = kP - 1;  // index of the lo part (the hi part for kP = 1)
  const int lane = ftid & 31, pf = ftid >> 5, j = 2 * lane, t0 = 4 * pf;
  float2 wv[4], av[4], rv[4], bv[4], dyv[4];
  if constexpr (kEpi) {  // epilogue: the stage holds dout and nv; dy replaces dout (the step-by-step path reads it)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int o = (t0 + e) * kN + j;
      *reinterpret_cast<__nv_bfloat162*>(rs + C_DY * kTile + o) =
          gn_backward_row(bf2(rs + C_DY * kTile + o), bf2(rs + C_NV * kTile + o), epi_lw, epi_rstd[e]);
    }
  }
  bool safe = true;
  float2 pb = make_float2(1.f, 1.f);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int o = (t0 + e) * kN + j;
    wv[e] = t0 + e < len ? decay_value2<kLogit>(bf2(rs + C_W * kTile + o)) : make_float2(1.f, 1.f);
    safe &= decay_is_safe(wv[e].x) && decay_is_safe(wv[e].y);
    pb = fmul2(pb, wv[e]);
  }
  *reinterpret_cast<float2*>(&Pc[pf][j]) = pb;
  // the other vectors are read before the group barrier, so their loads overlap it
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int o = (t0 + e) * kN + j;
    av[e] = bf2(rs + C_A * kTile + o);
    rv[e] = bf2(rs + C_R * kTile + o);
    bv[e] = bf2(rs + C_B * kTile + o);
    dyv[e] = bf2(rs + C_DY * kTile + o);
  }
  if (named_bar_or(1, 128, !safe)) return true;
  float2 cL = make_float2(1.f, 1.f), cpre = cL;  // cpre = c(t0 - 1)
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    cL = fmul2(cL, *reinterpret_cast<const float2*>(&Pc[q][j]));
    if (q < pf) cpre = cL;
  }
  if (pf == 0) *reinterpret_cast<float2*>(op.cL + j) = cL;
  float2 c = cpre;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int t = t0 + e;
    const float2 cprev = c;
    c = fmul2(c, wv[e]);
    const float2 ic = make_float2(rcp_approx(c.x), rcp_approx(c.y));
    const int q = t * kB64 + j;
    st_pair_p<kP>(op.Ah[0] + q, op.Ah[kLo] + q, fmul2(av[e], cprev));
    st_pair_p<kP>(op.Rh[0] + q, op.Rh[kLo] + q, fmul2(rv[e], c));
    st_pair_p<kP>(sc.Bt[0] + q, sc.Bt[kLo] + q, fmul2(bv[e], ic));
    st_pair_p<kP>(op.Bb[0] + q, op.Bb[kLo] + q, fmul2(bv[e], fmul2(cL, ic)));
    st_pair_p<kP>(op.DYs[0] + q, op.DYs[kLo] + q, dyv[e]);  // bf16 inputs: exact
  }
  return false;
}

// n-tile nt of P Q^T (16 x 8, K = 64, bf16 tiles of stride kB64 in kP parts: P and Q the
// hi parts, Pl and Ql the lo parts), masked to s < t (strict) or s <= t, stored as fp32
// (stride kLD16, to M) or in kP bf16 parts (stride kB16, to M and Ml).
__device__ __forceinline__ void ldsm2(uint32_t (&r)[2], const bf16_t* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r[0]), "=r"(r[1]) : "r"(smem_addr(p)));
}
template <int kP, typename TOut>
__device__ __forceinline__ void gram_tile16(TOut* M, TOut* Ml, const bf16_t* P, const bf16_t* Pl, const bf16_t* Q,
                                            const bf16_t* Ql, int nt, bool strict, int lane) {
  const int g = lane >> 2, t4 = lane & 3;
  float acc[4];
  zero4(acc);
  const int qo = (8 * nt + (lane & 7)) * kB64 + ((lane >> 3) & 1) * 8;
#pragma unroll
  for (int kb = 0; kb < kN / 16; ++kb) {
    uint32_t a[4], b[2];
    a_mk(a, P, kB64, 0, 16 * kb, lane);
    ldsm2(b, Q + qo + 16 * kb);
    if constexpr (kP == 2) {  // lo parts: a_lo b_hi + a_hi b_lo
      uint32_t al[4], bl[2];
      a_mk(al, Pl, kB64, 0, 16 * kb, lane);
      ldsm2(bl, Ql + qo + 16 * kb);
      mma16(acc, al, b[0], b[1]);
      mma16(acc, a, bl[0], bl[1]);
    }
    mma16(acc, a, b[0], b[1]);
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int t = g + 8 * h, s = 8 * nt + 2 * t4;
    const bool k0 = strict ? s < t : s <= t, k1 = strict ? s + 1 < t : s + 1 <= t;
    const float2 x = make_float2(k0 ? acc[2 * h] : 0.f, k1 ? acc[2 * h + 1] : 0.f);
    if constexpr (sizeof(TOut) == 4)
      *reinterpret_cast<float2*>(M + t * kLD16 + s) = x;
    else
      st_pair_p<kP>(M + t * kB16 + s, Ml + t * kB16 + s, x);
  }
}

// Where the carry's Gram blocks Mba and Mbr are made: in the products group with bf16 operands
// (the forming group has the longest round: about 1,390 cycles against 520-970 for the
// products warps), in the forming group with split-bf16 operands (three products each, which
// would make the products warp that forms T the longest).
template <int kP>
constexpr bool kGramsInProducts = kP == 1;

// Forming group: wait for a chunk's inputs and form its operands. A timeout
// raises the CTA's abort flag and returns false, after forming the operands
// all the same (from whatever the stage holds) so that the group's named
// barriers stay matched; every thread reads the flag after the round's barrier.
template <typename TIn, bool kLogit, bool kEpi>
__device__ bool front_form(CarrySmemT<TIn>& sm, ScratchC16<kCarryParts<TIn>>& sc, OpC16<kCarryParts<TIn>>& op,
                           TIn* rs, uint64_t* bar, uint32_t parity, int len, unsigned* status, const float* epi_rstd,
                           float2 epi_lw) {
  constexpr int kP = kCarryParts<TIn>, kLo = kP - 1;
  const int ftid = threadIdx.x - 128;
  const bool ok = mbar_wait_bounded(status, bar, parity);
  if (!ok) *reinterpret_cast<volatile int*>(&sm.abort_flag) = 1;
  const bool unsafe = form_carry<TIn, kLogit, kEpi>(sc, sm.Pc, rs, op, len, ftid, epi_rstd, epi_lw);
  if (ftid == 0) op.unsafe = unsafe;
  if (unsafe || kGramsInProducts<kP>) return ok;
  named_bar(1, 128);
  const int pf = ftid >> 5;
  // n-tile pf of Mba = A^ B~^T (warps 0, 1; fp32, strictly lower) or pf - 2 of Mbr = R^ B~^T
  // (warps 2, 3; kP bf16 parts, with the diagonal)
  if (pf < 2)
    gram_tile16<kP>(sc.Mba, sc.Mba, op.Ah[0], op.Ah[kLo], sc.Bt[0], sc.Bt[kLo], pf, true, ftid & 31);
  else
    gram_tile16<kP>(op.Mbr[0], op.Mbr[kLo], op.Rh[0], op.Rh[kLo], sc.Bt[0], sc.Bt[kLo], pf - 2, false, ftid & 31);
  return ok;
}

// Products group (128 threads), a round after the forming group: with bf16 operands the Gram
// blocks Mba = A^ B~^T (n-tile pp of warps 0, 1; fp32, strictly lower) and Mbr = R^ B~^T
// (n-tile pp - 2 of warps 2, 3, with the diagonal) first; then T = (I - Mba)^-1 by fp32 forward
// substitution on warp 0 (once warp 1's n-tile is in: named barrier 2), stored in kP bf16 parts.
template <int kP>
__device__ void front_products16(ScratchC16<kP>& sc, OpC16<kP>& op) {
  const int pp = (threadIdx.x >> 5) - 8, lane = threadIdx.x & 31;
  if constexpr (kGramsInProducts<kP>) {
    if (pp < 2)
      gram_tile16<kP>(sc.Mba, sc.Mba, op.Ah[0], op.Ah[0], sc.Bt[0], sc.Bt[0], pp, true, lane);
    else
      gram_tile16<kP>(op.Mbr[0], op.Mbr[0], op.Rh[0], op.Rh[0], sc.Bt[0], sc.Bt[0], pp - 2, false, lane);
    if (pp == 1) named_arrive(2, 64);
    if (pp != 0) return;
    named_bar(2, 64);
  } else {
    if (pp != 0) return;
  }
  const int s = lane & 15;
  float col[kL];
  unit_lower_inverse_col16<kLD16>(sc.Mba, s, col);
  if (lane < 16) {
#pragma unroll
    for (int tt = 0; tt < kL; ++tt) put_p<kP>(op.Tm[0] + tt * kB16 + s, op.Tm[kP - 1] + tt * kB16 + s, col[tt]);
  }
}

// One chunk of the carry (state warp, rows i0 .. i0+15 of G), T applied last:
//   DSA^T = (G Bb^T + DY^T Mbr) T;  G <- G diag(c(L)) + DY^T R^ + DSA^T A^
// Every operand enters in kP bf16 parts (G, X and DSA^T split from their fp32 accumulator
// tiles); G stays fp32 in its accumulator tiles.
template <int kP>
__device__ __forceinline__ void carry_chunk16(float (&G)[8][4], const OpC16<kP>& op, int i0, int t4, int lane) {
  constexpr int kLo = kP - 1;
  using Acc2 = float[2][4];
  FragP<kP> aD, b;
  a_km_p<kP>(aD, op.DYs[0], op.DYs[kLo], kB64, i0, 0, lane);  // DY^T rows i0.., k = s (DY stored [s][i])
  float X[2][4];
  zero4(X[0]);
  zero4(X[1]);
  b_kn_p<kP>(b, op.Mbr[0], op.Mbr[kLo], kB16, 0, 0, lane);  // Mbr [u][s]
  mma_pp<kP, kP>(X, aD, b);
#pragma unroll
  for (int kb = 0; kb < 4; ++kb) {
    FragP<kP> aG;
    c2a_p<kP>(aG, G[2 * kb], G[2 * kb + 1]);
    b_nk_p<kP>(b, op.Bb[0], op.Bb[kLo], kB64, 0, 16 * kb, lane);  // Bb^T: Bb stored [s][j]
    mma_pp<kP, kP>(X, aG, b);
  }
  float DS[2][4];
  zero4(DS[0]);
  zero4(DS[1]);
  {
    FragP<kP> aX;
    c2a_p<kP>(aX, X[0], X[1]);
    b_kn_p<kP>(b, op.Tm[0], op.Tm[kLo], kB16, 0, 0, lane);  // T [s][t]
    mma_pp<kP, kP>(DS, aX, b);
  }
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) {
    const float2 cl = *reinterpret_cast<const float2*>(op.cL + 8 * nt + 2 * t4);
    G[nt][0] *= cl.x;
    G[nt][1] *= cl.y;
    G[nt][2] *= cl.x;
    G[nt][3] *= cl.y;
  }
#pragma unroll
  for (int np = 0; np < 4; ++np) {  // + DY^T R^ (R^ stored [t][j])
    b_kn_p<kP>(b, op.Rh[0], op.Rh[kLo], kB64, 16 * np, 0, lane);
    mma_pp<kP, kP>(reinterpret_cast<Acc2&>(G[2 * np]), aD, b);
  }
  FragP<kP> aS;
  c2a_p<kP>(aS, DS[0], DS[1]);
#pragma unroll
  for (int np = 0; np < 4; ++np) {  // + DSA^T A^
    b_kn_p<kP>(b, op.Ah[0], op.Ah[kLo], kB64, 16 * np, 0, lane);
    mma_pp<kP, kP>(reinterpret_cast<Acc2&>(G[2 * np]), aS, b);
  }
}

// The same chunk step by step in fp32 (a chunk outside the scaled form's
// range): G += dy r^T ; dsa = G b ; G <- G diag(w) + dsa a^T.
template <typename TIn, bool kLogit>
__device__ void carry_direct(float (&G)[8][4], const TIn* rs, int len, int i0, int g, int t4) {
  for (int t = len - 1; t >= 0; --t) {
    const TIn* row = rs + t * kN;
    const float dy0 = bf(row + C_DY * kTile + i0 + g), dy1 = bf(row + C_DY * kTile + i0 + g + 8);
    float ds0 = 0.f, ds1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const int col = 8 * nt + 2 * t4;
      const float2 r = bf2(row + C_R * kTile + col), b = bf2(row + C_B * kTile + col);
      G[nt][0] = fmaf(dy0, r.x, G[nt][0]);
      G[nt][1] = fmaf(dy0, r.y, G[nt][1]);
      G[nt][2] = fmaf(dy1, r.x, G[nt][2]);
      G[nt][3] = fmaf(dy1, r.y, G[nt][3]);
      ds0 = fmaf(G[nt][0], b.x, fmaf(G[nt][1], b.y, ds0));
      ds1 = fmaf(G[nt][2], b.x, fmaf(G[nt][3], b.y, ds1));
    }
    ds0 = quad_sum(ds0);
    ds1 = quad_sum(ds1);
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const int col = 8 * nt + 2 * t4;
      const float2 w = decay_value2<kLogit>(bf2(row + C_W * kTile + col)), a = bf2(row + C_A * kTile + col);
      G[nt][0] = fmaf(ds0, a.x, G[nt][0] * w.x);
      G[nt][1] = fmaf(ds0, a.y, G[nt][1] * w.y);
      G[nt][2] = fmaf(ds1, a.x, G[nt][2] * w.x);
      G[nt][3] = fmaf(ds1, a.y, G[nt][3] * w.y);
    }
  }
}

// A staged 64 x 64 carry (rows of 72) to global memory, kT threads, whole rows per
// instruction: fp32 (64 rows of 16 pieces of 16 bytes) or bf16 (64 rows of 8 pieces).
template <int kT>
__device__ __forceinline__ void flush_carry(const float* src, float* dst, int ptid, const Extent& x, unsigned* status) {
#pragma unroll
  for (int q = 0; q < (kN * 16 + kT - 1) / kT; ++q) {
    const int idx = ptid + kT * q;  // row idx / 16, columns 4 (idx % 16) ..
    if (kT * (q + 1) > kN * 16 && idx >= kN * 16) break;
    uint4* p = reinterpret_cast<uint4*>(dst + 4 * idx);
    if (in_extent(status, x, p)) *p = *reinterpret_cast<const uint4*>(src + (idx >> 4) * 72 + 4 * (idx & 15));
  }
}

template <int kT>
__device__ __forceinline__ void flush_carry(const bf16_t* src, bf16_t* dst, int ptid, const Extent& x,
                                            unsigned* status) {
#pragma unroll
  for (int q = 0; q < (kN * 8 + kT - 1) / kT; ++q) {
    const int idx = ptid + kT * q;  // row idx / 8, columns 8 (idx % 8) ..
    if (kT * (q + 1) > kN * 8 && idx >= kN * 8) break;
    uint4* p = reinterpret_cast<uint4*>(dst + 8 * idx);
    if (in_extent(status, x, p)) *p = *reinterpret_cast<const uint4*>(src + (idx >> 3) * 72 + 8 * (idx & 7));
  }
}

template <typename TIn, bool kLogit, bool kEpi>
__global__ void __launch_bounds__(kCarryThreads, 1) wkv7_bwd4_carry_kernel(const __grid_constant__ BwdArgs args) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  using Smem = CarrySmemT<TIn>;
  constexpr bool kX3 = sizeof(TIn) == 4;
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
  const int T = args.T, H = args.H;
  const int head = blockIdx.x, bi = head / H, hi = head % H;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t4 = lane & 3;
  const int role = warp < 4 ? 0 : warp < 8 ? 1 : 2;  // state, forming, products
  const int i0 = 16 * warp;                          // state warps: rows of the carry
  const int nchunks = (T + kL - 1) / kL;
  const int nvec = kEpi ? 6 : 5;
  const uint32_t stage_bytes = (uint32_t)(nvec * kTile * sizeof(TIn));
  TIn* carry_head = reinterpret_cast<TIn*>(args.carry) + (size_t)head * nchunks * kN * kN;

  // Chunks are visited in reverse: visit v is chunk nchunks-1-v. In visit m the state warps
  // advance the carry through chunk m, the products group finishes chunk m+1 and the
  // forming group forms chunk m+2 (visit numbers); inputs arrive by TMA four visits ahead.
  auto chunk_of = [&](int v) { return nchunks - 1 - v; };
  auto len_of = [&](int v) { return min(kL, T - chunk_of(v) * kL); };
  auto issue = [&](int v) {
    const int st = v % kCarryStages;
    const int vmap[5] = {V_R, V_W, V_A, V_B, V_DY};
    mbar_arrive_expect_tx(&sm.full[st], stage_bytes);
    for (int q = 0; q < 5; ++q)
      tma_load_4d(sm.raw[st][q], &args.map[vmap[q]], &sm.full[st], 0, hi, chunk_of(v) * kL, bi);
    if constexpr (kEpi) tma_load_4d(sm.raw[st][C_NV], &args.map_nv, &sm.full[st], 0, hi, chunk_of(v) * kL, bi);
  };
  // Epilogue: the forming threads' rstd (rows 4 pf .. 4 pf + 3 of the chunk they form next),
  // requested a visit ahead, and ln_w of their two channels.
  float rs_next[4] = {0.f, 0.f, 0.f, 0.f}, rs_cur[4];
  float2 epi_lw = make_float2(0.f, 0.f);
  auto load_rstd = [&](int v) {
    const int t0 = chunk_of(v) * kL + 4 * ((tid - 128) >> 5);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float* p = args.epi_stats + 2 * (((size_t)bi * T + t0 + e) * H + hi);
      rs_next[e] = t0 + e < T && in_extent(args.status, args.ext.stats, p) ? *p : 0.f;
    }
  };
  if (kEpi && role == 1) {
    const float2* p = reinterpret_cast<const float2*>(args.epi_ln_w + (size_t)hi * kN + 2 * (lane));
    if (in_extent(args.status, args.ext.ln_w, p)) epi_lw = *p;
    load_rstd(0);
  }
  int waited = 0, issued = 0;
  auto form = [&](int v) {  // forming group; false on a timeout
    const int c = chunk_of(v);
    const float* rst = nullptr;
    if constexpr (kEpi) {
#pragma unroll
      for (int e = 0; e < 4; ++e) rs_cur[e] = rs_next[e];
      if (v + 1 < nchunks) load_rstd(v + 1);
      rst = rs_cur;
    }
    if (!front_form<TIn, kLogit, kEpi>(sm, sm.sc[c & 1], sm.op[c % 3], sm.raw[v % kCarryStages][0],
                                       &sm.full[v % kCarryStages], (v / kCarryStages) & 1, len_of(v), args.status, rst,
                                       epi_lw))
      return false;
    waited = v + 1;
    return true;
  };
  auto products = [&](int v) {  // products group
    const int c = chunk_of(v);
    if (!sm.op[c % 3].unsafe) front_products16<Smem::kP>(sm.sc[c & 1], sm.op[c % 3]);
  };
  // TMA copies are issued by a products-group thread (that group has the most slack); the
  // forming group waits for them
  constexpr int kIssuer = 352;
  if (tid == kIssuer) {
    for (int s = 0; s < kCarryStages; ++s) mbar_init(&sm.full[s], 1);
    fence_mbar_init();
    for (int q = 0; q < 7; ++q) prefetch_tensormap(&args.map[q]);
    if (kEpi) prefetch_tensormap(&args.map_nv);
    for (int v = 0; v < kCarryStages && v < nchunks; ++v) issue(v);
  }
  issued = min(kCarryStages, nchunks);
  if (tid == 0) sm.abort_flag = 0;
  // the carry after the last chunk: the gradient entering through the final state (or zero)
  float G[8][4];
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) zero4(G[nt]);
  if (args.dS_final && warp < 4) {
    const float* src = args.dS_final + (size_t)head * kN * kN;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const int col = 8 * nt + 2 * t4;
      const float2* p0 = reinterpret_cast<const float2*>(src + (i0 + g) * kN + col);
      const float2* p1 = reinterpret_cast<const float2*>(src + (i0 + g + 8) * kN + col);
      const float2 lo = in_extent(args.status, args.ext.dS_final, p0) ? *p0 : make_float2(0.f, 0.f);
      const float2 hi = in_extent(args.status, args.ext.dS_final, p1) ? *p1 : make_float2(0.f, 0.f);
      G[nt][0] = lo.x;
      G[nt][1] = lo.y;
      G[nt][2] = hi.x;
      G[nt][3] = hi.y;
    }
  }
  __syncthreads();

  bool aborted = false;
  // pipeline fill: form visits 0 and 1, products of visit 0
  if (role == 1 && !form(0)) aborted = true;
  if (__syncthreads_or(sm.abort_flag)) aborted = true;
  if (!aborted) {
    if (role == 1 && nchunks > 1) form(1);
    if (role == 2) products(0);
    if (__syncthreads_or(sm.abort_flag)) aborted = true;
  }

  for (int m = 0; m < nchunks && !aborted; ++m) {
    const int n = chunk_of(m), st = m % kCarryStages;
    if (role == 0) {
      const auto& op = sm.op[n % 3];
      // the carry entering this chunk (gradient w.r.t. the state after it), as the output
      // pass multiplies with it (bf16, or fp32 for fp32 inputs); the products group stores it
      // next round
      TIn* dst = sm.gst[m & 1];
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const int col = 8 * nt + 2 * t4;
        if constexpr (kX3) {
          *reinterpret_cast<float2*>(dst + (i0 + g) * 72 + col) = make_float2(G[nt][0], G[nt][1]);
          *reinterpret_cast<float2*>(dst + (i0 + g + 8) * 72 + col) = make_float2(G[nt][2], G[nt][3]);
        } else {
          *reinterpret_cast<uint32_t*>(dst + (i0 + g) * 72 + col) = pack_bf16(G[nt][0], G[nt][1]);
          *reinterpret_cast<uint32_t*>(dst + (i0 + g + 8) * 72 + col) = pack_bf16(G[nt][2], G[nt][3]);
        }
      }
      if (op.unsafe)
        carry_direct<TIn, kLogit>(G, sm.raw[st][0], len_of(m), i0, g, t4);
      else
        carry_chunk16<Smem::kP>(G, op, i0, t4, lane);
    } else if (role == 1) {
      if (m + 2 < nchunks) form(m + 2);
    } else {
      if (m + 1 < nchunks) products(m + 1);
      // the carry the state warps staged last round, stored by the products warps other than
      // the one forming T
      if (m > 0 && tid >= 288)
        flush_carry<96>(sm.gst[(m - 1) & 1], carry_head + (size_t)chunk_of(m - 1) * kN * kN, tid - 288,
                        args.ext.carry, args.status);
    }
    // the stage of visit m is free (formed two visits ago, direct steps done); refill it
    __syncthreads();
    if (*reinterpret_cast<volatile int*>(&sm.abort_flag)) {
      aborted = true;
      break;
    }
    if (tid == kIssuer && m + kCarryStages < nchunks) {
      fence_proxy_async_smem();
      issue(m + kCarryStages);
    }
    issued = min(m + 1 + kCarryStages, nchunks);
  }
  if (aborted) {
    if (tid == 128)
      for (int v = waited; v < issued; ++v)
        mbar_wait_bounded(nullptr, &sm.full[v % kCarryStages], (v / kCarryStages) & 1, 200000000ull);
    __syncthreads();
    return;
  }
  if (role == 2) flush_carry<128>(sm.gst[(nchunks - 1) & 1], carry_head, tid - 256, args.ext.carry, args.status);  // chunk 0's
  if (role == 0 && args.dS_init) {
    float* dst = args.dS_init + (size_t)head * kN * kN;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const int col = 8 * nt + 2 * t4;
      float2* p0 = reinterpret_cast<float2*>(dst + (i0 + g) * kN + col);
      float2* p1 = reinterpret_cast<float2*>(dst + (i0 + g + 8) * kN + col);
      if (in_extent(args.status, args.ext.dS_init, p0)) *p0 = make_float2(G[nt][0], G[nt][1]);
      if (in_extent(args.status, args.ext.dS_init, p1)) *p1 = make_float2(G[nt][2], G[nt][3]);
    }
  }
}

// =============================================================== output ===
//
// The output kernel multiplies bf16 operands (mma.sync m16n8k16, fp32
// accumulation): the inputs are bf16 already, the scaled operands, the
// checkpoint and the carry are rounded to bf16 once, every sum is fp32.
// Operands live once, row-major, in shared memory; ldmatrix (.trans where
// the product reads a matrix down its columns) forms the fragments, so no
// transposed copies are kept. Row strides of 72 (64-wide) and 24 (16-wide)
// bf16 elements put the eight 16-byte rows of an 8 x 8 matrix on distinct
// banks.

struct OutSmem {
  bf16_t raw[7][kL * kB64];  // r, w, k, v, a, b, dy of the chunk [t][j] (V, DY: [t][i])
  union {
    struct {
      bf16_t S0[kN * kB64];  // checkpoint [i][j]
      bf16_t Gc[kN * kB64];  // carry after the chunk [i][j]
    } st;
    float xch[3][kL * kLD64];  // the dw exchange, once the column products are done
    float red[8 * 5 * kN];     // column sums of a direct chunk
  } u;
  bf16_t Ah[kL * kB64], Rh[kL * kB64], Kt[kL * kB64], Bt[kL * kB64];  // [t][j]
  bf16_t Kb[kL * kB64], Bb[kL * kB64];
  bf16_t SA[kL * kB64], DSA[kL * kB64];  // sa(t), dsa(t) [t][i]
  // Mka, Mkr, Mbr [t][s]; T = (I - Mba)^-1 [t][s]; U0 = triu(V DY^T), U1 = triu(V DSA^T, 1),
  // U2 = triu(SA DY^T), U3 = triu(SA DSA^T, 1) [t][s]
  bf16_t M[3][kL * kB16], Tm[kL * kB16], U[4][kL * kB16];
  float Mba[kL * kLD16];  // fp32, for the substitution
  float cS[kL * kLD64];   // c(t) [t][j], fp32
  float Epart[4][kN];     // colsum(Gc o S0) over the rows of each row block
  float Ppart[8][kN];     // products of the decays of steps 2 q, 2 q + 1
  float cLs[kN];          // c(L) = product of the chunk's decays
  float anc[2][kN];  // the chunk's parts of colsum(carry o state) at its start and end, without c(L) colsum(Gc o S0)
};
static_assert(offsetof(OutSmem, Mba) % 16 == 0, "Mba rows are read 16 bytes at a time");

// Extra shared memory of the output pass with the epilogue's backward fused (after OutSmem).
struct OutEpiSmem {
  bf16_t dout[kL * kB64];  // the gradient of the epilogue's output [t][i]
  bf16_t nv[kL * kB64];    // the normalized y [t][i]
  float stat[kL][2];       // (rstd, bonus) per step
  float dbon[kL];          // gradient of each step's bonus: sum_i dout_i v_i
  float lnw[kN], rk[kN];
};

// The epilogue's bonus terms for the chunk's stored dr, dk, dv (a chunk run step by step:
// added to what out_direct wrote): dr += dbon k r_k, dk += dbon r r_k, dv += dout bonus.
__device__ void epi_bonus_direct(const OutEpiSmem& ep, const bf16_t* rs, int len, const BwdArgs& args, size_t base,
                                 size_t vstep) {
  constexpr int RS = kL * kB64;
  for (int idx = threadIdx.x; idx < len * kN; idx += kThreads) {
    const int t = idx / kN, c = idx % kN;
    const size_t off = base + (size_t)t * vstep + c;
    const float db = ep.dbon[t];
    if (in_extent(args.status, args.ext.dr, args.dr + off)) args.dr[off] += db * bf(rs + V_K * RS + t * kB64 + c) * ep.rk[c];
    if (in_extent(args.status, args.ext.dk, args.dk + off)) args.dk[off] += db * bf(rs + V_R * RS + t * kB64 + c) * ep.rk[c];
    if (in_extent(args.status, args.ext.dv, args.dv + off)) args.dv[off] += bf(ep.dout + t * kB64 + c) * ep.stat[t][1];
  }
}

// This chunk's terms of the epilogue's parameter gradients, from every thread's partial
// sums over its steps (columns 2 lane, 2 lane + 1): sum_t dout nv, sum_t dout,
// sum_t dbon r k, summed over the warps in order into epi_part.
__device__ void epi_params_chunk(float* scratch, const float (&pp)[3][2], const BwdArgs& args, int head, int n,
                                 int nchunks) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int q = 0; q < 3; ++q)
    *reinterpret_cast<float2*>(scratch + (warp * 3 + q) * kN + 2 * lane) = make_float2(pp[q][0], pp[q][1]);
  __syncthreads();
  for (int i = threadIdx.x; i < 3 * kN; i += kThreads) {
    float x = 0.f;
#pragma unroll
    for (int w8 = 0; w8 < 8; ++w8) x += scratch[w8 * 3 * kN + i];
    float* p = args.epi_part + ((size_t)head * nchunks + n) * 3 * kN + i;
    if (in_extent(args.status, args.ext.part, p)) *p = x;
  }
}

// Step-by-step reverse scan of one chunk (all eight warps, fp32; warp w owns
// rows 8 w .. 8 w + 7 of the state and the carry, lane (g, t) row 8 w + g and
// columns 8 nt + 2 t, + 1): the carry starts at the stored Gc, S_prev of step
// t is recomputed from the checkpoint (fp32, read from global memory).
// `rs` holds the chunk's r, w, k, v, a, b, dy rows ([t][j], row stride kB64,
// kL * kB64 elements apart); `red` is 8 * 5 * kN floats of scratch.
template <bool kLogit>
__device__ void out_direct(const bf16_t* rs, float* red, const float* S0, const bf16_t* Gcg, int len,
                           const BwdArgs& args, size_t base, size_t vstep, int warp, int lane) {
  const int g = lane >> 2, t4 = lane & 3, i = 8 * warp + g, tid = threadIdx.x;  // red: [8 warps][5][64]
  constexpr int RS = kL * kB64;
  float G[8][2];
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) {
    const uint32_t* p = reinterpret_cast<const uint32_t*>(Gcg + i * kN + 8 * nt + 2 * t4);
    const float2 x = unpack_bf16(in_extent(args.status, args.ext.carry, p) ? *p : 0u);
    G[nt][0] = x.x;
    G[nt][1] = x.y;
  }
  for (int t = len - 1; t >= 0; --t) {
    float sp[8][2];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const float2* p = reinterpret_cast<const float2*>(S0 + i * kN + 8 * nt + 2 * t4);
      const float2 x = in_extent(args.status, args.ext.ckpt, p) ? *p : make_float2(0.f, 0.f);
      sp[nt][0] = x.x;
      sp[nt][1] = x.y;
    }
    float sa = 0.f;
    for (int u = 0; u <= t; ++u) {
      const bf16_t* row = rs + u * kB64;
      float s = 0.f;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const float2 a = bf2(row + V_A * RS + 8 * nt + 2 * t4);
        s = fmaf(sp[nt][0], a.x, fmaf(sp[nt][1], a.y, s));
      }
      sa = quad_sum(s);
      if (u == t) break;  // sp = S_prev(t), sa = sa(t)
      const float v = bf(row + V_V * RS + i);
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const int col = 8 * nt + 2 * t4;
        const float2 w = decay_value2<kLogit>(bf2(row + V_W * RS + col)), k = bf2(row + V_K * RS + col),
                     b = bf2(row + V_B * RS + col);
        sp[nt][0] = fmaf(sa, b.x, fmaf(sp[nt][0], w.x, v * k.x));
        sp[nt][1] = fmaf(sa, b.y, fmaf(sp[nt][1], w.y, v * k.y));
      }
    }
    const bf16_t* row = rs + t * kB64;
    const float v = bf(row + V_V * RS + i), dy = bf(row + V_DY * RS + i);
    // column sums (over this warp's rows) of dr (from S_t), then G += dy r^T, dk, db, dw; row sums dv, dsa
    float dv = 0.f, ds = 0.f;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const int col = 8 * nt + 2 * t4;
      const float2 w = decay_value2<kLogit>(bf2(row + V_W * RS + col)), k = bf2(row + V_K * RS + col);
      const float2 b = bf2(row + V_B * RS + col), r = bf2(row + V_R * RS + col);
      const float wv[2] = {w.x, w.y}, kv[2] = {k.x, k.y}, bv[2] = {b.x, b.y}, rv[2] = {r.x, r.y};
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float st = fmaf(sa, bv[e], fmaf(sp[nt][e], wv[e], v * kv[e]));
        G[nt][e] = fmaf(dy, rv[e], G[nt][e]);
        const float sums[4] = {col_sum(st * dy), col_sum(G[nt][e] * v), col_sum(G[nt][e] * sa),
                               col_sum(G[nt][e] * sp[nt][e])};
        if (g == 0) {
#pragma unroll
          for (int q = 0; q < 4; ++q) red[(warp * 5 + q) * kN + col + e] = sums[q];
        }
        dv = fmaf(G[nt][e], kv[e], dv);
        ds = fmaf(G[nt][e], bv[e], ds);
      }
    }
    dv = quad_sum(dv);
    ds = quad_sum(ds);
    if (t4 == 0 && in_extent(args.status, args.ext.dv, args.dv + base + (size_t)t * vstep + i))
      args.dv[base + (size_t)t * vstep + i] = dv;
    // da = S_prev^T dsa; carry G <- G diag(w) + dsa a^T
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const int col = 8 * nt + 2 * t4;
      const float2 w = decay_value2<kLogit>(bf2(row + V_W * RS + col)), a = bf2(row + V_A * RS + col);
      const float wv[2] = {w.x, w.y}, av[2] = {a.x, a.y};
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float pa = col_sum(sp[nt][e] * ds);
        G[nt][e] = fmaf(ds, av[e], G[nt][e] * wv[e]);
        if (g == 0) red[(warp * 5 + 4) * kN + col + e] = pa;
      }
    }
    __syncthreads();
    for (int idx = tid; idx < 5 * kN; idx += kThreads) {
      const int q = idx / kN, col = idx % kN;
      float x = 0.f;
#pragma unroll
      for (int w8 = 0; w8 < 8; ++w8) x += red[(w8 * 5 + q) * kN + col];
      float* dst = q == 0 ? args.dr : q == 1 ? args.dk : q == 2 ? args.db : q == 3 ? args.dw : args.da;
      const Extent& xe = q == 0 ? args.ext.dr : q == 1 ? args.ext.dk : q == 2 ? args.ext.db : q == 3 ? args.ext.dw
                                                                                                  : args.ext.da;
      if constexpr (kLogit) {
        if (q == 3) {  // dL/dz from dL/dw
          const float z = bf(rs + V_W * RS + t * kB64 + col);
          x = logit_grad_from_wdw(x * decay_value<true>(z), z);
        }
      }
      if (in_extent(args.status, xe, dst + base + (size_t)t * vstep + col)) dst[base + (size_t)t * vstep + col] = x;
    }
    __syncthreads();
  }
}

// T = (I - M)^-1 for a strictly lower 16 x 16 fp32 M (stride kLD16) by
// forward substitution, one warp; lane s < 16 owns column s. Writes T
// row-major as bf16.
__device__ __forceinline__ void unit_lower_inverse16(const float* M, bf16_t* Tout, int lane) {
  const int s = lane & 15;
  float col[kL];
  unit_lower_inverse_col16<kLD16>(M, s, col);
  if (lane < 16) {
#pragma unroll
    for (int t = 0; t < kL; ++t) Tout[t * kB16 + s] = __float2bfloat16_rn(col[t]);
  }
}

template <bool kLogit, bool kEpi>
__global__ void __launch_bounds__(kThreads, 3) wkv7_bwd4_out_kernel(const __grid_constant__ BwdArgs args) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  OutSmem& sm = *reinterpret_cast<OutSmem*>(smem_raw);
  OutEpiSmem& ep = *reinterpret_cast<OutEpiSmem*>(smem_raw + sizeof(OutSmem));  // epilogue only
  constexpr bool epi = kEpi;
  const int T = args.T, H = args.H, nchunks = (T + kL - 1) / kL;
  const int head = blockIdx.x / nchunks, n = blockIdx.x % nchunks, bi = head / H, hi = head % H;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t4 = lane & 3;
  const int t0 = n * kL, len = min(kL, T - t0);
  const size_t vstep = (size_t)H * kN, base = ((size_t)bi * T + t0) * vstep + (size_t)hi * kN;
  const float* S0g = args.ckpt + ((size_t)head * args.nck + n) * kN * kN;
  const bf16_t* Gcg = reinterpret_cast<const bf16_t*>(args.carry) + ((size_t)head * nchunks + n) * kN * kN;
  constexpr int RS = kL * kB64;  // elements between staged vectors

  // ---- loads: the chunk's rows (zeros past T) and the carry by cp.async, the checkpoint through registers.
  //      Epilogue: dout (in the place of dy) and nv to their own tiles, dy is formed below.
  for (int idx = tid; idx < (epi ? 8 : 7) * kL * 8; idx += kThreads) {
    const int v = idx / (kL * 8), t = (idx >> 3) % kL, c = idx & 7;
    const bf16_t* src = static_cast<const bf16_t*>(v == 7 ? args.epi_nv : args.in[v]) + base +
                        (size_t)min(t, len - 1) * vstep + 8 * c;
    bf16_t* dst = !epi || v < V_DY ? sm.raw[v] : v == V_DY ? ep.dout : ep.nv;
    cp_async16_zfill(dst + t * kB64 + 8 * c, src,
                     t < len && in_extent(args.status, args.ext.in[v], reinterpret_cast<const uint4*>(src)));
  }
  if (epi) {
    if (tid < kL) {
      const float2* p = reinterpret_cast<const float2*>(args.epi_stats + 2 * (((size_t)bi * T + t0 + tid) * H + hi));
      const float2 st = tid < len && in_extent(args.status, args.ext.stats, p) ? *p : make_float2(0.f, 0.f);
      ep.stat[tid][0] = st.x;
      ep.stat[tid][1] = st.y;
    } else if (tid >= 64 && tid < 64 + kN) {
      const float* pl = args.epi_ln_w + (size_t)hi * kN + tid - 64;
      const float* pr = args.epi_r_k + (size_t)hi * kN + tid - 64;
      ep.lnw[tid - 64] = in_extent(args.status, args.ext.ln_w, pl) ? *pl : 0.f;
      ep.rk[tid - 64] = in_extent(args.status, args.ext.r_k, pr) ? *pr : 0.f;
    }
  }
#pragma unroll
  for (int q = 0; q < kN * 8 / kThreads; ++q) {
    const int idx = tid + kThreads * q;  // row idx / 8, columns 8 (idx % 8) ..
    if (in_extent(args.status, args.ext.carry, reinterpret_cast<const uint4*>(Gcg + 8 * idx)))
      cp_async16(sm.u.st.Gc + (idx >> 3) * kB64 + 8 * (idx & 7), Gcg + 8 * idx);
  }
  cp_async_commit();
  float4 s0v[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float4* p = reinterpret_cast<const float4*>(S0g + 4 * (tid + kThreads * q));
    s0v[q] = in_extent(args.status, args.ext.ckpt, p) ? *p : make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int idx = tid + kThreads * q;  // row idx / 16, columns 4 (idx % 16) ..
    *reinterpret_cast<uint2*>(sm.u.st.S0 + (idx >> 4) * kB64 + 4 * (idx & 15)) =
        make_uint2(pack_bf16(s0v[q].x, s0v[q].y), pack_bf16(s0v[q].z, s0v[q].w));
  }
  cp_async_wait_all();
  __syncthreads();
  const bf16_t* rs = sm.raw[0];
  // Epilogue: the scan's dy (rows of the step pairs 2 warp, 2 warp + 1, lane's channels
  // 2 lane, 2 lane + 1), each step's dbon, and this thread's parameter terms.
  float pp[3][2] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
  if (epi) {
    const int j = 2 * lane;
    const float2 lw = make_float2(ep.lnw[j], ep.lnw[j + 1]);
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int t = 2 * warp + e, q = t * kB64 + j;
      const float2 d = bf2(ep.dout + q), nv = bf2(ep.nv + q), v = bf2(rs + V_V * RS + q);
      *reinterpret_cast<__nv_bfloat162*>(sm.raw[V_DY] + q) = gn_backward_row(d, nv, lw, ep.stat[t][0]);
      const float dbon = warp_sum(fmaf(d.x, v.x, d.y * v.y));
      if (lane == 0) ep.dbon[t] = dbon;
      const float2 r = bf2(rs + V_R * RS + q), k = bf2(rs + V_K * RS + q);
      pp[0][0] = fmaf(d.x, nv.x, pp[0][0]);
      pp[0][1] = fmaf(d.y, nv.y, pp[0][1]);
      pp[1][0] += d.x;
      pp[1][1] += d.y;
      pp[2][0] = fmaf(dbon, r.x * k.x, pp[2][0]);
      pp[2][1] = fmaf(dbon, r.y * k.y, pp[2][1]);
    }
  }

  // ---- A: scaled operands; thread (lane, warp) forms columns 2 lane, 2 lane + 1 of steps
  //      2 warp, 2 warp + 1. The running products c(t) are taken per pair of steps and the
  //      pairs' products chained in step order.
  {
    const int j = 2 * lane, ta = 2 * warp;
    float2 wv[2];
#pragma unroll
    for (int e = 0; e < 2; ++e)
      wv[e] = ta + e < len ? decay_value2<kLogit>(bf2(rs + V_W * RS + (ta + e) * kB64 + j)) : make_float2(1.f, 1.f);
    const bool safe = decay_is_safe(wv[0].x) && decay_is_safe(wv[0].y) && decay_is_safe(wv[1].x) &&
                      decay_is_safe(wv[1].y);
    *reinterpret_cast<float2*>(&sm.Ppart[warp][j]) = fmul2(wv[0], wv[1]);
    if (__syncthreads_or(!safe)) {
      out_direct<kLogit>(sm.raw[0], sm.u.red, S0g, Gcg, len, args, base, vstep, warp, lane);
      if (epi) {
        epi_bonus_direct(ep, rs, len, args, base, vstep);
        epi_params_chunk(sm.u.red, pp, args, head, n, nchunks);
      }
      return;
    }
    float2 cL = make_float2(1.f, 1.f), cpre = cL;  // cpre = c(ta - 1)
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      cL = fmul2(cL, *reinterpret_cast<const float2*>(&sm.Ppart[q][j]));
      if (q < warp) cpre = cL;
    }
    if (warp == 0) *reinterpret_cast<float2*>(&sm.cLs[j]) = cL;
    float2 c = cpre;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int t = ta + e, q = t * kB64 + j;
      const float2 w = wv[e];
      const float2 a = bf2(rs + V_A * RS + q), r = bf2(rs + V_R * RS + q);
      const float2 k = bf2(rs + V_K * RS + q), b = bf2(rs + V_B * RS + q);
      const float2 cprev = c;
      c = fmul2(c, w);
      const float2 ic = make_float2(rcp_approx(c.x), rcp_approx(c.y)), s = fmul2(cL, ic);
      st_pair(sm.Ah + q, fmul2(a, cprev));
      st_pair(sm.Rh + q, fmul2(r, c));
      st_pair(sm.Kt + q, fmul2(k, ic));
      st_pair(sm.Bt + q, fmul2(b, ic));
      st_pair(sm.Kb + q, fmul2(k, s));
      st_pair(sm.Bb + q, fmul2(b, s));
      *reinterpret_cast<float2*>(sm.cS + t * kLD64 + j) = c;
    }
  }
  __syncthreads();

  // ---- B: L x L products and T (warps 0-3), the K = 64 parts of sa, dsa, dv (rows i of block rb)
  const int rb = warp & 3, r0 = 16 * rb;
  float X1[2][4], X2[2][4];  // warps 0-3: RDSA^T, DV^T; warps 4-7: RSA^T (rows i, columns t)
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    zero4(X1[q]);
    zero4(X2[q]);
  }
  if (warp < 4) {
    // Mka = A^ K~^T, Mba = A^ B~^T (strictly lower); Mkr = R^ K~^T, Mbr = R^ B~^T (with diagonal)
    float acc[2][4];
    zero4(acc[0]);
    zero4(acc[1]);
    mm_mk_nk<4>(acc, warp < 2 ? sm.Ah : sm.Rh, kB64, 0, (warp & 1) ? sm.Bt : sm.Kt, kB64, 0, lane);
    if (warp == 1) {
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int t = g + 8 * h, s = 8 * nt + 2 * t4;
          sm.Mba[t * kLD16 + s] = s < t ? acc[nt][2 * h] : 0.f;
          sm.Mba[t * kLD16 + s + 1] = s + 1 < t ? acc[nt][2 * h + 1] : 0.f;
        }
      __syncwarp();
      unit_lower_inverse16(sm.Mba, sm.Tm, lane);
    } else {
      store_masked16(acc, sm.M[warp == 0 ? 0 : warp - 1], true, warp >= 2, g, t4);
    }
#pragma unroll
    for (int kb = 0; kb < 4; ++kb) {  // Gc Bb^T and Gc Kb^T, one A fragment for both
      uint32_t a[4], b[4];
      a_mk(a, sm.u.st.Gc, kB64, r0, 16 * kb, lane);
      b_nk(b, sm.Bb, kB64, 0, 16 * kb, lane);
      mma16(X1[0], a, b[0], b[1]);
      mma16(X1[1], a, b[2], b[3]);
      b_nk(b, sm.Kb, kB64, 0, 16 * kb, lane);
      mma16(X2[0], a, b[0], b[1]);
      mma16(X2[1], a, b[2], b[3]);
    }
  } else {
    mm_mk_nk<4>(X1, sm.u.st.S0, kB64, r0, sm.Ah, kB64, 0, lane);  // S0 A^T
    // this row block's part of colsum(Gc o S0), columns 2 lane, 2 lane + 1
    float2 ep = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = r0; i < r0 + 16; ++i) {
      const float2 gc = bf2(sm.u.st.Gc + i * kB64 + 2 * lane), s0 = bf2(sm.u.st.S0 + i * kB64 + 2 * lane);
      ep = ffma2(gc, s0, ep);
    }
    *reinterpret_cast<float2*>(&sm.Epart[rb][2 * lane]) = ep;
  }
  __syncthreads();

  // ---- C: DSA^T = (Gc Bb^T + DY^T Mbr) T, DV^T += DY^T Mkr + DSA^T Mka and dv (warps 0-3);
  //      SA^T = (S0 A^T + V^T Mka^T) T^T (warps 4-7); sa and dsa stored as bf16 [t][i]
  {
    uint32_t b[4], p[4];
    float Y[2][4];
    zero4(Y[0]);
    zero4(Y[1]);
    if (warp < 4) {
      uint32_t aD[4];
      a_km(aD, sm.raw[V_DY], kB64, r0, 0, lane);  // DY^T
      b_kn(b, sm.M[2], kB16, 0, 0, lane);         // Mbr
      mma16(X1[0], aD, b[0], b[1]);
      mma16(X1[1], aD, b[2], b[3]);
      b_kn(b, sm.M[1], kB16, 0, 0, lane);  // Mkr
      mma16(X2[0], aD, b[0], b[1]);
      mma16(X2[1], aD, b[2], b[3]);
      c2a16(p, X1[0], X1[1]);
      b_kn(b, sm.Tm, kB16, 0, 0, lane);  // T
      mma16(Y[0], p, b[0], b[1]);
      mma16(Y[1], p, b[2], b[3]);
    } else {
      uint32_t aV[4];
      a_km(aV, sm.raw[V_V], kB64, r0, 0, lane);  // V^T
      b_nk(b, sm.M[0], kB16, 0, 0, lane);        // Mka^T
      mma16(X1[0], aV, b[0], b[1]);
      mma16(X1[1], aV, b[2], b[3]);
      c2a16(p, X1[0], X1[1]);
      b_nk(b, sm.Tm, kB16, 0, 0, lane);  // T^T
      mma16(Y[0], p, b[0], b[1]);
      mma16(Y[1], p, b[2], b[3]);
    }
    c2a16(p, Y[0], Y[1]);
    stsm4t((warp < 4 ? sm.DSA : sm.SA) + ((lane & 7) + (lane >> 4) * 8) * kB64 + r0 + ((lane >> 3) & 1) * 8, p);
    if (warp < 4) {  // DV^T += DSA^T Mka (DSA^T from the registers just stored), then dv
      b_kn(b, sm.M[0], kB16, 0, 0, lane);  // Mka
      mma16(X2[0], p, b[0], b[1]);
      mma16(X2[1], p, b[2], b[3]);
#pragma unroll
      for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int t = 8 * q + 2 * t4 + e;
          if (t < len) {
            float* dst = args.dv + base + (size_t)t * vstep + r0 + g;
            float x0 = X2[q][e], x1 = X2[q][2 + e];
            if (epi) {  // + dout bonus
              x0 = fmaf(bf(ep.dout + t * kB64 + r0 + g), ep.stat[t][1], x0);
              x1 = fmaf(bf(ep.dout + t * kB64 + r0 + g + 8), ep.stat[t][1], x1);
            }
            if (in_extent(args.status, args.ext.dv, dst)) dst[0] = x0;
            if (in_extent(args.status, args.ext.dv, dst + 8)) dst[8] = x1;
          }
        }
    }
  }
  __syncthreads();

  // ---- D: U0 = triu(V DY^T), U1 = triu(V DSA^T, 1), U2 = triu(SA DY^T), U3 = triu(SA DSA^T, 1)
  //      (warps 4-7), while warps 0-3 go on to the column products; the barrier after the
  //      column products orders them before the triangular terms read them
  if (warp >= 4) {
    const int u = warp - 4;
    float acc[2][4];
    zero4(acc[0]);
    zero4(acc[1]);
    mm_mk_nk<4>(acc, u < 2 ? sm.raw[V_V] : sm.SA, kB64, 0, u % 2 == 0 ? sm.raw[V_DY] : sm.DSA, kB64, 0, lane);
    store_masked16(acc, sm.U[u], false, u % 2 == 0, g, t4);
  }

  // ---- E: column products, 8 warps: warp (grp, jb) covers columns j0 .. j0+15 of
  //      dk~, db~ (grp 0) or dr^, da^ (grp 1)
  const int grp = warp >> 2, jb = warp & 3, j0 = 16 * jb;
  float P0[2][4], P1[2][4];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    zero4(P0[nt]);
    zero4(P1[nt]);
  }
  {  // sums over the rows i: V Gc, SA Gc (grp 0); DY S0, DSA S0 (grp 1)
    const bf16_t* Bm = grp ? sm.u.st.S0 : sm.u.st.Gc;
    const bf16_t* X = grp ? sm.raw[V_DY] : sm.raw[V_V];
    const bf16_t* Y = grp ? sm.DSA : sm.SA;
#pragma unroll
    for (int kb = 0; kb < 4; ++kb) {
      uint32_t a0[4], a1[4], b[4];
      a_mk(a0, X, kB64, 0, 16 * kb, lane);
      a_mk(a1, Y, kB64, 0, 16 * kb, lane);
      b_kn(b, Bm, kB64, j0, 16 * kb, lane);
      mma16(P0[0], a0, b[0], b[1]);
      mma16(P0[1], a0, b[2], b[3]);
      mma16(P1[0], a1, b[0], b[1]);
      mma16(P1[1], a1, b[2], b[3]);
    }
  }
  // per element (t, j) of this warp: grp 0: 1/c, k, b; grp 1: c, c(t-1), r, a
  auto load_q = [&](float2 (&q0)[2][2], float2 (&q1)[2][2], float2 (&q2)[2][2], float2 (&q3)[2][2]) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int t = g + 8 * h, col = j0 + 8 * nt + 2 * t4;
        const float2 c = *reinterpret_cast<const float2*>(sm.cS + t * kLD64 + col);
        if (grp == 0) {
          q0[nt][h] = make_float2(rcp_approx(c.x), rcp_approx(c.y));
          q1[nt][h] = bf2(rs + V_K * RS + t * kB64 + col);
          q2[nt][h] = bf2(rs + V_B * RS + t * kB64 + col);
          q3[nt][h] = make_float2(0.f, 0.f);
        } else {
          q0[nt][h] = c;
          q1[nt][h] = t ? *reinterpret_cast<const float2*>(sm.cS + (t - 1) * kLD64 + col) : make_float2(1.f, 1.f);
          q2[nt][h] = bf2(rs + V_R * RS + t * kB64 + col);
          q3[nt][h] = bf2(rs + V_A * RS + t * kB64 + col);
        }
      }
  };
  {
    float2 q0[2][2], q1[2][2], q2[2][2], q3[2][2];
    load_q(q0, q1, q2, q3);
    // This warp's part of the dw anchors, from the column products (c(L) colsum(Gc o S0) is
    // added later):
    //   colsum(Gc o S(L)) = c(L) colsum(Gc o S0) + sum_t (Kb o V Gc + Bb o SA Gc)       (grp 0)
    //   colsum(Gc' o S0)  = c(L) colsum(Gc o S0) + sum_t (R^ o DY S0 + A^ o DSA S0)     (grp 1)
    // with S(L) = S0 diag(c(L)) + V^T Kb + SA^T Bb and Gc' = Gc diag(c(L)) + DY^T R^ + DSA^T A^.
    float v[4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      float2 acc = make_float2(0.f, 0.f);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        // grp 0: Kb = k c(L) / c, Bb = b c(L) / c (c(L) applied after the sum); grp 1: R^ = r c, A^ = a c(t-1)
        const float2 m0 = grp ? fmul2(q2[nt][h], q0[nt][h]) : fmul2(q1[nt][h], q0[nt][h]);
        const float2 m1 = grp ? fmul2(q3[nt][h], q1[nt][h]) : fmul2(q2[nt][h], q0[nt][h]);
        acc = ffma2(m0, make_float2(P0[nt][2 * h], P0[nt][2 * h + 1]), acc);
        acc = ffma2(m1, make_float2(P1[nt][2 * h], P1[nt][2 * h + 1]), acc);
      }
      v[2 * nt] = acc.x;
      v[2 * nt + 1] = acc.y;
    }
    // sum over the 8 row groups: reduce-scatter over xor 16 (n-tile), 8 (column parity), then 4
    const bool up16 = (g & 4) != 0, up8 = (g & 2) != 0;
    const float x0 = (up16 ? v[2] : v[0]) + __shfl_xor_sync(0xffffffffu, up16 ? v[0] : v[2], 16);
    const float x1 = (up16 ? v[3] : v[1]) + __shfl_xor_sync(0xffffffffu, up16 ? v[1] : v[3], 16);
    float y = (up8 ? x1 : x0) + __shfl_xor_sync(0xffffffffu, up8 ? x0 : x1, 8);
    y += __shfl_xor_sync(0xffffffffu, y, 4);
    if ((g & 1) == 0) {
      const int col = j0 + 8 * (up16 ? 1 : 0) + 2 * t4 + (up8 ? 1 : 0);
      const float cl = sm.cLs[col];
      sm.anc[grp ? 0 : 1][col] = grp ? y : cl * y;
    }
  }
  __syncthreads();  // checkpoint and carry tiles are free from here on (the dw exchange below)
  // triangular terms (U0 = triu(V DY^T), U1 = triu(V DSA^T, 1), U2 = triu(SA DY^T), U3 = triu(SA DSA^T, 1)):
  //   dk~ = (V Gc) c(L) + U0 R^ + U1 A^        db~ = (SA Gc) c(L) + U2 R^ + U3 A^
  //   dr^ = DY S0 + U0^T K~ + U2^T B~          da^ = DSA S0 + U1^T K~ + U3^T B~
  {
    uint32_t u0[4], u1[4], u2[4], u3[4], b[4];
    if (grp == 0) {
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const float2 cl = *reinterpret_cast<const float2*>(sm.cLs + j0 + 8 * nt + 2 * t4);
        P0[nt][0] *= cl.x;
        P0[nt][1] *= cl.y;
        P0[nt][2] *= cl.x;
        P0[nt][3] *= cl.y;
        P1[nt][0] *= cl.x;
        P1[nt][1] *= cl.y;
        P1[nt][2] *= cl.x;
        P1[nt][3] *= cl.y;
      }
      a_mk(u0, sm.U[0], kB16, 0, 0, lane);
      a_mk(u1, sm.U[1], kB16, 0, 0, lane);
      a_mk(u2, sm.U[2], kB16, 0, 0, lane);
      a_mk(u3, sm.U[3], kB16, 0, 0, lane);
      b_kn(b, sm.Rh, kB64, j0, 0, lane);
      mma16(P0[0], u0, b[0], b[1]);
      mma16(P0[1], u0, b[2], b[3]);
      mma16(P1[0], u2, b[0], b[1]);
      mma16(P1[1], u2, b[2], b[3]);
      b_kn(b, sm.Ah, kB64, j0, 0, lane);
      mma16(P0[0], u1, b[0], b[1]);
      mma16(P0[1], u1, b[2], b[3]);
      mma16(P1[0], u3, b[0], b[1]);
      mma16(P1[1], u3, b[2], b[3]);
    } else {
      a_km(u0, sm.U[0], kB16, 0, 0, lane);
      a_km(u1, sm.U[1], kB16, 0, 0, lane);
      a_km(u2, sm.U[2], kB16, 0, 0, lane);
      a_km(u3, sm.U[3], kB16, 0, 0, lane);
      b_kn(b, sm.Kt, kB64, j0, 0, lane);
      mma16(P0[0], u0, b[0], b[1]);
      mma16(P0[1], u0, b[2], b[3]);
      mma16(P1[0], u1, b[0], b[1]);
      mma16(P1[1], u1, b[2], b[3]);
      b_kn(b, sm.Bt, kB64, j0, 0, lane);
      mma16(P0[0], u2, b[0], b[1]);
      mma16(P0[1], u2, b[2], b[3]);
      mma16(P1[0], u3, b[0], b[1]);
      mma16(P1[1], u3, b[2], b[3]);
    }
  }
  // unscale: dk = dk~ / c, db = db~ / c (grp 0); dr = dr^ c, da = da^ c(t-1) (grp 1); and this
  // group's part of x = r dr - k dk - b db + a da
  float X[2][4], AD[2][4];
  float2 q0[2][2], q1[2][2], q2[2][2], q3[2][2];
  load_q(q0, q1, q2, q3);
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (grp == 0) {
        const float ic[2] = {q0[nt][h].x, q0[nt][h].y}, kv[2] = {q1[nt][h].x, q1[nt][h].y},
                    bv[2] = {q2[nt][h].x, q2[nt][h].y};
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          P0[nt][2 * h + e] *= ic[e];
          P1[nt][2 * h + e] *= ic[e];
          X[nt][2 * h + e] = -kv[e] * P0[nt][2 * h + e] - bv[e] * P1[nt][2 * h + e];
          AD[nt][2 * h + e] = 0.f;
        }
      } else {
        const float cv[2] = {q0[nt][h].x, q0[nt][h].y}, cpv[2] = {q1[nt][h].x, q1[nt][h].y},
                    rv[2] = {q2[nt][h].x, q2[nt][h].y}, av[2] = {q3[nt][h].x, q3[nt][h].y};
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          P0[nt][2 * h + e] *= cv[e];
          P1[nt][2 * h + e] *= cpv[e];
          AD[nt][2 * h + e] = av[e] * P1[nt][2 * h + e];
          X[nt][2 * h + e] = rv[e] * P0[nt][2 * h + e] + AD[nt][2 * h + e];
        }
      }
    }
  // this warp's outputs, and its part of x for dw: grp 0 -k dk - b db, grp 1 r dr + a da and a da
  float* XK = sm.u.xch[0];  // [t][j] stride 72
  float* XR = sm.u.xch[1];
  float* XA = sm.u.xch[2];
  float* out0 = grp ? args.dr : args.dk;
  float* out1 = grp ? args.da : args.db;
  const Extent& x0 = grp ? args.ext.dr : args.ext.dk;
  const Extent& x1 = grp ? args.ext.da : args.ext.db;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int t = g + 8 * h;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int col = j0 + 8 * nt + 2 * t4;
      *reinterpret_cast<float2*>((grp ? XR : XK) + t * kLD64 + col) = make_float2(X[nt][2 * h], X[nt][2 * h + 1]);
      if (grp) *reinterpret_cast<float2*>(XA + t * kLD64 + col) = make_float2(AD[nt][2 * h], AD[nt][2 * h + 1]);
      if (t < len) {
        const size_t off = base + (size_t)t * vstep + col;
        float2 o0 = make_float2(P0[nt][2 * h], P0[nt][2 * h + 1]);
        if (epi) {  // the bonus terms: dk += dbon r r_k (grp 0), dr += dbon k r_k (grp 1)
          const float db = ep.dbon[t];
          const float2 x = bf2(rs + (grp ? V_K : V_R) * RS + t * kB64 + col);
          o0.x = fmaf(db * x.x, ep.rk[col], o0.x);
          o0.y = fmaf(db * x.y, ep.rk[col + 1], o0.y);
        }
        float2* p0 = reinterpret_cast<float2*>(out0 + off);
        float2* p1 = reinterpret_cast<float2*>(out1 + off);
        if (in_extent(args.status, x0, p0)) *p0 = o0;
        if (in_extent(args.status, x1, p1)) *p1 = make_float2(P1[nt][2 * h], P1[nt][2 * h + 1]);
      }
    }
  }
  __syncthreads();
  // w dw from the identity, anchored where fewer terms are summed, thread (column, half):
  //   t < 8:  colsum(carry at the chunk start o S0) - sum_{u<t} x(u) - a(t) da(t)
  //   t >= 8: sum_{u>=t} x(u) - a(t) da(t) + colsum(carry at the chunk end o S(L))
  if (tid < 2 * kN) {
    const int col = tid & 63, upper = tid >> 6;
    const float cge = sm.cLs[col] * (sm.Epart[0][col] + sm.Epart[1][col] + sm.Epart[2][col] + sm.Epart[3][col]);
    float run = cge + sm.anc[upper][col];
#pragma unroll
    for (int e = 0; e < kL / 2; ++e) {
      const int t = upper ? kL - 1 - e : e;
      const float x = XK[t * kLD64 + col] + XR[t * kLD64 + col];
      if (upper) run += x;  // end anchor plus the x of the steps from t on
      float v;
      if constexpr (kLogit)  // dL/dz straight from w dw: no division by w
        v = logit_grad_from_wdw(run - XA[t * kLD64 + col], bf(rs + V_W * RS + t * kB64 + col));
      else
        v = (run - XA[t * kLD64 + col]) * rcp_approx(bf(rs + V_W * RS + t * kB64 + col));
      float* pw = args.dw + base + (size_t)t * vstep + col;
      if (t < len && in_extent(args.status, args.ext.dw, pw)) *pw = v;
      if (!upper) run -= x;  // start anchor minus the x of the steps before t
    }
  }
  if (epi) {
    __syncthreads();  // the dw exchange is read; its space takes the parameter terms
    epi_params_chunk(sm.u.xch[0], pp, args, head, n, nchunks);
  }
}


// ========================================== output kernel on tcgen05 ===
//
// The same per-chunk output pass as wkv7_bwd4_out_kernel, with every product
// on the 5th-generation tensor cores: tcgen05.mma kind::f16 (bf16 operands,
// fp32 accumulators in tensor memory), issued by one thread, operands read
// by the tensor core from shared memory through matrix descriptors. The
// chunk's rows and its carry arrive by TMA (cp.async.bulk.tensor) straight
// into the 128-byte-swizzled layout the descriptors describe. Five rounds of
// products, each followed by the threads reading the accumulators back (rows
// i of the state or columns j, as tensor-memory lanes):
//   1. Gram blocks [A^; R^] [K~; B~]^T                                (M = 64)
//   2. [S0; Gc] [Bb; Kb; A^]^T + [V^T; DY^T] (Mka, [Mbr | Mkr]):
//      S0 A^T + V^T Mka^T, Gc Bb^T + DY^T Mbr, Gc Kb^T + DY^T Mkr      (M = 128)
//   3. the same rounds' SA and DSA parts times T^T and T: SA^T, DSA^T   (M = 128)
//   4. DV^T += DSA^T Mka; the triangular factors [V; SA; DY; DSA] [DY; DSA]^T
//      (M = 64); the column products [S0^T; Gc^T] [V; SA; DY; DSA]^T    (M = 128)
//   5. the triangular terms [K~^T; R^T] U + [B~^T; A^T] U'              (M = 128)
// T = (I - Mba)^-1 is formed by one warp from the Gram rows it holds while
// round 2 runs. Each tile is stored once and read K-major or MN-major
// (transposed) as a product needs it. 128 tensor-memory columns per CTA,
// three CTAs per SM.

namespace tcout {

constexpr int kThreads = 256;
constexpr int kCtasPerSm = 4;
constexpr uint32_t kTmemCols = 128;

// Shared memory (byte offsets from a 1024-byte-aligned base). 128B-swizzled
// tiles of rows of 64 bf16 (128 bytes), 16 rows (2 KB) or 64 rows (8 KB).
// Tiles whose lifetimes do not overlap share space (noted at each).
enum : uint32_t {
  OFF_S0 = 0x0000,   // checkpoint [i][j] (rounded to bf16); after round 4: U tiles, dw exchange
  OFF_GC = 0x2000,   // carry after the chunk [i][j] (TMA); follows S0
  OFF_UA = 0x0000,   // (after round 4) [U0 | U1] rows p (columns 0-15, 16-31)
  OFF_UB = 0x0800,   // (after round 4) [U2 | U3]
  OFF_XK = 0x1000,   // (after round 5) the dw exchange XK, XR, XA [16][64] fp32 (12 KB)
  OFF_KT = 0x4000,   // K~ = k / c [t][j]
  OFF_BT = 0x4800,   // B~ = b / c
  OFF_BB = 0x5000,   // Bb = b c(L) / c
  OFF_KB = 0x5800,   // Kb = k c(L) / c
  OFF_PA = 0x5000,   // (after round 2) [SA_pre; DSA_pre], then [.; DSA^T]: 128 x 16 bf16, unswizzled core-matrix layout
  OFF_AH = 0x6000,   // A^ = a c(t - 1)
  OFF_RH = 0x6800,   // R^ = r c
  OFF_V = 0x7000,    // v [t][i] (TMA)
  OFF_SA = 0x7800,   // sa [t][i]
  OFF_DY = 0x8000,   // dy [t][i] (TMA)
  OFF_DSA = 0x8800,  // dsa [t][i]; before phase 3: the Mba rows [16][16] fp32 for T
  OFF_MA = 0x9000,   // Mka [t][s]; before phase 1: the decay pair products [8][64] fp32
  OFF_MB = 0x9800,   // [Mbr | Mkr] rows s
  OFF_X = 0x9800,    // (after round 2) T^T: row s = column s of T
  OFF_RAW = 0xA000,  // r, w, k, a, b [t][j] (TMA, plain row-major), 2 KB apart
  OFF_EPART = 0xC800,  // colsum(Gc o S0), one partial per warp [8][64] fp32
  OFF_ANC = 0xD000,    // the chunk's parts of the dw anchors [start, end][half][64] fp32
  OFF_CL = 0xD400,     // c(L) [64] fp32
  OFF_C7 = 0xD500,     // c(7) [64] fp32, the running decay product after the first 8 steps
  OFF_BAR = 0xD600,    // two mbarriers and the tensor-memory address
  SMEM_USED = 0xD640,
};
// A chunk run step by step: its rows with padded stride (16,128 B) and the
// reduction scratch (10,240 B) from OFF_S0, below every tile the copy reads.
constexpr uint32_t kSmemBytes = SMEM_USED + 1024;  // + alignment slack
constexpr uint32_t OFF_RED = 0x3F00;
enum { RAW_R = 0, RAW_W = 1, RAW_K = 2, RAW_A = 3, RAW_B = 4 };

// Byte offset of element (row, col) in a 128B-swizzled tile of 64-element
// rows (the tile 1024-byte aligned): 16-byte chunks permuted by row mod 8.
__device__ __forceinline__ uint32_t swz(int row, int col) {
  return (uint32_t)(row * 128 + ((((col >> 3) ^ row) & 7) << 4) + ((col & 7) << 1));
}
// Byte offset of element (t, j) in a plain row-major tile of 64-element rows
// (the chunk's r, w, k, a, b, which only the threads read).
__device__ __forceinline__ uint32_t rowo(int t, int j) { return (uint32_t)(t * 128 + j * 2); }
// Byte offset of element (r, c) in a 16-column tile in the unswizzled
// core-matrix layout (8 x 8 blocks of 128 contiguous bytes).
__device__ __forceinline__ uint32_t core16(int r, int c) {
  return (uint32_t)(((r >> 3) * 2 + (c >> 3)) * 128 + (r & 7) * 16 + (c & 7) * 2);
}

// Shared-memory matrix descriptor (sm_100 form): start, leading and stride
// byte offsets (>> 4), descriptor version 1, layout type (2 = 128B swizzle,
// 0 = none).
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t layout) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46) | ((uint64_t)layout << 61);
}
// K-major 128B-swizzled operand (rows of 64 elements, 8-row groups 1024 bytes
// apart), K step ks of 16 elements.
__device__ __forceinline__ uint64_t desc_k(uint32_t addr, int ks) { return sdesc(addr + 32u * ks, 16, 1024, 2); }
// MN-major 128B-swizzled operand: stored [k][mn] with 64 mn per row; atoms of
// 64 (M or N) x 8 (K), the next 64 along M or N `lbo` bytes on; K step ks.
__device__ __forceinline__ uint64_t desc_mn(uint32_t addr, uint32_t lbo, int ks) {
  return sdesc(addr + 2048u * ks, lbo, 1024, 2);
}
// K-major unswizzled 16-column operand (core16 layout), K = 16.
__device__ __forceinline__ uint64_t desc_k16(uint32_t addr) { return sdesc(addr, 128, 256, 0); }
// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, A/B
// MN-major flags, N and M.
__host__ __device__ constexpr uint32_t idesc(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// D[tmem] (+)= A[smem] B[smem]^T
__device__ __forceinline__ void mma(uint32_t d, uint64_t a, uint64_t b, uint32_t id, bool acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d),
      "l"(a), "l"(b), "r"(id), "r"((uint32_t)acc)
      : "memory");
}
__device__ __forceinline__ void commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}
__device__ __forceinline__ void ld8(uint32_t taddr, float (&v)[8]) { tmem_ld<8>(taddr, v); }
__device__ __forceinline__ void ld16(uint32_t taddr, float (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, "
      "[%16];"
      : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]), "=f"(v[7]), "=f"(v[8]),
        "=f"(v[9]), "=f"(v[10]), "=f"(v[11]), "=f"(v[12]), "=f"(v[13]), "=f"(v[14]), "=f"(v[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ float bfs(const unsigned char* sb, uint32_t off) {
  return __bfloat162float(*reinterpret_cast<const bf16_t*>(sb + off));
}
__device__ __forceinline__ float2 bfs2(const unsigned char* sb, uint32_t off) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(sb + off));
}
__device__ __forceinline__ void sts_bf(unsigned char* sb, uint32_t off, float x) {
  *reinterpret_cast<bf16_t*>(sb + off) = __float2bfloat16_rn(x);
}
// Every thread waits for the phase; all leave together, false if any gave up
// (after draining: a second bounded wait).
__device__ __forceinline__ bool cta_wait(unsigned* status, uint64_t* bar, uint32_t parity) {
  bool ok = mbar_wait_bounded(status, bar, parity);
  if (!ok) mbar_wait_bounded(status, bar, parity);
  return __syncthreads_and(ok) != 0;
}
// Smem writes by the threads become visible to the tensor core's reads, and
// tensor-memory reads finish before the next product is issued.
__device__ __forceinline__ void to_mma_sync() {
  fence_proxy_async_smem();
  tmem_fence_before_sync();
  __syncthreads();
  tmem_fence_after_sync();
}

// The v, dy and carry tiles of `task` (one of the two arrivals of the load barrier's phase).
__device__ __forceinline__ void issue_loads_vdg(unsigned char* sb, const BwdArgs& args, int task, int nchunks,
                                                uint64_t* bar) {
  const int head = task / nchunks, n = task % nchunks, bi = head / args.H, hi = head % args.H;
  mbar_arrive_expect_tx(bar, 2 * 2048 + 8192);
  tma_load_4d(sb + OFF_V, &args.swmap[3], bar, 0, hi, n * kL, bi);
  tma_load_4d(sb + OFF_DY, &args.swmap[6], bar, 0, hi, n * kL, bi);
  tma_load_3d(sb + OFF_GC, &args.gcmap, bar, 0, 0, task);
}
// The r, w, k, a, b rows of `task`, row-major (the other arrival).
__device__ __forceinline__ void issue_loads_raw(unsigned char* sb, const BwdArgs& args, int task, int nchunks,
                                                uint64_t* bar) {
  const int head = task / nchunks, n = task % nchunks, bi = head / args.H, hi = head % args.H;
  mbar_arrive_expect_tx(bar, 5 * 2048);
  const int vec[5] = {0, 1, 2, 4, 5};  // r w k a b
#pragma unroll
  for (int q = 0; q < 5; ++q) tma_load_4d(sb + OFF_RAW + 0x800 * q, &args.map[vec[q]], bar, 0, hi, n * kL, bi);
}
// The checkpoint S0 (fp32 [i][j]) rounded to bf16 into its swizzled tile, four float4 per thread.
__device__ __forceinline__ void stage_checkpoint(unsigned char* sb, const float* S0g, int tid, const BwdArgs& args) {
  float4 x[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float4* p = reinterpret_cast<const float4*>(S0g + 4 * (tid + kThreads * q));
    x[q] = in_extent(args.status, args.ext.ckpt, p) ? *p : make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int idx = tid + kThreads * q, i = idx >> 4, c4 = idx & 15;
    *reinterpret_cast<uint2*>(sb + OFF_S0 + swz(i, 4 * c4)) = make_uint2(pack_bf16(x[q].x, x[q].y), pack_bf16(x[q].z, x[q].w));
  }
}

// One chunk (task = (b, h) head * nchunks + chunk). The load barrier completes once per
// task (ld_it counts them), the product barrier five times per task run on the tensor
// cores (mma_it counts those) and never for a chunk run step by step. Returns 1 for a
// tensor-core task, 0 for a step-by-step one, -1 if a wait gave up (the CTA then leaves).
template <bool kLogit>
__device__ __forceinline__ int body(unsigned char* sb, uint32_t tb, const BwdArgs& args, int task, int ld_it,
                                    int mma_it) {
  const int T = args.T, H = args.H, nchunks = (T + kL - 1) / kL;
  const int head = task / nchunks, n = task % nchunks, bi = head / H, hi = head % H;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t0 = n * kL, len = min(kL, T - t0);
  const size_t vstep = (size_t)H * kN, base = ((size_t)bi * T + t0) * vstep + (size_t)hi * kN;
  const float* S0g = args.ckpt + ((size_t)head * args.nck + n) * kN * kN;
  const bf16_t* Gcg = reinterpret_cast<const bf16_t*>(args.carry) + ((size_t)head * nchunks + n) * kN * kN;
  const uint32_t sa_ = smem_addr(sb);
  uint64_t* bar_load = reinterpret_cast<uint64_t*>(sb + OFF_BAR);
  uint64_t* bar_mma = bar_load + 1;
  float* c7s = reinterpret_cast<float*>(sb + OFF_C7);
  float* cLs = reinterpret_cast<float*>(sb + OFF_CL);
  float* Epart = reinterpret_cast<float*>(sb + OFF_EPART);
  float* anc = reinterpret_cast<float*>(sb + OFF_ANC);
  const unsigned char* raw = sb + OFF_RAW;
  // this warp's quarter of tensor-memory lanes
  const uint32_t tq = tb + ((uint32_t)(32 * (warp & 3)) << 16);

  // ---- loads: the chunk's rows and its carry by TMA (rows past T read as zeros), the
  //      checkpoint rounded to bf16
  if (tid == 0) {
    issue_loads_vdg(sb, args, task, nchunks, bar_load);
    issue_loads_raw(sb, args, task, nchunks, bar_load);
  }
  stage_checkpoint(sb, S0g, tid, args);
  // five product rounds per task: round r (from 0) waits on parity par ^ (r & 1)
  const uint32_t par = (uint32_t)mma_it & 1u;
  if (!cta_wait(args.status, bar_load, (uint32_t)ld_it & 1u)) return -1;
  {  // colsum(Gc o S0) of the bf16 tiles: thread rows tid / 16 + 16 q, columns 4 (tid % 16) ..;
     // then lanes l, l ^ 16 (the same columns); one partial per warp and column
    float4 e = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int idx = tid + kThreads * q, i = idx >> 4, c4 = idx & 15;
      const uint2 gv = *reinterpret_cast<const uint2*>(sb + OFF_GC + swz(i, 4 * c4));
      const uint2 sv = *reinterpret_cast<const uint2*>(sb + OFF_S0 + swz(i, 4 * c4));
      const float2 g0 = unpack_bf16(gv.x), g1 = unpack_bf16(gv.y), s0 = unpack_bf16(sv.x), s1 = unpack_bf16(sv.y);
      e.x = fmaf(g0.x, s0.x, e.x);
      e.y = fmaf(g0.y, s0.y, e.y);
      e.z = fmaf(g1.x, s1.x, e.z);
      e.w = fmaf(g1.y, s1.y, e.w);
    }
    e.x += __shfl_xor_sync(0xffffffffu, e.x, 16);
    e.y += __shfl_xor_sync(0xffffffffu, e.y, 16);
    e.z += __shfl_xor_sync(0xffffffffu, e.z, 16);
    e.w += __shfl_xor_sync(0xffffffffu, e.w, 16);
    if (lane < 16) *reinterpret_cast<float4*>(Epart + warp * kN + 4 * lane) = e;
  }

  // ---- A: scaled operands; thread (lane, warp) forms columns 2 lane, 2 lane + 1 of steps
  //      2 warp, 2 warp + 1 (the pairs' decay products chained in step order)
  {
    const int j = 2 * lane, ta = 2 * warp;
    float* Ppart = reinterpret_cast<float*>(sb + OFF_MA);  // [8][64]
    float2 wv[2];
#pragma unroll
    for (int e = 0; e < 2; ++e)
      wv[e] = ta + e < len ? decay_value2<kLogit>(bfs2(raw + RAW_W * 0x800, rowo(ta + e, j))) : make_float2(1.f, 1.f);
    const bool safe = decay_is_safe(wv[0].x) && decay_is_safe(wv[0].y) && decay_is_safe(wv[1].x) &&
                      decay_is_safe(wv[1].y);
    *reinterpret_cast<float2*>(&Ppart[warp * kN + j]) = fmul2(wv[0], wv[1]);
    if (__syncthreads_or(!safe)) {
      // A chunk whose decays leave the scaled form's range: step by step, from the rows
      // copied with the padded stride of out_direct into the (dead) checkpoint and carry
      // tiles, which no source tile overlaps.
      const uint32_t src[7] = {OFF_RAW + 0x000, OFF_RAW + 0x800, OFF_RAW + 0x1000, OFF_V, OFF_RAW + 0x1800,
                               OFF_RAW + 0x2000, OFF_DY};
      bf16_t* pad = reinterpret_cast<bf16_t*>(sb + OFF_S0);
#pragma unroll 1
      for (int v = 0; v < 7; ++v)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int e = 4 * (tid + kThreads * h), t = e >> 6, c = e & 63;
          *reinterpret_cast<uint2*>(pad + v * kL * kB64 + t * kB64 + c) =
              *reinterpret_cast<const uint2*>(sb + src[v] + ((v == 3 || v == 6) ? swz(t, c) : rowo(t, c)));
        }
      __syncthreads();
      out_direct<kLogit>(pad, reinterpret_cast<float*>(sb + OFF_RED), S0g, Gcg, len, args, base, vstep, warp, lane);
      return 0;
    }
    float2 cL = make_float2(1.f, 1.f), cpre = cL;  // cpre = c(ta - 1)
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      cL = fmul2(cL, *reinterpret_cast<const float2*>(&Ppart[q * kN + j]));
      if (q < warp) cpre = cL;
    }
    if (warp == 0) *reinterpret_cast<float2*>(&cLs[j]) = cL;
    if (warp == 4) *reinterpret_cast<float2*>(&c7s[j]) = cpre;  // c(7)
    float2 c = cpre;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int t = ta + e;
      const uint32_t o = swz(t, j), ro = rowo(t, j);
      const float2 w = wv[e];
      const float2 a = bfs2(raw + RAW_A * 0x800, ro), r = bfs2(raw + RAW_R * 0x800, ro);
      const float2 k = bfs2(raw + RAW_K * 0x800, ro), b = bfs2(raw + RAW_B * 0x800, ro);
      const float2 cprev = c;
      c = fmul2(c, w);
      const float2 ic = make_float2(rcp_approx(c.x), rcp_approx(c.y)), sc = fmul2(cL, ic);
      *reinterpret_cast<uint32_t*>(sb + OFF_AH + o) = pack_bf16(a.x * cprev.x, a.y * cprev.y);
      *reinterpret_cast<uint32_t*>(sb + OFF_RH + o) = pack_bf16(r.x * c.x, r.y * c.y);
      *reinterpret_cast<uint32_t*>(sb + OFF_KT + o) = pack_bf16(k.x * ic.x, k.y * ic.y);
      *reinterpret_cast<uint32_t*>(sb + OFF_BT + o) = pack_bf16(b.x * ic.x, b.y * ic.y);
      *reinterpret_cast<uint32_t*>(sb + OFF_KB + o) = pack_bf16(k.x * sc.x, k.y * sc.y);
      *reinterpret_cast<uint32_t*>(sb + OFF_BB + o) = pack_bf16(b.x * sc.x, b.y * sc.y);
    }
  }
  to_mma_sync();

  // ---- round 1: the Gram blocks (columns 0-31, M = 64: lanes 0-15 A^, 32-47 R^; columns
  //      0-15 = . K~^T, 16-31 = . B~^T): Mka, Mba (lanes 0-15), Mkr, Mbr (lanes 32-47)
  if (tid == 0) {
#pragma unroll
    for (int ks = 0; ks < 4; ++ks)
      mma(tb, desc_k(sa_ + OFF_AH, ks), desc_k(sa_ + OFF_KT, ks), idesc(64, 32, 0, 0), ks > 0);
    commit(bar_mma);
  }
  if (!cta_wait(args.status, bar_mma, par)) return -1;
  tmem_fence_after_sync();

  // ---- phase 1: Mka rows (masked s < t) to the tile Mka [t][s]; [Mbr | Mkr] rows (s <= t) to
  //      [Mbr | Mkr] [s][.]; warp 0 keeps the Mba rows for T
  if (warp < 2) {
    float g[32];
    ld16(tq, *reinterpret_cast<float(*)[16]>(&g[0]));
    ld16(tq + 16, *reinterpret_cast<float(*)[16]>(&g[16]));
    tmem_wait_ld();
    if (lane < 16) {
      const int t = lane;
      uint32_t pk[16];
      if (warp == 0) {
        float* mba = reinterpret_cast<float*>(sb + OFF_DSA);  // Mba rows, fp32, for T
#pragma unroll
        for (int q = 0; q < 4; ++q)
          *reinterpret_cast<float4*>(mba + t * 16 + 4 * q) =
              make_float4(4 * q < t ? g[16 + 4 * q] : 0.f, 4 * q + 1 < t ? g[17 + 4 * q] : 0.f,
                          4 * q + 2 < t ? g[18 + 4 * q] : 0.f, 4 * q + 3 < t ? g[19 + 4 * q] : 0.f);
#pragma unroll
        for (int s = 0; s < 16; s += 2) pk[s / 2] = pack_bf16(s < t ? g[s] : 0.f, s + 1 < t ? g[s + 1] : 0.f);
#pragma unroll
        for (int c = 0; c < 2; ++c)
          *reinterpret_cast<uint4*>(sb + OFF_MA + swz(t, 8 * c)) =
              make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      } else {
#pragma unroll
        for (int s = 0; s < 16; s += 2) {
          pk[s / 2] = pack_bf16(s <= t ? g[16 + s] : 0.f, s + 1 <= t ? g[16 + s + 1] : 0.f);  // Mbr
          pk[8 + s / 2] = pack_bf16(s <= t ? g[s] : 0.f, s + 1 <= t ? g[s + 1] : 0.f);       // Mkr
        }
#pragma unroll
        for (int c = 0; c < 4; ++c)
          *reinterpret_cast<uint4*>(sb + OFF_MB + swz(t, 8 * c)) =
              make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      }
    }
  }
  to_mma_sync();

  // ---- round 2 (columns 32-79, M = 128; B = [Bb; Kb; A^]): rows 0-63 (S0) columns 64-79 =
  //      SA_pre^T = S0 A^T + V^T Mka^T; rows 64-127 (Gc) columns 32-47 = DSA_pre^T = Gc Bb^T +
  //      DY^T Mbr, columns 48-63 = DV_pre^T = Gc Kb^T + DY^T Mkr
  if (tid == 0) {
#pragma unroll
    for (int ks = 0; ks < 4; ++ks)
      mma(tb + 32, desc_k(sa_ + OFF_S0, ks), desc_k(sa_ + OFF_BB, ks), idesc(128, 48, 0, 0), ks > 0);
    mma(tb + 64, desc_mn(sa_ + OFF_V, OFF_DY - OFF_V, 0), desc_k(sa_ + OFF_MA, 0), idesc(128, 16, 1, 0), true);
    mma(tb + 32, desc_mn(sa_ + OFF_V, OFF_DY - OFF_V, 0), desc_mn(sa_ + OFF_MB, 8192, 0), idesc(128, 32, 1, 1), true);
    commit(bar_mma);
  }
  float col[kL];  // warp 0: column (lane & 15) of T
  if (warp == 0) {  // meanwhile: T = (I - Mba)^-1, lane s owning column s (rows of Mba broadcast)
    const int s = lane & 15;
    const float* mba = reinterpret_cast<const float*>(sb + OFF_DSA);
#pragma unroll
    for (int t = 0; t < kL; ++t) {
      float m[16];
#pragma unroll
      for (int q = 0; q < (t + 3) / 4; ++q) {
        const float4 r4 = *reinterpret_cast<const float4*>(mba + t * 16 + 4 * q);
        m[4 * q] = r4.x;
        m[4 * q + 1] = r4.y;
        m[4 * q + 2] = r4.z;
        m[4 * q + 3] = r4.w;
      }
      float x = t == s ? 1.f : 0.f;
#pragma unroll
      for (int u = 0; u < t; ++u) x = fmaf(m[u], col[u], x);
      col[t] = x;
    }
  }
  if (!cta_wait(args.status, bar_mma, par ^ 1u)) return -1;
  tmem_fence_after_sync();

  // ---- phase 2: T^T rows over [Mbr | Mkr] (read by round 2); SA_pre (rows 0-63) and
  //      DSA_pre (rows 64-127) to the A tile [i][t] over Bb, Kb (read by round 2)
  if (warp == 0 && lane < 16) {  // row s of T^T
    const int s = lane;
    uint32_t pk[8];
#pragma unroll
    for (int t = 0; t < kL; t += 2) pk[t / 2] = pack_bf16(col[t], col[t + 1]);
#pragma unroll
    for (int c = 0; c < 2; ++c)
      *reinterpret_cast<uint4*>(sb + OFF_X + swz(s, 8 * c)) = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
  }
  if (warp < 4) {
    float v[16];
    ld16(tq + (warp < 2 ? 64 : 32), v);
    tmem_wait_ld();
    const int r = 32 * warp + lane;
    uint32_t pk[8];
#pragma unroll
    for (int t = 0; t < kL; t += 2) pk[t / 2] = pack_bf16(v[t], v[t + 1]);
    *reinterpret_cast<uint4*>(sb + OFF_PA + core16(r, 0)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    *reinterpret_cast<uint4*>(sb + OFF_PA + core16(r, 8)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
  }
  to_mma_sync();

  // ---- round 3 (columns 0-31, M = 128): columns 0-15 rows 0-63 = SA^T = SA_pre^T T^T
  //      (T^T read MN-major); columns 16-31 rows 64-127 = DSA^T = DSA_pre^T T (K-major)
  if (tid == 0) {
    mma(tb, desc_k16(sa_ + OFF_PA), desc_mn(sa_ + OFF_X, 8192, 0), idesc(128, 16, 0, 1), false);
    mma(tb + 16, desc_k16(sa_ + OFF_PA), desc_k(sa_ + OFF_X, 0), idesc(128, 16, 0, 0), false);
    commit(bar_mma);
  }
  if (!cta_wait(args.status, bar_mma, par)) return -1;
  tmem_fence_after_sync();

  // ---- phase 3: sa, dsa to bf16 tiles [t][i]; dsa^T also to rows 64-127 of the A tile.
  //      Warps 0, 1 / 4, 5: sa steps 0-7 / 8-15; warps 2, 3 / 6, 7: dsa steps 0-7 / 8-15.
  {
    const int i = lane + 32 * (warp & 1), tbeg = warp >= 4 ? 8 : 0;
    float v[8];
    ld8(tq + ((warp & 2) ? 16 : 0) + tbeg, v);
    tmem_wait_ld();
    const uint32_t dst = (warp & 2) ? OFF_DSA : OFF_SA;
#pragma unroll
    for (int e = 0; e < 8; ++e) sts_bf(sb + dst, swz(tbeg + e, i), v[e]);
    if (warp & 2) {
      *reinterpret_cast<uint4*>(sb + OFF_PA + core16(64 + i, tbeg)) =
          make_uint4(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]), pack_bf16(v[4], v[5]), pack_bf16(v[6], v[7]));
    }
  }
  to_mma_sync();

  // ---- round 4: DV^T += DSA^T Mka (columns 48-63, rows 64-127; Mka read MN-major); the
  //      triangular factors (columns 0-31, M = 64: lanes 0-15 V, 32-47 SA; columns 0-15 =
  //      . DY^T, 16-31 = . DSA^T); the column products (columns 64-127, M = 128: rows 0-63
  //      S0^T, 64-127 Gc^T; columns 64-79 . V^T, 80-95 . SA^T, 96-111 . DY^T, 112-127 . DSA^T)
  if (tid == 0) {
    mma(tb + 48, desc_k16(sa_ + OFF_PA), desc_mn(sa_ + OFF_MA, 8192, 0), idesc(128, 16, 0, 1), true);
#pragma unroll
    for (int ks = 0; ks < 4; ++ks)
      mma(tb, desc_k(sa_ + OFF_V, ks), desc_k(sa_ + OFF_DY, ks), idesc(64, 32, 0, 0), ks > 0);
#pragma unroll
    for (int ks = 0; ks < 4; ++ks)
      mma(tb + 64, desc_mn(sa_ + OFF_S0, OFF_GC - OFF_S0, ks), desc_k(sa_ + OFF_V, ks), idesc(128, 64, 1, 0), ks > 0);
    commit(bar_mma);
  }
  if (!cta_wait(args.status, bar_mma, par ^ 1u)) return -1;
  tmem_fence_after_sync();

  // ---- phase 4: U0 = triu(V DY^T), U1 = triu(V DSA^T, 1) into [U0 | U1] rows p; U2 =
  //      triu(SA DY^T), U3 = triu(SA DSA^T, 1) into [U2 | U3]; dv out
  if (warp < 2) {
    float v[32];
    ld16(tq, *reinterpret_cast<float(*)[16]>(&v[0]));
    ld16(tq + 16, *reinterpret_cast<float(*)[16]>(&v[16]));
    tmem_wait_ld();
    if (lane < 16) {
      const int p = lane;
      uint32_t pk[16];
#pragma unroll
      for (int q = 0; q < 16; q += 2) {
        pk[q / 2] = pack_bf16(q >= p ? v[q] : 0.f, q + 1 >= p ? v[q + 1] : 0.f);
        pk[8 + q / 2] = pack_bf16(q > p ? v[16 + q] : 0.f, q + 1 > p ? v[16 + q + 1] : 0.f);
      }
      unsigned char* dst = sb + (warp == 0 ? OFF_UA : OFF_UB);
#pragma unroll
      for (int c = 0; c < 4; ++c)
        *reinterpret_cast<uint4*>(dst + swz(p, 8 * c)) = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
    }
  } else if (warp >= 6) {  // dv (rows 64-127 = i, columns 48-63)
    const int i = lane + 32 * (warp & 1);
    float v[16];
    ld16(tq + 48, v);
    tmem_wait_ld();
#pragma unroll
    for (int t = 0; t < kL; ++t)
      if (t < len && in_extent(args.status, args.ext.dv, args.dv + base + (size_t)t * vstep + i))
        args.dv[base + (size_t)t * vstep + i] = v[t];
  }
  to_mma_sync();

  // ---- round 5: the triangular terms. Columns 0-31 (rows 64-127): (U0 R^ + U1 A^)^T and
  //      (U2 R^ + U3 A^)^T; columns 32-63 (rows 0-63): (U0^T K~ + U2^T B~)^T and
  //      (U1^T K~ + U3^T B~)^T
  if (tid == 0) {
    mma(tb, desc_mn(sa_ + OFF_KT, OFF_RH - OFF_KT, 0), desc_k(sa_ + OFF_UA, 0), idesc(128, 32, 1, 0), false);
    mma(tb, desc_mn(sa_ + OFF_BT, OFF_AH - OFF_BT, 0), desc_k(sa_ + OFF_UA, 1), idesc(128, 32, 1, 0), true);
    mma(tb + 32, desc_mn(sa_ + OFF_KT, OFF_RH - OFF_KT, 0), desc_mn(sa_ + OFF_UA, 8192, 0), idesc(128, 32, 1, 1), false);
    mma(tb + 32, desc_mn(sa_ + OFF_BT, OFF_AH - OFF_BT, 0), desc_mn(sa_ + OFF_UB, 8192, 0), idesc(128, 32, 1, 1), true);
    commit(bar_mma);
  }
  if (!cta_wait(args.status, bar_mma, par)) return -1;
  tmem_fence_after_sync();

  // ---- E: the gradients, thread = column j, warp w and w + 4 take steps 0-7 and 8-15;
  //      warps 2, 3, 6, 7 dk, db (rows 64-127), warps 0, 1, 4, 5 dr, da (rows 0-63); and the
  //      chunk's parts of the dw anchors over those steps (anc [grp][half][64]):
  //      end   c(L) sum_t (k V Gc + b SA Gc) / c        start  sum_t (r c DY S0 + a c(t-1) DSA S0)
  float* XK = reinterpret_cast<float*>(sb + OFF_XK);  // [t][j]: -k dk - b db
  float* XR = XK + kL * kN;                          // r dr + a da
  float* XA = XR + kL * kN;                          // a da
  {
    const int j = lane + 32 * (warp & 1), h = warp >> 2, tbeg = 8 * h;
    float p0[8], p1[8], y0[8], y1[8];
    // c(t) of this column for the steps tbeg - 1 .. tbeg + 7, as the forming warps formed it
    float cc[9];
    cc[0] = h ? c7s[j] : 1.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int t = tbeg + e;
      const float w = t < len ? decay_value<kLogit>(__bfloat162float(
                                    *reinterpret_cast<const bf16_t*>(raw + RAW_W * 0x800 + rowo(t, j))))
                              : 1.f;
      cc[e + 1] = cc[e] * w;
    }
    if (warp & 2) {  // dk, db
      ld8(tq + 64 + tbeg, p0);  // (V Gc)^T
      ld8(tq + 80 + tbeg, p1);  // (SA Gc)^T
      ld8(tq + tbeg, y0);
      ld8(tq + 16 + tbeg, y1);
      tmem_wait_ld();
      const float cl = cLs[j];
      float an = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int t = tbeg + e;
        const float ic = rcp_approx(cc[e + 1]);
        const float kv = bfs(raw + RAW_K * 0x800, rowo(t, j)), bv = bfs(raw + RAW_B * 0x800, rowo(t, j));
        an = fmaf(kv * ic, p0[e], fmaf(bv * ic, p1[e], an));
        const float dk = fmaf(cl, p0[e], y0[e]) * ic, db = fmaf(cl, p1[e], y1[e]) * ic;
        XK[t * kN + j] = -kv * dk - bv * db;
        if (t < len) {
          const size_t o = base + (size_t)t * vstep + j;
          if (in_extent(args.status, args.ext.dk, args.dk + o)) args.dk[o] = dk;
          if (in_extent(args.status, args.ext.db, args.db + o)) args.db[o] = db;
        }
      }
      anc[(2 + h) * kN + j] = cl * an;
    } else {  // dr, da
      ld8(tq + 96 + tbeg, p0);   // (DY S0)^T
      ld8(tq + 112 + tbeg, p1);  // (DSA S0)^T
      ld8(tq + 32 + tbeg, y0);
      ld8(tq + 48 + tbeg, y1);
      tmem_wait_ld();
      float an = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int t = tbeg + e;
        const float c = cc[e + 1], cp = cc[e];
        const float rv = bfs(raw + RAW_R * 0x800, rowo(t, j)), av = bfs(raw + RAW_A * 0x800, rowo(t, j));
        an = fmaf(rv * c, p0[e], fmaf(av * cp, p1[e], an));
        const float dr = (p0[e] + y0[e]) * c, da = (p1[e] + y1[e]) * cp;
        const float ad = av * da;
        XR[t * kN + j] = fmaf(rv, dr, ad);
        XA[t * kN + j] = ad;
        if (t < len) {
          const size_t o = base + (size_t)t * vstep + j;
          if (in_extent(args.status, args.ext.dr, args.dr + o)) args.dr[o] = dr;
          if (in_extent(args.status, args.ext.da, args.da + o)) args.da[o] = da;
        }
      }
      anc[h * kN + j] = an;
    }
  }
  __syncthreads();
  // w dw from the identity, anchored where fewer terms are summed; thread (column, quarter
  // of the steps q), the quarters' partial sums of x taken from the steps between:
  //   t < 8:  colsum(carry at the chunk start o S0) - sum_{u<t} x(u) - a(t) da(t)
  //   t >= 8: sum_{u>=t} x(u) - a(t) da(t) + colsum(carry at the chunk end o S(L))
  {
    const int col = tid & 63, q = tid >> 6, upper = q >> 1;
    float eg = 0.f;
#pragma unroll
    for (int w8 = 0; w8 < 8; ++w8) eg += Epart[w8 * kN + col];
    const float cge = cLs[col] * eg;
    float run = cge + anc[2 * upper * kN + col] + anc[(2 * upper + 1) * kN + col];
    if (q == 1) {
#pragma unroll
      for (int u = 0; u < 4; ++u) run -= XK[u * kN + col] + XR[u * kN + col];
    } else if (q == 2) {
#pragma unroll
      for (int u = 12; u < kL; ++u) run += XK[u * kN + col] + XR[u * kN + col];
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int t = upper ? 4 * q + 3 - e : 4 * q + e;
      const float x = XK[t * kN + col] + XR[t * kN + col];
      if (upper) run += x;
      const float wraw = bfs(raw + RAW_W * 0x800, rowo(t, col));
      float v;
      if constexpr (kLogit)
        v = logit_grad_from_wdw(run - XA[t * kN + col], wraw);
      else
        v = (run - XA[t * kN + col]) * rcp_approx(wraw);
      if (t < len && in_extent(args.status, args.ext.dw, args.dw + base + (size_t)t * vstep + col))
        args.dw[base + (size_t)t * vstep + col] = v;
      if (!upper) run -= x;
    }
  }
  return 1;
}

template <bool kLogit>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) wkv7_bwd4_tc_kernel(const __grid_constant__ BwdArgs args, int ntasks) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sb = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sb + OFF_BAR);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sb + OFF_BAR + 16);
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(bars, 2);  // loads: two arrivals per task (v, dy, carry; the rows)
    mbar_init(bars + 1, 1);
    fence_mbar_init();
#pragma unroll
    for (int v = 0; v < 7; ++v) prefetch_tensormap(&args.swmap[v]);
    prefetch_tensormap(&args.gcmap);
  }
  if (warp == 0) tmem_alloc(tslot, kTmemCols);
  tmem_fence_before_sync();
  __syncthreads();
  tmem_fence_after_sync();
  const uint32_t tb = *tslot;
  // Persistent: this CTA takes tasks blockIdx.x, + gridDim.x, ...
  int ld_it = 0, mma_it = 0;
  for (int task = blockIdx.x; task < ntasks; task += gridDim.x) {
    const int r = body<kLogit>(sb, tb, args, task, ld_it, mma_it);
    if (r < 0) break;
    ld_it += 1;
    mma_it += r;
    // every thread's reads of this task's tiles are ordered before the next task's TMA
    // writes (another proxy) land in them
    fence_proxy_async_smem();
    __syncthreads();
  }
  tmem_fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tb, kTmemCols);
}

}  // namespace tcout

}  // namespace

size_t bwd4_workspace_bytes(int B, int T, int H, bool bf16) {
  const size_t nchunks = ((size_t)T + kL - 1) / kL, heads = (size_t)B * H;
  return heads * nchunks * kN * kN * (bf16 ? sizeof(__nv_bfloat16) : sizeof(float));
}

template <bool kLogit, bool kEpi>
cudaError_t launch_bwd4_impl(const BwdArgs& args, cudaStream_t stream) {
  const size_t smem_c = sizeof(CarrySmem), smem_o = sizeof(OutSmem) + (kEpi ? sizeof(OutEpiSmem) : 0);
  cudaError_t e = cudaFuncSetAttribute(wkv7_bwd4_carry_kernel<bf16_t, kLogit, kEpi>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_c);
  if (e != cudaSuccess) return e;
  const unsigned heads = (unsigned)(args.B * args.H), nchunks = (unsigned)((args.T + kL - 1) / kL);
  wkv7_bwd4_carry_kernel<bf16_t, kLogit, kEpi><<<heads, kCarryThreads, smem_c, stream>>>(args);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (args.out_kernel != 1 || kEpi) {
    e = cudaFuncSetAttribute(wkv7_bwd4_out_kernel<kLogit, kEpi>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem_o);
    if (e != cudaSuccess) return e;
    wkv7_bwd4_out_kernel<kLogit, kEpi><<<heads * nchunks, kThreads, smem_o, stream>>>(args);
    return cudaGetLastError();
  }
  e = cudaFuncSetAttribute(tcout::wkv7_bwd4_tc_kernel<kLogit>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)tcout::kSmemBytes);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const unsigned ntasks = heads * nchunks, grid = std::min<unsigned>(ntasks, (unsigned)tcout::kCtasPerSm * (unsigned)sms);
  tcout::wkv7_bwd4_tc_kernel<kLogit><<<grid, tcout::kThreads, tcout::kSmemBytes, stream>>>(args, (int)ntasks);
  return cudaGetLastError();
}

// fp32 inputs: the carry chain alone, in split bf16, storing fp32 carries.
cudaError_t launch_bwd4_carry_f32(const BwdArgs& args, cudaStream_t stream) {
  const size_t smem = sizeof(CarrySmemT<float>);
  static_assert(sizeof(CarrySmemT<float>) <= 227 * 1024, "shared memory over budget");
  cudaError_t e = cudaFuncSetAttribute(wkv7_bwd4_carry_kernel<float, false, false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  wkv7_bwd4_carry_kernel<float, false, false><<<(unsigned)(args.B * args.H), kCarryThreads, smem, stream>>>(args);
  return cudaGetLastError();
}

cudaError_t launch_bwd4(const BwdArgs& args, cudaStream_t stream) {
  if (args.epilogue)
    return args.w_logit ? launch_bwd4_impl<true, true>(args, stream) : launch_bwd4_impl<false, true>(args, stream);
  return args.w_logit ? launch_bwd4_impl<true, false>(args, stream) : launch_bwd4_impl<false, false>(args, stream);
}

}  // namespace wkv7
