// WKV7 backward-through-time for fp32 inputs (sm_103a), N = 64, 16-step
// checkpoints: the per-chunk output pass of the split backward.
//
// Same result as "rx_pretrain.c", rx_wkv7_backward (the reverse scan of its
// equations (1)-(3)). The carry kernel (wkv7_bwd4.cu, fp32 instantiation) has
// stored Gc, the gradient w.r.t. the state after each chunk, in fp32; with it
// and the chunk's checkpoint S0, every chunk's gradients follow from its own
// inputs (the chunked algebra of the fused backward, wkv7_bwd3.cu):
//   SA  = T (A^ S0^T + Mka V),  DSA = T^T (Bb Gc^T + Mbr^T DY)
//   DV  = Kb Gc^T + Mkr^T DY + Mka^T DSA
//   DK~ = (V Gc) diag(c(L)) + triu(V DY^T) R^ + triu(V DSA^T, 1) A^,   dk = DK~ / c
//   DB~ = (SA Gc) diag(c(L)) + triu(SA DY^T) R^ + triu(SA DSA^T, 1) A^, db = DB~ / c
//   DR^ = DY S0 + tril(DY V^T) K~ + tril(DY SA^T) B~,                   dr = DR^ c
//   DA^ = DSA S0 + tril(DSA V^T, -1) K~ + tril(DSA SA^T, -1) B~,        da = DA^ c(t-1)
// and dw from w(t) dw(t) = start - sum_{u<t} x(u) - a(t) da(t)
//                        = sum_{u>=t} x(u) - a(t) da(t) + end,
// x = r dr - k dk - b db + a da, with the two anchors taken from the chunk's
// own column products (E = colsum(Gc o S0)):
//   start = colsum(carry at the chunk start o S0) = c(L) E + colsum(R^ o (DY S0) + A^ o (DSA S0))
//   end   = colsum(Gc o S(L))                     = c(L) E + colsum(Kb o (V Gc) + Bb o (SA Gc))
// (S(L) = S0 diag(c(L)) + V^T Kb + SA^T Bb, and the carry at the chunk start
// = Gc diag(c(L)) + DY^T R^ + DSA^T A^). The first form is taken for the
// first 8 steps, the second for the last 8.
//
// Every product runs on the tensor cores (mma.sync m16n8k8) in split tf32:
// three tf32 products per fp32 product (wkv7_mma.cuh, mma_x), fp32
// accumulation; the decay scaling, T and the sums are fp32.
//
// One CTA of 256 threads per (b, h, chunk) task, tasks strided over the grid.
// Per task: the chunk's rows, checkpoint and carry arrive by cp.async; warps
// 4..7 form the scaled operands, the L x L products, T and triu(V DY^T);
// warps 0..3 meanwhile take colsum(Gc o S0), then make SA, DSA and DV; all
// eight warps then make dk, db, dr, da and dw, 16 columns per warp pair.
// A chunk whose decays leave [1/16, 16] (or hold a NaN) runs step by step in
// fp32 (warps 0..3).
#include "wkv7_launch.h"
#include "wkv7_mma.cuh"
#include "wkv7_scaled.cuh"

namespace wkv7 {
namespace {

constexpr int kN = 64, kL = 16;
constexpr int kLD64 = 72;  // row stride of 64-wide operands read along k
constexpr int kLD16 = 24;  // row stride of 16-wide operands
constexpr int kLDT = 68;   // row stride of operands read only as [k][n] B operands
constexpr int kLDS = 72;   // row stride of the checkpoint
constexpr int kThreads = 256;
constexpr int kTile = kL * kN;
enum { V_R = 0, V_W = 1, V_K = 2, V_V = 3, V_A = 4, V_B = 5, V_DY = 6 };

// Operands of the chunk (fp32 values), formed by warps 4..7.
struct OpF {
  float Ah[kL * kLD64], Rh[kL * kLD64], Kt[kL * kLD64], Bt[kL * kLD64];  // [t][j]
  float Kb[kL * kLD64], Bb[kL * kLD64], Vs[kL * kLD64], DYs[kL * kLD64];  // [t][j], V and DY [t][i]
  float Ah68[kL * kLDT], Rh68[kL * kLDT];  // A^ and R^ again (read only as [k][n] B operands)
  float cS[kTile];                        // c(t) [t][j]
  float cL[kN];
  float M[3][kL * kLD16];  // Mka (strictly lower), Mkr, Mbr (lower)   [t][s]
  float Tinv[kL * kLD16];  // (I - Mba)^-1                            [t][s]
  float TinvT[kL * kLD16];
  float U0[kL * kLD16];    // triu(V DY^T)                            [t][s]
  int unsafe;
  int pad_[3];
};

// A chunk's inputs: its rows, checkpoint and carry (two sets: the next task's arrive while
// the current one is processed).
struct InF32 {
  float raw[7][kTile];   // r, w, k, v, a, b, dy of the chunk [t][j], zero past the sequence
  float GcS[kN * kLDT];  // the carry after the chunk [i][j]; in the output phase, the dw exchange
  float S0s[kN * kLDS];  // the checkpoint [i][j]
};

struct OutF32Smem {
  InF32 in[2];
  OpF op;
  float U[3][kL * kLD16];                    // triu(V DSA^T, 1), triu(SA DY^T), triu(SA DSA^T, 1)
  float SAs[kL * kLD64], DSAs[kL * kLD64];  // sa(t), dsa(t) [t][i]
  float Epart[4][kN];                       // colsum(Gc o S0) over each state warp's rows
  float anc[2][kN];                         // colsum(R^ o DY S0 + A^ o DSA S0), colsum(Kb o V Gc + Bb o SA Gc)
};

template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ float quad_sum(float x) {
  x += __shfl_xor_sync(0xffffffffu, x, 1);
  return x + __shfl_xor_sync(0xffffffffu, x, 2);
}
__device__ __forceinline__ float col_sum(float x) {  // over the 8 row groups g of the warp
  x += __shfl_xor_sync(0xffffffffu, x, 4);
  x += __shfl_xor_sync(0xffffffffu, x, 8);
  return x + __shfl_xor_sync(0xffffffffu, x, 16);
}
__device__ __forceinline__ float2 f2at(const float* p) { return *reinterpret_cast<const float2*>(p); }

// Scaled operands (128 threads; thread (j, half) forms column j of steps
// 8 half .. 8 half + 7). Returns, uniformly over the 128 threads, whether
// some decay leaves the range of the scaled form.
__device__ bool prep_f32(const float* rs, OpF& op, int len, int ptid) {
  const int j = ptid & 63, half = ptid >> 6;
  float wm[8], wo[8];
  const int tm = 8 * half, to = 8 - tm;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    wm[e] = tm + e < len ? rs[V_W * kTile + (tm + e) * kN + j] : 1.f;
    wo[e] = to + e < len ? rs[V_W * kTile + (to + e) * kN + j] : 1.f;
  }
  bool unsafe = false;
#pragma unroll
  for (int e = 0; e < 8; ++e) unsafe |= !decay_is_safe(wm[e]);
  unsafe = named_bar_or(1, 128, unsafe);
  if (unsafe) return true;
  float pm = 1.f, po = 1.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    pm *= wm[e];
    po *= wo[e];
  }
  const float cL = half ? po * pm : pm * po;
  float c = half ? po : 1.f;
  if (half == 0) op.cL[j] = cL;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const int t = tm + e, o = t * kN + j, q = t * kLD64 + j;
    const float cprev = c;
    c *= wm[e];
    const float ic = rcp_approx(c);
    const float a = rs[V_A * kTile + o], r = rs[V_R * kTile + o], k = rs[V_K * kTile + o], b = rs[V_B * kTile + o];
    const float ah = a * cprev, rh = r * c;
    op.Ah[q] = ah;
    op.Rh[q] = rh;
    op.Ah68[t * kLDT + j] = ah;
    op.Rh68[t * kLDT + j] = rh;
    op.Kt[q] = k * ic;
    op.Bt[q] = b * ic;
    const float s = cL * ic;
    op.Kb[q] = k * s;
    op.Bb[q] = b * s;
    op.Vs[q] = rs[V_V * kTile + o];
    op.DYs[q] = rs[V_DY * kTile + o];
    op.cS[o] = c;
  }
  return false;
}

// acc = P Q^T for 16-row P, Q (stride kLD64), K = 64, split tf32.
__device__ __forceinline__ void gram16(float (&acc)[2][4], const float* P, const float* Q, int g, int t4) {
  zero4(acc[0]);
  zero4(acc[1]);
#pragma unroll
  for (int kb = 0; kb < kN / 8; ++kb) {
    FragA<true> a;
    ld_a(a, P, kLD64, 0, 8 * kb, g, t4);
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      FragB<true> b;
      ld_b(b, Q, kLD64, 8 * nt, 8 * kb, g, t4);
      mma_x(acc[nt], a, b);
    }
  }
}

// A 16 x 16 accumulator stored (stride kLD16), keeping (t, s) with
// lower: s < t (+ s == t if incl); upper: s > t (+ s == t if incl).
__device__ __forceinline__ void store_masked(const float (&acc)[2][4], float* dst, bool lower, bool incl, int g,
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
      *reinterpret_cast<float2*>(dst + t * kLD16 + s) = make_float2(x[0], x[1]);
    }
}

// Warps 4..7: the operands, the masked L x L products, T and triu(V DY^T).
__device__ void front_f32(OutF32Smem& sm, const InF32& in, int len) {
  const int ptid = threadIdx.x - 128, pw = ptid >> 5, lane = threadIdx.x & 31, g = lane >> 2, t4 = lane & 3;
  OpF& op = sm.op;
  const bool unsafe = prep_f32(&in.raw[0][0], op, len, ptid);
  if (ptid == 0) op.unsafe = unsafe;
  if (unsafe) return;
  named_bar(1, 128);
  float acc[2][4];
  const int mt = pw >> 1, nb = pw & 1;
  zero4(acc[0]);
  zero4(acc[1]);
#pragma unroll
  for (int kb = 0; kb < kN / 8; ++kb) {
    FragA<true> a;
    ld_a(a, mt ? op.Rh : op.Ah, kLD64, 0, 8 * kb, g, t4);
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      FragB<true> b;
      ld_b(b, nb ? op.Bt : op.Kt, kLD64, 8 * nt, 8 * kb, g, t4);
      mma_x(acc[nt], a, b);
    }
  }
  // Mba goes to U1's tile, which is free until the output phase
  store_masked(acc, pw == 1 ? sm.U[0] : op.M[pw == 0 ? 0 : pw - 1], true, mt == 1, g, t4);
  if (pw == 1) {  // T = (I - Mba)^-1, lane s < 16 owns column s
    __syncwarp();
    const float* Mba = sm.U[0];
    const int s = lane & 15;
    float col[kL];
#pragma unroll
    for (int t = 0; t < kL; ++t) {
      float x = t == s ? 1.f : 0.f;
#pragma unroll
      for (int u = 0; u < t; ++u) x = fmaf(Mba[t * kLD16 + u], col[u], x);
      col[t] = x;
    }
    if (lane < 16) {
#pragma unroll
      for (int t = 0; t < kL; ++t) {
        op.Tinv[t * kLD16 + s] = col[t];
        op.TinvT[s * kLD16 + t] = col[t];
      }
    }
  } else if (pw == 2) {  // U0 = triu(V DY^T)
    gram16(acc, op.Vs, op.DYs, g, t4);
    store_masked(acc, op.U0, false, true, g, t4);
  }
}

struct OutPtrs {
  const BwdArgs* a;
  size_t base;   // element offset of (b, t0, h, 0)
  size_t vstep;  // elements between consecutive steps
};

__device__ __forceinline__ void put(const BwdArgs& a, float* dst, const Extent& x, size_t off, float v) {
  float* p = dst + off;
  if (in_extent(a.status, x, p)) *p = v;
}

// Step-by-step reverse scan of the chunk (warps 0..3, fp32): the carry G
// starts at Gc, S_prev of step t is recomputed from the checkpoint.
__device__ void direct_f32(OutF32Smem& sm, const InF32& in, int len, const OutPtrs& o, float (&G)[8][4], int warp,
                           int lane) {
  const BwdArgs& a = *o.a;
  const int g = lane >> 2, t4 = lane & 3, i0 = 16 * warp, tid = threadIdx.x;
  const float* rs = &in.raw[0][0];
  const float* S0 = in.S0s;
  float* red = sm.SAs;  // [4 warps][5][64], in SAs and DSAs (unused by a direct chunk)
  for (int t = len - 1; t >= 0; --t) {
    float sp[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const int col = 8 * nt + 2 * t4;
      const float2 lo = f2at(S0 + (i0 + g) * kLDS + col), hi = f2at(S0 + (i0 + g + 8) * kLDS + col);
      sp[nt][0] = lo.x;
      sp[nt][1] = lo.y;
      sp[nt][2] = hi.x;
      sp[nt][3] = hi.y;
    }
    float sa0 = 0.f, sa1 = 0.f;
    for (int u = 0; u <= t; ++u) {
      const float* row = rs + u * kN;
      float s0 = 0.f, s1 = 0.f;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const float2 av = f2at(row + V_A * kTile + 8 * nt + 2 * t4);
        s0 = fmaf(sp[nt][0], av.x, fmaf(sp[nt][1], av.y, s0));
        s1 = fmaf(sp[nt][2], av.x, fmaf(sp[nt][3], av.y, s1));
      }
      sa0 = quad_sum(s0);
      sa1 = quad_sum(s1);
      if (u == t) break;  // sp = S_prev(t), sa = sa(t)
      const float v0 = row[V_V * kTile + i0 + g], v1 = row[V_V * kTile + i0 + g + 8];
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const int col = 8 * nt + 2 * t4;
        const float2 w = f2at(row + V_W * kTile + col), k = f2at(row + V_K * kTile + col),
                     b = f2at(row + V_B * kTile + col);
        sp[nt][0] = fmaf(sa0, b.x, fmaf(sp[nt][0], w.x, v0 * k.x));
        sp[nt][1] = fmaf(sa0, b.y, fmaf(sp[nt][1], w.y, v0 * k.y));
        sp[nt][2] = fmaf(sa1, b.x, fmaf(sp[nt][2], w.x, v1 * k.x));
        sp[nt][3] = fmaf(sa1, b.y, fmaf(sp[nt][3], w.y, v1 * k.y));
      }
    }
    const float* row = rs + t * kN;
    const float v0 = row[V_V * kTile + i0 + g], v1 = row[V_V * kTile + i0 + g + 8];
    const float dy0 = row[V_DY * kTile + i0 + g], dy1 = row[V_DY * kTile + i0 + g + 8];
    // column partials: dr (from S_t), then G += dy r^T, dk, db, dw; row sums dv, dsa
    float pr[8][2], pk[8][2], pb[8][2], pwv[8][2];
    float dv0 = 0.f, dv1 = 0.f, ds0 = 0.f, ds1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const int col = 8 * nt + 2 * t4;
      const float2 w = f2at(row + V_W * kTile + col), k = f2at(row + V_K * kTile + col);
      const float2 b = f2at(row + V_B * kTile + col), r = f2at(row + V_R * kTile + col);
      const float wv[2] = {w.x, w.y}, kv[2] = {k.x, k.y}, bv[2] = {b.x, b.y}, rv[2] = {r.x, r.y};
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float st0 = fmaf(sa0, bv[e], fmaf(sp[nt][e], wv[e], v0 * kv[e]));
        const float st1 = fmaf(sa1, bv[e], fmaf(sp[nt][2 + e], wv[e], v1 * kv[e]));
        pr[nt][e] = fmaf(st0, dy0, st1 * dy1);
        G[nt][e] = fmaf(dy0, rv[e], G[nt][e]);
        G[nt][2 + e] = fmaf(dy1, rv[e], G[nt][2 + e]);
        pk[nt][e] = fmaf(G[nt][e], v0, G[nt][2 + e] * v1);
        pb[nt][e] = fmaf(G[nt][e], sa0, G[nt][2 + e] * sa1);
        pwv[nt][e] = fmaf(G[nt][e], sp[nt][e], G[nt][2 + e] * sp[nt][2 + e]);
        dv0 = fmaf(G[nt][e], kv[e], dv0);
        dv1 = fmaf(G[nt][2 + e], kv[e], dv1);
        ds0 = fmaf(G[nt][e], bv[e], ds0);
        ds1 = fmaf(G[nt][2 + e], bv[e], ds1);
      }
    }
    dv0 = quad_sum(dv0);
    dv1 = quad_sum(dv1);
    ds0 = quad_sum(ds0);
    ds1 = quad_sum(ds1);
    if (t4 == 0) {
      put(a, a.dv, a.ext.dv, o.base + (size_t)t * o.vstep + i0 + g, dv0);
      put(a, a.dv, a.ext.dv, o.base + (size_t)t * o.vstep + i0 + g + 8, dv1);
    }
    // da = S_prev^T dsa; carry G <- G diag(w) + dsa a^T; column sums to shared memory
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const int col = 8 * nt + 2 * t4;
      const float2 w = f2at(row + V_W * kTile + col), av = f2at(row + V_A * kTile + col);
      const float wv[2] = {w.x, w.y}, aa[2] = {av.x, av.y};
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float pa = fmaf(sp[nt][e], ds0, sp[nt][2 + e] * ds1);
        G[nt][e] = fmaf(ds0, aa[e], G[nt][e] * wv[e]);
        G[nt][2 + e] = fmaf(ds1, aa[e], G[nt][2 + e] * wv[e]);
        const float sums[5] = {col_sum(pr[nt][e]), col_sum(pk[nt][e]), col_sum(pb[nt][e]), col_sum(pwv[nt][e]),
                               col_sum(pa)};
        if (g == 0) {
#pragma unroll
          for (int q = 0; q < 5; ++q) red[(warp * 5 + q) * kN + col + e] = sums[q];
        }
      }
    }
    named_bar(2, 128);
    for (int idx = tid; idx < 5 * kN; idx += 128) {
      const int q = idx / kN, col = idx % kN;
      const float x = red[q * kN + col] + red[(5 + q) * kN + col] + red[(10 + q) * kN + col] + red[(15 + q) * kN + col];
      float* dst = q == 0 ? a.dr : q == 1 ? a.dk : q == 2 ? a.db : q == 3 ? a.dw : a.da;
      const Extent& xe = q == 0 ? a.ext.dr : q == 1 ? a.ext.dk : q == 2 ? a.ext.db : q == 3 ? a.ext.dw : a.ext.da;
      put(a, dst, xe, o.base + (size_t)t * o.vstep + col, x);
    }
    named_bar(2, 128);
  }
}

// Warps 0..3: SA, DSA (to shared memory) and dv of the chunk (rows i0 .. i0+15).
__device__ void state_f32(OutF32Smem& sm, const InF32& in, const float (&G)[8][4], int len, const OutPtrs& o, int warp,
                          int lane) {
  const BwdArgs& a = *o.a;
  const int g = lane >> 2, t4 = lane & 3, i0 = 16 * warp;
  const OpF& op = sm.op;
  float RSA[2][4], RDSA[2][4], DV[2][4];
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    zero4(RSA[q]);
    zero4(RDSA[q]);
    zero4(DV[q]);
  }
#pragma unroll
  for (int kb = 0; kb < 8; ++kb) {
    FragA<true> aS, aG;
    ld_a(aS, in.S0s, kLDS, i0, 8 * kb, g, t4);
    acc_to_a(aG, G[kb]);
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      FragB<true> b;
      ld_b(b, op.Ah, kLD64, 8 * q, 8 * kb, g, t4);
      mma_x(RSA[q], aS, b);
      ld_b(b, op.Bb, kLD64, 8 * q, 8 * kb, g, t4);
      mma_x(RDSA[q], aG, b);
      ld_b(b, op.Kb, kLD64, 8 * q, 8 * kb, g, t4);  // dv^T: Gc Kb^T
      mma_x(DV[q], aG, b);
    }
  }
  FragA<true> aV[2], aD[2];
#pragma unroll
  for (int kb = 0; kb < 2; ++kb) {
    ld_a_t(aV[kb], op.Vs, kLD64, i0, 8 * kb, g, t4);    // V^T
    ld_a_ts(aD[kb], op.DYs, kLD64, i0, 8 * kb, g, t4);  // DY^T (hardware k order)
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      FragB<true> b;
      ld_b(b, op.M[0], kLD16, 8 * q, 8 * kb, g, t4);  // + V^T Mka^T
      mma_x(RSA[q], aV[kb], b);
      ld_b_ts(b, op.M[2], kLD16, 8 * q, 8 * kb, g, t4);  // + DY^T Mbr
      mma_x(RDSA[q], aD[kb], b);
    }
  }
  float SA[2][4], DSA[2][4];
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    zero4(SA[q]);
    zero4(DSA[q]);
  }
#pragma unroll
  for (int kb = 0; kb < 2; ++kb) {
    FragA<true> a1, a2;
    acc_to_a(a1, RSA[kb]);
    acc_to_a(a2, RDSA[kb]);
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      FragB<true> b;
      ld_b(b, op.Tinv, kLD16, 8 * q, 8 * kb, g, t4);  // SA^T = RSA T^T
      mma_x(SA[q], a1, b);
      ld_b(b, op.TinvT, kLD16, 8 * q, 8 * kb, g, t4);  // DSA^T = RDSA T
      mma_x(DSA[q], a2, b);
    }
  }
  FragA<true> aDS[2];
  acc_to_a(aDS[0], DSA[0]);
  acc_to_a(aDS[1], DSA[1]);
  // dv^T (rows i, columns t) += DY^T Mkr + DSA^T Mka
#pragma unroll
  for (int kb = 0; kb < 2; ++kb)
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      FragB<true> b;
      ld_b_ts(b, op.M[1], kLD16, 8 * q, 8 * kb, g, t4);
      mma_x(DV[q], aD[kb], b);
      ld_b_t(b, op.M[0], kLD16, 8 * q, 8 * kb, g, t4);
      mma_x(DV[q], aDS[kb], b);
    }
#pragma unroll
  for (int q = 0; q < 2; ++q)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int t = 8 * q + 2 * t4 + e;
      if (t < len) {
        put(a, a.dv, a.ext.dv, o.base + (size_t)t * o.vstep + i0 + g, DV[q][e]);
        put(a, a.dv, a.ext.dv, o.base + (size_t)t * o.vstep + i0 + g + 8, DV[q][2 + e]);
      }
    }
#pragma unroll
  for (int q = 0; q < 2; ++q)
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int i = i0 + g + 8 * h, t = 8 * q + 2 * t4 + e;
        sm.SAs[t * kLD64 + i] = SA[q][2 * h + e];
        sm.DSAs[t * kLD64 + i] = DSA[q][2 * h + e];
      }
}

// All eight warps: dk, db (warps 0..3), dr, da (warps 4..7) and dw. Warp
// (grp, jb) covers columns j0 .. j0+15, j0 = 16 jb.
__device__ void outputs_f32(OutF32Smem& sm, InF32& in, int len, const OutPtrs& o) {
  const BwdArgs& a = *o.a;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t4 = lane & 3;
  const int grp = warp >> 2, jb = warp & 3, j0 = 16 * jb;
  const OpF& op = sm.op;
  if (grp == 1 && jb < 3) {  // U1 = triu(V DSA^T, 1), U2 = triu(SA DY^T), U3 = triu(SA DSA^T, 1)
    float acc[2][4];
    gram16(acc, jb == 0 ? op.Vs : sm.SAs, jb == 1 ? op.DYs : sm.DSAs, g, t4);
    store_masked(acc, sm.U[jb], false, jb == 1, g, t4);
  }
  // sums over the rows i: V Gc, SA Gc (grp 0); DY S0, DSA S0 (grp 1)
  float P0[2][4], P1[2][4];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    zero4(P0[nt]);
    zero4(P1[nt]);
  }
  const float* Bm = grp ? in.S0s : in.GcS;
  const int ldb = grp ? kLDS : kLDT;
#pragma unroll
  for (int kb = 0; kb < 8; ++kb) {
    FragA<true> a0, a1;
    ld_a(a0, grp ? op.DYs : op.Vs, kLD64, 0, 8 * kb, g, t4);
    ld_a(a1, grp ? sm.DSAs : sm.SAs, kLD64, 0, 8 * kb, g, t4);
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      FragB<true> b;
      ld_b_t(b, Bm, ldb, j0 + 8 * nt, 8 * kb, g, t4);
      mma_x(P0[nt], a0, b);
      mma_x(P1[nt], a1, b);
    }
  }
  // the anchors' column sums over the steps: grp 1 colsum(R^ o DY S0 + A^ o DSA S0),
  // grp 0 colsum(Kb o V Gc + Bb o SA Gc)
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int col = j0 + 8 * nt + 2 * t4 + e;
      const float* X0 = grp ? op.Rh : op.Kb;
      const float* X1 = grp ? op.Ah : op.Bb;
      float s = 0.f;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int t = g + 8 * h;
        s = fmaf(X0[t * kLD64 + col], P0[nt][2 * h + e], fmaf(X1[t * kLD64 + col], P1[nt][2 * h + e], s));
      }
      s = col_sum(s);
      if (g == 0) sm.anc[grp ? 0 : 1][col] = s;
    }
  __syncthreads();  // U1..U3 and the anchors complete; every read of GcS done
  // triangular terms (U0 = triu(V DY^T), U1 = triu(V DSA^T, 1), U2 = triu(SA DY^T), U3 = triu(SA DSA^T, 1)):
  //   dk~ = (V Gc) c(L) + U0 R^ + U1 A^        db~ = (SA Gc) c(L) + U2 R^ + U3 A^
  //   dr^ = DY S0 + U0^T K~ + U2^T B~          da^ = DSA S0 + U1^T K~ + U3^T B~
  const float* Uq[4] = {op.U0, sm.U[0], sm.U[1], sm.U[2]};
  if (grp == 0) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const float2 cl = f2at(op.cL + j0 + 8 * nt + 2 * t4);
      P0[nt][0] *= cl.x;
      P0[nt][1] *= cl.y;
      P0[nt][2] *= cl.x;
      P0[nt][3] *= cl.y;
      P1[nt][0] *= cl.x;
      P1[nt][1] *= cl.y;
      P1[nt][2] *= cl.x;
      P1[nt][3] *= cl.y;
    }
#pragma unroll
    for (int kb = 0; kb < 2; ++kb) {
      FragA<true> u0, u1, u2, u3;
      ld_a(u0, Uq[0], kLD16, 0, 8 * kb, g, t4);
      ld_a(u1, Uq[1], kLD16, 0, 8 * kb, g, t4);
      ld_a(u2, Uq[2], kLD16, 0, 8 * kb, g, t4);
      ld_a(u3, Uq[3], kLD16, 0, 8 * kb, g, t4);
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        FragB<true> b;
        ld_b_t(b, op.Rh68, kLDT, j0 + 8 * nt, 8 * kb, g, t4);
        mma_x(P0[nt], u0, b);
        mma_x(P1[nt], u2, b);
        ld_b_t(b, op.Ah68, kLDT, j0 + 8 * nt, 8 * kb, g, t4);
        mma_x(P0[nt], u1, b);
        mma_x(P1[nt], u3, b);
      }
    }
  } else {
#pragma unroll
    for (int kb = 0; kb < 2; ++kb) {
      FragA<true> u0, u1, u2, u3;
      ld_a_ts(u0, Uq[0], kLD16, 0, 8 * kb, g, t4);
      ld_a_ts(u1, Uq[1], kLD16, 0, 8 * kb, g, t4);
      ld_a_ts(u2, Uq[2], kLD16, 0, 8 * kb, g, t4);
      ld_a_ts(u3, Uq[3], kLD16, 0, 8 * kb, g, t4);
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        FragB<true> b;
        ld_b_ts(b, op.Kt, kLD64, j0 + 8 * nt, 8 * kb, g, t4);
        mma_x(P0[nt], u0, b);
        mma_x(P1[nt], u1, b);
        ld_b_ts(b, op.Bt, kLD64, j0 + 8 * nt, 8 * kb, g, t4);
        mma_x(P0[nt], u2, b);
        mma_x(P1[nt], u3, b);
      }
    }
  }
  // unscale: dk = dk~ / c, db = db~ / c (grp 0); dr = dr^ c, da = da^ c(t-1) (grp 1); and this
  // group's part of x = r dr - k dk - b db + a da
  const float* rs = &in.raw[0][0];
  float X[2][4], AD[2][4];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int t = g + 8 * h, col = j0 + 8 * nt + 2 * t4;
      const float2 c = f2at(op.cS + t * kN + col);
      if (grp == 0) {
        const float2 k = f2at(rs + V_K * kTile + t * kN + col), b = f2at(rs + V_B * kTile + t * kN + col);
        const float ic[2] = {rcp_approx(c.x), rcp_approx(c.y)}, kv[2] = {k.x, k.y}, bv[2] = {b.x, b.y};
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          P0[nt][2 * h + e] *= ic[e];
          P1[nt][2 * h + e] *= ic[e];
          X[nt][2 * h + e] = -kv[e] * P0[nt][2 * h + e] - bv[e] * P1[nt][2 * h + e];
          AD[nt][2 * h + e] = 0.f;
        }
      } else {
        const float2 cp = t ? f2at(op.cS + (t - 1) * kN + col) : make_float2(1.f, 1.f);
        const float2 r = f2at(rs + V_R * kTile + t * kN + col), av = f2at(rs + V_A * kTile + t * kN + col);
        const float cv[2] = {c.x, c.y}, cpv[2] = {cp.x, cp.y}, rv[2] = {r.x, r.y}, aa[2] = {av.x, av.y};
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          P0[nt][2 * h + e] *= cv[e];
          P1[nt][2 * h + e] *= cpv[e];
          AD[nt][2 * h + e] = aa[e] * P1[nt][2 * h + e];
          X[nt][2 * h + e] = rv[e] * P0[nt][2 * h + e] + AD[nt][2 * h + e];
        }
      }
    }
  // exchange with the partner warp of the other group (same columns): grp 0 keeps dw of
  // n-tile 0, grp 1 of n-tile 1. The carry tile is free in this phase.
  float* XK = in.GcS;                   // grp 0's x part, [t][j] stride 72
  float* XR = in.GcS + kL * kLD64;      // grp 1's x part
  float* XA = in.GcS + 2 * kL * kLD64;  // grp 1's a da
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int t = g + 8 * h;
    if (grp == 0) {
      *reinterpret_cast<float2*>(XK + t * kLD64 + j0 + 8 + 2 * t4) = make_float2(X[1][2 * h], X[1][2 * h + 1]);
    } else {
      *reinterpret_cast<float2*>(XR + t * kLD64 + j0 + 2 * t4) = make_float2(X[0][2 * h], X[0][2 * h + 1]);
      *reinterpret_cast<float2*>(XA + t * kLD64 + j0 + 2 * t4) = make_float2(AD[0][2 * h], AD[0][2 * h + 1]);
    }
  }
  named_bar(3 + jb, 64);
  const int nw = grp, jw = j0 + 8 * nw;  // this warp's dw columns jw .. jw+7
  float xw[4], adw[4];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int t = g + 8 * h;
    if (grp == 0) {
      const float2 xr = f2at(XR + t * kLD64 + jw + 2 * t4), xa = f2at(XA + t * kLD64 + jw + 2 * t4);
      xw[2 * h] = X[0][2 * h] + xr.x;
      xw[2 * h + 1] = X[0][2 * h + 1] + xr.y;
      adw[2 * h] = xa.x;
      adw[2 * h + 1] = xa.y;
    } else {
      const float2 xk = f2at(XK + t * kLD64 + jw + 2 * t4);
      xw[2 * h] = X[1][2 * h] + xk.x;
      xw[2 * h + 1] = X[1][2 * h + 1] + xk.y;
      adw[2 * h] = AD[1][2 * h];
      adw[2 * h + 1] = AD[1][2 * h + 1];
    }
  }
  // w dw from the identity, anchored where fewer terms are summed:
  // rows t < 8: start - sum_{u<t} x(u) - a(t) da(t); rows t >= 8: sum_{u>=t} x(u) - a(t) da(t) + end
  float dw[4];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    float hi2 = xw[2 + e], lo = xw[e];
#pragma unroll
    for (int d = 1; d < 8; d <<= 1) {
      const float oh = __shfl_down_sync(0xffffffffu, hi2, 4 * d);
      const float ol = __shfl_up_sync(0xffffffffu, lo, 4 * d);
      if (g + d < 8) hi2 += oh;
      if (g >= d) lo += ol;
    }
    const int col = jw + 2 * t4 + e;
    const float ce = op.cL[col] * (sm.Epart[0][col] + sm.Epart[1][col] + sm.Epart[2][col] + sm.Epart[3][col]);
    const float start = ce + sm.anc[0][col], end = ce + sm.anc[1][col];
    const float w0 = rs[V_W * kTile + g * kN + col], w1 = rs[V_W * kTile + (g + 8) * kN + col];
    dw[e] = (start - (lo - xw[e]) - adw[e]) * rcp_approx(w0);
    dw[2 + e] = (hi2 - adw[2 + e] + end) * rcp_approx(w1);
  }
  float* out0 = grp ? a.dr : a.dk;
  float* out1 = grp ? a.da : a.db;
  const Extent& x0 = grp ? a.ext.dr : a.ext.dk;
  const Extent& x1 = grp ? a.ext.da : a.ext.db;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int t = g + 8 * h;
    if (t < len) {
      const size_t off = o.base + (size_t)t * o.vstep + j0 + 2 * t4;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        float2* p0 = reinterpret_cast<float2*>(out0 + off + 8 * nt);
        float2* p1 = reinterpret_cast<float2*>(out1 + off + 8 * nt);
        if (in_extent(a.status, x0, p0)) *p0 = make_float2(P0[nt][2 * h], P0[nt][2 * h + 1]);
        if (in_extent(a.status, x1, p1)) *p1 = make_float2(P1[nt][2 * h], P1[nt][2 * h + 1]);
      }
      float2* pw = reinterpret_cast<float2*>(a.dw + off + 8 * nw);
      if (in_extent(a.status, a.ext.dw, pw)) *pw = make_float2(dw[2 * h], dw[2 * h + 1]);
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1) wkv7_bwd4_out_f32_kernel(const __grid_constant__ BwdArgs args,
                                                                        long long ntasks) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  OutF32Smem& sm = *reinterpret_cast<OutF32Smem*>(smem_raw);
  const int T = args.T, H = args.H, nchunks = (T + kL - 1) / kL;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t4 = lane & 3;
  const size_t vstep = (size_t)H * kN;
  // The rows (zeros past T), checkpoint and carry of `task` into input set `in`, as one
  // cp.async group (empty past the last task).
  auto load = [&](InF32& in, long long task) {
    if (task < ntasks) {
      const int head = (int)(task / nchunks), n = (int)(task % nchunks), bi = head / H, hi = head % H;
      const int t0 = n * kL, len = min(kL, T - t0);
      const size_t base = ((size_t)bi * T + t0) * vstep + (size_t)hi * kN;
      const float* S0g = args.ckpt + ((size_t)head * args.nck + n) * kN * kN;
      const float* Gcg = reinterpret_cast<const float*>(args.carry) + ((size_t)head * nchunks + n) * kN * kN;
      for (int idx = tid; idx < 7 * kL * (kN / 4); idx += kThreads) {
        const int v = idx / (kL * kN / 4), t = (idx / (kN / 4)) % kL, c4 = idx % (kN / 4);
        float* dst = &in.raw[v][t * kN + 4 * c4];
        const float* src = static_cast<const float*>(args.in[v]) + base + (size_t)t * vstep + 4 * c4;
        if (t < len && in_extent(args.status, args.ext.in[v], reinterpret_cast<const float4*>(src)))
          cp_async16(dst, src);
        else
          *reinterpret_cast<float4*>(dst) = make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int q = 0; q < kN * kN / 4 / kThreads; ++q) {
        const int idx = tid + kThreads * q, r = idx >> 4, c4 = idx & 15;  // row r, columns 4 c4 ..
        if (in_extent(args.status, args.ext.ckpt, reinterpret_cast<const float4*>(S0g + 4 * idx)))
          cp_async16(in.S0s + r * kLDS + 4 * c4, S0g + 4 * idx);
        if (in_extent(args.status, args.ext.carry, reinterpret_cast<const float4*>(Gcg + 4 * idx)))
          cp_async16(in.GcS + r * kLDT + 4 * c4, Gcg + 4 * idx);
      }
    }
    cp_async_commit();
  };
  load(sm.in[0], blockIdx.x);
  int cur = 0;
  for (long long task = blockIdx.x; task < ntasks; task += gridDim.x, cur ^= 1) {
    const int head = (int)(task / nchunks), n = (int)(task % nchunks), bi = head / H, hi = head % H;
    const int t0 = n * kL, len = min(kL, T - t0);
    const OutPtrs o{&args, ((size_t)bi * T + t0) * vstep + (size_t)hi * kN, vstep};
    InF32& in = sm.in[cur];
    __syncthreads();  // the previous task is done with shared memory (and its input set)
    load(sm.in[cur ^ 1], task + gridDim.x);  // the next task's inputs, while this one runs
    cp_async_wait_group<1>();                // this task's group complete
    __syncthreads();

    // ---- warps 4..7: operands and products; warps 0..3: the carry into registers and
    //      colsum(Gc o S0) over their rows
    float G[8][4];
    if (warp >= 4) {
      front_f32(sm, in, len);
    } else {
      const int i0 = 16 * warp;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const int col = 8 * nt + 2 * t4;
        const float2 lo = f2at(in.GcS + (i0 + g) * kLDT + col), hi = f2at(in.GcS + (i0 + g + 8) * kLDT + col);
        const float2 s_lo = f2at(in.S0s + (i0 + g) * kLDS + col), s_hi = f2at(in.S0s + (i0 + g + 8) * kLDS + col);
        G[nt][0] = lo.x;
        G[nt][1] = lo.y;
        G[nt][2] = hi.x;
        G[nt][3] = hi.y;
        const float p0 = col_sum(fmaf(lo.x, s_lo.x, hi.x * s_hi.x));
        const float p1 = col_sum(fmaf(lo.y, s_lo.y, hi.y * s_hi.y));
        if (g == 0) *reinterpret_cast<float2*>(&sm.Epart[warp][col]) = make_float2(p0, p1);
      }
    }
    __syncthreads();
    const bool unsafe = sm.op.unsafe;
    // ---- warps 0..3: SA, DSA and dv (or the whole chunk step by step)
    if (warp < 4) {
      if (unsafe)
        direct_f32(sm, in, len, o, G, warp, lane);
      else
        state_f32(sm, in, G, len, o, warp, lane);
    }
    __syncthreads();
    // ---- all warps: dk, db, dr, da, dw
    if (!unsafe) outputs_f32(sm, in, len, o);
  }
  cp_async_wait_all();  // the trailing (empty) group
}

}  // namespace

cudaError_t launch_bwd4_out_f32(const BwdArgs& args, cudaStream_t stream) {
  const size_t smem = sizeof(OutF32Smem);
  static_assert(sizeof(OutF32Smem) <= 227 * 1024, "shared memory over budget");
  cudaError_t e =
      cudaFuncSetAttribute(wkv7_bwd4_out_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const long long ntasks = (long long)args.B * args.H * ((args.T + kL - 1) / kL);
  const unsigned grid = (unsigned)(ntasks < (1ll << 30) ? ntasks : (1ll << 30));
  wkv7_bwd4_out_f32_kernel<<<grid, kThreads, smem, stream>>>(args, ntasks);
  return cudaGetLastError();
}

}  // namespace wkv7
