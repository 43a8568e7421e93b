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
//  * wkv7_bwd4_carry_kernel - one CTA per (b, h), chunks in reverse: eight
//    "prep" warps form the next chunk's R^, A^, DY, T^T Bb and Mbr T while
//    four "state" warps (16 rows of Gc each, as accumulator tiles) advance
//    the carry with three small products. It stores Gc for every chunk (as
//    tf32 values) and dS_init.
//  * wkv7_bwd4_out_kernel - one CTA per (b, h, chunk), all independent: from
//    the chunk's inputs, checkpoint and stored carry it forms every gradient
//    of the chunk. Two CTAs share an SM. The dw anchors come from the
//    chunk's own column products: with S(L) = S0 diag(c(L)) + V^T Kb + SA^T Bb,
//      colsum(Gc o S(L)) = c(L) colsum(Gc o S0) + sum_t (Kb o V Gc + Bb o SA Gc)
//      colsum(Gc' o S0)  = c(L) colsum(Gc o S0) + sum_t (R^ o DY S0 + A^ o DSA S0).
// All products run on tf32 tensor cores (mma.sync m16n8k8) with fp32
// accumulation. A chunk whose decays leave [1/16, 16] (or hold a NaN) is run
// step by step in fp32 by both kernels.
#include "wkv7_launch.h"
#include "wkv7_mma.cuh"
#include "wkv7_scaled.cuh"

namespace wkv7 {
namespace {

constexpr int kN = 64, kL = 16;
constexpr int kLD64 = 72;  // row stride (floats) of 64-wide operands read along k
constexpr int kLD16 = 24;  // row stride of 16-wide operands
constexpr int kLDT = 68;   // row stride of operands read only as [k][n] B operands
constexpr int kLDS = 72;   // row stride of checkpoints in the carry kernel (read along rows)
constexpr int kLDG = 68;   // row stride of checkpoint and carry in the output kernel (read down columns)
constexpr int kTile = kL * kN;
constexpr int kThreads = 256;
enum { V_R = 0, V_W = 1, V_K = 2, V_V = 3, V_A = 4, V_B = 5, V_DY = 6 };

__device__ __forceinline__ float bf(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ float2 bf2(const __nv_bfloat16* p) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
}
__device__ __forceinline__ float2 tf32r2(float2 x) { return make_float2(tf32r(x.x), tf32r(x.y)); }

// acc = P Q^T for 16-row P, Q (ld kLD64, tf32 values), K = 64.
__device__ __forceinline__ void gram16(float (&acc)[2][4], const float* P, const float* Q, int g, int t4) {
  zero4(acc[0]);
  zero4(acc[1]);
#pragma unroll
  for (int kb = 0; kb < kN / 8; ++kb) {
    uint32_t a[4];
    frag_a(a, P, kLD64, 0, 8 * kb, g, t4);
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      uint32_t b0, b1;
      frag_b(b0, b1, Q, kLD64, 8 * nt, 8 * kb, g, t4);
      mma_tf32(acc[nt], a, b0, b1);
    }
  }
}

// Store a 16 x 16 accumulator as tf32, keeping (t, s) with
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
      *reinterpret_cast<float2*>(dst + t * kLD16 + s) = make_float2(tf32r(x[0]), tf32r(x[1]));
    }
}

// T = (I - M)^-1 for a strictly lower 16 x 16 M (stride kLD16) by forward
// substitution, one warp; lane s < 16 owns column s. Writes T (row-major)
// and/or its transpose as tf32 values.
__device__ __forceinline__ void unit_lower_inverse(const float* M, float* Tout, float* TTout, int lane) {
  const int s = lane & 15;
  float col[kL];
#pragma unroll
  for (int t = 0; t < kL; ++t) {
    float x = t == s ? 1.f : 0.f;
#pragma unroll
    for (int u = 0; u < t; ++u) x = fmaf(M[t * kLD16 + u], col[u], x);
    col[t] = x;
  }
  if (lane < 16) {
#pragma unroll
    for (int t = 0; t < kL; ++t) {
      const float x = tf32r(col[t]);
      if (Tout) Tout[t * kLD16 + s] = x;
      if (TTout) TTout[s * kLD16 + t] = x;
    }
  }
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

// 16 KB state (64 x 64 fp32, row-major) global -> shared rows of stride LD
// by cp.async, spread over NT threads (this one is number `tid`), as one
// commit group (empty unless `any`).
template <int LD, int NT>
__device__ __forceinline__ void fetch_state(float* dst, const float* src, int tid, bool any) {
  if (any) {
#pragma unroll
    for (int q = 0; q < kN * kN / 4 / NT; ++q) {
      const int idx = tid + NT * q;  // 16-byte piece: row idx / 16, column 4 * (idx % 16)
      cp_async16(dst + (idx >> 4) * LD + 4 * (idx & 15), src + 4 * idx);
    }
  }
  cp_async_commit();
}

// ================================================================ carry ===

enum { C_R = 0, C_W = 1, C_A = 2, C_B = 3, C_DY = 4 };  // vectors staged for the carry
constexpr int kCarryStages = 3;
constexpr int kCarryThreads = 384;  // warps 0-3: state; warps 4-11: prep
constexpr int kPrepThreads = 256;

// Operands of one chunk for the carry update (tf32 values unless noted).
struct OpC {
  float Rh[kL * kLD64];   // R^ [t][j]
  float DYs[kL * kLD64];  // DY [t][i] (bf16 values)
  float Btp[kL * kLD64];  // T^T Bb [t][j]
  float Ah68[kL * kLDT];  // A^ [t][j]
  float W[kL * kLD16];    // Mbr T [s][t]
  float cL[kN];           // c(L), fp32
  int unsafe;
  int pad_[3];
};

struct CarrySmem {
  __nv_bfloat16 raw[kCarryStages][5][kTile];  // r, w, a, b, dy of one chunk per stage
  OpC op[2];
  // prep scratch (one chunk at a time)
  float Ah[kL * kLD64], Bt[kL * kLD64];                   // A^, B~ [t][j]
  float Bb68[kL * kLDT];                                  // Bb [t][j]
  float Mbr[kL * kLD16], Mba[kL * kLD16], TT[kL * kLD16];  // [t][s]; TT = T^T
  uint64_t full[kCarryStages];
  int abort_flag;
};

// Scaled operands of a chunk for the carry. 256 prep threads; thread
// (lane, pw) forms columns 2 lane, 2 lane + 1 of steps 2 pw, 2 pw + 1. The
// running products c(t) are taken in step order from t = 0 in every thread
// (the output kernel forms the same values). Returns (uniformly over the
// prep warps) whether some decay leaves the range of the scaled form.
__device__ bool prep_carry(CarrySmem& sm, const __nv_bfloat16* rs, OpC& op, int len, int ptid) {
  const int lane = ptid & 31, pw = ptid >> 5, j = 2 * lane, t0 = 2 * pw;
  bool safe = true;
  float2 cL = make_float2(1.f, 1.f), cpre = cL;  // cpre = c(t0 - 1)
#pragma unroll
  for (int t = 0; t < kL; ++t) {
    const float2 w = t < len ? bf2(rs + C_W * kTile + t * kN + j) : make_float2(1.f, 1.f);
    safe &= decay_is_safe(w.x) && decay_is_safe(w.y);
    cL = fmul2(cL, w);
    if (t < t0) cpre = cL;
  }
  if (named_bar_or(1, kPrepThreads, !safe)) return true;
  if (pw == 0) *reinterpret_cast<float2*>(op.cL + j) = cL;
  float2 wv[2], av[2], rv[2], bv[2], dyv[2];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int o = (t0 + e) * kN + j;
    wv[e] = t0 + e < len ? bf2(rs + C_W * kTile + o) : make_float2(1.f, 1.f);
    av[e] = bf2(rs + C_A * kTile + o);
    rv[e] = bf2(rs + C_R * kTile + o);
    bv[e] = bf2(rs + C_B * kTile + o);
    dyv[e] = bf2(rs + C_DY * kTile + o);
  }
  float2 c = cpre;
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int t = t0 + e, q = t * kLD64 + j, q68 = t * kLDT + j;
    const float2 cprev = c;
    c = fmul2(c, wv[e]);
    const float2 ic = make_float2(rcp_approx(c.x), rcp_approx(c.y));
    const float2 ah = tf32r2(fmul2(av[e], cprev));
    *reinterpret_cast<float2*>(sm.Ah + q) = ah;
    *reinterpret_cast<float2*>(op.Ah68 + q68) = ah;
    *reinterpret_cast<float2*>(op.Rh + q) = tf32r2(fmul2(rv[e], c));
    *reinterpret_cast<float2*>(sm.Bt + q) = tf32r2(fmul2(bv[e], ic));
    *reinterpret_cast<float2*>(sm.Bb68 + q68) = tf32r2(fmul2(bv[e], fmul2(cL, ic)));
    *reinterpret_cast<float2*>(op.DYs + q) = dyv[e];
  }
  return false;
}

// Prep warps: wait for a chunk's inputs, form its operands, Mbr, Mba, T,
// T^T Bb and Mbr T. Returns false on a timeout.
__device__ bool front_carry(CarrySmem& sm, OpC& op, const __nv_bfloat16* rs, uint64_t* bar, uint32_t parity, int len,
                            unsigned* status) {
  const int ptid = threadIdx.x - 128, pw = ptid >> 5, lane = threadIdx.x & 31, g = lane >> 2, t4 = lane & 3;
  const bool ok = mbar_wait_bounded(status, bar, parity);
  if (named_bar_or(1, kPrepThreads, !ok)) {
    if (ptid == 0) sm.abort_flag = 1;
    return false;
  }
  const bool unsafe = prep_carry(sm, rs, op, len, ptid);
  if (ptid == 0) op.unsafe = unsafe;
  if (unsafe) return true;
  named_bar(1, kPrepThreads);
  if (pw < 2) {  // Mbr = R^ B~^T (with diagonal), Mba = A^ B~^T (strictly lower), then T
    float acc[2][4];
    gram16(acc, pw ? sm.Ah : op.Rh, sm.Bt, g, t4);
    store_masked(acc, pw ? sm.Mba : sm.Mbr, true, pw == 0, g, t4);
    if (pw == 1) {
      __syncwarp();
      unit_lower_inverse(sm.Mba, nullptr, sm.TT, lane);
    }
  }
  named_bar(1, kPrepThreads);
  {  // T^T Bb, n-tile pw
    float acc[4];
    zero4(acc);
#pragma unroll
    for (int kb = 0; kb < 2; ++kb) {
      uint32_t a[4], b0, b1;
      frag_a(a, sm.TT, kLD16, 0, 8 * kb, g, t4);
      frag_b_t(b0, b1, sm.Bb68, kLDT, 8 * pw, 8 * kb, g, t4);
      mma_tf32(acc, a, b0, b1);
    }
#pragma unroll
    for (int h = 0; h < 2; ++h)
      *reinterpret_cast<float2*>(op.Btp + (g + 8 * h) * kLD64 + 8 * pw + 2 * t4) =
          make_float2(tf32r(acc[2 * h]), tf32r(acc[2 * h + 1]));
  }
  if (pw >= 6) {  // W = Mbr T, n-tile pw - 6
    const int q = pw - 6;
    float acc[4];
    zero4(acc);
#pragma unroll
    for (int kb = 0; kb < 2; ++kb) {
      uint32_t a[4], b0, b1;
      frag_a(a, sm.Mbr, kLD16, 0, 8 * kb, g, t4);
      frag_b(b0, b1, sm.TT, kLD16, 8 * q, 8 * kb, g, t4);
      mma_tf32(acc, a, b0, b1);
    }
#pragma unroll
    for (int h = 0; h < 2; ++h)
      *reinterpret_cast<float2*>(op.W + (g + 8 * h) * kLD16 + 8 * q + 2 * t4) =
          make_float2(tf32r(acc[2 * h]), tf32r(acc[2 * h + 1]));
  }
  return true;
}

// One chunk of the carry (state warp, rows i0 .. i0+15 of G):
//   DSA^T = G (T^T Bb)^T + DY^T (Mbr T);  G <- G diag(c(L)) + DY^T R^ + DSA^T A^
__device__ __forceinline__ void carry_chunk(float (&G)[8][4], const OpC& op, int i0, int g, int t4) {
  uint32_t aG[8][4];
#pragma unroll
  for (int kb = 0; kb < 8; ++kb) c2a(aG[kb], G[kb]);
  uint32_t aD[2][4];
#pragma unroll
  for (int kb = 0; kb < 2; ++kb) frag_a_ts(aD[kb], op.DYs, kLD64, i0, 8 * kb, g, t4);  // DY^T (hardware k order)
  float DS[2][4];
  zero4(DS[0]);
  zero4(DS[1]);
#pragma unroll
  for (int kb = 0; kb < 2; ++kb)
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      uint32_t b0, b1;
      frag_b_ts(b0, b1, op.W, kLD16, 8 * q, 8 * kb, g, t4);
      mma_tf32(DS[q], aD[kb], b0, b1);
    }
#pragma unroll
  for (int kb = 0; kb < 8; ++kb)
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      uint32_t b0, b1;
      frag_b(b0, b1, op.Btp, kLD64, 8 * q, 8 * kb, g, t4);
      mma_tf32(DS[q], aG[kb], b0, b1);
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
  for (int kb = 0; kb < 2; ++kb)
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      uint32_t b0, b1;
      frag_b_ts(b0, b1, op.Rh, kLD64, 8 * nt, 8 * kb, g, t4);
      mma_tf32(G[nt], aD[kb], b0, b1);
    }
  uint32_t aS[2][4];
  c2a(aS[0], DS[0]);
  c2a(aS[1], DS[1]);
#pragma unroll
  for (int kb = 0; kb < 2; ++kb)
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      uint32_t b0, b1;
      frag_b_t(b0, b1, op.Ah68, kLDT, 8 * nt, 8 * kb, g, t4);
      mma_tf32(G[nt], aS[kb], b0, b1);
    }
}

// The same chunk step by step in fp32 (a chunk outside the scaled form's
// range): G += dy r^T ; dsa = G b ; G <- G diag(w) + dsa a^T.
__device__ void carry_direct(float (&G)[8][4], const __nv_bfloat16* rs, int len, int i0, int g, int t4) {
  for (int t = len - 1; t >= 0; --t) {
    const __nv_bfloat16* row = rs + t * kN;
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
      const float2 w = bf2(row + C_W * kTile + col), a = bf2(row + C_A * kTile + col);
      G[nt][0] = fmaf(ds0, a.x, G[nt][0] * w.x);
      G[nt][1] = fmaf(ds0, a.y, G[nt][1] * w.y);
      G[nt][2] = fmaf(ds1, a.x, G[nt][2] * w.x);
      G[nt][3] = fmaf(ds1, a.y, G[nt][3] * w.y);
    }
  }
}

__global__ void __launch_bounds__(kCarryThreads, 1) wkv7_bwd4_carry_kernel(const __grid_constant__ BwdArgs args) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  CarrySmem& sm = *reinterpret_cast<CarrySmem*>(smem_raw);
  const int T = args.T, H = args.H;
  const int head = blockIdx.x, bi = head / H, hi = head % H;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t4 = lane & 3;
  const bool is_prep = warp >= 4;
  const int i0 = 16 * warp;  // state warps: rows of the carry
  const int nchunks = (T + kL - 1) / kL;
  constexpr int kStageBytes = 5 * kTile * 2;
  float* carry_head = args.carry + (size_t)head * nchunks * kN * kN;

  // chunks are visited in reverse; visit m handles chunk nchunks-1-m
  auto issue = [&](int m) {
    const int st = m % kCarryStages, chunk = nchunks - 1 - m;
    const int vmap[5] = {V_R, V_W, V_A, V_B, V_DY};
    mbar_arrive_expect_tx(&sm.full[st], kStageBytes);
    for (int v = 0; v < 5; ++v) tma_load_4d(sm.raw[st][v], &args.map[vmap[v]], &sm.full[st], 0, hi, chunk * kL, bi);
  };
  if (tid == 128) {
    for (int s = 0; s < kCarryStages; ++s) mbar_init(&sm.full[s], 1);
    fence_mbar_init();
    for (int v = 0; v < 7; ++v) prefetch_tensormap(&args.map[v]);
    for (int m = 0; m < kCarryStages && m < nchunks; ++m) issue(m);
  }
  if (tid == 0) sm.abort_flag = 0;
  float G[8][4];
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) zero4(G[nt]);
  __syncthreads();

  int waited = 0, issued = min(kCarryStages, nchunks);
  bool aborted = false;
  if (is_prep) {  // front half of the first visited chunk
    const int n = nchunks - 1;
    if (front_carry(sm, sm.op[n & 1], sm.raw[0][0], &sm.full[0], 0, min(kL, T - n * kL), args.status)) waited = 1;
  }
  if (__syncthreads_or(sm.abort_flag)) aborted = true;

  for (int m = 0; m < nchunks && !aborted; ++m) {
    const int n = nchunks - 1 - m, st = m % kCarryStages, len = min(kL, T - n * kL);
    if (!is_prep) {
      const OpC& op = sm.op[n & 1];
      // the carry entering this chunk (gradient w.r.t. the state after it), as the tf32
      // operand the output kernel multiplies with
      float* dst = carry_head + (size_t)n * kN * kN;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const int col = 8 * nt + 2 * t4;
        *reinterpret_cast<float2*>(dst + (i0 + g) * kN + col) = make_float2(tf32r(G[nt][0]), tf32r(G[nt][1]));
        *reinterpret_cast<float2*>(dst + (i0 + g + 8) * kN + col) = make_float2(tf32r(G[nt][2]), tf32r(G[nt][3]));
      }
      if (op.unsafe)
        carry_direct(G, sm.raw[st][0], len, i0, g, t4);
      else
        carry_chunk(G, op, i0, g, t4);
    } else if (n > 0) {
      const int st1 = (m + 1) % kCarryStages;
      if (front_carry(sm, sm.op[(n - 1) & 1], sm.raw[st1][0], &sm.full[st1], ((m + 1) / kCarryStages) & 1,
                      min(kL, T - (n - 1) * kL), args.status))
        waited = m + 2;
    }
    // the stage of chunk n is free (front half and direct steps done); refill it
    if (__syncthreads_or(sm.abort_flag)) {
      aborted = true;
      break;
    }
    if (tid == 128 && m + kCarryStages < nchunks) {
      fence_proxy_async_smem();
      issue(m + kCarryStages);
      issued = m + kCarryStages + 1;
    }
  }
  if (aborted) {
    if (tid == 128)
      for (int mm = waited; mm < issued; ++mm)
        mbar_wait_bounded(nullptr, &sm.full[mm % kCarryStages], (mm / kCarryStages) & 1, 200000000ull);
    __syncthreads();
    return;
  }
  if (!is_prep && args.dS_init) {
    float* dst = args.dS_init + (size_t)head * kN * kN;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const int col = 8 * nt + 2 * t4;
      *reinterpret_cast<float2*>(dst + (i0 + g) * kN + col) = make_float2(G[nt][0], G[nt][1]);
      *reinterpret_cast<float2*>(dst + (i0 + g + 8) * kN + col) = make_float2(G[nt][2], G[nt][3]);
    }
  }
}

// =============================================================== output ===

struct OpsB {  // phases A-B
  float Ah[kL * kLD64], Rh[kL * kLD64], Kb[kL * kLD64], Bb[kL * kLD64];  // [t][j]
};
struct OpsD {  // phases C-E
  float SAs[kL * kLD64], DSAs[kL * kLD64];  // sa(t), dsa(t) [t][i] (tf32)
  // triu(V DY^T), triu(V DSA^T, 1), triu(SA DY^T), triu(SA DSA^T, 1) [t][s]
  // (their transposes are the tril(...) factors)
  float U[4][kL * kLD16];
};
struct OpsE {  // phases A-E
  float Kt[kL * kLD64], Bt[kL * kLD64], Vs[kL * kLD64], DYs[kL * kLD64];  // [t][j], V and DY [t][i]
  float Ah68[kL * kLDT], Rh68[kL * kLDT];                                 // A^, R^ [t][j]
};

struct OutSmem {
  __nv_bfloat16 raw[7][kTile];  // r, w, k, v, a, b, dy of the chunk
  float S0s[kN * kLDG];         // checkpoint [i][j]
  float GcS[kN * kLDG];         // carry after the chunk [i][j] (tf32 values); the dw exchange later
  union {
    OpsB b;
    OpsD d;
    float red[4 * 5 * kN];  // column sums of a direct chunk
  } u;
  OpsE e;
  float cS[kTile];                            // c(t) [t][j], fp32
  float M[4][kL * kLD16];                     // Mka, Mkr, Mbr (with diagonal), Mba [t][s]
  float Tinv[kL * kLD16], TinvT[kL * kLD16];  // T and T^T
  float Epart[4][kN];                         // colsum(Gc o S0) over quarters of the rows
  float anc[2][kN];  // the chunk's parts of colsum(carry o state) at its start and end, without c(L) colsum(Gc o S0)
  uint64_t bar;
  int pad_[2];
};

// Step-by-step reverse scan of one chunk (warps 0..3, fp32): the carry
// starts at the stored Gc, S_prev of step t is recomputed from the
// checkpoint.
__device__ void out_direct(OutSmem& sm, int len, const BwdArgs& args, size_t base, size_t vstep, int warp,
                           int lane) {
  const int g = lane >> 2, t4 = lane & 3, i0 = 16 * warp, tid = threadIdx.x;
  const __nv_bfloat16* rs = sm.raw[0];
  const float* S0 = sm.S0s;
  float* red = sm.u.red;
  float G[8][4];
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) {
    const int col = 8 * nt + 2 * t4;
    const float2 lo = *reinterpret_cast<const float2*>(sm.GcS + (i0 + g) * kLDG + col);
    const float2 hi = *reinterpret_cast<const float2*>(sm.GcS + (i0 + g + 8) * kLDG + col);
    G[nt][0] = lo.x;
    G[nt][1] = lo.y;
    G[nt][2] = hi.x;
    G[nt][3] = hi.y;
  }
  for (int t = len - 1; t >= 0; --t) {
    float sp[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const int col = 8 * nt + 2 * t4;
      const float2 lo = *reinterpret_cast<const float2*>(S0 + (i0 + g) * kLDG + col);
      const float2 hi = *reinterpret_cast<const float2*>(S0 + (i0 + g + 8) * kLDG + col);
      sp[nt][0] = lo.x;
      sp[nt][1] = lo.y;
      sp[nt][2] = hi.x;
      sp[nt][3] = hi.y;
    }
    float sa0 = 0.f, sa1 = 0.f;
    for (int u = 0; u <= t; ++u) {
      const __nv_bfloat16* row = rs + u * kN;
      float s0 = 0.f, s1 = 0.f;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const float2 a = bf2(row + V_A * kTile + 8 * nt + 2 * t4);
        s0 = fmaf(sp[nt][0], a.x, fmaf(sp[nt][1], a.y, s0));
        s1 = fmaf(sp[nt][2], a.x, fmaf(sp[nt][3], a.y, s1));
      }
      sa0 = quad_sum(s0);
      sa1 = quad_sum(s1);
      if (u == t) break;  // sp = S_prev(t), sa = sa(t)
      const float v0 = bf(row + V_V * kTile + i0 + g), v1 = bf(row + V_V * kTile + i0 + g + 8);
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const int col = 8 * nt + 2 * t4;
        const float2 w = bf2(row + V_W * kTile + col), k = bf2(row + V_K * kTile + col);
        const float2 b = bf2(row + V_B * kTile + col);
        sp[nt][0] = fmaf(sa0, b.x, fmaf(sp[nt][0], w.x, v0 * k.x));
        sp[nt][1] = fmaf(sa0, b.y, fmaf(sp[nt][1], w.y, v0 * k.y));
        sp[nt][2] = fmaf(sa1, b.x, fmaf(sp[nt][2], w.x, v1 * k.x));
        sp[nt][3] = fmaf(sa1, b.y, fmaf(sp[nt][3], w.y, v1 * k.y));
      }
    }
    const __nv_bfloat16* row = rs + t * kN;
    const float v0 = bf(row + V_V * kTile + i0 + g), v1 = bf(row + V_V * kTile + i0 + g + 8);
    const float dy0 = bf(row + V_DY * kTile + i0 + g), dy1 = bf(row + V_DY * kTile + i0 + g + 8);
    // column partials: dr (from S_t), then G += dy r^T, dk, db, dw; row sums dv, dsa
    float pr[8][2], pk[8][2], pb[8][2], pw[8][2];
    float dv0 = 0.f, dv1 = 0.f, ds0 = 0.f, ds1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const int col = 8 * nt + 2 * t4;
      const float2 w = bf2(row + V_W * kTile + col), k = bf2(row + V_K * kTile + col);
      const float2 b = bf2(row + V_B * kTile + col), r = bf2(row + V_R * kTile + col);
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
        pw[nt][e] = fmaf(G[nt][e], sp[nt][e], G[nt][2 + e] * sp[nt][2 + e]);
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
      args.dv[base + (size_t)t * vstep + i0 + g] = dv0;
      args.dv[base + (size_t)t * vstep + i0 + g + 8] = dv1;
    }
    // da = S_prev^T dsa; carry G <- G diag(w) + dsa a^T; column sums to shared memory
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const int col = 8 * nt + 2 * t4;
      const float2 w = bf2(row + V_W * kTile + col), a = bf2(row + V_A * kTile + col);
      const float wv[2] = {w.x, w.y}, av[2] = {a.x, a.y};
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float pa = fmaf(sp[nt][e], ds0, sp[nt][2 + e] * ds1);
        G[nt][e] = fmaf(ds0, av[e], G[nt][e] * wv[e]);
        G[nt][2 + e] = fmaf(ds1, av[e], G[nt][2 + e] * wv[e]);
        const float sums[5] = {col_sum(pr[nt][e]), col_sum(pk[nt][e]), col_sum(pb[nt][e]), col_sum(pw[nt][e]),
                               col_sum(pa)};
        if (g == 0) {
#pragma unroll
          for (int q = 0; q < 5; ++q) red[(warp * 5 + q) * kN + col + e] = sums[q];
        }
      }
    }
    named_bar(5, 128);
    for (int idx = tid; idx < 5 * kN; idx += 128) {
      const int q = idx / kN, col = idx % kN;
      const float x = red[q * kN + col] + red[(5 + q) * kN + col] + red[(10 + q) * kN + col] + red[(15 + q) * kN + col];
      float* dst = q == 0 ? args.dr : q == 1 ? args.dk : q == 2 ? args.db : q == 3 ? args.dw : args.da;
      dst[base + (size_t)t * vstep + col] = x;
    }
    named_bar(5, 128);
  }
}

// P0 += X M[:, j0 .. j0+15], P1 += Y M[:, j0 .. j0+15] for 16-row X, Y (stride
// kLD64, tf32 values) and a 64 x 64 M (stride kLDG; fp32 values that need
// rounding if kRound).
template <bool kRound>
__device__ __forceinline__ void column_products(float (&P0)[2][4], float (&P1)[2][4], const float* X, const float* Y,
                                                const float* M, int j0, int g, int t4) {
#pragma unroll
  for (int kb = 0; kb < 8; ++kb) {
    uint32_t a0[4], a1[4];
    frag_a(a0, X, kLD64, 0, 8 * kb, g, t4);
    frag_a(a1, Y, kLD64, 0, 8 * kb, g, t4);
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      uint32_t b0, b1;
      if (kRound)
        frag_b_t_r(b0, b1, M, kLDG, j0 + 8 * nt, 8 * kb, g, t4);
      else
        frag_b_t(b0, b1, M, kLDG, j0 + 8 * nt, 8 * kb, g, t4);
      mma_tf32(P0[nt], a0, b0, b1);
      mma_tf32(P1[nt], a1, b0, b1);
    }
  }
}

__global__ void __launch_bounds__(kThreads, 2) wkv7_bwd4_out_kernel(const __grid_constant__ BwdArgs args) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  OutSmem& sm = *reinterpret_cast<OutSmem*>(smem_raw);
  const int T = args.T, H = args.H, nchunks = (T + kL - 1) / kL;
  const int head = blockIdx.x / nchunks, n = blockIdx.x % nchunks, bi = head / H, hi = head % H;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t4 = lane & 3;
  const int t0 = n * kL, len = min(kL, T - t0);
  const size_t vstep = (size_t)H * kN, base = ((size_t)bi * T + t0) * vstep + (size_t)hi * kN;

  // ---- loads: inputs by TMA, checkpoint and carry by cp.async
  if (tid == 0) {
    mbar_init(&sm.bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(&sm.bar, 7 * kTile * 2);
    for (int v = 0; v < 7; ++v) tma_load_4d(sm.raw[v], &args.map[v], &sm.bar, 0, hi, t0, bi);
  }
  fetch_state<kLDG, kThreads>(sm.S0s, args.ckpt + ((size_t)head * args.nck + n) * kN * kN, tid, true);
  fetch_state<kLDG, kThreads>(sm.GcS, args.carry + ((size_t)head * nchunks + n) * kN * kN, tid, true);
  __syncthreads();  // barrier initialised
  const bool ok = mbar_wait_bounded(args.status, &sm.bar, 0);
  cp_async_wait_all();
  if (__syncthreads_or(!ok)) {
    if (tid == 0) mbar_wait_bounded(nullptr, &sm.bar, 0, 200000000ull);
    __syncthreads();
    return;
  }
  const __nv_bfloat16* rs = sm.raw[0];

  // ---- A: scaled operands; thread (lane, warp) forms columns 2 lane, 2 lane + 1 of steps
  //      2 warp, 2 warp + 1 (running products c in step order from t = 0, as in the carry kernel)
  {
    const int j = 2 * lane, t0 = 2 * warp;
    bool safe = true;
    float2 cL = make_float2(1.f, 1.f), cpre = cL;  // cpre = c(t0 - 1)
#pragma unroll
    for (int t = 0; t < kL; ++t) {
      const float2 w = t < len ? bf2(rs + V_W * kTile + t * kN + j) : make_float2(1.f, 1.f);
      safe &= decay_is_safe(w.x) && decay_is_safe(w.y);
      cL = fmul2(cL, w);
      if (t < t0) cpre = cL;
    }
    if (__syncthreads_or(!safe)) {
      if (warp < 4) out_direct(sm, len, args, base, vstep, warp, lane);
      return;
    }
    float2 wv[2], av[2], rv[2], kv[2], bv[2], vv[2], dyv[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int o = (t0 + e) * kN + j;
      wv[e] = t0 + e < len ? bf2(rs + V_W * kTile + o) : make_float2(1.f, 1.f);
      av[e] = bf2(rs + V_A * kTile + o);
      rv[e] = bf2(rs + V_R * kTile + o);
      kv[e] = bf2(rs + V_K * kTile + o);
      bv[e] = bf2(rs + V_B * kTile + o);
      vv[e] = bf2(rs + V_V * kTile + o);
      dyv[e] = bf2(rs + V_DY * kTile + o);
    }
    float2 c = cpre;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int t = t0 + e, o = t * kN + j, q = t * kLD64 + j, q68 = t * kLDT + j;
      const float2 cprev = c;
      c = fmul2(c, wv[e]);
      const float2 ic = make_float2(rcp_approx(c.x), rcp_approx(c.y)), s = fmul2(cL, ic);
      const float2 ah = tf32r2(fmul2(av[e], cprev)), rh = tf32r2(fmul2(rv[e], c));
      *reinterpret_cast<float2*>(sm.u.b.Ah + q) = ah;
      *reinterpret_cast<float2*>(sm.e.Ah68 + q68) = ah;
      *reinterpret_cast<float2*>(sm.u.b.Rh + q) = rh;
      *reinterpret_cast<float2*>(sm.e.Rh68 + q68) = rh;
      *reinterpret_cast<float2*>(sm.e.Kt + q) = tf32r2(fmul2(kv[e], ic));
      *reinterpret_cast<float2*>(sm.e.Bt + q) = tf32r2(fmul2(bv[e], ic));
      *reinterpret_cast<float2*>(sm.u.b.Kb + q) = tf32r2(fmul2(kv[e], s));
      *reinterpret_cast<float2*>(sm.u.b.Bb + q) = tf32r2(fmul2(bv[e], s));
      *reinterpret_cast<float2*>(sm.e.Vs + q) = vv[e];  // bf16 values are tf32 values
      *reinterpret_cast<float2*>(sm.e.DYs + q) = dyv[e];
      *reinterpret_cast<float2*>(sm.cS + o) = c;
    }
    // colsum(Gc o S0) over rows 16 q .. 16 q + 15, column j = tid % 64 (both anchors of dw start from it)
    const int jc = tid & 63, q = tid >> 6;
    float ep = 0.f;
#pragma unroll
    for (int i = 16 * q; i < 16 * q + 16; ++i) ep = fmaf(sm.GcS[i * kLDG + jc], sm.S0s[i * kLDG + jc], ep);
    sm.Epart[q][jc] = ep;
  }
  __syncthreads();

  // ---- B: L x L products and T (warps 0-3), the K = 64 parts of sa, dsa, dv
  const int rb = warp & 3, r0 = 16 * rb;  // row block of the state-sized products
  float X1[2][4], X2[2][4];               // warps 0-3: RDSA^T; warps 4-7: RSA^T, DV^T (rows i, columns t)
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    zero4(X1[q]);
    zero4(X2[q]);
  }
  if (warp < 4) {
    // Mka = A^ K~^T, Mba = A^ B~^T (strictly lower); Mkr = R^ K~^T, Mbr = R^ B~^T (with diagonal)
    float acc[2][4];
    gram16(acc, warp < 2 ? sm.u.b.Ah : sm.u.b.Rh, (warp & 1) ? sm.e.Bt : sm.e.Kt, g, t4);
    store_masked(acc, sm.M[warp == 0 ? 0 : warp == 1 ? 3 : warp - 1], true, warp >= 2, g, t4);
    if (warp == 1) {
      __syncwarp();
      unit_lower_inverse(sm.M[3], sm.Tinv, sm.TinvT, lane);
    }
#pragma unroll
    for (int kb = 0; kb < 8; ++kb) {  // Gc Bb^T
      uint32_t aG[4];
      frag_a(aG, sm.GcS, kLDG, r0, 8 * kb, g, t4);
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        uint32_t b0, b1;
        frag_b(b0, b1, sm.u.b.Bb, kLD64, 8 * q, 8 * kb, g, t4);
        mma_tf32(X1[q], aG, b0, b1);
      }
    }
  } else {
#pragma unroll
    for (int kb = 0; kb < 8; ++kb) {  // S0 A^T, Gc Kb^T
      uint32_t aS[4], aG[4];
      frag_a_r(aS, sm.S0s, kLDG, r0, 8 * kb, g, t4);
      frag_a(aG, sm.GcS, kLDG, r0, 8 * kb, g, t4);
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        uint32_t b0, b1;
        frag_b(b0, b1, sm.u.b.Ah, kLD64, 8 * q, 8 * kb, g, t4);
        mma_tf32(X1[q], aS, b0, b1);
        frag_b(b0, b1, sm.u.b.Kb, kLD64, 8 * q, 8 * kb, g, t4);
        mma_tf32(X2[q], aG, b0, b1);
      }
    }
  }
  __syncthreads();

  // ---- C: DSA^T = (Gc Bb^T + DY^T Mbr) T (warps 0-3); SA^T = (S0 A^T + V^T Mka^T) T^T and
  //      DV^T += DY^T Mkr (warps 4-7). SAs/DSAs overwrite operands of phase B.
  {
    uint32_t aD[2][4];
#pragma unroll
    for (int kb = 0; kb < 2; ++kb) frag_a_ts(aD[kb], sm.e.DYs, kLD64, r0, 8 * kb, g, t4);  // DY^T
    float Y[2][4];
    zero4(Y[0]);
    zero4(Y[1]);
    if (warp < 4) {
#pragma unroll
      for (int kb = 0; kb < 2; ++kb)
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          uint32_t b0, b1;
          frag_b_ts(b0, b1, sm.M[2], kLD16, 8 * q, 8 * kb, g, t4);
          mma_tf32(X1[q], aD[kb], b0, b1);
        }
#pragma unroll
      for (int kb = 0; kb < 2; ++kb) {
        uint32_t a2[4];
        c2a(a2, X1[kb]);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          uint32_t b0, b1;
          frag_b(b0, b1, sm.TinvT, kLD16, 8 * q, 8 * kb, g, t4);
          mma_tf32(Y[q], a2, b0, b1);
        }
      }
    } else {
#pragma unroll
      for (int kb = 0; kb < 2; ++kb) {
        uint32_t aV[4];
        frag_a_t(aV, sm.e.Vs, kLD64, r0, 8 * kb, g, t4);  // V^T
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          uint32_t b0, b1;
          frag_b(b0, b1, sm.M[0], kLD16, 8 * q, 8 * kb, g, t4);
          mma_tf32(X1[q], aV, b0, b1);
          frag_b_ts(b0, b1, sm.M[1], kLD16, 8 * q, 8 * kb, g, t4);
          mma_tf32(X2[q], aD[kb], b0, b1);
        }
      }
#pragma unroll
      for (int kb = 0; kb < 2; ++kb) {
        uint32_t a1[4];
        c2a(a1, X1[kb]);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          uint32_t b0, b1;
          frag_b(b0, b1, sm.Tinv, kLD16, 8 * q, 8 * kb, g, t4);
          mma_tf32(Y[q], a1, b0, b1);
        }
      }
    }
    float* dst = warp < 4 ? sm.u.d.DSAs : sm.u.d.SAs;
#pragma unroll
    for (int q = 0; q < 2; ++q)
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int e = 0; e < 2; ++e) dst[(8 * q + 2 * t4 + e) * kLD64 + r0 + g + 8 * h] = tf32r(Y[q][2 * h + e]);
  }
  __syncthreads();

  // ---- D: DV^T += DSA^T Mka and dv (warps 4-7); the four triangular L x L factors (warps 0-3)
  if (warp >= 4) {
#pragma unroll
    for (int kb = 0; kb < 2; ++kb) {
      uint32_t aS[4];
      frag_a_t(aS, sm.u.d.DSAs, kLD64, r0, 8 * kb, g, t4);  // DSA^T
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        uint32_t b0, b1;
        frag_b_t(b0, b1, sm.M[0], kLD16, 8 * q, 8 * kb, g, t4);
        mma_tf32(X2[q], aS, b0, b1);
      }
    }
#pragma unroll
    for (int q = 0; q < 2; ++q)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int t = 8 * q + 2 * t4 + e;
        if (t < len) {
          float* dst = args.dv + base + (size_t)t * vstep + r0 + g;
          dst[0] = X2[q][e];
          dst[8] = X2[q][2 + e];
        }
      }
  } else {
    // U0 = triu(V DY^T), U1 = triu(V DSA^T, 1), U2 = triu(SA DY^T), U3 = triu(SA DSA^T, 1)
    float acc[2][4];
    gram16(acc, warp < 2 ? sm.e.Vs : sm.u.d.SAs, (warp & 1) ? sm.u.d.DSAs : sm.e.DYs, g, t4);
    store_masked(acc, sm.u.d.U[warp], false, (warp & 1) == 0, g, t4);
  }
  __syncthreads();

  // ---- E: column products, 8 warps: warp (grp, jb) covers columns j0 .. j0+15 of
  //      dk~, db~ (grp 0) or dr^, da^ (grp 1)
  const int grp = warp >> 2, jb = warp & 3, j0 = 16 * jb;
  float P0[2][4], P1[2][4];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    zero4(P0[nt]);
    zero4(P1[nt]);
  }
  // sums over the rows i: V Gc, SA Gc (grp 0); DY S0, DSA S0 (grp 1)
  if (grp == 0)
    column_products<false>(P0, P1, sm.e.Vs, sm.u.d.SAs, sm.GcS, j0, g, t4);
  else
    column_products<true>(P0, P1, sm.e.DYs, sm.u.d.DSAs, sm.S0s, j0, g, t4);
  {
    // This warp's part of the dw anchors, from the column products (c(L) colsum(Gc o S0) is
    // added later):
    //   colsum(Gc o S(L)) = c(L) colsum(Gc o S0) + sum_t (Kb o V Gc + Bb o SA Gc)       (grp 0)
    //   colsum(Gc' o S0)  = c(L) colsum(Gc o S0) + sum_t (R^ o DY S0 + A^ o DSA S0)     (grp 1)
    // with S(L) = S0 diag(c(L)) + V^T Kb + SA^T Bb and Gc' = Gc diag(c(L)) + DY^T R^ + DSA^T A^.
    const __nv_bfloat16* rs0 = sm.raw[0];
    float v[4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int col = j0 + 8 * nt + 2 * t4;
      float2 acc = make_float2(0.f, 0.f);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int t = g + 8 * h;
        const float2 c = *reinterpret_cast<const float2*>(sm.cS + t * kN + col);
        if (grp == 0) {
          const float2 k = bf2(rs0 + V_K * kTile + t * kN + col), b = bf2(rs0 + V_B * kTile + t * kN + col);
          acc.x += fmaf(k.x, P0[nt][2 * h], b.x * P1[nt][2 * h]) * rcp_approx(c.x);
          acc.y += fmaf(k.y, P0[nt][2 * h + 1], b.y * P1[nt][2 * h + 1]) * rcp_approx(c.y);
        } else {
          const float2 cp = t ? *reinterpret_cast<const float2*>(sm.cS + (t - 1) * kN + col) : make_float2(1.f, 1.f);
          const float2 r = bf2(rs0 + V_R * kTile + t * kN + col), a = bf2(rs0 + V_A * kTile + t * kN + col);
          acc.x += fmaf(r.x * c.x, P0[nt][2 * h], a.x * cp.x * P1[nt][2 * h]);
          acc.y += fmaf(r.y * c.y, P0[nt][2 * h + 1], a.y * cp.y * P1[nt][2 * h + 1]);
        }
      }
      v[2 * nt] = acc.x;
      v[2 * nt + 1] = acc.y;
    }
    // sum over the 8 row groups: reduce-scatter over xor 16 (n-tile), 8 (column parity), then 4
    const bool up16 = (g & 4) != 0, up8 = (g & 2) != 0;
    float x0 = (up16 ? v[2] : v[0]) + __shfl_xor_sync(0xffffffffu, up16 ? v[0] : v[2], 16);
    float x1 = (up16 ? v[3] : v[1]) + __shfl_xor_sync(0xffffffffu, up16 ? v[1] : v[3], 16);
    float y = (up8 ? x1 : x0) + __shfl_xor_sync(0xffffffffu, up8 ? x0 : x1, 8);
    y += __shfl_xor_sync(0xffffffffu, y, 4);
    if ((g & 1) == 0) {
      const int col = j0 + 8 * (up16 ? 1 : 0) + 2 * t4 + (up8 ? 1 : 0);
      const float cl = sm.cS[(kL - 1) * kN + col];
      sm.anc[grp ? 0 : 1][col] = grp ? y : cl * y;
    }
  }
  __syncthreads();  // the carry tile is free from here on (the dw exchange below)
  // triangular terms (U0 = triu(V DY^T), U1 = triu(V DSA^T, 1), U2 = triu(SA DY^T), U3 = triu(SA DSA^T, 1)):
  //   dk~ = (V Gc) c(L) + U0 R^ + U1 A^        db~ = (SA Gc) c(L) + U2 R^ + U3 A^
  //   dr^ = DY S0 + U0^T K~ + U2^T B~          da^ = DSA S0 + U1^T K~ + U3^T B~
  const float* U0 = sm.u.d.U[0];
  const float* U1 = sm.u.d.U[1];
  const float* U2 = sm.u.d.U[2];
  const float* U3 = sm.u.d.U[3];
  if (grp == 0) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      // c(L) = c(15), the last row of cS
      const float2 cl = *reinterpret_cast<const float2*>(sm.cS + (kL - 1) * kN + j0 + 8 * nt + 2 * t4);
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
      uint32_t u0[4], u1[4], u2[4], u3[4];
      frag_a(u0, U0, kLD16, 0, 8 * kb, g, t4);
      frag_a(u1, U1, kLD16, 0, 8 * kb, g, t4);
      frag_a(u2, U2, kLD16, 0, 8 * kb, g, t4);
      frag_a(u3, U3, kLD16, 0, 8 * kb, g, t4);
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        uint32_t b0, b1;
        frag_b_t(b0, b1, sm.e.Rh68, kLDT, j0 + 8 * nt, 8 * kb, g, t4);
        mma_tf32(P0[nt], u0, b0, b1);
        mma_tf32(P1[nt], u2, b0, b1);
        frag_b_t(b0, b1, sm.e.Ah68, kLDT, j0 + 8 * nt, 8 * kb, g, t4);
        mma_tf32(P0[nt], u1, b0, b1);
        mma_tf32(P1[nt], u3, b0, b1);
      }
    }
  } else {
#pragma unroll
    for (int kb = 0; kb < 2; ++kb) {
      uint32_t u0[4], u1[4], u2[4], u3[4];
      frag_a_ts(u0, U0, kLD16, 0, 8 * kb, g, t4);
      frag_a_ts(u1, U1, kLD16, 0, 8 * kb, g, t4);
      frag_a_ts(u2, U2, kLD16, 0, 8 * kb, g, t4);
      frag_a_ts(u3, U3, kLD16, 0, 8 * kb, g, t4);
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        uint32_t b0, b1;
        frag_b_ts(b0, b1, sm.e.Kt, kLD64, j0 + 8 * nt, 8 * kb, g, t4);
        mma_tf32(P0[nt], u0, b0, b1);
        mma_tf32(P1[nt], u1, b0, b1);
        frag_b_ts(b0, b1, sm.e.Bt, kLD64, j0 + 8 * nt, 8 * kb, g, t4);
        mma_tf32(P0[nt], u2, b0, b1);
        mma_tf32(P1[nt], u3, b0, b1);
      }
    }
  }
  // unscale: dk = dk~ / c, db = db~ / c (grp 0); dr = dr^ c, da = da^ c(t-1) (grp 1); and this
  // group's part of x = r dr - k dk - b db + a da
  float X[2][4], AD[2][4];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int t = g + 8 * h, col = j0 + 8 * nt + 2 * t4;
      const float2 c = *reinterpret_cast<const float2*>(sm.cS + t * kN + col);
      if (grp == 0) {
        const float2 k = bf2(rs + V_K * kTile + t * kN + col), b = bf2(rs + V_B * kTile + t * kN + col);
        const float ic[2] = {rcp_approx(c.x), rcp_approx(c.y)}, kv[2] = {k.x, k.y}, bv[2] = {b.x, b.y};
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          P0[nt][2 * h + e] *= ic[e];
          P1[nt][2 * h + e] *= ic[e];
          X[nt][2 * h + e] = -kv[e] * P0[nt][2 * h + e] - bv[e] * P1[nt][2 * h + e];
          AD[nt][2 * h + e] = 0.f;
        }
      } else {
        const float2 cp = t ? *reinterpret_cast<const float2*>(sm.cS + (t - 1) * kN + col) : make_float2(1.f, 1.f);
        const float2 r = bf2(rs + V_R * kTile + t * kN + col), a = bf2(rs + V_A * kTile + t * kN + col);
        const float cv[2] = {c.x, c.y}, cpv[2] = {cp.x, cp.y}, rv[2] = {r.x, r.y}, av[2] = {a.x, a.y};
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          P0[nt][2 * h + e] *= cv[e];
          P1[nt][2 * h + e] *= cpv[e];
          AD[nt][2 * h + e] = av[e] * P1[nt][2 * h + e];
          X[nt][2 * h + e] = rv[e] * P0[nt][2 * h + e] + AD[nt][2 * h + e];
        }
      }
    }
  // exchange with the partner warp of the other group (same columns): grp 0 keeps
  // dw of n-tile 0, grp 1 of n-tile 1
  float* XK = sm.GcS;                   // grp 0's x part, [t][j] stride 72
  float* XR = sm.GcS + kL * kLD64;      // grp 1's x part
  float* XA = sm.GcS + 2 * kL * kLD64;  // grp 1's a da
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
  named_bar(1 + jb, 64);
  const int nw = grp, jw = j0 + 8 * nw;  // this warp's dw columns jw .. jw+7
  float xw[4], adw[4];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int t = g + 8 * h;
    if (grp == 0) {
      const float2 xr = *reinterpret_cast<const float2*>(XR + t * kLD64 + jw + 2 * t4);
      const float2 xa = *reinterpret_cast<const float2*>(XA + t * kLD64 + jw + 2 * t4);
      xw[2 * h] = X[0][2 * h] + xr.x;
      xw[2 * h + 1] = X[0][2 * h + 1] + xr.y;
      adw[2 * h] = xa.x;
      adw[2 * h + 1] = xa.y;
    } else {
      const float2 xk = *reinterpret_cast<const float2*>(XK + t * kLD64 + jw + 2 * t4);
      xw[2 * h] = X[1][2 * h] + xk.x;
      xw[2 * h + 1] = X[1][2 * h + 1] + xk.y;
      adw[2 * h] = AD[1][2 * h];
      adw[2 * h + 1] = AD[1][2 * h + 1];
    }
  }
  // w dw from the identity, anchored where fewer terms are summed:
  // rows t < 8: colsum(carry at the chunk start o S0) - sum_{u<t} x(u) - a(t) da(t);
  // rows t >= 8: sum_{u>=t} x(u) - a(t) da(t) + colsum(carry at the chunk end o S(L)).
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
    const float2 w0 = bf2(rs + V_W * kTile + g * kN + jw + 2 * t4);
    const float2 w1 = bf2(rs + V_W * kTile + (g + 8) * kN + jw + 2 * t4);
    const float cge = sm.cS[(kL - 1) * kN + col] * (sm.Epart[0][col] + sm.Epart[1][col] + sm.Epart[2][col] + sm.Epart[3][col]);
    dw[e] = (cge + sm.anc[0][col] - (lo - xw[e]) - adw[e]) * rcp_approx(e ? w0.y : w0.x);
    dw[2 + e] = (hi2 - adw[2 + e] + cge + sm.anc[1][col]) * rcp_approx(e ? w1.y : w1.x);
  }
  float* out0 = grp ? args.dr : args.dk;
  float* out1 = grp ? args.da : args.db;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int t = g + 8 * h;
    if (t < len) {
      const size_t off = base + (size_t)t * vstep + j0 + 2 * t4;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        *reinterpret_cast<float2*>(out0 + off + 8 * nt) = make_float2(P0[nt][2 * h], P0[nt][2 * h + 1]);
        *reinterpret_cast<float2*>(out1 + off + 8 * nt) = make_float2(P1[nt][2 * h], P1[nt][2 * h + 1]);
      }
      *reinterpret_cast<float2*>(args.dw + off + 8 * nw) = make_float2(dw[2 * h], dw[2 * h + 1]);
    }
  }
}

}  // namespace

size_t bwd4_workspace_bytes(int B, int T, int H) {
  const size_t nchunks = ((size_t)T + kL - 1) / kL, heads = (size_t)B * H;
  return heads * nchunks * kN * kN * sizeof(float);
}

cudaError_t launch_bwd4(const BwdArgs& args, cudaStream_t stream) {
  const size_t smem_c = sizeof(CarrySmem), smem_o = sizeof(OutSmem);
  cudaError_t e = cudaFuncSetAttribute(wkv7_bwd4_carry_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_c);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(wkv7_bwd4_out_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_o);
  if (e != cudaSuccess) return e;
  const unsigned heads = (unsigned)(args.B * args.H), nchunks = (unsigned)((args.T + kL - 1) / kL);
  wkv7_bwd4_carry_kernel<<<heads, kCarryThreads, smem_c, stream>>>(args);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  wkv7_bwd4_out_kernel<<<heads * nchunks, kThreads, smem_o, stream>>>(args);
  return cudaGetLastError();
}

}  // namespace wkv7
