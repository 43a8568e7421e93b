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
// Every product runs on the tensor cores in split bf16: each operand is a
// pair of bf16 values hi + lo (hi = x rounded to bf16, lo = the remainder
// rounded to bf16), formed once per chunk, and a b is taken as a_lo b_hi +
// a_hi b_lo + a_hi b_hi, three mma.sync m16n8k16 with fp32 accumulation
// (wkv7_mma16.cuh). E is summed from the fp32 checkpoint and carry; the decay
// scaling, T and every other sum are fp32.
//
// One CTA of 256 threads per (b, h, chunk) task, two CTAs per SM, in the
// phases of the bf16 output pass (wkv7_bwd4.cu): loads (the rows by cp.async,
// the checkpoint and the carry through registers, split into bf16 tiles, with
// E); the scaled operands; the L x L products, T, the K = 64 parts of SA, DSA
// and DV; SA, DSA and dv; the triangular factors; the column products and
// every column output. The fp32 rows are read only until the operands are
// formed: their space then holds the later tiles, and the unscaling reads the
// few values it needs from global memory. A chunk whose decays leave
// [1/16, 16] (or hold a NaN) runs step by step in fp32.
#include "wkv7_launch.h"
#include "wkv7_mma.cuh"
#include "wkv7_mma16.cuh"
#include "wkv7_scaled.cuh"

namespace wkv7 {
namespace {

constexpr int kN = 64, kL = 16;
constexpr int kLD64 = 72;  // row stride of fp32 [t][j] rows (c(t), the dw exchange)
constexpr int kLD16 = 24;  // row stride of 16-wide fp32 rows
constexpr int kThreads = 256;
constexpr int kTile = kL * kN;
constexpr int kT64 = kL * kB64;  // elements of a 16-row bf16 tile of 64 columns
constexpr int kT16 = kL * kB16;  // elements of a 16 x 16 bf16 tile
enum { V_R = 0, V_W = 1, V_K = 2, V_V = 3, V_A = 4, V_B = 5, V_DY = 6 };

// Shared memory of one task; the first index of every bf16 tile is the part (0 hi, 1 lo).
struct F2Smem {
  union {
    float raw[7][kTile];  // r, w, k, v, a, b, dy of the chunk [t][j], zero past the sequence (loads, forming)
    struct {              // from the L x L products on
      bf16_t SA[2][kT64], DSA[2][kT64];  // sa(t), dsa(t) [t][i]
      bf16_t M[2][3][kT16];              // Mka (strictly lower), Mkr, Mbr (lower) [t][s]
      bf16_t Tm[2][kT16];                // T = (I - Mba)^-1 [t][s]
      // U0 = triu(V DY^T), U1 = triu(V DSA^T, 1), U2 = triu(SA DY^T), U3 = triu(SA DSA^T, 1) [t][s]
      bf16_t U[2][4][kT16];
    } t;
  } a;
  union {
    struct {
      bf16_t S0[2][kN * kB64];  // checkpoint [i][j]
      bf16_t Gc[2][kN * kB64];  // carry after the chunk [i][j]
    } st;
    float xch[3][kL * kLD64];  // the dw exchange, once the column products are done
    float red[8 * 5 * kN];     // column sums of a direct chunk
  } u;
  bf16_t V[2][kT64], DY[2][kT64];  // v(t), dy(t) [t][i]
  bf16_t Ah[2][kT64], Rh[2][kT64], Kt[2][kT64], Bt[2][kT64], Kb[2][kT64], Bb[2][kT64];  // [t][j]
  float Mba[kL * kLD16];  // fp32, for the substitution
  float cS[kL * kLD64];   // c(t) [t][j], fp32
  float Epart[8][kN];     // E over the rows each warp loaded
  float Ppart[8][kN];     // products of the decays of steps 2 q, 2 q + 1
  float cLs[kN];          // c(L)
  float anc[2][kN];       // the chunk's parts of colsum(carry o state) at its start and end, without c(L) E
};
static_assert(offsetof(F2Smem, Mba) % 16 == 0, "Mba rows are read 16 bytes at a time");

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

// Four fp32 values as bf16 hi and lo parts (8 bytes each) at hi, lo.
__device__ __forceinline__ void put4_split(bf16_t* hi, bf16_t* lo, float4 x) {
  const uint32_t h0 = pack_bf16(x.x, x.y), h1 = pack_bf16(x.z, x.w);
  const float2 u0 = unpack_bf16(h0), u1 = unpack_bf16(h1);
  *reinterpret_cast<uint2*>(hi) = make_uint2(h0, h1);
  *reinterpret_cast<uint2*>(lo) = make_uint2(pack_bf16(x.x - u0.x, x.y - u0.y), pack_bf16(x.z - u1.x, x.w - u1.y));
}

// Step-by-step reverse scan of one chunk (all eight warps, fp32; warp w owns
// rows 8 w .. 8 w + 7 of the state and the carry, lane (g, t) row 8 w + g and
// columns 8 nt + 2 t, + 1): the carry starts at the stored Gc, S_prev of step
// t is recomputed from the checkpoint (both read from global memory). `rs`
// holds the chunk's rows (fp32 [t][j], kTile floats apart); `red` is
// 8 * 5 * kN floats of scratch.
__device__ void out_direct_f32(const float* rs, float* red, const float* S0, const float* Gcg, int len,
                               const BwdArgs& args, size_t base, size_t vstep, int warp, int lane) {
  const int g = lane >> 2, t4 = lane & 3, i = 8 * warp + g, tid = threadIdx.x;  // red: [8 warps][5][64]
  float G[8][2];
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) {
    const float2* p = reinterpret_cast<const float2*>(Gcg + i * kN + 8 * nt + 2 * t4);
    const float2 x = in_extent(args.status, args.ext.carry, p) ? *p : make_float2(0.f, 0.f);
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
      const float* row = rs + u * kN;
      float s = 0.f;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const float2 a = f2at(row + V_A * kTile + 8 * nt + 2 * t4);
        s = fmaf(sp[nt][0], a.x, fmaf(sp[nt][1], a.y, s));
      }
      sa = quad_sum(s);
      if (u == t) break;  // sp = S_prev(t), sa = sa(t)
      const float v = row[V_V * kTile + i];
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const int col = 8 * nt + 2 * t4;
        const float2 w = f2at(row + V_W * kTile + col), k = f2at(row + V_K * kTile + col),
                     b = f2at(row + V_B * kTile + col);
        sp[nt][0] = fmaf(sa, b.x, fmaf(sp[nt][0], w.x, v * k.x));
        sp[nt][1] = fmaf(sa, b.y, fmaf(sp[nt][1], w.y, v * k.y));
      }
    }
    const float* row = rs + t * kN;
    const float v = row[V_V * kTile + i], dy = row[V_DY * kTile + i];
    // column sums (over this warp's rows) of dr (from S_t), then G += dy r^T, dk, db, dw; row sums dv, dsa
    float dv = 0.f, ds = 0.f;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const int col = 8 * nt + 2 * t4;
      const float2 w = f2at(row + V_W * kTile + col), k = f2at(row + V_K * kTile + col);
      const float2 b = f2at(row + V_B * kTile + col), r = f2at(row + V_R * kTile + col);
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
      const float2 w = f2at(row + V_W * kTile + col), a = f2at(row + V_A * kTile + col);
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
      if (in_extent(args.status, xe, dst + base + (size_t)t * vstep + col)) dst[base + (size_t)t * vstep + col] = x;
    }
    __syncthreads();
  }
}

__global__ void __launch_bounds__(kThreads, 2) wkv7_bwd4_out_f32_kernel(const __grid_constant__ BwdArgs args) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  F2Smem& sm = *reinterpret_cast<F2Smem*>(smem_raw);
  const int T = args.T, H = args.H, nchunks = (T + kL - 1) / kL;
  const int head = blockIdx.x / nchunks, n = blockIdx.x % nchunks, bi = head / H, hi = head % H;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t4 = lane & 3;
  const int t0 = n * kL, len = min(kL, T - t0);
  const size_t vstep = (size_t)H * kN, base = ((size_t)bi * T + t0) * vstep + (size_t)hi * kN;
  const float* S0g = args.ckpt + ((size_t)head * args.nck + n) * kN * kN;
  const float* Gcg = static_cast<const float*>(args.carry) + ((size_t)head * nchunks + n) * kN * kN;
  auto gin = [&](int v) { return static_cast<const float*>(args.in[v]); };

  // ---- loads: the chunk's rows (zeros past T) by cp.async; the checkpoint and the carry
  //      through registers (thread rows tid / 16 + 16 q, columns 4 (tid % 16) ..), split into
  //      bf16 tiles, and this warp's part of E = colsum(Gc o S0) from the fp32 values (lanes
  //      l and l ^ 16 hold the same columns)
  for (int idx = tid; idx < 7 * kL * 16; idx += kThreads) {
    const int v = idx / (kL * 16), t = (idx >> 4) % kL, c = idx & 15;
    const float* src = gin(v) + base + (size_t)min(t, len - 1) * vstep + 4 * c;
    cp_async16_zfill(sm.a.raw[v] + t * kN + 4 * c, src,
                     t < len && in_extent(args.status, args.ext.in[v], reinterpret_cast<const float4*>(src)));
  }
  cp_async_commit();
  {
    float4 e = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int idx = tid + kThreads * q, o = (idx >> 4) * kB64 + 4 * (idx & 15);
      const float4* ps = reinterpret_cast<const float4*>(S0g + 4 * idx);
      const float4* pg = reinterpret_cast<const float4*>(Gcg + 4 * idx);
      const float4 s = in_extent(args.status, args.ext.ckpt, ps) ? *ps : make_float4(0.f, 0.f, 0.f, 0.f);
      const float4 gc = in_extent(args.status, args.ext.carry, pg) ? *pg : make_float4(0.f, 0.f, 0.f, 0.f);
      put4_split(sm.u.st.S0[0] + o, sm.u.st.S0[1] + o, s);
      put4_split(sm.u.st.Gc[0] + o, sm.u.st.Gc[1] + o, gc);
      e.x = fmaf(gc.x, s.x, e.x);
      e.y = fmaf(gc.y, s.y, e.y);
      e.z = fmaf(gc.z, s.z, e.z);
      e.w = fmaf(gc.w, s.w, e.w);
    }
    e.x += __shfl_xor_sync(0xffffffffu, e.x, 16);
    e.y += __shfl_xor_sync(0xffffffffu, e.y, 16);
    e.z += __shfl_xor_sync(0xffffffffu, e.z, 16);
    e.w += __shfl_xor_sync(0xffffffffu, e.w, 16);
    if (lane < 16) *reinterpret_cast<float4*>(&sm.Epart[warp][4 * lane]) = e;
  }
  cp_async_wait_all();
  __syncthreads();

  // ---- A: scaled operands, v and dy, in hi and lo parts; thread (lane, warp) forms columns
  //      2 lane, 2 lane + 1 of steps 2 warp, 2 warp + 1. The running products c(t) are taken
  //      per pair of steps and the pairs' products chained in step order.
  {
    const int j = 2 * lane, ta = 2 * warp;
    float2 wv[2];
#pragma unroll
    for (int e = 0; e < 2; ++e)
      wv[e] = ta + e < len ? f2at(sm.a.raw[V_W] + (ta + e) * kN + j) : make_float2(1.f, 1.f);
    const bool safe = decay_is_safe(wv[0].x) && decay_is_safe(wv[0].y) && decay_is_safe(wv[1].x) &&
                      decay_is_safe(wv[1].y);
    *reinterpret_cast<float2*>(&sm.Ppart[warp][j]) = fmul2(wv[0], wv[1]);
    if (__syncthreads_or(!safe)) {
      out_direct_f32(sm.a.raw[0], sm.u.red, S0g, Gcg, len, args, base, vstep, warp, lane);
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
    float2 row[2][6];  // a, r, k, b, v, dy of this thread's two steps
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int o = (ta + e) * kN + j;
      row[e][0] = f2at(sm.a.raw[V_A] + o);
      row[e][1] = f2at(sm.a.raw[V_R] + o);
      row[e][2] = f2at(sm.a.raw[V_K] + o);
      row[e][3] = f2at(sm.a.raw[V_B] + o);
      row[e][4] = f2at(sm.a.raw[V_V] + o);
      row[e][5] = f2at(sm.a.raw[V_DY] + o);
    }
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int t = ta + e, q = t * kB64 + j;
      const float2 w = wv[e], a = row[e][0], r = row[e][1], k = row[e][2], b = row[e][3];
      const float2 cprev = c;
      c = fmul2(c, w);
      const float2 ic = make_float2(rcp_approx(c.x), rcp_approx(c.y)), s = fmul2(cL, ic);
      st_pair_p<2>(sm.Ah[0] + q, sm.Ah[1] + q, fmul2(a, cprev));
      st_pair_p<2>(sm.Rh[0] + q, sm.Rh[1] + q, fmul2(r, c));
      st_pair_p<2>(sm.Kt[0] + q, sm.Kt[1] + q, fmul2(k, ic));
      st_pair_p<2>(sm.Bt[0] + q, sm.Bt[1] + q, fmul2(b, ic));
      st_pair_p<2>(sm.Kb[0] + q, sm.Kb[1] + q, fmul2(k, s));
      st_pair_p<2>(sm.Bb[0] + q, sm.Bb[1] + q, fmul2(b, s));
      st_pair_p<2>(sm.V[0] + q, sm.V[1] + q, row[e][4]);
      st_pair_p<2>(sm.DY[0] + q, sm.DY[1] + q, row[e][5]);
      *reinterpret_cast<float2*>(sm.cS + t * kLD64 + j) = c;
    }
  }
  __syncthreads();  // the fp32 rows are dead from here on: their space takes the tiles below

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
    const bf16_t(*A)[kT64] = warp < 2 ? sm.Ah : sm.Rh;
    const bf16_t(*B)[kT64] = (warp & 1) ? sm.Bt : sm.Kt;
    mm_mk_nk_p<4, 2>(acc, A[0], A[1], kB64, 0, B[0], B[1], kB64, 0, lane);
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
      // T = (I - Mba)^-1 by forward substitution in fp32; lane s (< 16) owns column s
      const int s = lane & 15;
      float col[kL];
      unit_lower_inverse_col16<kLD16>(sm.Mba, s, col);
      if (lane < 16) {
#pragma unroll
        for (int t = 0; t < kL; ++t) put_p<2>(sm.a.t.Tm[0] + t * kB16 + s, sm.a.t.Tm[1] + t * kB16 + s, col[t]);
      }
    } else {
      const int m = warp == 0 ? 0 : warp - 1;  // Mka; Mkr, Mbr
      store_masked16_p<2>(acc, sm.a.t.M[0][m], sm.a.t.M[1][m], true, warp >= 2, g, t4);
    }
#pragma unroll
    for (int kb = 0; kb < 4; ++kb) {  // Gc Bb^T and Gc Kb^T, one A fragment for both
      FragP<2> a, b;
      a_mk_p<2>(a, sm.u.st.Gc[0], sm.u.st.Gc[1], kB64, r0, 16 * kb, lane);
      b_nk_p<2>(b, sm.Bb[0], sm.Bb[1], kB64, 0, 16 * kb, lane);
      mma_pp<2, 2>(X1, a, b);
      b_nk_p<2>(b, sm.Kb[0], sm.Kb[1], kB64, 0, 16 * kb, lane);
      mma_pp<2, 2>(X2, a, b);
    }
  } else {
    mm_mk_nk_p<4, 2>(X1, sm.u.st.S0[0], sm.u.st.S0[1], kB64, r0, sm.Ah[0], sm.Ah[1], kB64, 0, lane);  // S0 A^T
    if (warp == 4) {  // U0 = triu(V DY^T)
      float acc[2][4];
      zero4(acc[0]);
      zero4(acc[1]);
      mm_mk_nk_p<4, 2>(acc, sm.V[0], sm.V[1], kB64, 0, sm.DY[0], sm.DY[1], kB64, 0, lane);
      store_masked16_p<2>(acc, sm.a.t.U[0][0], sm.a.t.U[1][0], false, true, g, t4);
    }
  }
  __syncthreads();

  // ---- C: DSA^T = (Gc Bb^T + DY^T Mbr) T, DV^T += DY^T Mkr + DSA^T Mka and dv (warps 0-3);
  //      SA^T = (S0 A^T + V^T Mka^T) T^T (warps 4-7); sa and dsa stored [t][i] in two parts
  {
    FragP<2> b, p;
    float Y[2][4];
    zero4(Y[0]);
    zero4(Y[1]);
    if (warp < 4) {
      FragP<2> aD;
      a_km_p<2>(aD, sm.DY[0], sm.DY[1], kB64, r0, 0, lane);           // DY^T
      b_kn_p<2>(b, sm.a.t.M[0][2], sm.a.t.M[1][2], kB16, 0, 0, lane);  // Mbr
      mma_pp<2, 2>(X1, aD, b);
      b_kn_p<2>(b, sm.a.t.M[0][1], sm.a.t.M[1][1], kB16, 0, 0, lane);  // Mkr
      mma_pp<2, 2>(X2, aD, b);
      c2a_p<2>(p, X1[0], X1[1]);
      b_kn_p<2>(b, sm.a.t.Tm[0], sm.a.t.Tm[1], kB16, 0, 0, lane);  // T
      mma_pp<2, 2>(Y, p, b);
    } else {
      FragP<2> aV;
      a_km_p<2>(aV, sm.V[0], sm.V[1], kB64, r0, 0, lane);              // V^T
      b_nk_p<2>(b, sm.a.t.M[0][0], sm.a.t.M[1][0], kB16, 0, 0, lane);  // Mka^T
      mma_pp<2, 2>(X1, aV, b);
      c2a_p<2>(p, X1[0], X1[1]);
      b_nk_p<2>(b, sm.a.t.Tm[0], sm.a.t.Tm[1], kB16, 0, 0, lane);  // T^T
      mma_pp<2, 2>(Y, p, b);
    }
    c2a_p<2>(p, Y[0], Y[1]);
    const int so = ((lane & 7) + (lane >> 4) * 8) * kB64 + r0 + ((lane >> 3) & 1) * 8;
    stsm4t((warp < 4 ? sm.a.t.DSA[0] : sm.a.t.SA[0]) + so, p.h);
    stsm4t((warp < 4 ? sm.a.t.DSA[1] : sm.a.t.SA[1]) + so, p.l);
    if (warp < 4) {  // DV^T += DSA^T Mka (DSA^T from the registers just stored), then dv
      b_kn_p<2>(b, sm.a.t.M[0][0], sm.a.t.M[1][0], kB16, 0, 0, lane);  // Mka
      mma_pp<2, 2>(X2, p, b);
#pragma unroll
      for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int t = 8 * q + 2 * t4 + e;
          if (t < len) {
            float* dst = args.dv + base + (size_t)t * vstep + r0 + g;
            if (in_extent(args.status, args.ext.dv, dst)) dst[0] = X2[q][e];
            if (in_extent(args.status, args.ext.dv, dst + 8)) dst[8] = X2[q][2 + e];
          }
        }
    }
  }
  __syncthreads();

  // ---- D: U1 = triu(V DSA^T, 1), U2 = triu(SA DY^T), U3 = triu(SA DSA^T, 1) (warps 5-7)
  if (warp >= 5) {
    const int u = warp - 4;
    float acc[2][4];
    zero4(acc[0]);
    zero4(acc[1]);
    const bf16_t(*A)[kT64] = u == 1 ? sm.V : sm.a.t.SA;
    const bf16_t(*B)[kT64] = u == 2 ? sm.DY : sm.a.t.DSA;
    mm_mk_nk_p<4, 2>(acc, A[0], A[1], kB64, 0, B[0], B[1], kB64, 0, lane);
    store_masked16_p<2>(acc, sm.a.t.U[0][u], sm.a.t.U[1][u], false, u == 2, g, t4);
  }
  __syncthreads();

  // ---- E: column products, 8 warps: warp (grp, jb) covers columns j0 .. j0+15 of
  //      dk~, db~ (grp 0) or dr^, da^ (grp 1)
  const int grp = warp >> 2, jb = warp & 3, j0 = 16 * jb;
  // per element (t, j) of this warp: grp 0: 1/c, k, b; grp 1: c, c(t-1), r, a (k, b, r, a from
  // global memory; zero past the sequence), requested before the column products
  float2 q0[2][2], q1[2][2], q2[2][2], q3[2][2];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int t = g + 8 * h, col = j0 + 8 * nt + 2 * t4;
      const size_t off = base + (size_t)t * vstep + col;
      auto ld = [&](int v) {
        const float2* p = reinterpret_cast<const float2*>(gin(v) + off);
        return t < len && in_extent(args.status, args.ext.in[v], p) ? *p : make_float2(0.f, 0.f);
      };
      const float2 c = *reinterpret_cast<const float2*>(sm.cS + t * kLD64 + col);
      if (grp == 0) {
        q0[nt][h] = make_float2(rcp_approx(c.x), rcp_approx(c.y));
        q1[nt][h] = ld(V_K);
        q2[nt][h] = ld(V_B);
        q3[nt][h] = make_float2(0.f, 0.f);
      } else {
        q0[nt][h] = c;
        q1[nt][h] = t ? *reinterpret_cast<const float2*>(sm.cS + (t - 1) * kLD64 + col) : make_float2(1.f, 1.f);
        q2[nt][h] = ld(V_R);
        q3[nt][h] = ld(V_A);
      }
    }
  float P0[2][4], P1[2][4];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    zero4(P0[nt]);
    zero4(P1[nt]);
  }
  {  // sums over the rows i: V Gc, SA Gc (grp 0); DY S0, DSA S0 (grp 1)
    const bf16_t(*Bm)[kN * kB64] = grp ? sm.u.st.S0 : sm.u.st.Gc;
    const bf16_t(*X)[kT64] = grp ? sm.DY : sm.V;
    const bf16_t(*Y)[kT64] = grp ? sm.a.t.DSA : sm.a.t.SA;
#pragma unroll
    for (int kb = 0; kb < 4; ++kb) {
      FragP<2> a0, a1, b;
      a_mk_p<2>(a0, X[0], X[1], kB64, 0, 16 * kb, lane);
      a_mk_p<2>(a1, Y[0], Y[1], kB64, 0, 16 * kb, lane);
      b_kn_p<2>(b, Bm[0], Bm[1], kB64, j0, 16 * kb, lane);
      mma_pp<2, 2>(P0, a0, b);
      mma_pp<2, 2>(P1, a1, b);
    }
  }
  {
    // This warp's part of the dw anchors, from the column products (c(L) E is added later):
    //   colsum(Gc o S(L)) = c(L) E + sum_t (Kb o V Gc + Bb o SA Gc)       (grp 0)
    //   colsum(Gc' o S0)  = c(L) E + sum_t (R^ o DY S0 + A^ o DSA S0)     (grp 1)
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
    FragP<2> u0, u1, u2, u3, b;
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
      a_mk_p<2>(u0, sm.a.t.U[0][0], sm.a.t.U[1][0], kB16, 0, 0, lane);
      a_mk_p<2>(u1, sm.a.t.U[0][1], sm.a.t.U[1][1], kB16, 0, 0, lane);
      a_mk_p<2>(u2, sm.a.t.U[0][2], sm.a.t.U[1][2], kB16, 0, 0, lane);
      a_mk_p<2>(u3, sm.a.t.U[0][3], sm.a.t.U[1][3], kB16, 0, 0, lane);
      b_kn_p<2>(b, sm.Rh[0], sm.Rh[1], kB64, j0, 0, lane);
      mma_pp<2, 2>(P0, u0, b);
      mma_pp<2, 2>(P1, u2, b);
      b_kn_p<2>(b, sm.Ah[0], sm.Ah[1], kB64, j0, 0, lane);
      mma_pp<2, 2>(P0, u1, b);
      mma_pp<2, 2>(P1, u3, b);
    } else {
      a_km_p<2>(u0, sm.a.t.U[0][0], sm.a.t.U[1][0], kB16, 0, 0, lane);
      a_km_p<2>(u1, sm.a.t.U[0][1], sm.a.t.U[1][1], kB16, 0, 0, lane);
      a_km_p<2>(u2, sm.a.t.U[0][2], sm.a.t.U[1][2], kB16, 0, 0, lane);
      a_km_p<2>(u3, sm.a.t.U[0][3], sm.a.t.U[1][3], kB16, 0, 0, lane);
      b_kn_p<2>(b, sm.Kt[0], sm.Kt[1], kB64, j0, 0, lane);
      mma_pp<2, 2>(P0, u0, b);
      mma_pp<2, 2>(P1, u1, b);
      b_kn_p<2>(b, sm.Bt[0], sm.Bt[1], kB64, j0, 0, lane);
      mma_pp<2, 2>(P0, u2, b);
      mma_pp<2, 2>(P1, u3, b);
    }
  }
  // unscale: dk = dk~ / c, db = db~ / c (grp 0); dr = dr^ c, da = da^ c(t-1) (grp 1); and this
  // group's part of x = r dr - k dk - b db + a da
  float X[2][4], AD[2][4];
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
  float* XK = sm.u.xch[0];  // [t][j] stride kLD64
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
        float2* p0 = reinterpret_cast<float2*>(out0 + off);
        float2* p1 = reinterpret_cast<float2*>(out1 + off);
        if (in_extent(args.status, x0, p0)) *p0 = make_float2(P0[nt][2 * h], P0[nt][2 * h + 1]);
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
    float e = 0.f;
#pragma unroll
    for (int w8 = 0; w8 < 8; ++w8) e += sm.Epart[w8][col];
    float run = sm.cLs[col] * e + sm.anc[upper][col];
    float wv[kL / 2];
#pragma unroll
    for (int q = 0; q < kL / 2; ++q) {  // this thread's decays, requested at once
      const int t = upper ? kL - 1 - q : q;
      const float* p = gin(V_W) + base + (size_t)t * vstep + col;
      wv[q] = t < len && in_extent(args.status, args.ext.in[V_W], p) ? *p : 1.f;
    }
#pragma unroll
    for (int q = 0; q < kL / 2; ++q) {
      const int t = upper ? kL - 1 - q : q;
      const float x = XK[t * kLD64 + col] + XR[t * kLD64 + col];
      if (upper) run += x;  // end anchor plus the x of the steps from t on
      const float v = (run - XA[t * kLD64 + col]) * rcp_approx(wv[q]);
      float* pw = args.dw + base + (size_t)t * vstep + col;
      if (t < len && in_extent(args.status, args.ext.dw, pw)) *pw = v;
      if (!upper) run -= x;  // start anchor minus the x of the steps before t
    }
  }
}

}  // namespace

cudaError_t launch_bwd4_out_f32(const BwdArgs& args, cudaStream_t stream) {
  const size_t smem = sizeof(F2Smem);
  static_assert(sizeof(F2Smem) <= 113 * 1024, "two CTAs per SM need at most 113 KB each");
  cudaError_t e =
      cudaFuncSetAttribute(wkv7_bwd4_out_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const long long ntasks = (long long)args.B * args.H * ((args.T + kL - 1) / kL);
  if (ntasks <= 0) return cudaSuccess;
  if (ntasks >= (1ll << 31)) return cudaErrorInvalidValue;
  wkv7_bwd4_out_f32_kernel<<<(unsigned)ntasks, kThreads, smem, stream>>>(args);
  return cudaGetLastError();
}

}  // namespace wkv7
