// RWKV-8 normalized recurrence, backward-through-time, in chunks of 16 steps.
//
// Gradient formulas of backward_chunk_impl (burn_dragon_kernel,
// "src/sequence/rwkv8/backward.rs"), with G_t = dL/d rho_after_t and
// Gn_t = dL/d n_after_t carried backwards:
//     g_qw[t][l] = <rho_t[l], dy_t> / (n_t[l] + EPS)          (rho_t, n_t: state before step t)
//     g_n[t][l]  = -U[t][l] <rho_t[l], dy_t> / (n_t[l] + EPS),  U = qw / (n + EPS)
//     dq_t = (g_qw - <g_qw, qw>) / (sum q_t + EPS) + G_t v_t + Gn_t
//     dv_t = G_t^T q_t
//     ddecay += sum_e G_t (.) rho_t + Gn_t (.) n_t
//     G_{t-1} = d (.) G_t + U[t] dy_t^T,   Gn_{t-1} = d (.) Gn_t + g_n[t]
// In a chunk (tau = 0 .. len-1 from the chunk start, G15 = G at its last step,
// rho0 / n0 = the checkpointed state at its first step), with M = DY V^T:
//     R[tau]  = <rho_tau, dy_tau> = d^tau R0[tau] + sum_{s<tau} d^(tau-1-s) q_s M[tau][s],  R0 = DY rho0^T
//     Gv[tau] = (G_tau v_tau)    = d^(len-1-tau) W[tau] + sum_{s>tau} d^(s-1-tau) U[s] M[s][tau],  W = V G15^T
//     dv      = (q d^(len-1-tau)) G15 + A^T DY,  A[s][tau] = sum_l U[s] q_tau d^(s-1-tau)
//     Gn_tau  = d^(len-1-tau) Gn15 + sum_{s>tau} d^(s-1-tau) g_n[s]
//     G_start = d^len G15 + sum_s (U[s] d^s) dy_s^T
// and the decay gradient of the chunk, sum_tau sum_e G_tau rho_tau, in four
// closed-form terms (the products of the two affine expansions):
//     len d^(len-1) <G15[l], rho0[l]> + sum_s s d^(s-1) U[s] R0[s]
//   + sum_s (len-1-s) d^(len-2-s) q_s W[s] + sum_{s'<s-1} (s-1-s') d^(s-2-s') q_s' U[s] M[s][s'].
// (d^k is per latent l; every exponent is >= 0, so no power of d is divided.)
//
// One CTA of 256 threads per (b, h) walks the chunks from the last to the
// first, fp32 FFMA on the CUDA cores. The carried G lives in registers (4 x 4
// per thread) with a copy in shared memory for the products that read it;
// the checkpointed state and the next chunk's inputs are copied in with
// cp.async while the current chunk is processed. ddecay is accumulated per
// thread over all chunks and reduced once, in a fixed order, at the end.
#include <cuda_runtime.h>

#include "rwkv8.h"
#include "rwkv8_launch.h"

namespace rwkv8 {
namespace {

constexpr int kThreads = 256;
constexpr int kP = 68;  // row pitch (floats) of 64-wide tiles read by row

struct BwdSmem {
  float qs[2][kC][kP];
  float vs[2][kC][kP];
  float dys[2][kC][kP];
  float rho0[2][kL][kP];
  float n0[2][kL];
  float G[kL][kP];       // carried G (last step of the current chunk)
  float pw[kC + 1][kL];  // d_l^k
  float U[kC][kL];
  float Ut[kC][kL];      // U[s][l] d_l^s
  float QG[kC][kL];      // q_s[l] d_l^(len-1-s), zero for s >= len
  float NB[kC][kL];      // n before every step
  float R0[kC][kL];
  float W[kC][kL];
  float gn[kC][kL];      // g_n
  float M[kC][kC + 1];
  float A[kC][kC + 1];   // strictly lower; the rest stays zero
  float mend[4][kL];
  float sqp[2][kC];
  float rowp[2][kC];
  float gnst[2][kL];     // carried Gn, by chunk parity
  float ddpart[16 + 4][kL];
};

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<unsigned>(__cvta_generic_to_shared(dst))),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Sum of a 4 x 4 tile over the four lanes that share it (lane bits 3 and 4,
// kq = lane >> 3), leaving row kq of the sum in `out`: a reduce-scatter in two
// exchange steps instead of an all-reduce of all sixteen values.
__device__ __forceinline__ void reduce_scatter4(const float (&a)[4][4], int kq, float (&out)[4]) {
  const bool hi = (kq & 2) != 0;
  float k2[2][4];
#pragma unroll
  for (int ii = 0; ii < 2; ++ii)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float keep = hi ? a[2 + ii][j] : a[ii][j];
      const float send = hi ? a[ii][j] : a[2 + ii][j];
      k2[ii][j] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
  const bool odd = (kq & 1) != 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float keep = odd ? k2[1][j] : k2[0][j];
    const float send = odd ? k2[0][j] : k2[1][j];
    out[j] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
  }
}

__device__ __forceinline__ float dot4(const float4 a, const float4 b) {
  return fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, a.w * b.w)));
}

struct Heads {
  const float *q, *v, *dy, *ck_rho, *ck_n;
  int T;
};

// Chunk c of q, v, dy and its checkpointed state into buffer `buf` (rows past
// the end of the sequence zero-filled).
__device__ __forceinline__ void load_chunk(BwdSmem& sm, int buf, const Heads& hd, int c, int tid) {
  const int row = tid >> 4, col = (tid & 15) * 4;
  const int t = c * kC + row;
  if (t < hd.T) {
    cp_async16(&sm.qs[buf][row][col], hd.q + (size_t)t * kL + col);
    cp_async16(&sm.vs[buf][row][col], hd.v + (size_t)t * kE + col);
    cp_async16(&sm.dys[buf][row][col], hd.dy + (size_t)t * kE + col);
  } else {
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    *reinterpret_cast<float4*>(&sm.qs[buf][row][col]) = z;
    *reinterpret_cast<float4*>(&sm.vs[buf][row][col]) = z;
    *reinterpret_cast<float4*>(&sm.dys[buf][row][col]) = z;
  }
  const float* ck = hd.ck_rho + (size_t)c * kL * kE;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = row + 16 * i;
    cp_async16(&sm.rho0[buf][r][col], ck + (size_t)r * kE + col);
  }
  if (tid < kL / 4) cp_async16(&sm.n0[buf][4 * tid], hd.ck_n + (size_t)c * kL + 4 * tid);
  cp_async_commit();
}

// Per-element work of one chunk for the rows tau = SEG + 4 j of latent l:
// R, the weights' gradient, g_n, Gv and the decay-gradient terms that need
// them. Every register index is a compile-time constant.
template <int SEG>
__device__ __forceinline__ void chunk_elements(BwdSmem& sm, int buf, int l, int len, const float (&pcol)[kC + 1],
                                               float (&gq)[4], float (&gv)[4], float (&nb)[4], float (&qwv)[4],
                                               float& dd) {
  float qcol[kC], ucol[kC];
#pragma unroll
  for (int s = 0; s < kC; ++s) {
    qcol[s] = sm.qs[buf][s][l];
    ucol[s] = sm.U[s][l];
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int tau = SEG + 4 * j;
    const float r0 = sm.R0[tau][l];
    const float wv = sm.W[tau][l];
    float R = pcol[tau] * r0;
    float d4 = 0.f;
#pragma unroll
    for (int s = 0; s < kC; ++s) {
      if (s < tau) {
        const float m = sm.M[tau][s];
        const float qm = qcol[s] * m;
        R = fmaf(pcol[tau - 1 - s], qm, R);
        if (s <= tau - 2) d4 = fmaf((float)(tau - 1 - s) * pcol[tau - 2 - s], qm, d4);
      }
    }
    float G = 0.f;
#pragma unroll
    for (int s = 0; s < kC; ++s)
      if (s > tau) G = fmaf(pcol[s - 1 - tau] * ucol[s], sm.M[s][tau], G);
    if (tau < len) G = fmaf(sm.pw[len - 1 - tau][l], wv, G);
    const float n = sm.NB[tau][l];
    const float g = __fdividef(R, n + kEps);  // denominator >= 1e-6
    gq[j] = g;
    gv[j] = G;
    nb[j] = n;
    qwv[j] = qcol[tau];
    sm.gn[tau][l] = -ucol[tau] * g;
    float ddj = ucol[tau] * d4;
    if (tau >= 1) ddj = fmaf((float)tau * pcol[tau - 1] * ucol[tau], r0, ddj);
    if (tau <= len - 2) ddj = fmaf((float)(len - 1 - tau) * sm.pw[len - 2 - tau][l] * qcol[tau], wv, ddj);
    dd += ddj;
  }
}

template <int SEG>
__device__ __forceinline__ void chunk_outputs(BwdSmem& sm, int buf, int l, int len, int c, const float (&pcol)[kC + 1],
                                              const float (&gq)[4], const float (&gv)[4], const float (&nb)[4],
                                              const float (&qv)[4], float& dd, float* dqh) {
  float gcol[kC];
#pragma unroll
  for (int s = 0; s < kC; ++s) gcol[s] = sm.gn[s][l];
  const float gn15 = sm.gnst[buf][l];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int tau = SEG + 4 * j;
    if (tau < len) {
      float gnt = sm.pw[len - 1 - tau][l] * gn15;
#pragma unroll
      for (int s = 0; s < kC; ++s)
        if (s > tau) gnt = fmaf(pcol[s - 1 - tau], gcol[s], gnt);
      dd = fmaf(gnt, nb[j], dd);
      const float sq = sm.sqp[0][tau] + sm.sqp[1][tau] + kEps;
      const float rowsum = sm.rowp[0][tau] + sm.rowp[1][tau];
      dqh[((size_t)c * kC + tau) * kL + l] = (gq[j] - rowsum) / sq + gv[j] + gnt;
    }
  }
  (void)qv;
  if (SEG == 0) {
    // Gn at the chunk start: d^len Gn15 + sum_s d^s g_n[s]
    float g0 = sm.pw[len][l] * gn15;
#pragma unroll
    for (int s = 0; s < kC; ++s) g0 = fmaf(pcol[s], gcol[s], g0);
    sm.gnst[buf ^ 1][l] = g0;
  }
}

__global__ void __launch_bounds__(kThreads, 1) rwkv8_bwd_kernel(const Args a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  BwdSmem& sm = *reinterpret_cast<BwdSmem*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int bh = blockIdx.x, h = bh % a.H, b = bh / a.H;
  const int T = a.T, nck = (T + kC - 1) / kC;
  Heads hd;
  hd.T = T;
  hd.q = a.q + (size_t)bh * T * kL;
  hd.v = a.v + ((size_t)b * a.Hv + (a.Hv == 1 ? 0 : h)) * T * kE;
  hd.dy = a.dy + (size_t)bh * T * kE;
  hd.ck_rho = a.ckpt + (size_t)bh * nck * kL * kE;
  hd.ck_n = a.ckpt + ckpt_norm_offset(a.B, T, a.H) + (size_t)bh * nck * kL;
  float* dqh = a.dq + (size_t)bh * T * kL;
  float* dvh = a.dv + (size_t)bh * T * kE;

  load_chunk(sm, 0, hd, nck - 1, tid);

  // Roles (see the forward for the scan, A and state-tile roles).
  const int l_s = tid & 63, seg = tid >> 6;
  // A role: the 120 pairs (at, as), as < at, in four rounds; in round r the
  // eight lanes of group ag of warp w take pair p = 4 (8 r + w) + ag and split
  // the latent range between them (conflict-free rows). Pairs past 119 are
  // computed on a valid pair and not stored.
  const int ag = lane >> 3, a8 = lane & 7;
  int apair[4];
#pragma unroll
  for (int rr = 0; rr < 4; ++rr) {
    const int p = 4 * (8 * rr + w) + ag;
    int at = 1, as = min(p, 119);
    while (as >= at) {
      as -= at;
      ++at;
    }
    apair[rr] = p < 120 ? (at << 8) | as : -((at << 8) | as) - 1;
  }
  const int ec = (lane & 7) | ((w & 1) << 3);  // 4 columns of a 64-wide output
  const int kq = lane >> 3, rt = w >> 1;
  const int lt = (lane >> 3) + 4 * (w >> 1);
  const int mt = tid >> 4, ms = tid & 15;  // M role

  if (tid < kL) {
    const float d = a.decay[(size_t)h * kL + tid];
    float p = 1.f;
    for (int k = 0; k <= kC; ++k) {
      sm.pw[k][tid] = p;
      p *= d;
    }
    sm.gnst[0][tid] = a.d_rho_norm_final ? a.d_rho_norm_final[(size_t)bh * kL + tid] : 0.f;
  }
  for (int i = tid; i < kC * (kC + 1); i += kThreads) (&sm.A[0][0])[i] = 0.f;
  float r[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (a.d_rho_final)
      x = *reinterpret_cast<const float4*>(a.d_rho_final + ((size_t)bh * kL + 4 * lt + i) * kE + 4 * ec);
    r[i][0] = x.x, r[i][1] = x.y, r[i][2] = x.z, r[i][3] = x.w;
    *reinterpret_cast<float4*>(&sm.G[4 * lt + i][4 * ec]) = x;
  }
  __syncthreads();
  float pcol[kC + 1];
#pragma unroll
  for (int k = 0; k <= kC; ++k) pcol[k] = sm.pw[k][l_s];
  float dd_tile[4] = {0.f, 0.f, 0.f, 0.f};  // ddecay of rows 4 lt + i (state-tile role)
  float dd_col = 0.f;                       // ddecay of latent l_s (scan role)

  for (int it = 0; it < nck; ++it) {
    const int c = nck - 1 - it;
    const int buf = it & 1;
    const int len = min(kC, T - c * kC);
    cp_async_wait_all();
    __syncthreads();

    // ---- phase 1: local norm scan, row sums, M, R0 = DY rho0^T, W = V G^T,
    //      <G, rho0> per row, prefetch of the previous chunk
    float x[4], loc[4];
    {
      const float d = pcol[1];
      float m = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        x[j] = sm.qs[buf][4 * seg + j][l_s];
        loc[j] = m;
        m = fmaf(d, m, x[j]);
      }
      sm.mend[seg][l_s] = m;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float s = x[j];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0) sm.sqp[w & 1][4 * seg + j] = s;
      }
    }
    {
      float acc = 0.f;
#pragma unroll
      for (int e = 0; e < kE; e += 4)
        acc += dot4(*reinterpret_cast<const float4*>(&sm.dys[buf][mt][e]),
                    *reinterpret_cast<const float4*>(&sm.vs[buf][ms][e]));
      sm.M[mt][ms] = acc;
    }
    {
      float ar[4][4], aw[4][4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) ar[i][j] = aw[i][j] = 0.f;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const int e = 16 * kq + 4 * kk;
        float4 dyv[4], vv[4], rv[4], gv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          dyv[i] = *reinterpret_cast<const float4*>(&sm.dys[buf][4 * rt + i][e]);
          vv[i] = *reinterpret_cast<const float4*>(&sm.vs[buf][4 * rt + i][e]);
          rv[i] = *reinterpret_cast<const float4*>(&sm.rho0[buf][ec + 16 * i][e]);
          gv[i] = *reinterpret_cast<const float4*>(&sm.G[ec + 16 * i][e]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            ar[i][j] += dot4(dyv[i], rv[j]);
            aw[i][j] += dot4(vv[i], gv[j]);
          }
      }
      // lane group kq keeps and stores row 4 rt + kq
      float vr[4], vw[4];
      reduce_scatter4(ar, kq, vr);
      reduce_scatter4(aw, kq, vw);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        sm.R0[4 * rt + kq][ec + 16 * j] = vr[j];
        sm.W[4 * rt + kq][ec + 16 * j] = vw[j];
      }
    }
    {
      const float4 pl = *reinterpret_cast<const float4*>(&sm.pw[len - 1][4 * lt]);
      const float pd[4] = {pl.x, pl.y, pl.z, pl.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 s0 = *reinterpret_cast<const float4*>(&sm.rho0[buf][4 * lt + i][4 * ec]);
        const float p = r[i][0] * s0.x + r[i][1] * s0.y + r[i][2] * s0.z + r[i][3] * s0.w;
        dd_tile[i] = fmaf((float)len * pd[i], p, dd_tile[i]);
      }
    }
    if (c > 0) load_chunk(sm, buf ^ 1, hd, c - 1, tid);
    __syncthreads();

    // ---- phase 2: n before every step, U, U d^s, q d^(len-1-s)
    {
      const float n0 = sm.n0[buf][l_s];
      float start = n0;
      for (int s2 = 0; s2 < seg; ++s2) start = fmaf(pcol[4], start, sm.mend[s2][l_s]);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int tau = 4 * seg + j;
        const float nbv = fmaf(sm.pw[j][l_s], start, loc[j]);
        const float sq = sm.sqp[0][tau] + sm.sqp[1][tau] + kEps;
        const float u = __fdividef(x[j], sq * (nbv + kEps));  // denominator >= 1e-12
        sm.NB[tau][l_s] = nbv;
        sm.U[tau][l_s] = u;
        sm.Ut[tau][l_s] = u * sm.pw[tau][l_s];
        sm.QG[tau][l_s] = tau < len ? x[j] * sm.pw[len - 1 - tau][l_s] : 0.f;
      }
    }
    __syncthreads();

    // ---- phase 3: per-element terms, A, dv = QG G (partial sums over l)
    float gq[4], gvv[4], nb[4], qv[4];
    switch (seg) {
      case 0: chunk_elements<0>(sm, buf, l_s, len, pcol, gq, gvv, nb, qv, dd_col); break;
      case 1: chunk_elements<1>(sm, buf, l_s, len, pcol, gq, gvv, nb, qv, dd_col); break;
      case 2: chunk_elements<2>(sm, buf, l_s, len, pcol, gq, gvv, nb, qv, dd_col); break;
      default: chunk_elements<3>(sm, buf, l_s, len, pcol, gq, gvv, nb, qv, dd_col); break;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int tau = seg + 4 * j;
      const float sq = sm.sqp[0][tau] + sm.sqp[1][tau] + kEps;
      float s = gq[j] * (qv[j] / sq);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      if (lane == 0) sm.rowp[w & 1][tau] = s;
    }
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      const int code = apair[rr] >= 0 ? apair[rr] : -apair[rr] - 1;
      const int at = code >> 8, as = code & 255, k = at - 1 - as;
      float acc = 0.f;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int l = 32 * hh + 4 * a8;
        const float4 u = *reinterpret_cast<const float4*>(&sm.U[at][l]);
        const float4 q = *reinterpret_cast<const float4*>(&sm.qs[buf][as][l]);
        const float4 p = *reinterpret_cast<const float4*>(&sm.pw[k][l]);
        acc = fmaf(u.x * q.x, p.x, acc);
        acc = fmaf(u.y * q.y, p.y, acc);
        acc = fmaf(u.z * q.z, p.z, acc);
        acc = fmaf(u.w * q.w, p.w, acc);
      }
      acc += __shfl_xor_sync(0xffffffffu, acc, 1);
      acc += __shfl_xor_sync(0xffffffffu, acc, 2);
      acc += __shfl_xor_sync(0xffffffffu, acc, 4);
      if (a8 == 0 && apair[rr] >= 0) sm.A[at][as] = acc;
    }
    float dv4[4];
    {
      float acc[4][4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const int l = 16 * kq + 4 * kk;
        float4 qg[4], gr[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          qg[i] = *reinterpret_cast<const float4*>(&sm.QG[4 * rt + i][l]);
          gr[i] = *reinterpret_cast<const float4*>(&sm.G[l + i][4 * ec]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float qq[4] = {qg[i].x, qg[i].y, qg[i].z, qg[i].w};
#pragma unroll
          for (int k2 = 0; k2 < 4; ++k2) {
            acc[i][0] = fmaf(qq[k2], gr[k2].x, acc[i][0]);
            acc[i][1] = fmaf(qq[k2], gr[k2].y, acc[i][1]);
            acc[i][2] = fmaf(qq[k2], gr[k2].z, acc[i][2]);
            acc[i][3] = fmaf(qq[k2], gr[k2].w, acc[i][3]);
          }
        }
      }
      reduce_scatter4(acc, kq, dv4);
    }
    __syncthreads();  // A, g_n and the row sums complete; every read of G done

    // ---- phase 4: dq, dv, the carried Gn and G
    switch (seg) {
      case 0: chunk_outputs<0>(sm, buf, l_s, len, c, pcol, gq, gvv, nb, qv, dd_col, dqh); break;
      case 1: chunk_outputs<1>(sm, buf, l_s, len, c, pcol, gq, gvv, nb, qv, dd_col, dqh); break;
      case 2: chunk_outputs<2>(sm, buf, l_s, len, c, pcol, gq, gvv, nb, qv, dd_col, dqh); break;
      default: chunk_outputs<3>(sm, buf, l_s, len, c, pcol, gq, gvv, nb, qv, dd_col, dqh); break;
    }
    {
      const int tau = 4 * rt + kq;
      // A[s][tau] is zero for s <= tau; the warp's rows start at 4 rt
#pragma unroll 4
      for (int s = 4 * rt + 1; s < kC; ++s) {
        const float al = sm.A[s][tau];
        const float4 dd = *reinterpret_cast<const float4*>(&sm.dys[buf][s][4 * ec]);
        dv4[0] = fmaf(al, dd.x, dv4[0]);
        dv4[1] = fmaf(al, dd.y, dv4[1]);
        dv4[2] = fmaf(al, dd.z, dv4[2]);
        dv4[3] = fmaf(al, dd.w, dv4[3]);
      }
      if (tau < len)
        *reinterpret_cast<float4*>(dvh + ((size_t)c * kC + tau) * kE + 4 * ec) = make_float4(dv4[0], dv4[1], dv4[2], dv4[3]);
    }
    {
      const float4 pl = *reinterpret_cast<const float4*>(&sm.pw[len][4 * lt]);
      const float pd[4] = {pl.x, pl.y, pl.z, pl.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) r[i][j] *= pd[i];
#pragma unroll 4
      for (int s = 0; s < kC; ++s) {
        const float4 ut = *reinterpret_cast<const float4*>(&sm.Ut[s][4 * lt]);
        const float4 dd = *reinterpret_cast<const float4*>(&sm.dys[buf][s][4 * ec]);
        const float uu[4] = {ut.x, ut.y, ut.z, ut.w}, yy[4] = {dd.x, dd.y, dd.z, dd.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) r[i][j] = fmaf(uu[i], yy[j], r[i][j]);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
        *reinterpret_cast<float4*>(&sm.G[4 * lt + i][4 * ec]) = make_float4(r[i][0], r[i][1], r[i][2], r[i][3]);
    }
  }
  __syncthreads();
  if (a.d_rho_init) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
      *reinterpret_cast<float4*>(a.d_rho_init + ((size_t)bh * kL + 4 * lt + i) * kE + 4 * ec) =
          make_float4(r[i][0], r[i][1], r[i][2], r[i][3]);
  }
  if (a.d_rho_norm_init && tid < kL) a.d_rho_norm_init[(size_t)bh * kL + tid] = sm.gnst[nck & 1][tid];
  // ddecay of this (b, h): a fixed-order sum of every thread's share
#pragma unroll
  for (int i = 0; i < 4; ++i) sm.ddpart[ec][4 * lt + i] = dd_tile[i];
  sm.ddpart[16 + seg][l_s] = dd_col;
  __syncthreads();
  if (tid < kL) {
    float s = 0.f;
    for (int p = 0; p < 20; ++p) s += sm.ddpart[p][tid];
    a.ddecay_bh[(size_t)bh * kL + tid] = s;
  }
}

// out[i] = sum_g in[g * stride + i], g in order.
__global__ void group_sum_kernel(const float* __restrict__ in, float* __restrict__ out, size_t n, size_t stride,
                                 int groups) {
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    float s = 0.f;
    for (int g = 0; g < groups; ++g) s += in[(size_t)g * stride + i];
    out[i] = s;
  }
}

}  // namespace

cudaError_t launch_backward(const Args& a, cudaStream_t s) {
  const size_t smem = sizeof(BwdSmem);
  cudaError_t e = cudaFuncSetAttribute(rwkv8_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  rwkv8_bwd_kernel<<<a.B * a.H, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_group_sum(const float* in, float* out, size_t n, size_t stride, int groups, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const int threads = 256;
  size_t blocks = (n + threads - 1) / threads;
  if (blocks > 152 * 8) blocks = 152 * 8;
  group_sum_kernel<<<(unsigned)blocks, threads, 0, s>>>(in, out, n, stride, groups);
  return cudaGetLastError();
}

cudaError_t launch_head_sum(const float* part, float* dv, int B, int H, int T, cudaStream_t s) {
  // dv[b][0][t][e] = sum_h part[b][h][t][e]: one group sum per batch row
  const size_t per = (size_t)T * kE;
  for (int b = 0; b < B; ++b) {
    cudaError_t e = launch_group_sum(part + (size_t)b * H * per, dv + (size_t)b * per, per, per, H, s);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace rwkv8
