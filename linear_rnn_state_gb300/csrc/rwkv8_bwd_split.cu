// RWKV-8 normalized recurrence, backward-through-time, split the way the
// forward is: the carried gradients alone, then every chunk at once.
//
// With G15, Gn15 the gradients w.r.t. the state (rho, n) after a chunk's last
// step, the formulas of backward_chunk_impl (burn_dragon_kernel,
// "src/sequence/rwkv8/backward.rs") over a chunk of len steps (tau, s from
// its start; d^k per latent l) give the gradients at its start as
//     G_start  = d^len (.) G15  + sum_s (U[s] d^s) dy_s^T
//     Gn_start = d^len (.) Gn15 + sum_s d^s (.) g_n[s],   g_n[s] = -U[s] R[s] / (n_s + EPS)
//     R[tau]   = d^tau R0[tau] + sum_{s<tau} d^(tau-1-s) q_s M[tau][s]
// with R0 = DY rho0^T (rho0 the checkpointed state at the chunk start) and
// M = DY V^T. Neither chain term depends on the carried gradients, so between
// chunks the chain is one multiply-add per element; and once G15, Gn15 of
// every chunk are known, its dq, dv and decay terms need nothing from any
// other chunk.
//
// rwkv8_bwd_r0_kernel: R0 of every chunk at once (one CTA per chunk), fp32 FFMA.
// rwkv8_bwd_chain_kernel: one CTA of 256 threads per (b, h), chunks from the
// last to the first, inputs, checkpoints and R0 through a four-chunk cp.async
// ring. Per chunk it stores G15, Gn15 and <G15[l], rho0[l]> to the workspace,
// then advances G (accumulator tiles) and Gn.
// rwkv8_bwd_chunk_kernel: one CTA of 256 threads per (b, h, chunk): the rest
// of the chunk's formulas (rwkv8_bwd.cu lists them) from its own q, v, dy and
// n0 and those four stored values; the checkpointed rho0 is not read again.
// The G update, W = V G15^T and dv run on the tensor cores (mma.sync
// m16n8k8) in split tf32 (rwkv8_split.cuh). R0 and M stay fp32 FFMA: R =
// <rho_tau, dy_tau> can cancel to a small fraction of its terms, and dq
// divides it by sum q + EPS, which is EPS itself for a query row of zeros;
// split tf32's error per product (near 2^-21) is then too large where fp32's
// (2^-24) is not. The norm scans, U, A and the sums along a chunk's steps are
// fp32 FFMA too.
#include <cuda_runtime.h>
#include <stdint.h>

#include "rwkv8.h"
#include "rwkv8_launch.h"
#include "rwkv8_split.cuh"
#include "wkv7_mma.cuh"

namespace rwkv8 {
namespace {

using wkv7::cp_async16;
using wkv7::cp_async_commit;
using wkv7::cp_async_wait_all;
using wkv7::mma_tf32;

constexpr int kThreads = 256;
constexpr int kP8 = 72;  // row pitch 8 mod 32: float2 fragments along a row, scalar ones down a column
constexpr int kP4 = 68;  // row pitch 4 mod 32: scalar fragments along a row
constexpr int kPM = 24;  // row pitch of M
constexpr int kPA = 20;  // row pitch of A^T (16 wide)
constexpr int kRing = 4; // chain: chunks in flight

template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ------------------------------------------------------- split products ---

__device__ __forceinline__ void split4(const float (&x)[4], uint32_t (&h)[4], uint32_t (&l)[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) split_tf32(x[i], h[i], l[i]);
}

// d += a b for one 16 x 8 x 8 tile from fp32 fragment values: the two small
// cross terms first, then the main product.
__device__ __forceinline__ void mma3(float (&d)[4], const uint32_t (&ah)[4], const uint32_t (&al)[4], float2 b) {
  uint32_t bh0, bl0, bh1, bl1;
  split_tf32(b.x, bh0, bl0);
  split_tf32(b.y, bh1, bl1);
  mma_tf32(d, al, bh0, bh1);
  mma_tf32(d, ah, bl0, bl1);
  mma_tf32(d, ah, bh0, bh1);
}

// Fragments of lane (g, t). Both operands of one product bind the k slots
// the same way. "row": A[m][k] and B^T[n][k] row-major, read as float2 (slot
// t <-> column 2 t, slot t + 4 <-> 2 t + 1; pitch 8 mod 32). "col": A from
// storage [k][m] and B from storage [k][n], the hardware's own slots (pitch
// 8 mod 32). "rowk": A[m][k] row-major in the hardware's slots (pitch 4 mod
// 32, or 20 for a 16-wide matrix).
__device__ __forceinline__ void fa_row(float (&a)[4], const float* A, int ld, int k0, int g, int t) {
  const float2 lo = *reinterpret_cast<const float2*>(A + g * ld + k0 + 2 * t);
  const float2 hi = *reinterpret_cast<const float2*>(A + (g + 8) * ld + k0 + 2 * t);
  a[0] = lo.x, a[1] = hi.x, a[2] = lo.y, a[3] = hi.y;
}
__device__ __forceinline__ float2 fb_row(const float* BT, int ld, int n0, int k0, int g, int t) {
  return *reinterpret_cast<const float2*>(BT + (n0 + g) * ld + k0 + 2 * t);
}
__device__ __forceinline__ void fa_col(float (&a)[4], const float* S, int ld, int m0, int k0, int g, int t) {
  const float* p = S + (k0 + t) * ld + m0 + g;
  a[0] = p[0], a[1] = p[8], a[2] = p[4 * ld], a[3] = p[4 * ld + 8];
}
__device__ __forceinline__ float2 fb_col(const float* S, int ld, int n0, int k0, int g, int t) {
  const float* p = S + (k0 + t) * ld + n0 + g;
  return make_float2(p[0], p[4 * ld]);
}
__device__ __forceinline__ void fa_rowk(float (&a)[4], const float* A, int ld, int k0, int g, int t) {
  const float* p = A + g * ld + k0 + t;
  a[0] = p[0], a[1] = p[8 * ld], a[2] = p[4], a[3] = p[8 * ld + 4];
}

__device__ __forceinline__ void zero16(void* dst) {
  *reinterpret_cast<float4*>(dst) = make_float4(0.f, 0.f, 0.f, 0.f);
}

// Local norm scan of the 4-step segment `seg` of latent l (q from rows
// [t][l] of qs), and the row sums of q over each half of l: as the forward's
// per-chunk kernel. x holds q, loc the scan from zero within the segment.
__device__ __forceinline__ void local_scan(const float* qs, float d, int l, int seg, int lane, int w, float (&x)[4],
                                           float (&loc)[4], float* mend, float* sqp) {
  float m = 0.f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    x[j] = qs[(4 * seg + j) * kL + l];
    loc[j] = m;
    m = fmaf(d, m, x[j]);
  }
  mend[seg * kL + l] = m;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float s = x[j];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) sqp[(w & 1) * kC + 4 * seg + j] = s;
  }
}

// R0[tau][l] = <rho0[l], dy_tau> for the steps tau = 4 q4 .. 4 q4 + 3 of latent l (rows of
// rho0 at pitch 4 mod 32: conflict-free float4 loads along a row; dy rows broadcast).
__device__ __forceinline__ void r0_rows(const float* rho, const float* dys, int l, int q4, float (&r)[4]) {
  r[0] = r[1] = r[2] = r[3] = 0.f;
#pragma unroll 4
  for (int e = 0; e < kE; e += 4) {
    const float4 x = *reinterpret_cast<const float4*>(rho + l * kP4 + e);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 y = *reinterpret_cast<const float4*>(dys + (4 * q4 + i) * kP8 + e);
      r[i] = fmaf(x.x, y.x, fmaf(x.y, y.y, fmaf(x.z, y.z, fmaf(x.w, y.w, r[i]))));
    }
  }
}

// M[tau][s] = <dy_tau, v_s> for tau = tid / 16, s = tid % 16.
__device__ __forceinline__ float m_entry(const float* dys, const float* vs, int tid) {
  const float* a = dys + (tid >> 4) * kP8;
  const float* b = vs + (tid & 15) * kP8;
  float m = 0.f;
#pragma unroll 4
  for (int e = 0; e < kE; e += 4) {
    const float4 x = *reinterpret_cast<const float4*>(a + e), y = *reinterpret_cast<const float4*>(b + e);
    m = fmaf(x.x, y.x, fmaf(x.y, y.y, fmaf(x.z, y.z, fmaf(x.w, y.w, m))));
  }
  return m;
}

// ================================================================== R0 ===

// R0[tau][l] = <rho0[l], dy_tau> of one chunk per CTA (256 threads: latent l = tid % 64,
// steps 4 (tid / 64) ..), the same FFMA sequence as everywhere it is formed.
__global__ void __launch_bounds__(kThreads) rwkv8_bwd_r0_kernel(const Args a) {
  __shared__ __align__(16) float rho[kL][kP4];
  __shared__ __align__(16) float dys[kC][kP8];
  const int tid = threadIdx.x, T = a.T, nck = (T + kC - 1) / kC;
  const long long task = blockIdx.x;
  const int bh = (int)(task / nck), c = (int)(task % nck);
  {
    const int row = tid >> 4, col = 4 * (tid & 15), tt = c * kC + row;
    const float* ck = a.ckpt + (size_t)task * kL * kE;
#pragma unroll
    for (int i = 0; i < 4; ++i) cp_async16(&rho[row + 16 * i][col], ck + (size_t)(row + 16 * i) * kE + col);
    if (tt < T)
      cp_async16(&dys[row][col], a.dy + ((size_t)bh * T + tt) * kE + col);
    else
      zero16(&dys[row][col]);
    cp_async_commit();
    cp_async_wait_all();
  }
  __syncthreads();
  const int l = tid & 63, q4 = tid >> 6;
  float r[4];
  r0_rows(&rho[0][0], &dys[0][0], l, q4, r);
  float* dst = a.r0 + (size_t)task * kC * kL;
#pragma unroll
  for (int i = 0; i < 4; ++i) dst[(4 * q4 + i) * kL + l] = r[i];
}

// ================================================================ chain ===

struct ChainSmem {
  float qs[kRing][kC][kL];
  float vs[kRing][kC][kP8];
  float dys[kRing][kC][kP8];
  float rho[kRing][kL][kP4];  // the checkpointed state at the chunk start
  float n0[kRing][kL];
  float pw[kC + 1][kL];       // d_l^k
  float Ut[kC][kP8];          // U[s][l] d_l^s: the G update's A operand, stored [k = s][m = l]
  float U[kC][kL];
  float NB[kC][kL];           // n before every step
  float R0[kRing][kC][kL];     // R0 of the chunk (the pre-pass's)
  float M[kC][kPM];
  float mend[4][kL];
  float sqp[2][kC];
  float xnp[4][kL];           // sum of d^tau g_n[tau] over each thread's steps
  float gdp[2][kL];           // <G15[l], rho0[l]> over each half of the columns
};

struct HeadPtrs {
  const float *q, *v, *dy, *ck_rho, *ck_n, *r0;
  int T;
};

// Chunk c (if >= 0) of q, v, dy and its checkpointed state into ring slot
// `slot` (rows past the end of the sequence zero). Always commits one copy
// group, so groups and visits stay paired.
__device__ __forceinline__ void chain_load(ChainSmem& sm, int slot, const HeadPtrs& hp, int c, int tid) {
  if (c >= 0) {
    const int row = tid >> 4, col = 4 * (tid & 15), t = c * kC + row;
    if (t < hp.T) {
      cp_async16(&sm.qs[slot][row][col], hp.q + (size_t)t * kL + col);
      cp_async16(&sm.vs[slot][row][col], hp.v + (size_t)t * kE + col);
      cp_async16(&sm.dys[slot][row][col], hp.dy + (size_t)t * kE + col);
    } else {
      zero16(&sm.qs[slot][row][col]);
      zero16(&sm.vs[slot][row][col]);
      zero16(&sm.dys[slot][row][col]);
    }
    const float* ck = hp.ck_rho + (size_t)c * kL * kE;
#pragma unroll
    for (int i = 0; i < 4; ++i) cp_async16(&sm.rho[slot][row + 16 * i][col], ck + (size_t)(row + 16 * i) * kE + col);
    if (tid < kL / 4) cp_async16(&sm.n0[slot][4 * tid], hp.ck_n + (size_t)c * kL + 4 * tid);
    cp_async16(&sm.R0[slot][row][col], hp.r0 + ((size_t)c * kC + row) * kL + col);
  }
  cp_async_commit();
}

// g_n of the steps tau = SEG + 4 j of latent l, summed with weights d^tau.
template <int SEG>
__device__ __forceinline__ float chain_elements(const ChainSmem& sm, int slot, int l, const float (&pcol)[kC + 1]) {
  float qcol[kC];
#pragma unroll
  for (int s = 0; s < kC; ++s) qcol[s] = sm.qs[slot][s][l];
  float xn = 0.f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int tau = SEG + 4 * j;
    float R = pcol[tau] * sm.R0[slot][tau][l];
#pragma unroll
    for (int s = 0; s < tau; ++s) R = fmaf(pcol[tau - 1 - s], qcol[s] * sm.M[tau][s], R);
    const float gn = -sm.U[tau][l] * __fdividef(R, sm.NB[tau][l] + kEps);  // denominator >= 1e-6
    xn = fmaf(pcol[tau], gn, xn);
  }
  return xn;
}

// grid B*H. Warp w holds G over latents m0 .. m0+15 (m0 = 16 (w % 4)) and
// columns n0 .. n0+31 (n0 = 32 (w / 4)) as four 16 x 8 accumulator tiles;
// thread tid < 64 holds Gn of latent tid.
__global__ void __launch_bounds__(kThreads, 1) rwkv8_bwd_chain_kernel(const Args a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  ChainSmem& sm = *reinterpret_cast<ChainSmem*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5, g = lane >> 2, t = lane & 3;
  const int bh = blockIdx.x, h = bh % a.H, b = bh / a.H;
  const int T = a.T, nck = (T + kC - 1) / kC;
  const int l_s = tid & 63, seg = tid >> 6;
  const int m0 = 16 * (w & 3), n0 = 32 * (w >> 2), rowa = m0 + g, rowb = m0 + g + 8;
  HeadPtrs hp;
  hp.T = T;
  hp.q = a.q + (size_t)bh * T * kL;
  hp.v = a.v + ((size_t)b * a.Hv + (a.Hv == 1 ? 0 : h)) * T * kE;
  hp.dy = a.dy + (size_t)bh * T * kE;
  hp.ck_rho = a.ckpt + (size_t)bh * nck * kL * kE;
  hp.ck_n = a.ckpt + ckpt_norm_offset(a.B, T, a.H) + (size_t)bh * nck * kL;
  hp.r0 = a.r0 + (size_t)bh * nck * kC * kL;

  // visit v handles chunk nck - 1 - v
#pragma unroll
  for (int k = 0; k < kRing - 1; ++k) chain_load(sm, k, hp, nck - 1 - k, tid);
  if (tid < kL) {
    const float d = a.decay[(size_t)h * kL + tid];
    float p = 1.f;
    for (int k = 0; k <= kC; ++k) {
      sm.pw[k][tid] = p;
      p *= d;
    }
  }
  float acc[4][4];
#pragma unroll
  for (int nt = 0; nt < 4; ++nt) {
    float2 x = make_float2(0.f, 0.f), y = x;
    if (a.d_rho_final) {
      x = *reinterpret_cast<const float2*>(a.d_rho_final + ((size_t)bh * kL + rowa) * kE + n0 + 8 * nt + 2 * t);
      y = *reinterpret_cast<const float2*>(a.d_rho_final + ((size_t)bh * kL + rowb) * kE + n0 + 8 * nt + 2 * t);
    }
    acc[nt][0] = x.x, acc[nt][1] = x.y, acc[nt][2] = y.x, acc[nt][3] = y.y;
  }
  float gn = tid < kL && a.d_rho_norm_final ? a.d_rho_norm_final[(size_t)bh * kL + tid] : 0.f;
  __syncthreads();
  float pcol[kC + 1];
#pragma unroll
  for (int k = 0; k <= kC; ++k) pcol[k] = sm.pw[k][l_s];

  for (int v = 0; v < nck; ++v) {
    const int c = nck - 1 - v, slot = v % kRing, len = min(kC, T - c * kC);
    const size_t task = (size_t)bh * nck + c;
    cp_async_wait_group<kRing - 2>();  // visit v's group (and every older one) complete
    __syncthreads();                   // staged; every thread is done with visit v - 1

    // ---- the carried gradients entering the chunk from its end
    float* gdst = a.g15 + task * kL * kE;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const int col = n0 + 8 * nt + 2 * t;
      *reinterpret_cast<float2*>(gdst + (size_t)rowa * kE + col) = make_float2(acc[nt][0], acc[nt][1]);
      *reinterpret_cast<float2*>(gdst + (size_t)rowb * kE + col) = make_float2(acc[nt][2], acc[nt][3]);
    }
    if (tid < kL) a.gn15[task * kL + tid] = gn;
    {  // <G15[l], rho0[l]>: this thread's eight columns of rows rowa, rowb, then the row's four lanes
      float pa = 0.f, pb = 0.f;
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const int col = n0 + 8 * nt + 2 * t;
        const float2 ra = *reinterpret_cast<const float2*>(&sm.rho[slot][rowa][col]);
        const float2 rb = *reinterpret_cast<const float2*>(&sm.rho[slot][rowb][col]);
        pa = fmaf(acc[nt][0], ra.x, fmaf(acc[nt][1], ra.y, pa));
        pb = fmaf(acc[nt][2], rb.x, fmaf(acc[nt][3], rb.y, pb));
      }
      pa += __shfl_xor_sync(0xffffffffu, pa, 1);
      pa += __shfl_xor_sync(0xffffffffu, pa, 2);
      pb += __shfl_xor_sync(0xffffffffu, pb, 1);
      pb += __shfl_xor_sync(0xffffffffu, pb, 2);
      if (t == 0) {
        sm.gdp[w >> 2][rowa] = pa;
        sm.gdp[w >> 2][rowb] = pb;
      }
    }
    // the chunk kRing - 1 visits ahead, into the slot visit v - 1 used
    chain_load(sm, (v + kRing - 1) % kRing, hp, c - (kRing - 1), tid);

    float x[4], loc[4];
    local_scan(&sm.qs[slot][0][0], pcol[1], l_s, seg, lane, w, x, loc, &sm.mend[0][0], &sm.sqp[0][0]);
    sm.M[tid >> 4][tid & 15] = m_entry(&sm.dys[slot][0][0], &sm.vs[slot][0][0], tid);  // M = DY V^T (fp32 FFMA)
    __syncthreads();

    // ---- n before every step, U, U d^tau; <G15, rho0> to the workspace
    {
      float start = sm.n0[slot][l_s];
      for (int s2 = 0; s2 < seg; ++s2) start = fmaf(pcol[4], start, sm.mend[s2][l_s]);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int tau = 4 * seg + j;
        const float nb = fmaf(pcol[j], start, loc[j]);
        const float sq = sm.sqp[0][tau] + sm.sqp[1][tau] + kEps;
        const float u = __fdividef(x[j], sq * (nb + kEps));  // denominator >= 1e-12
        sm.NB[tau][l_s] = nb;
        sm.U[tau][l_s] = u;
        sm.Ut[tau][l_s] = u * sm.pw[tau][l_s];
      }
    }
    if (tid < kL) a.gdot[task * kL + tid] = sm.gdp[0][tid] + sm.gdp[1][tid];
    __syncthreads();

    // ---- G <- d^len (.) G + (U d^s)^T DY; this thread's share of sum_tau d^tau g_n[tau]
    {
      const float dla = sm.pw[len][rowa], dlb = sm.pw[len][rowb];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        acc[nt][0] *= dla, acc[nt][1] *= dla;
        acc[nt][2] *= dlb, acc[nt][3] *= dlb;
      }
#pragma unroll
      for (int kb = 0; kb < kC / 8; ++kb) {
        float af[4];
        uint32_t ah[4], al[4];
        fa_col(af, &sm.Ut[0][0], kP8, m0, 8 * kb, g, t);
        split4(af, ah, al);
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) mma3(acc[nt], ah, al, fb_col(&sm.dys[slot][0][0], kP8, n0 + 8 * nt, 8 * kb, g, t));
      }
    }
    float xn;
    switch (seg) {
      case 0: xn = chain_elements<0>(sm, slot, l_s, pcol); break;
      case 1: xn = chain_elements<1>(sm, slot, l_s, pcol); break;
      case 2: xn = chain_elements<2>(sm, slot, l_s, pcol); break;
      default: xn = chain_elements<3>(sm, slot, l_s, pcol); break;
    }
    sm.xnp[seg][l_s] = xn;
    __syncthreads();
    // ---- Gn <- d^len Gn + sum_tau d^tau g_n[tau]
    if (tid < kL) gn = fmaf(sm.pw[len][tid], gn, (sm.xnp[0][tid] + sm.xnp[1][tid]) + (sm.xnp[2][tid] + sm.xnp[3][tid]));
  }
  cp_async_wait_all();  // the empty trailing groups
  if (a.d_rho_init) {
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const int col = n0 + 8 * nt + 2 * t;
      *reinterpret_cast<float2*>(a.d_rho_init + ((size_t)bh * kL + rowa) * kE + col) = make_float2(acc[nt][0], acc[nt][1]);
      *reinterpret_cast<float2*>(a.d_rho_init + ((size_t)bh * kL + rowb) * kE + col) = make_float2(acc[nt][2], acc[nt][3]);
    }
  }
  if (a.d_rho_norm_init && tid < kL) a.d_rho_norm_init[(size_t)bh * kL + tid] = gn;
}

// ============================================================ per chunk ===

struct ChunkSmem {
  float qs[kC][kL];
  float vs[kC][kP8];
  float dys[kC][kP8];
  float G[kL][kP8];      // G15 [l][e]
  float R0[kC][kL];
  float pw[kC + 1][kL];
  float U[kC][kL];
  float NB[kC][kL];
  float W[kC][kP8];      // W = V G15^T [tau][l]
  float gn[kC][kL];      // g_n
  float QG[kC][kP4];     // q_tau d^(len-1-tau), zero for tau >= len
  float M[kC][kPM];
  float At[kC][kPA];     // At[tau][s] = A[s][tau] (s > tau), zero elsewhere
  float mend[4][kL];
  float sqp[2][kC];
  float rowp[2][kC];
  float n0[kL], gn15[kL], gdot[kL];
  float ddp[4][kL];
};

// The 120 pairs (at, as), as < at, in four rounds; in round r the eight lanes
// of group ag of warp w take pair p = 4 (8 r + w) + ag and split the latent
// range between them. A pair past 119 is computed on a valid pair and not
// stored (encoded negative).
__device__ __forceinline__ void a_pairs(int (&apair)[4], int w, int ag) {
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
}

// R, the weights' gradient, g_n, Gv and the decay terms that need them, for
// the steps tau = SEG + 4 j of latent l.
template <int SEG>
__device__ __forceinline__ void chunk_elements(ChunkSmem& sm, int l, int len, const float (&pcol)[kC + 1],
                                               float (&gq)[4], float (&gv)[4], float (&nb)[4], float& dd) {
  float qcol[kC], ucol[kC];
#pragma unroll
  for (int s = 0; s < kC; ++s) {
    qcol[s] = sm.qs[s][l];
    ucol[s] = sm.U[s][l];
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int tau = SEG + 4 * j;
    const float r0 = sm.R0[tau][l], wv = sm.W[tau][l];
    float R = pcol[tau] * r0, d4 = 0.f;
#pragma unroll
    for (int s = 0; s < tau; ++s) {
      const float qm = qcol[s] * sm.M[tau][s];
      R = fmaf(pcol[tau - 1 - s], qm, R);
      if (s <= tau - 2) d4 = fmaf((float)(tau - 1 - s) * pcol[tau - 2 - s], qm, d4);
    }
    float G = 0.f;
#pragma unroll
    for (int s = tau + 1; s < kC; ++s) G = fmaf(pcol[s - 1 - tau] * ucol[s], sm.M[s][tau], G);
    if (tau < len) G = fmaf(sm.pw[len - 1 - tau][l], wv, G);
    const float n = sm.NB[tau][l];
    const float gqv = __fdividef(R, n + kEps);  // denominator >= 1e-6
    gq[j] = gqv;
    gv[j] = G;
    nb[j] = n;
    sm.gn[tau][l] = -ucol[tau] * gqv;
    float ddj = ucol[tau] * d4;
    if (tau >= 1) ddj = fmaf((float)tau * pcol[tau - 1] * ucol[tau], r0, ddj);
    if (tau <= len - 2) ddj = fmaf((float)(len - 1 - tau) * sm.pw[len - 2 - tau][l] * qcol[tau], wv, ddj);
    dd += ddj;
  }
}

// dq of the steps tau = SEG + 4 j of latent l, with Gn at each step and the
// norm's decay term.
template <int SEG>
__device__ __forceinline__ void chunk_dq(const ChunkSmem& sm, int l, int len, const float (&pcol)[kC + 1],
                                        const float (&gq)[4], const float (&gv)[4], const float (&nb)[4], float& dd,
                                        float* dqc) {
  float gcol[kC];
#pragma unroll
  for (int s = 0; s < kC; ++s) gcol[s] = sm.gn[s][l];
  const float gn15 = sm.gn15[l];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int tau = SEG + 4 * j;
    if (tau < len) {
      float gnt = sm.pw[len - 1 - tau][l] * gn15;
#pragma unroll
      for (int s = tau + 1; s < kC; ++s) gnt = fmaf(pcol[s - 1 - tau], gcol[s], gnt);
      dd = fmaf(gnt, nb[j], dd);
      const float sq = sm.sqp[0][tau] + sm.sqp[1][tau] + kEps;
      const float rowsum = sm.rowp[0][tau] + sm.rowp[1][tau];
      dqc[(size_t)tau * kL + l] = (gq[j] - rowsum) / sq + gv[j] + gnt;
    }
  }
}

__global__ void __launch_bounds__(kThreads, 2) rwkv8_bwd_chunk_kernel(const Args a, long long ntasks) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  ChunkSmem& sm = *reinterpret_cast<ChunkSmem*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5, g = lane >> 2, t = lane & 3;
  const int T = a.T, nck = (T + kC - 1) / kC;
  const int l_s = tid & 63, seg = tid >> 6;
  const int ag = lane >> 3, a8 = lane & 7;
  int apair[4];
  a_pairs(apair, w, ag);

  for (long long task = blockIdx.x; task < ntasks; task += gridDim.x) {
    const int bh = (int)(task / nck), c = (int)(task % nck), h = bh % a.H, b = bh / a.H;
    const int len = min(kC, T - c * kC);
    const float* qh = a.q + (size_t)bh * T * kL;
    const float* vh = a.v + ((size_t)b * a.Hv + (a.Hv == 1 ? 0 : h)) * T * kE;
    const float* dyh = a.dy + (size_t)bh * T * kE;
    const float* g15 = a.g15 + (size_t)task * kL * kE;
    const float* r0 = a.r0 + (size_t)task * kC * kL;
    __syncthreads();  // the previous task is done with shared memory
    {
      const int row = tid >> 4, col = 4 * (tid & 15), tt = c * kC + row;
      if (tt < T) {
        cp_async16(&sm.qs[row][col], qh + (size_t)tt * kL + col);
        cp_async16(&sm.vs[row][col], vh + (size_t)tt * kE + col);
        cp_async16(&sm.dys[row][col], dyh + (size_t)tt * kE + col);
      } else {
        zero16(&sm.qs[row][col]);
        zero16(&sm.vs[row][col]);
        zero16(&sm.dys[row][col]);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) cp_async16(&sm.G[row + 16 * i][col], g15 + (size_t)(row + 16 * i) * kE + col);
      cp_async16(&sm.R0[row][col], r0 + (size_t)row * kL + col);
      if (tid < 16)
        cp_async16(&sm.n0[4 * tid], a.ckpt + ckpt_norm_offset(a.B, T, a.H) + (size_t)task * kL + 4 * tid);
      else if (tid < 32)
        cp_async16(&sm.gn15[4 * (tid - 16)], a.gn15 + (size_t)task * kL + 4 * (tid - 16));
      else if (tid < 48)
        cp_async16(&sm.gdot[4 * (tid - 32)], a.gdot + (size_t)task * kL + 4 * (tid - 32));
      cp_async_commit();
    }
    if (tid < kL) {
      const float d = a.decay[(size_t)h * kL + tid];
      float p = 1.f;
      for (int k = 0; k <= kC; ++k) {
        sm.pw[k][tid] = p;
        p *= d;
      }
    }
    for (int i = tid; i < kC * kPA; i += kThreads) (&sm.At[0][0])[i] = 0.f;
    cp_async_wait_all();
    __syncthreads();
    float pcol[kC + 1];
#pragma unroll
    for (int k = 0; k <= kC; ++k) pcol[k] = sm.pw[k][l_s];

    // ---- phase 1: local norm scan, row sums; W = V G15^T (warp w: latents 8 w ..),
    //      M = DY V^T (fp32 FFMA)
    float x[4], loc[4];
    local_scan(&sm.qs[0][0], pcol[1], l_s, seg, lane, w, x, loc, &sm.mend[0][0], &sm.sqp[0][0]);
    {
      float wa[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kb = 0; kb < kE / 8; ++kb) {
        float af[4];
        uint32_t ah[4], al[4];
        fa_row(af, &sm.vs[0][0], kP8, 8 * kb, g, t);
        split4(af, ah, al);
        mma3(wa, ah, al, fb_row(&sm.G[0][0], kP8, 8 * w, 8 * kb, g, t));
      }
      *reinterpret_cast<float2*>(&sm.W[g][8 * w + 2 * t]) = make_float2(wa[0], wa[1]);
      *reinterpret_cast<float2*>(&sm.W[g + 8][8 * w + 2 * t]) = make_float2(wa[2], wa[3]);
      sm.M[tid >> 4][tid & 15] = m_entry(&sm.dys[0][0], &sm.vs[0][0], tid);
    }
    __syncthreads();

    // ---- phase 2: n before every step, U, q d^(len-1-tau)
    {
      float start = sm.n0[l_s];
      for (int s2 = 0; s2 < seg; ++s2) start = fmaf(pcol[4], start, sm.mend[s2][l_s]);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int tau = 4 * seg + j;
        const float nbv = fmaf(pcol[j], start, loc[j]);
        const float sq = sm.sqp[0][tau] + sm.sqp[1][tau] + kEps;
        sm.NB[tau][l_s] = nbv;
        sm.U[tau][l_s] = __fdividef(x[j], sq * (nbv + kEps));  // denominator >= 1e-12
        sm.QG[tau][l_s] = tau < len ? x[j] * sm.pw[len - 1 - tau][l_s] : 0.f;
      }
    }
    __syncthreads();

    // ---- phase 3: per-element terms, the weights' row sums, A
    float gq[4], gvv[4], nb[4], dd = 0.f;
    switch (seg) {
      case 0: chunk_elements<0>(sm, l_s, len, pcol, gq, gvv, nb, dd); break;
      case 1: chunk_elements<1>(sm, l_s, len, pcol, gq, gvv, nb, dd); break;
      case 2: chunk_elements<2>(sm, l_s, len, pcol, gq, gvv, nb, dd); break;
      default: chunk_elements<3>(sm, l_s, len, pcol, gq, gvv, nb, dd); break;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int tau = seg + 4 * j;
      const float sq = sm.sqp[0][tau] + sm.sqp[1][tau] + kEps;
      float s = gq[j] * (sm.qs[tau][l_s] / sq);
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
        const float4 q = *reinterpret_cast<const float4*>(&sm.qs[as][l]);
        const float4 p = *reinterpret_cast<const float4*>(&sm.pw[k][l]);
        acc = fmaf(u.x * q.x, p.x, acc);
        acc = fmaf(u.y * q.y, p.y, acc);
        acc = fmaf(u.z * q.z, p.z, acc);
        acc = fmaf(u.w * q.w, p.w, acc);
      }
      acc += __shfl_xor_sync(0xffffffffu, acc, 1);
      acc += __shfl_xor_sync(0xffffffffu, acc, 2);
      acc += __shfl_xor_sync(0xffffffffu, acc, 4);
      if (a8 == 0 && apair[rr] >= 0) sm.At[as][at] = acc;
    }
    __syncthreads();

    // ---- phase 4: dq (with Gn); dv = (q d^(len-1-tau)) G15 + A^T DY (warp w: columns 8 w ..)
    float* dqc = a.dq + ((size_t)bh * T + (size_t)c * kC) * kL;
    switch (seg) {
      case 0: chunk_dq<0>(sm, l_s, len, pcol, gq, gvv, nb, dd, dqc); break;
      case 1: chunk_dq<1>(sm, l_s, len, pcol, gq, gvv, nb, dd, dqc); break;
      case 2: chunk_dq<2>(sm, l_s, len, pcol, gq, gvv, nb, dd, dqc); break;
      default: chunk_dq<3>(sm, l_s, len, pcol, gq, gvv, nb, dd, dqc); break;
    }
    if (seg == 0) dd = fmaf((float)len * sm.pw[len - 1][l_s], sm.gdot[l_s], dd);
    {
      float dva[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kb = 0; kb < kL / 8; ++kb) {
        float af[4];
        uint32_t ah[4], al[4];
        fa_rowk(af, &sm.QG[0][0], kP4, 8 * kb, g, t);
        split4(af, ah, al);
        mma3(dva, ah, al, fb_col(&sm.G[0][0], kP8, 8 * w, 8 * kb, g, t));
      }
#pragma unroll
      for (int kb = 0; kb < kC / 8; ++kb) {
        float af[4];
        uint32_t ah[4], al[4];
        fa_rowk(af, &sm.At[0][0], kPA, 8 * kb, g, t);
        split4(af, ah, al);
        mma3(dva, ah, al, fb_col(&sm.dys[0][0], kP8, 8 * w, 8 * kb, g, t));
      }
      float* dvc = a.dv + ((size_t)bh * T + (size_t)c * kC) * kE + 8 * w + 2 * t;
      if (g < len) *reinterpret_cast<float2*>(dvc + (size_t)g * kE) = make_float2(dva[0], dva[1]);
      if (g + 8 < len) *reinterpret_cast<float2*>(dvc + (size_t)(g + 8) * kE) = make_float2(dva[2], dva[3]);
    }
    sm.ddp[seg][l_s] = dd;
    __syncthreads();
    if (tid < kL)
      a.ddecay_part[(size_t)task * kL + tid] = (sm.ddp[0][tid] + sm.ddp[1][tid]) + (sm.ddp[2][tid] + sm.ddp[3][tid]);
  }
}

// out[bh][l] = sum over the chunks c, in order, of part[bh][c][l].
__global__ void chunk_sum_kernel(const float* __restrict__ part, float* __restrict__ out, int BH, int nck) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= BH * kL) return;
  const float* p = part + (size_t)(i / kL) * nck * kL + (i % kL);
  float s = 0.f;
  for (int c = 0; c < nck; ++c) s += p[(size_t)c * kL];
  out[i] = s;
}

}  // namespace

cudaError_t launch_backward_chain(const Args& a, cudaStream_t s) {
  const long long ntasks = (long long)a.B * a.H * (long long)nchunks(a.T);
  if (ntasks <= 0) return cudaSuccess;
  if (ntasks >= (1ll << 31)) return cudaErrorInvalidValue;
  rwkv8_bwd_r0_kernel<<<(unsigned)ntasks, kThreads, 0, s>>>(a);  // R0 of every chunk, before the chain reads it
  const size_t smem = sizeof(ChainSmem);
  cudaError_t e = cudaFuncSetAttribute(rwkv8_bwd_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  rwkv8_bwd_chain_kernel<<<(unsigned)(a.B * a.H), kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_backward_chunks(const Args& a, cudaStream_t s) {
  const size_t smem = sizeof(ChunkSmem);
  cudaError_t e = cudaFuncSetAttribute(rwkv8_bwd_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const long long ntasks = (long long)a.B * a.H * (long long)nchunks(a.T);
  const unsigned grid = (unsigned)(ntasks < (1ll << 30) ? ntasks : (1ll << 30));
  rwkv8_bwd_chunk_kernel<<<grid, kThreads, smem, s>>>(a, ntasks);
  return cudaGetLastError();
}

cudaError_t launch_chunk_sum(const Args& a, cudaStream_t s) {
  const int n = a.B * a.H * kL;
  chunk_sum_kernel<<<(n + 255) / 256, 256, 0, s>>>(a.ddecay_part, a.ddecay_bh, a.B * a.H, (int)nchunks(a.T));
  return cudaGetLastError();
}

}  // namespace rwkv8
