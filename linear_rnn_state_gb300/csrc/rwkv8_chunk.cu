// RWKV-8 normalized recurrence: the per-chunk work, every chunk at once.
//
// With the state at every chunk start written by the chain kernel
// (rwkv8_state.cu), the readout of a chunk of steps t0 .. t0+len-1
// ("src/sequence/rwkv8/backward.rs", burn_dragon_kernel: the readout of
// backward_chunk_impl) needs nothing from any other chunk:
//     n_tau   = d^tau n0 + sum_{s<tau} d^(tau-1-s) q_s
//     U[tau]  = qw_tau / (n_tau + EPS),  qw_tau = q_tau / (sum q_tau + EPS)
//     y_tau   = (U[tau] d^tau)^T rho0 + sum_{s<tau} A[tau][s] v_s,
//     A[tau][s] = sum_l U[tau][l] q_s[l] d_l^(tau-1-s)            (s < tau)
// One CTA of 256 threads per (b, h, chunk): the chunk's q, v and checkpoint
// arrive by cp.async, then four phases (norm scan and row sums; n before
// every step, U and U d^tau; A and the readout of rho0; y = readout + A v).
// The scans, U and A are fp32 FFMA on the CUDA cores; the two dense products
// (the readout, [16 x 64] x [64 x 64], and A v, [16 x 16] x [16 x 64]) run on
// the tensor cores (mma.sync m16n8k8) in split tf32 (rwkv8_split.cuh: three
// tf32 products per fp32 one, fp32 accumulation), warp w producing columns
// 8 w .. 8 w + 7 of y.
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

constexpr int kThreads = 256;
constexpr int kP = 72;   // row pitch of rho0 and v (8 mod 32: conflict-free B fragments)
constexpr int kUT = 68;  // row pitch of U d^tau (4 mod 32: conflict-free A fragments and row stores)
constexpr int kAP = 20;  // row pitch of A (conflict-free A fragments)



// The A role: the 120 pairs (at, as), as < at, in four rounds; in round r
// the eight lanes of group ag of warp w take pair p = 4 (8 r + w) + ag and
// split the latent range between them. A pair past 119 is computed on a
// valid pair and not stored (encoded negative).
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

// ------------------------------------------------------------ forward ---

struct FwdOutSmem {
  float qs[kC][kL];
  float vs[kC][kP];
  float rho[kL][kP];     // the state at the chunk start
  float pw[kC + 1][kL];  // pw[k][l] = d_l^k
  float U[kC][kL];       // U[tau][l]
  float Ut[kC][kUT];     // U[tau][l] d_l^tau
  float A[kC][kAP];      // strictly lower part of A; the rest stays zero
  float mend[4][kL];     // end of each 4-step segment of the local norm scan
  float sqp[2][kC];      // row sums of q over each half of l
  float n0[kL];
};

__global__ void __launch_bounds__(kThreads, 3) rwkv8_fwd_chunk_kernel(const Args a, long long ntasks) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  FwdOutSmem& sm = *reinterpret_cast<FwdOutSmem*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int T = a.T, nck = (T + kC - 1) / kC;
  const int l_s = tid & 63, seg = tid >> 6;
  const int ag = lane >> 3, a8 = lane & 7;
  int apair[4];
  a_pairs(apair, w, ag);
  const int g = lane >> 2, t = lane & 3, e0 = 8 * w;  // fragment roles

  for (long long task = blockIdx.x; task < ntasks; task += gridDim.x) {
    const int bh = (int)(task / nck), c = (int)(task % nck), h = bh % a.H, b = bh / a.H;
    const int len = min(kC, T - c * kC);
    const float* qh = a.q + (size_t)bh * T * kL;
    const float* vh = a.v + ((size_t)b * a.Hv + (a.Hv == 1 ? 0 : h)) * T * kE;
    const float* ck = a.ckpt + ((size_t)bh * nck + c) * kL * kE;
    const float* ckn = a.ckpt + ckpt_norm_offset(a.B, T, a.H) + ((size_t)bh * nck + c) * kL;
    __syncthreads();  // the previous task is done with shared memory
    {
      const int row = tid >> 4, col = 4 * (tid & 15), t = c * kC + row;
      if (t < T) {
        cp_async16(&sm.qs[row][col], qh + (size_t)t * kL + col);
        cp_async16(&sm.vs[row][col], vh + (size_t)t * kE + col);
      } else {
        *reinterpret_cast<float4*>(&sm.qs[row][col]) = make_float4(0.f, 0.f, 0.f, 0.f);
        *reinterpret_cast<float4*>(&sm.vs[row][col]) = make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) cp_async16(&sm.rho[row + 16 * i][col], ck + (size_t)(row + 16 * i) * kE + col);
      if (tid < kL / 4) cp_async16(&sm.n0[4 * tid], ckn + 4 * tid);
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
    for (int i = tid; i < kC * kAP; i += kThreads) (&sm.A[0][0])[i] = 0.f;
    cp_async_wait_all();
    __syncthreads();

    // ---- phase 1: local norm scan in 4-step segments, row sums of q
    float x[4], loc[4];
    {
      const float d = sm.pw[1][l_s];
      float m = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        x[j] = sm.qs[4 * seg + j][l_s];
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
    __syncthreads();

    // ---- phase 2: n before every step, U, U d^tau
    {
      float start = sm.n0[l_s];
      for (int s2 = 0; s2 < seg; ++s2) start = fmaf(sm.pw[4][l_s], start, sm.mend[s2][l_s]);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int tau = 4 * seg + j;
        const float nb = fmaf(sm.pw[j][l_s], start, loc[j]);
        const float sq = sm.sqp[0][tau] + sm.sqp[1][tau] + kEps;
        const float u = __fdividef(x[j], sq * (nb + kEps));  // denominator >= 1e-12
        sm.U[tau][l_s] = u;
        sm.Ut[tau][l_s] = u * sm.pw[tau][l_s];
      }
    }
    __syncthreads();

    // ---- phase 3: A (strictly lower) and the readout of rho0
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
      if (a8 == 0 && apair[rr] >= 0) sm.A[at][as] = acc;
    }
    // readout: Y = (U d^tau)^T rho0, rows tau, columns e0 .. e0 + 7, in four
    // partial sums over k blocks (independent product chains)
    float yk[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) yk[i][0] = yk[i][1] = yk[i][2] = yk[i][3] = 0.f;
#pragma unroll
    for (int kb = 0; kb < kL / 8; ++kb) {
      const float* ap = &sm.Ut[g][8 * kb + t];
      const float* bp = &sm.rho[8 * kb + t][e0 + g];
      const float af[4] = {ap[0], ap[8 * kUT], ap[4], ap[8 * kUT + 4]};
      mma_split(yk[kb & 3], af, bp[0], bp[4 * kP]);
    }
    __syncthreads();  // A complete

    // ---- phase 4: y += A v, then the stores
#pragma unroll
    for (int kb = 0; kb < kC / 8; ++kb) {
      const float* ap = &sm.A[g][8 * kb + t];
      const float* bp = &sm.vs[8 * kb + t][e0 + g];
      const float af[4] = {ap[0], ap[8 * kAP], ap[4], ap[8 * kAP + 4]};
      mma_split(yk[kb], af, bp[0], bp[4 * kP]);
    }
    float y[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) y[i] = (yk[0][i] + yk[1][i]) + (yk[2][i] + yk[3][i]);
    float* yc = a.y + ((size_t)bh * T + (size_t)c * kC) * kE + e0 + 2 * t;
    if (g < len) *reinterpret_cast<float2*>(yc + (size_t)g * kE) = make_float2(y[0], y[1]);
    if (g + 8 < len) *reinterpret_cast<float2*>(yc + (size_t)(g + 8) * kE) = make_float2(y[2], y[3]);
  }
}

long long chunk_tasks(const Args& a) { return (long long)a.B * a.H * (long long)nchunks(a.T); }

}  // namespace

cudaError_t launch_forward_chunks(const Args& a, cudaStream_t s) {
  const size_t smem = sizeof(FwdOutSmem);
  cudaError_t e = cudaFuncSetAttribute(rwkv8_fwd_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const long long ntasks = chunk_tasks(a);
  const unsigned grid = (unsigned)(ntasks < (1ll << 30) ? ntasks : (1ll << 30));
  rwkv8_fwd_chunk_kernel<<<grid, kThreads, smem, s>>>(a, ntasks);
  return cudaGetLastError();
}

}  // namespace rwkv8
