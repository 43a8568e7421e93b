// RWKV-8 normalized recurrence, forward: the chain between chunks, alone.
//
// The decay d[l] of "src/sequence/rwkv8/backward.rs" (burn_dragon_kernel)
// does not depend on t, so over a chunk of len steps the state moves by
//     rho_end = d^len (.) rho0 + sum_s (q_s d^(len-1-s)) v_s^T,
//     n_end   = d^len (.) n0   + sum_s  q_s d^(len-1-s)
// and the readout of a chunk depends only on its own inputs and its start
// state. This kernel runs only the chain, one CTA per (b, h): each element of
// rho evolves on its own, and the chain of one chunk is one multiply per
// element on top of a product that does not depend on it. It writes the
// state at every chunk start (the checkpoints); the per-chunk kernel
// (rwkv8_chunk.cu) then makes y for all chunks at once.
//
// The chunk's product is a dense [64 x 16] x [16 x 64] contraction, run on the
// tensor cores (mma.sync m16n8k8) in split tf32: each fp32 operand x is
// x_hi + x_lo, x_hi = x rounded to tf32 and x_lo = x - x_hi (exact, itself
// rounded to tf32 on the way in), and the product is a_lo b_hi + a_hi b_lo +
// a_hi b_hi (relative error near 2^-21, against 2^-11 for one tf32
// product), accumulated in fp32 straight into the state's accumulator tiles.
// Warp w holds latents 16 w .. 16 w + 15 of all 64 columns (eight 16 x 8
// tiles) and, as a ninth tile, the norm n: a 65th column whose value row is
// all ones (n <- d n + q is the state recurrence with v = 1).
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
using wkv7::mma_tf32;

constexpr int kSThreads = 128;  // four warps of 16 latents
constexpr int kStages = 8;      // chunks in flight: the chain runs far ahead of DRAM latency
constexpr int kQP = 72;         // row pitch of the staged rows (8 mod 32: conflict-free fragments)
constexpr int kNT = kE / 8;     // accumulator tiles of the state (the norm is tile kNT)

template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void zero16(void* dst) {
  *reinterpret_cast<float4*>(dst) = make_float4(0.f, 0.f, 0.f, 0.f);
}

// ------------------------------------------------------------ forward ---

struct StateSmem {
  float qs[kStages][kC][kQP];
  float vs[kStages][kC][kQP];
  float pw[kC + 1][kL];  // d^k, for a shorter last chunk
};

// Chunk c of q and v into ring slot `buf` (rows past the end of the sequence
// zero). Always commits one copy group (empty past the last chunk), so
// groups and chunks stay paired.
__device__ __forceinline__ void load_state_chunk(StateSmem& sm, int buf, const float* qh, const float* vh, int c,
                                                 int T, int tid) {
  if (c * kC < T) {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int idx = tid + kSThreads * k, row = idx >> 4, col = 4 * (idx & 15);
      const int t = c * kC + row;
      if (t < T) {
        cp_async16(&sm.qs[buf][row][col], qh + (size_t)t * kL + col);
        cp_async16(&sm.vs[buf][row][col], vh + (size_t)t * kE + col);
      } else {
        zero16(&sm.qs[buf][row][col]);
        zero16(&sm.vs[buf][row][col]);
      }
    }
  }
  cp_async_commit();
}

// grid B*H; lane (g, t) of warp w holds, in tile nt, rows m0 + g and m0 + g + 8
// (m0 = 16 w) and columns 8 nt + 2 t, + 1; tile kNT holds n in column 0
// (lanes with t = 0).
__global__ void __launch_bounds__(kSThreads) rwkv8_state_kernel(const Args a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  StateSmem& sm = *reinterpret_cast<StateSmem*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5, g = lane >> 2, t = lane & 3;
  const int bh = blockIdx.x, h = bh % a.H, b = bh / a.H;
  const int T = a.T, nck = (T + kC - 1) / kC;
  const int m0 = 16 * w, rowa = m0 + g, rowb = m0 + g + 8;
  const float* qh = a.q + (size_t)bh * T * kL;
  const float* vh = a.v + ((size_t)b * a.Hv + (a.Hv == 1 ? 0 : h)) * T * kE;
  float* ck_rho = a.ckpt ? a.ckpt + (size_t)bh * nck * kL * kE : nullptr;
  float* ck_n = a.ckpt ? a.ckpt + ckpt_norm_offset(a.B, T, a.H) + (size_t)bh * nck * kL : nullptr;

#pragma unroll
  for (int k = 0; k < kStages - 1; ++k) load_state_chunk(sm, k, qh, vh, k, T, tid);

  if (tid < kL) {
    const float d = a.decay[(size_t)h * kL + tid];
    float p = 1.f;
    for (int k = 0; k <= kC; ++k) {
      sm.pw[k][tid] = p;
      p *= d;
    }
  }
  __syncthreads();
  // The lane's A entries are steps s = 8 kb + t + 4 j (k block kb, slot half j)
  // of latents rowa and rowb; a full chunk scales them by d^(15 - s).
  float pa[2][2], pb[2][2];
#pragma unroll
  for (int kb = 0; kb < 2; ++kb)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int s = 8 * kb + t + 4 * j;
      pa[kb][j] = sm.pw[kC - 1 - s][rowa];
      pb[kb][j] = sm.pw[kC - 1 - s][rowb];
    }
  const float dla = sm.pw[kC][rowa], dlb = sm.pw[kC][rowb];

  float acc[kNT + 1][4];
#pragma unroll
  for (int nt = 0; nt < kNT; ++nt) {
    float2 x = make_float2(0.f, 0.f), y = x;
    if (a.rho_init) {
      x = *reinterpret_cast<const float2*>(a.rho_init + ((size_t)bh * kL + rowa) * kE + 8 * nt + 2 * t);
      y = *reinterpret_cast<const float2*>(a.rho_init + ((size_t)bh * kL + rowb) * kE + 8 * nt + 2 * t);
    }
    acc[nt][0] = x.x, acc[nt][1] = x.y, acc[nt][2] = y.x, acc[nt][3] = y.y;
  }
  acc[kNT][0] = acc[kNT][1] = acc[kNT][2] = acc[kNT][3] = 0.f;
  if (t == 0 && a.rho_norm_init) {
    acc[kNT][0] = a.rho_norm_init[(size_t)bh * kL + rowa];
    acc[kNT][2] = a.rho_norm_init[(size_t)bh * kL + rowb];
  }
  // the norm's value column: B[s][64] = 1, B[s][65 ..] = 0 (exact in tf32)
  const uint32_t one_b = g == 0 ? __float_as_uint(1.f) : 0u;

  for (int c = 0; c < nck; ++c) {
    const int buf = c % kStages, len = min(kC, T - c * kC);
    cp_async_wait_group<kStages - 2>();  // chunk c's group (and every older one) complete
    __syncthreads();  // chunk c staged; every thread is done with chunk c - 1's slot
    if (ck_rho) {
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt) {
        *reinterpret_cast<float2*>(ck_rho + ((size_t)c * kL + rowa) * kE + 8 * nt + 2 * t) =
            make_float2(acc[nt][0], acc[nt][1]);
        *reinterpret_cast<float2*>(ck_rho + ((size_t)c * kL + rowb) * kE + 8 * nt + 2 * t) =
            make_float2(acc[nt][2], acc[nt][3]);
      }
      if (t == 0) {
        ck_n[(size_t)c * kL + rowa] = acc[kNT][0];
        ck_n[(size_t)c * kL + rowb] = acc[kNT][2];
      }
    }
    load_state_chunk(sm, (c + kStages - 1) % kStages, qh, vh, c + kStages - 1, T, tid);

    // A = (q_s d^(len-1-s))^T: rows = latents, k = steps (zero for s >= len)
    float qa[2][2][2];  // [kb][j][row a / b]
    const float* qs = &sm.qs[buf][0][0];
    float sla = dla, slb = dlb;
    if (len == kC) {
#pragma unroll
      for (int kb = 0; kb < 2; ++kb)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int s = 8 * kb + t + 4 * j;
          qa[kb][j][0] = qs[s * kQP + rowa] * pa[kb][j];
          qa[kb][j][1] = qs[s * kQP + rowb] * pb[kb][j];
        }
    } else {
#pragma unroll
      for (int kb = 0; kb < 2; ++kb)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int s = 8 * kb + t + 4 * j;
          const int e = s < len ? len - 1 - s : 0;
          qa[kb][j][0] = s < len ? qs[s * kQP + rowa] * sm.pw[e][rowa] : 0.f;
          qa[kb][j][1] = s < len ? qs[s * kQP + rowb] * sm.pw[e][rowb] : 0.f;
        }
      sla = sm.pw[len][rowa], slb = sm.pw[len][rowb];
    }
#pragma unroll
    for (int nt = 0; nt <= kNT; ++nt) {
      acc[nt][0] *= sla, acc[nt][1] *= sla;
      acc[nt][2] *= slb, acc[nt][3] *= slb;
    }
    const float* vs = &sm.vs[buf][0][0];
#pragma unroll
    for (int kb = 0; kb < 2; ++kb) {
      uint32_t ah[4], al[4];
      split_tf32(qa[kb][0][0], ah[0], al[0]);
      split_tf32(qa[kb][0][1], ah[1], al[1]);
      split_tf32(qa[kb][1][0], ah[2], al[2]);
      split_tf32(qa[kb][1][1], ah[3], al[3]);
      const float* vp = vs + (8 * kb + t) * kQP + g;
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt) {
        uint32_t bh0, bl0, bh1, bl1;
        split_tf32(vp[8 * nt], bh0, bl0);
        split_tf32(vp[8 * nt + 4 * kQP], bh1, bl1);
        mma_tf32(acc[nt], al, bh0, bh1);
        mma_tf32(acc[nt], ah, bl0, bl1);
        mma_tf32(acc[nt], ah, bh0, bh1);
      }
      mma_tf32(acc[kNT], al, one_b, one_b);
      mma_tf32(acc[kNT], ah, one_b, one_b);
    }
  }
  if (a.rho_final) {
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) {
      *reinterpret_cast<float2*>(a.rho_final + ((size_t)bh * kL + rowa) * kE + 8 * nt + 2 * t) =
          make_float2(acc[nt][0], acc[nt][1]);
      *reinterpret_cast<float2*>(a.rho_final + ((size_t)bh * kL + rowb) * kE + 8 * nt + 2 * t) =
          make_float2(acc[nt][2], acc[nt][3]);
    }
  }
  if (t == 0 && a.rho_norm_final) {
    a.rho_norm_final[(size_t)bh * kL + rowa] = acc[kNT][0];
    a.rho_norm_final[(size_t)bh * kL + rowb] = acc[kNT][2];
  }
}

}  // namespace

cudaError_t launch_state(const Args& a, cudaStream_t s) {
  const size_t smem = sizeof(StateSmem);
  cudaError_t e = cudaFuncSetAttribute(rwkv8_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  rwkv8_state_kernel<<<(unsigned)(a.B * a.H), kSThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace rwkv8
