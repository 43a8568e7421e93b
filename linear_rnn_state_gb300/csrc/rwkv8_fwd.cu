// RWKV-8 normalized recurrence, forward, in chunks of 16 steps.
//
// The recurrence (burn_dragon_kernel, "src/sequence/rwkv8/backward.rs":
// compute_chunk_traces and the readout of backward_chunk_impl): per (b, h) a
// 64 x 64 state rho and a 64-vector n, a decay d[l] fixed in time,
//     y_t  = sum_l qw_t[l] rho[l][:] / (n[l] + EPS),  qw_t = q_t / (sum q_t + EPS)
//     rho <- d (.) rho + q_t v_t^T,   n <- d (.) n + q_t       (after the readout)
// Because d does not depend on t, a chunk of steps t0 .. t0+15 (tau = t - t0)
// is exact in closed form from the chunk-start state rho0, n0:
//     n_tau   = d^tau n0 + sum_{s<tau} d^(tau-1-s) q_s
//     U[tau]  = qw_tau / (n_tau + EPS)                          (per l)
//     y_tau   = (U[tau] d^tau)^T rho0 + sum_{s<tau} A[tau][s] v_s,
//     A[tau][s] = sum_l U[tau][l] q_s[l] d_l^(tau-1-s)          (s < tau)
//     rho_end = d^len (.) rho0 + sum_s (q_s d^(len-1-s)) v_s^T,  n_end likewise
// with len = 16 except a shorter last chunk. Only rho_end depends on rho0, and
// only elementwise, so the chain between chunks is one multiply-add per state
// element; the rest of a chunk is independent work.
//
// This is the one-pass form (RWKV8_SEQUENTIAL=1; by default the chain runs
// alone in rwkv8_state.cu and the readout per chunk in rwkv8_chunk.cu). One
// CTA of 256 threads per (b, h) runs the chunks in order, fp32 FFMA on the
// CUDA cores. The state lives in registers (a 4 x 4 tile per thread) with
// a copy in shared memory for the readout product; the next chunk's q and v
// are copied in with cp.async while the current one is processed. The state
// before every chunk (and n) is written out as the backward's checkpoint.
#include <cuda_runtime.h>

#include "rwkv8.h"
#include "rwkv8_launch.h"

namespace rwkv8 {
namespace {

constexpr int kThreads = 256;
constexpr int kP = kE + 4;   // row pitch of the state copy (16-byte units 17 apart)
constexpr int kUP = kC + 4;  // row pitch of U^T

struct FwdSmem {
  float qs[2][kC][kL];
  float vs[2][kC][kE];
  float rho[kL][kP];
  float pw[kC + 1][kL];  // pw[k][l] = d_l^k
  float U[kC][kL];       // U[tau][l]
  float UtT[kL][kUP];    // U[tau][l] d_l^tau, transposed
  float Qt[kC][kL];      // q_s[l] d_l^(len-1-s), zero for s >= len
  float A[kC][kC + 1];   // strictly lower part of A; the rest stays zero
  float mend[4][kL];     // end of each 4-step segment of the local norm scan
  float sqp[2][kC];      // row sums of q over each half of l
  float nst[2][kL];      // chunk-start n, by chunk parity
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

// Copies chunk `c` of q and v into buffer `buf`; rows past the end of the
// sequence are zero-filled. Each thread moves one 16-byte piece of each.
__device__ __forceinline__ void load_chunk(FwdSmem& sm, int buf, const float* qh, const float* vh, int c, int T,
                                           int tid) {
  const int row = tid >> 4, col = (tid & 15) * 4;
  const int t = c * kC + row;
  float* dq = &sm.qs[buf][row][col];
  float* dv = &sm.vs[buf][row][col];
  if (t < T) {
    cp_async16(dq, qh + (size_t)t * kL + col);
    cp_async16(dv, vh + (size_t)t * kE + col);
  } else {
    *reinterpret_cast<float4*>(dq) = make_float4(0.f, 0.f, 0.f, 0.f);
    *reinterpret_cast<float4*>(dv) = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  cp_async_commit();
}

__global__ void __launch_bounds__(kThreads, 1) rwkv8_fwd_kernel(const Args a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  FwdSmem& sm = *reinterpret_cast<FwdSmem*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int bh = blockIdx.x, h = bh % a.H, b = bh / a.H;
  const int T = a.T, nck = (T + kC - 1) / kC;
  const float* qh = a.q + (size_t)bh * T * kL;
  const float* vh = a.v + ((size_t)b * a.Hv + (a.Hv == 1 ? 0 : h)) * T * kE;
  float* yh = a.y ? a.y + (size_t)bh * T * kE : nullptr;
  float* ck_rho = a.ckpt ? a.ckpt + (size_t)bh * nck * kL * kE : nullptr;
  float* ck_n = a.ckpt ? a.ckpt + ckpt_norm_offset(a.B, T, a.H) + (size_t)bh * nck * kL : nullptr;

  load_chunk(sm, 0, qh, vh, 0, T, tid);

  // Per-thread roles.
  //  scan role:   latent l_s = tid & 63, rows 4 seg .. 4 seg + 3 of a chunk
  //  A role:      pairs of A (below)
  //  readout:     rows 4 rt .. 4 rt + 3 of y, columns 4 ec .. 4 ec + 3, latent quarter kq
  //  state tile:  rows 4 lt .. 4 lt + 3, columns 4 ec .. 4 ec + 3
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
  const int ec = (lane & 7) | ((w & 1) << 3);
  const int kq = lane >> 3, rt = w >> 1;
  const int lt = (lane >> 3) + 4 * (w >> 1);

  if (tid < kL) {
    const float d = a.decay[(size_t)h * kL + tid];
    float p = 1.f;
    for (int k = 0; k <= kC; ++k) {
      sm.pw[k][tid] = p;
      p *= d;
    }
    sm.nst[0][tid] = a.rho_norm_init ? a.rho_norm_init[(size_t)bh * kL + tid] : 0.f;
  }
  for (int i = tid; i < kC * (kC + 1); i += kThreads) (&sm.A[0][0])[i] = 0.f;

  float r[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (a.rho_init) x = *reinterpret_cast<const float4*>(a.rho_init + ((size_t)bh * kL + 4 * lt + i) * kE + 4 * ec);
    r[i][0] = x.x, r[i][1] = x.y, r[i][2] = x.z, r[i][3] = x.w;
    *reinterpret_cast<float4*>(&sm.rho[4 * lt + i][4 * ec]) = x;
  }

  for (int c = 0; c < nck; ++c) {
    const int buf = c & 1;
    const int len = min(kC, T - c * kC);
    cp_async_wait_all();
    __syncthreads();  // chunk c in shared memory; previous chunk fully done

    // ---- phase 1: local norm scan, row sums, checkpoint, prefetch
    float x[4], loc[4];
    const float d = sm.pw[1][l_s];
    {
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
    if (ck_rho) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        *reinterpret_cast<float4*>(ck_rho + ((size_t)c * kL + 4 * lt + i) * kE + 4 * ec) =
            make_float4(r[i][0], r[i][1], r[i][2], r[i][3]);
    }
    if (c + 1 < nck) load_chunk(sm, buf ^ 1, qh, vh, c + 1, T, tid);
    __syncthreads();

    // ---- phase 2: n before every step, U, U d^tau, q d^(len-1-s)
    {
      const float n0 = sm.nst[buf][l_s];
      if (seg == 0 && ck_n) ck_n[(size_t)c * kL + l_s] = n0;
      float start = n0;
      for (int s2 = 0; s2 < seg; ++s2) start = fmaf(sm.pw[4][l_s], start, sm.mend[s2][l_s]);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int tau = 4 * seg + j;
        const float nb = fmaf(sm.pw[j][l_s], start, loc[j]);
        const float sq = sm.sqp[0][tau] + sm.sqp[1][tau] + kEps;
        const float u = __fdividef(x[j], sq * (nb + kEps));  // denominator >= 1e-12
        sm.U[tau][l_s] = u;
        sm.UtT[l_s][tau] = u * sm.pw[tau][l_s];
        sm.Qt[tau][l_s] = tau < len ? x[j] * sm.pw[len - 1 - tau][l_s] : 0.f;
        if (tau == len - 1) sm.nst[buf ^ 1][l_s] = fmaf(d, nb, x[j]);
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
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
#pragma unroll 4
    for (int k = 0; k < 16; ++k) {
      const int l = 16 * kq + k;
      const float4 u = *reinterpret_cast<const float4*>(&sm.UtT[l][4 * rt]);
      const float4 s = *reinterpret_cast<const float4*>(&sm.rho[l][4 * ec]);
      const float uu[4] = {u.x, u.y, u.z, u.w}, ss[4] = {s.x, s.y, s.z, s.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(uu[i], ss[j], acc[i][j]);
    }
    float yv[4];
    reduce_scatter4(acc, kq, yv);
    __syncthreads();  // A complete; every read of rho0 done

    // ---- phase 4: y = readout + A v, then rho <- d^len rho + Qt^T v
    {
      const int tau = 4 * rt + kq;
      // A[tau][s] is zero for s >= tau; the warp's rows end at 4 rt + 3
#pragma unroll 4
      for (int s = 0; s < 4 * rt + 3; ++s) {
        const float al = sm.A[tau][s];
        const float4 vv = *reinterpret_cast<const float4*>(&sm.vs[buf][s][4 * ec]);
        yv[0] = fmaf(al, vv.x, yv[0]);
        yv[1] = fmaf(al, vv.y, yv[1]);
        yv[2] = fmaf(al, vv.z, yv[2]);
        yv[3] = fmaf(al, vv.w, yv[3]);
      }
      if (tau < len && yh)
        *reinterpret_cast<float4*>(yh + ((size_t)c * kC + tau) * kE + 4 * ec) = make_float4(yv[0], yv[1], yv[2], yv[3]);
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
        const float4 qt = *reinterpret_cast<const float4*>(&sm.Qt[s][4 * lt]);
        const float4 vv = *reinterpret_cast<const float4*>(&sm.vs[buf][s][4 * ec]);
        const float qq[4] = {qt.x, qt.y, qt.z, qt.w}, vw[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) r[i][j] = fmaf(qq[i], vw[j], r[i][j]);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
        *reinterpret_cast<float4*>(&sm.rho[4 * lt + i][4 * ec]) = make_float4(r[i][0], r[i][1], r[i][2], r[i][3]);
    }
  }
  __syncthreads();
  if (a.rho_final) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
      *reinterpret_cast<float4*>(a.rho_final + ((size_t)bh * kL + 4 * lt + i) * kE + 4 * ec) =
          make_float4(r[i][0], r[i][1], r[i][2], r[i][3]);
  }
  if (a.rho_norm_final && tid < kL) a.rho_norm_final[(size_t)bh * kL + tid] = sm.nst[nck & 1][tid];
}

}  // namespace

cudaError_t launch_forward(const Args& a, cudaStream_t s) {
  const size_t smem = sizeof(FwdSmem);
  cudaError_t e = cudaFuncSetAttribute(rwkv8_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  rwkv8_fwd_kernel<<<a.B * a.H, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace rwkv8
