// Backward of the time-mix epilogue ("rx_pretrain.c": the group-norm backward
// and the bonus backward of the time-mix) around the scan's backward.
//
// With out = (y - mean) rstd ln_w + ln_b + bonus v, bonus = sum_j r_j k_j r_k[j],
// nv = (y - mean) rstd and dout the gradient of out, per step and head:
//     dn = dout ln_w
//     dy = rstd (dn - mean(dn) - nv mean(dn nv))          (the scan's upstream gradient)
//     dbon = sum_i dout_i v_i
//     dv += dout bonus ;  dr += dbon k r_k ;  dk += dbon r r_k
//     dln_w += dout nv ;  dln_b += dout ;  dr_k += dbon r k    (summed over b and t)
// epi_grad_kernel makes dy (bf16, what the scan's backward reads), dbon per
// row and the parameter terms per block; epi_bonus_kernel adds the bonus terms
// to the scan's dr, dk, dv in one streaming pass (folded into the backward's
// output kernel instead, the scattered loads they need cost more there); and
// epi_param_kernel sums the parameter terms over the blocks in a fixed order.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "wkv7_epilogue.h"
#include "wkv7_launch.h"

namespace wkv7 {
namespace {

constexpr int kN = 64;
constexpr int kRowsPerBlock = 64;  // (b, t) rows of one head per block
constexpr int kEpiThreads = 256;

__device__ __forceinline__ float2 ld_bf2(const __nv_bfloat16* p) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// grid (blocks over B*T, H); warp w handles rows 8 w .. 8 w + 7 of the block,
// lane l channels 2 l, 2 l + 1.
__global__ void __launch_bounds__(kEpiThreads) epi_grad_kernel(const EpiBwdArgs a) {
  __shared__ float part[8][3][kN];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int h = blockIdx.y, c = 2 * lane;
  const size_t rows = (size_t)a.B * a.T;
  const float2 lw = *reinterpret_cast<const float2*>(a.ln_w + (size_t)h * kN + c);
  float acc_w[2] = {0.f, 0.f}, acc_b[2] = {0.f, 0.f}, acc_k[2] = {0.f, 0.f};
  for (int q = 0; q < kRowsPerBlock / 8; ++q) {
    const size_t bt = (size_t)blockIdx.x * kRowsPerBlock + 8 * warp + q;
    if (bt >= rows) break;
    const size_t row = bt * a.H + h, off = row * kN + c;
    const float2 d = ld_bf2(a.dout + off), nv = ld_bf2(a.nv + off), v = ld_bf2(a.v + off);
    const float2 r = ld_bf2(a.r + off), k = ld_bf2(a.k + off);
    const float rstd = a.stats[2 * row];
    const float dn0 = d.x * lw.x, dn1 = d.y * lw.y;
    const float s1 = warp_sum(dn0 + dn1);
    const float s2 = warp_sum(fmaf(dn0, nv.x, dn1 * nv.y));
    const float dbon = warp_sum(fmaf(d.x, v.x, d.y * v.y));
    const float m1 = s1 * (1.f / kN), m2 = s2 * (1.f / kN);
    const float dy0 = rstd * (dn0 - m1 - nv.x * m2), dy1 = rstd * (dn1 - m1 - nv.y * m2);
    *reinterpret_cast<__nv_bfloat162*>(a.dy + off) = __floats2bfloat162_rn(dy0, dy1);
    if (lane == 0) a.dbon[row] = dbon;
    acc_w[0] = fmaf(d.x, nv.x, acc_w[0]);
    acc_w[1] = fmaf(d.y, nv.y, acc_w[1]);
    acc_b[0] += d.x;
    acc_b[1] += d.y;
    acc_k[0] = fmaf(dbon, r.x * k.x, acc_k[0]);
    acc_k[1] = fmaf(dbon, r.y * k.y, acc_k[1]);
  }
  part[warp][0][c] = acc_w[0], part[warp][0][c + 1] = acc_w[1];
  part[warp][1][c] = acc_b[0], part[warp][1][c + 1] = acc_b[1];
  part[warp][2][c] = acc_k[0], part[warp][2][c + 1] = acc_k[1];
  __syncthreads();
  for (int i = threadIdx.x; i < 3 * kN; i += kEpiThreads) {
    float s = 0.f;
    for (int w = 0; w < 8; ++w) s += part[w][i / kN][i % kN];
    a.part[((size_t)h * gridDim.x + blockIdx.x) * 3 * kN + i] = s;
  }
}

// dr += dbon k r_k, dk += dbon r r_k, dv += dout bonus; grid as epi_grad_kernel.
__global__ void __launch_bounds__(kEpiThreads) epi_bonus_kernel(const EpiBwdArgs a) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int h = blockIdx.y, c = 2 * lane;
  const size_t rows = (size_t)a.B * a.T;
  const float2 rk = *reinterpret_cast<const float2*>(a.r_k + (size_t)h * kN + c);
  for (int q = 0; q < kRowsPerBlock / 8; ++q) {
    const size_t bt = (size_t)blockIdx.x * kRowsPerBlock + 8 * warp + q;
    if (bt >= rows) break;
    const size_t row = bt * a.H + h, off = row * kN + c;
    const float dbon = a.dbon[row], bonus = a.stats[2 * row + 1];
    const float2 r = ld_bf2(a.r + off), k = ld_bf2(a.k + off), d = ld_bf2(a.dout + off);
    float2 x = *reinterpret_cast<float2*>(a.dr + off);
    x.x = fmaf(dbon * k.x, rk.x, x.x), x.y = fmaf(dbon * k.y, rk.y, x.y);
    *reinterpret_cast<float2*>(a.dr + off) = x;
    x = *reinterpret_cast<float2*>(a.dk + off);
    x.x = fmaf(dbon * r.x, rk.x, x.x), x.y = fmaf(dbon * r.y, rk.y, x.y);
    *reinterpret_cast<float2*>(a.dk + off) = x;
    x = *reinterpret_cast<float2*>(a.dv + off);
    x.x = fmaf(d.x, bonus, x.x), x.y = fmaf(d.y, bonus, x.y);
    *reinterpret_cast<float2*>(a.dv + off) = x;
  }
}

// dln_w, dln_b, dr_k [H][N]: the blocks' terms summed in block order.
__global__ void epi_param_kernel(const EpiBwdArgs a, int nblk) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= a.H * 3 * kN) return;
  const int h = i / (3 * kN), which = (i / kN) % 3, col = i % kN;
  float s = 0.f;
  for (int b = 0; b < nblk; ++b) s += a.part[((size_t)h * nblk + b) * 3 * kN + which * kN + col];
  float* dst = which == 0 ? a.dln_w : which == 1 ? a.dln_b : a.dr_k;
  dst[(size_t)h * kN + col] = s;
}

}  // namespace

int epi_blocks(int B, int T) { return (int)(((size_t)B * T + kRowsPerBlock - 1) / kRowsPerBlock); }

cudaError_t launch_epi_grad(const EpiBwdArgs& a, cudaStream_t s) {
  const dim3 grid((unsigned)epi_blocks(a.B, a.T), (unsigned)a.H);
  epi_grad_kernel<<<grid, kEpiThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_epi_finish(const EpiBwdArgs& a, cudaStream_t s) {
  const dim3 grid((unsigned)epi_blocks(a.B, a.T), (unsigned)a.H);
  epi_bonus_kernel<<<grid, kEpiThreads, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int n = a.H * 3 * kN;
  epi_param_kernel<<<(n + 255) / 256, 256, 0, s>>>(a, epi_blocks(a.B, a.T));
  return cudaGetLastError();
}

}  // namespace wkv7
