// Backward of the time-mix epilogue ("rx_pretrain.c": the group-norm backward
// and the bonus backward of the time-mix), fused into the split backward.
//
// With out = (y - mean) rstd ln_w + ln_b + bonus v, bonus = sum_j r_j k_j r_k[j],
// nv = (y - mean) rstd and dout the gradient of out, per step and head:
//     dn = dout ln_w
//     dy = rstd (dn - mean(dn) - nv mean(dn nv))          (the scan's upstream gradient)
//     dbon = sum_i dout_i v_i
//     dv += dout bonus ;  dr += dbon k r_k ;  dk += dbon r r_k
//     dln_w += dout nv ;  dln_b += dout ;  dr_k += dbon r k    (summed over b and t)
// The split backward's kernels form dy where they read it (the carry kernel's
// forming warps and the output pass, wkv7_bwd4.cu); the output pass adds the
// bonus terms to its stores and writes each chunk's parameter terms. This file
// sums those terms over the chunks and the batch in a fixed order.
#include <cuda_runtime.h>

#include "wkv7_launch.h"

namespace wkv7 {
namespace {

constexpr int kN = 64;

// One thread per (h, quantity, column): the sum over b and the chunks, in order.
__global__ void epi_param_kernel(const float* part, float* dln_w, float* dln_b, float* dr_k, int B, int H,
                                 int nchunks) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= H * 3 * kN) return;
  const int h = i / (3 * kN), which = (i / kN) % 3, col = i % kN;
  float s = 0.f;
  for (int b = 0; b < B; ++b) {
    const float* p = part + ((size_t)(b * H + h) * nchunks) * 3 * kN + which * kN + col;
    for (int n = 0; n < nchunks; ++n) s += p[(size_t)n * 3 * kN];
  }
  float* dst = which == 0 ? dln_w : which == 1 ? dln_b : dr_k;
  dst[(size_t)h * kN + col] = s;
}

}  // namespace

cudaError_t launch_epi_params(const float* part, float* dln_w, float* dln_b, float* dr_k, int B, int H, int nchunks,
                              cudaStream_t stream) {
  const int n = H * 3 * kN;
  epi_param_kernel<<<(n + 127) / 128, 128, 0, stream>>>(part, dln_w, dln_b, dr_k, B, H, nchunks);
  return cudaGetLastError();
}

}  // namespace wkv7
