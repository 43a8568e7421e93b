// Launch interface of the time-mix epilogue's backward (wkv7_epilogue.cu).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace wkv7 {

// Backward of the time-mix epilogue (wkv7_epilogue.cu): bf16 [B][T][H][N]
// rows, N = 64.
struct EpiBwdArgs {
  const __nv_bfloat16 *dout, *nv, *r, *k, *v;
  const float* stats;  // [B][T][H][2] (rstd, bonus)
  const float *ln_w, *r_k;
  __nv_bfloat16* dy;   // out: the scan's upstream gradient
  float* dbon;         // [B][T][H] workspace: gradient of each row's bonus
  float* part;         // [H][blocks][3][N] workspace: per-block parameter terms
  float *dr, *dk, *dv; // the scan's gradients, to which the bonus terms are added
  float *dln_w, *dln_b, *dr_k;
  int B, T, H;
};
int epi_blocks(int B, int T);
cudaError_t launch_epi_grad(const EpiBwdArgs& a, cudaStream_t stream);
cudaError_t launch_epi_finish(const EpiBwdArgs& a, cudaStream_t stream);

}  // namespace wkv7
