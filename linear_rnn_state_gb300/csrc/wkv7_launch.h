// Internal launch interface between the C ABI (wkv7_api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>

namespace wkv7 {

// Records `msg` as the calling thread's last error and returns `code`.
int api_fail(int code, const char* msg);

// A buffer that a kernel reads or writes with plain (non-TMA) loads and
// stores: its first byte and its size. The debug build (WKV7_DEBUG) checks
// every such access against it (wkv7_common.cuh, in_extent); other builds
// carry it unused. TMA copies are bounded by their tensor maps instead.
struct Extent {
  const void* lo = nullptr;
  size_t bytes = 0;
};
struct FwdExtents {
  Extent in[6];  // r, w, k, v, a, b
  Extent y, nv, stats, s_init, s_final, ckpt, ln_w, ln_b, r_k;
};
struct BwdExtents {
  Extent in[8];  // r, w, k, v, a, b, dy (dout with the epilogue), nv
  Extent ckpt, carry, dr, dw, dk, dv, da, db, dS_init, dS_final, stats, ln_w, r_k, part;
};

// Forward kernel arguments. The tensor maps describe r, w, k, v, a, b as
// 4-D tensors (N, H, T, B) with a box of (N, 1, K, 1): K steps of one head.
struct FwdArgs {
  CUtensorMap map[6];
  const void* in[6];    // r, w, k, v, a, b ([B][T][H][N], the input type), the tensor maps'
                        // buffers: the chunked kernel's direct form reads fp32 rows here
  const float* s_init;  // [B][H][N][N] or null (zeros)
  void* y;              // [B][T][H][N] of the input type, or null
  float* s_final;       // [B][H][N][N] or null
  float* ckpt;          // [B][H][nck][N][N] or null
  unsigned* status;     // device status word (timeout flag)
  int w_logit = 0;      // 1: the w tiles hold logits z, w = exp(-0.606531 sigmoid(z)) (chunked kernels only)
  // epilogue (chunked forward only): y <- group_norm(y) ln_w + ln_b + (sum r k r_k) v per head
  int epilogue = 0;
  const float* ln_w = nullptr;  // [H][N]
  const float* ln_b = nullptr;  // [H][N]
  const float* r_k = nullptr;   // [H][N]
  void* nv = nullptr;           // [B][T][H][N] normalized y (input type), or null
  float* stats = nullptr;       // [B][T][H][2] (rstd, bonus), or null
  int C;                // checkpoint interval (steps)
  int nck;              // ceil(T / C)
  int B, T, H;
  FwdExtents ext;
  // Debug build only (WKV7_DEBUG): 1 makes the scalar forward issue no load
  // (and no expected-byte count) for its last chunk, so the wait for that
  // chunk runs out with nothing in flight. Ignored by every other build.
  int debug_skip_last_load = 0;
};

// Backward kernel arguments. Tensor maps for r, w, k, v, a, b, dy with a box
// of (N, 1, KS, 1).
struct BwdArgs {
  CUtensorMap map[7];
  CUtensorMap ckmap;  // checkpoints as (N, N, B*H*nck), box (N, N, 1)
  const float* ckpt;  // [B][H][nck][N][N], checkpoint c = state before step c*C
  float* dr;
  float* dw;
  float* dk;
  float* dv;
  float* da;
  float* db;
  float* dS_init;         // [B][H][N][N] or null
  const float* dS_final;  // [B][H][N][N] gradient entering through the final state, or null (zeros)
  const void* in[7];  // r, w, k, v, a, b, dy ([B][T][H][N], the input type)
  void* carry;        // split backward: [B*H][nchunks][N][N] carry after each chunk (bf16)
  // Split backward's tensor-core output kernel: the seven vectors as maps with a
  // (N, 1, 16, 1) box in 128-byte-swizzled shared-memory layout, and the carry
  // workspace as (N, N, B*H*nchunks) with an (N, N, 1) box, also swizzled.
  CUtensorMap swmap[7];
  CUtensorMap gcmap;
  int out_kernel = 0;  // split backward's output pass: 0 the mma.sync kernel, 1 the tcgen05 one
  // Backward of the time-mix epilogue fused into the split backward (mma.sync output pass):
  // the dy vector (map[6], in[6]) holds dout, the gradient of the epilogue's output, and the
  // kernels form the scan's dy = rstd (dn - mean(dn) - nv mean(dn nv)), dn = dout ln_w, where
  // they read it; the output pass also adds the bonus terms to dr, dk, dv and writes each
  // chunk's parameter terms.
  int epilogue = 0;
  CUtensorMap map_nv;          // nv [B][T][H][N] bf16, box (N, 1, 16, 1)
  const void* epi_nv = nullptr;
  const float* epi_stats = nullptr;  // [B][T][H][2] (rstd, bonus)
  const float* epi_ln_w = nullptr;   // [H][N]
  const float* epi_r_k = nullptr;    // [H][N]
  float* epi_part = nullptr;         // [B][H][nchunks][3][N]: sum_t dout nv, sum_t dout, sum_t dbon r k
  unsigned* status;
  int w_logit = 0;    // 1: the w tiles hold logits z and dw receives dL/dz (split backward only)
  int C, nck;
  int B, T, H;
  BwdExtents ext;
};

// Steps per TMA box of the forward kernels' input rows.
int fwd_steps_per_stage(int N, bool bf16);

cudaError_t launch_fwd2(const FwdArgs& args, bool bf16, int N, cudaStream_t stream);
// Chunked tensor-core forward: N = 64, checkpoints (if any) at a multiple of
// its 16-step chunk; bf16 inputs (bf16 operands, one product per product) or
// fp32 inputs (split bf16, three; the decay as w and no epilogue).
cudaError_t launch_fwd3(const FwdArgs& args, bool bf16, cudaStream_t stream);
// Chunked tensor-core backward: bf16 inputs, N = 64, checkpoints every 16 steps.
cudaError_t launch_bwd3(const BwdArgs& args, cudaStream_t stream);
// The same backward as a carry-chain kernel plus a parallel per-chunk output
// kernel; needs args.carry, a workspace of bwd4_workspace_bytes.
cudaError_t launch_bwd4(const BwdArgs& args, cudaStream_t stream);
// The same split for fp32 inputs: the carry chain (products in split bf16), storing fp32
// carries in the workspace, then the per-chunk output pass.
cudaError_t launch_bwd4_carry_f32(const BwdArgs& args, cudaStream_t stream);
cudaError_t launch_bwd4_out_f32(const BwdArgs& args, cudaStream_t stream);
size_t bwd4_workspace_bytes(int B, int T, int H, bool bf16);
// dln_w, dln_b, dr_k [H][N] from the output pass's per-chunk terms, summed in a fixed order.
cudaError_t launch_epi_params(const float* part, float* dln_w, float* dln_b, float* dr_k, int B, int H, int nchunks,
                              cudaStream_t stream);
constexpr int kChunk = 16;
inline bool use_chunked(bool bf16, int N, int C) { return bf16 && N == 64 && C % kChunk == 0; }
// The forward takes the chunked kernel for either input type.
inline bool use_chunked_fwd(int N, int C) { return N == 64 && C % kChunk == 0; }
cudaError_t launch_bwd2(const BwdArgs& args, bool bf16, int N, cudaStream_t stream);
int bwd2_steps_per_window(int N, bool bf16);

}  // namespace wkv7
