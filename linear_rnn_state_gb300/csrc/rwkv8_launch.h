// Kernel arguments and launchers of the RWKV-8 normalized recurrence (the
// C ABI in rwkv8.h validates everything before these run).
#pragma once

#include <cuda_runtime.h>

namespace rwkv8 {

constexpr int kL = 64;       // latent size (rows of the state)
constexpr int kE = 64;       // value size (columns of the state)
constexpr int kC = 16;       // chunk length = checkpoint interval
constexpr float kEps = 1e-6f;

struct Args {
  const float *q, *v, *decay, *dy;
  const float *rho_init, *rho_norm_init;       // NULL = zeros
  const float *d_rho_final, *d_rho_norm_final; // NULL = zeros
  float* y;                                    // NULL = skip (checkpointing pass)
  float *rho_final, *rho_norm_final;           // NULL = skip
  float* ckpt;                                 // forward: written; backward: read
  float* dq;
  float* dv;        // [B][H][T][E]: dv itself (Hv = H) or per-head terms to sum (Hv = 1)
  float* ddecay_bh; // [B][H][L] per-(b, h) terms of ddecay
  float *d_rho_init, *d_rho_norm_init;         // NULL = skip
  // Split backward's workspaces, per (b, h) and chunk c ([B*H][nchunks] ...):
  float* g15;          // [L][E] gradient w.r.t. the state after the chunk's last step
  float* gn15;         // [L] the same for the norm
  float* r0;           // [kC][L] R0[tau][l] = <rho0[l], dy_tau>, rho0 the checkpointed state
  float* gdot;         // [L] <G15[l], rho0[l]>
  float* ddecay_part;  // [L] the chunk's terms of ddecay
  int B, T, H, Hv;
};

__host__ __device__ inline size_t nchunks(int T) { return (size_t)((T + kC - 1) / kC); }
// Float offset of the rho_norm checkpoints inside the checkpoint buffer.
__host__ __device__ inline size_t ckpt_norm_offset(int B, int T, int H) { return (size_t)B * H * nchunks(T) * kL * kE; }

// One CTA per (b, h) through all chunks (RWKV8_SEQUENTIAL=1).
cudaError_t launch_forward(const Args& a, cudaStream_t s);
// The chain alone: checkpoints (if ckpt is set) and final states, no y.
cudaError_t launch_state(const Args& a, cudaStream_t s);
// y of every chunk at once from the checkpoints in a.ckpt.
cudaError_t launch_forward_chunks(const Args& a, cudaStream_t s);
// One CTA per (b, h) through all chunks (RWKV8_SEQUENTIAL=1).
cudaError_t launch_backward(const Args& a, cudaStream_t s);
// The split backward: the carried gradients alone (g15, gn15, r0, gdot for
// every chunk, d_rho_init, d_rho_norm_init), then every chunk's dq, dv and
// ddecay terms at once, then ddecay_bh = the chunk terms summed per (b, h).
cudaError_t launch_backward_chain(const Args& a, cudaStream_t s);
cudaError_t launch_backward_chunks(const Args& a, cudaStream_t s);
cudaError_t launch_chunk_sum(const Args& a, cudaStream_t s);
// out[i] = sum over g of in[g * stride + i], g = 0 .. groups-1, for i in [0, n).
cudaError_t launch_group_sum(const float* in, float* out, size_t n, size_t stride, int groups, cudaStream_t s);
// dv [B][1][T][E] = sum over h of part [B][H][T][E].
cudaError_t launch_head_sum(const float* part, float* dv, int B, int H, int T, cudaStream_t s);

}  // namespace rwkv8
