/*
 * rwkv8.h - C ABI of the RWKV-8 normalized linear recurrence and its
 * backward-through-time on one GPU (sm_103a), in the same library as wkv7.h
 * (libwkv7.so). Status codes, the error message (wkv7_last_error) and the
 * stream conventions are those of wkv7.h.
 *
 * The operation (the burn_dragon_kernel page "src/sequence/rwkv8/backward.rs":
 * compute_chunk_traces for the state traces, backward_chunk_impl for the
 * readout and its gradient). For every batch b and head h an L x E fp32 state
 * rho (row l = latent index, column e = value index) and an L-vector rho_norm
 * run over t = 0 .. T-1 with a decay that depends on (h, l) only:
 *     qw_t   = q_t / (sum_l q_t[l] + EPS)                       EPS = 1e-6
 *     y_t[e] = sum_l qw_t[l] rho[l][e] / (rho_norm[l] + EPS)     (state before step t)
 *     rho[l][e]   <- decay[l] rho[l][e] + q_t[l] v_t[e]
 *     rho_norm[l] <- decay[l] rho_norm[l] + q_t[l]
 * The backward returns the gradients of
 *     L = sum <dy, y> + <d_rho_final, rho_final> + <d_rho_norm_final, rho_norm_final>
 * with respect to q, v, decay (summed over batch and time, as the page's
 * grad_decay) and the initial states. The page's own backward starts its carry
 * at zero; the final-state gradients are optional inputs (NULL = zero) so that
 * a long sequence can be cut into segments.
 *
 * Layouts (the page's): q [B][H][T][L]; v [B][Hv][T][E] with Hv = 1 (one value
 * row shared by every head; its gradient is summed over heads) or Hv = H;
 * decay [H][L]; y, dy [B][H][T][E]; rho states [B][H][L][E]; rho_norm states
 * [B][H][L]. All fp32, row-major.
 *
 * Sizes: L = E = 64 (the kernels' tile), B, H >= 1 or 0 with B * H < 2^28,
 * T >= 0 with B * H * T * L * 4 < 2^46. Every pointer
 * is device memory owned by the caller, 16-byte aligned; outputs are
 * overwritten and must not overlap an input or another output. An invalid
 * argument returns WKV7_ERR_INVALID before anything is enqueued.
 */
#ifndef RWKV8_H
#define RWKV8_H

#include <stddef.h>

#include "wkv7.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Length of the chunks the kernels process (and the checkpoint interval). */
#define RWKV8_CHUNK 16

/*
 * Bytes of the checkpoint buffer of rwkv8_forward / rwkv8_backward: the
 * states before every chunk of RWKV8_CHUNK steps, rho [B][H][nck][L][E]
 * followed by rho_norm [B][H][nck][L], nck = ceil(T / RWKV8_CHUNK), fp32.
 * 0 for an unsupported size.
 */
size_t rwkv8_ckpt_bytes(int B, int T, int H, int L, int E);

/*
 * Forward scan.
 *   q, v, decay        inputs (required).
 *   rho_init           [B][H][L][E] or NULL (zeros).
 *   rho_norm_init      [B][H][L] or NULL (zeros).
 *   y                  [B][H][T][E] output (required).
 *   rho_final          [B][H][L][E] or NULL (skipped).
 *   rho_norm_final     [B][H][L] or NULL (skipped).
 *   ckpt               rwkv8_ckpt_bytes(...) bytes for rwkv8_backward, or NULL.
 * The state chain between chunks runs first and writes the state before
 * every chunk into ckpt; y of every chunk is then made from it. With ckpt
 * NULL those states go to a workspace taken with cudaMallocAsync on the
 * stream (WKV7_ERR_ALLOC if that fails). RWKV8_SEQUENTIAL=1 in the
 * environment selects one pass per (b, h) through its chunks instead, which
 * needs no workspace; the results agree to fp32 rounding.
 * Returns WKV7_OK, WKV7_ERR_INVALID, WKV7_ERR_ALLOC or WKV7_ERR_CUDA.
 */
int rwkv8_forward(const float* q, const float* v, const float* decay, const float* rho_init,
                  const float* rho_norm_init, float* y, float* rho_final, float* rho_norm_final, float* ckpt,
                  int B, int T, int H, int Hv, int L, int E, void* stream);

/*
 * Backward-through-time.
 *   q, v, decay, dy          inputs (required).
 *   rho_init, rho_norm_init  the forward's initial states, or NULL (zeros);
 *                            read only when ckpt is NULL.
 *   d_rho_final              [B][H][L][E] gradient entering through the final
 *                            state, or NULL (zero).
 *   d_rho_norm_final         [B][H][L], or NULL (zero).
 *   ckpt                     the checkpoints rwkv8_forward wrote for the same
 *                            inputs, or NULL: the library then runs the forward
 *                            itself into a workspace taken with cudaMallocAsync
 *                            on `stream` and freed on it.
 *   dq [B][H][T][L], dv (v's shape), ddecay [H][L]     outputs (required).
 *   d_rho_init [B][H][L][E], d_rho_norm_init [B][H][L]  outputs, or NULL.
 * One CTA per (b, h) walks its chunks from the last to the first.
 * RWKV8_SPLIT_BACKWARD=1 in the environment selects the split form instead:
 * the <rho0, dy> rows of every chunk first, then the carried gradients alone,
 * one CTA per (b, h), storing their value after every chunk in a workspace
 * (about 1.3 KB per token-head with those rows), then every chunk's dq, dv and
 * ddecay terms at once; the results agree to fp32 rounding. ddecay is summed over the chunks
 * and over b in a fixed order (deterministic); with Hv = 1, dv is summed over
 * h in a fixed order. The workspace is taken with cudaMallocAsync on `stream`
 * (WKV7_ERR_ALLOC if that fails).
 * Returns WKV7_OK, WKV7_ERR_INVALID, WKV7_ERR_ALLOC or WKV7_ERR_CUDA.
 */
int rwkv8_backward(const float* q, const float* v, const float* decay, const float* dy, const float* rho_init,
                   const float* rho_norm_init, const float* d_rho_final, const float* d_rho_norm_final,
                   const float* ckpt, float* dq, float* dv, float* ddecay, float* d_rho_init,
                   float* d_rho_norm_init, int B, int T, int H, int Hv, int L, int E, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* RWKV8_H */
