/*
 * wkv7.h - C ABI of the GB300 WKV7 library: the RWKV-7 matrix-state
 * recurrence and its backward-through-time on one GPU (sm_103a).
 *
 * The operation ("rx_pretrain.c", rx_wkv7_forward_seq and rx_wkv7_backward
 * with the reverse-scan equations (1)-(3) in the comment above it). For every
 * batch b and head h an N x N fp32 state S (row i = value index, column
 * j = key index) runs over t = 0 .. T-1:
 *     sa  = S a_t
 *     S  <- S diag(w_t) + v_t k_t^T + sa b_t^T
 *     y_t = S r_t                       (read after the update)
 * The backward carries G = dL/dS from t = T-1 down to 0, starting at zero
 * (no gradient enters through the final state):
 *     dr_t = S_t^T dy_t ;  G += dy_t r_t^T
 *     dk_t = G^T v_t ;  db_t = G^T sa_t ;  dw_t = colsum(G o S_prev)
 *     dv_t = G k_t ;    dsa = G b_t ;      da_t = S_prev^T dsa
 *     G <- G diag(w_t) + dsa a_t^T
 * and returns G after t = 0 as the gradient of the initial state. dw is the
 * gradient with respect to the effective decay w itself.
 *
 * Layout ("rx_pretrain.c", helpers vx and sx). Per-step vectors r, w, k, v,
 * a, b, y, dy and the six input gradients are row-major [B][T][H][N];
 * states s_init, s_final and dS_init are [B][H][N][N] with S_ij at
 * ((b*H + h)*N + i)*N + j. Checkpoints are [B][H][nck][N][N] with
 * nck = ceil(T / ckpt_every); checkpoint c is the state before step
 * c*ckpt_every (checkpoint 0 is the initial state).
 *
 * Memory and streams. Every pointer is device memory owned by the caller;
 * the library never frees or keeps it. Work is enqueued on `stream` (a
 * cudaStream_t; NULL is the legacy default stream) and the calls return
 * without waiting for it, except wkv7_status. Outputs are overwritten, not
 * accumulated, and must not overlap any input. Every pointer must be 16-byte
 * aligned. N must be 16, 32 or 64; B, T and H may be 0 (an empty problem:
 * with T = 0 the forward copies s_init, or zeros, to s_final and the backward
 * zeroes dS_init; buffers of zero size may be NULL).
 *
 * Status codes: WKV7_OK on success, otherwise a negative code; the message of
 * the calling thread's last error is in wkv7_last_error(). An invalid
 * argument is reported before anything is enqueued.
 */
#ifndef WKV7_H
#define WKV7_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define WKV7_OK 0
#define WKV7_ERR_ALLOC (-1)   /* a workspace could not be allocated */
#define WKV7_ERR_INVALID (-2) /* bad pointer, size, alignment or overlap */
#define WKV7_ERR_CUDA (-3)    /* a CUDA launch or runtime call failed */
#define WKV7_ERR_TIMEOUT (-4) /* a kernel gave up a bounded wait (wkv7_status) */
#define WKV7_ERR_BOUNDS (-5)  /* debug build only: a kernel skipped an access outside its buffer (wkv7_status) */

/* bfloat16 values are passed as their 16-bit patterns. */
typedef uint16_t wkv7_bf16;

/*
 * Forward scan, fp32 inputs.
 *   r, w, k, v, a, b  [B][T][H][N] inputs (required).
 *   s_init            [B][H][N][N] initial state, or NULL for zeros.
 *   y                 [B][T][H][N] output, or NULL to skip it.
 *   s_final           [B][H][N][N] final state, or NULL to skip it.
 *   ckpt              checkpoint buffer of wkv7_ckpt_bytes(B, T, H, N,
 *                     ckpt_every) bytes for wkv7_backward, or NULL.
 *   ckpt_every        checkpoint interval in steps (>= 1 when ckpt is set).
 * Arithmetic. At N = 64 with checkpoints every multiple of 16 steps (or none)
 * the chunked tensor-core form runs with every product taken in split
 * bfloat16: each fp32 operand x is x_hi + x_lo (x_hi = x rounded to bfloat16,
 * x_lo = x - x_hi rounded to bfloat16) and a b is a_lo b_hi + a_hi b_lo +
 * a_hi b_hi, three tensor-core products with fp32 accumulation (relative
 * error near 2^-16 per product); the state, its decay, the triangular solve
 * and y stay fp32.
 * Other N or checkpoint intervals run fp32 FMA throughout.
 * Returns WKV7_OK, WKV7_ERR_INVALID or WKV7_ERR_CUDA.
 */
int wkv7_forward(const float* r, const float* w, const float* k, const float* v, const float* a,
                 const float* b, const float* s_init, float* y, float* s_final, float* ckpt,
                 int ckpt_every, int B, int T, int H, int N, void* stream);

/* Forward scan with bfloat16 r, w, k, v, a, b and y; the state, s_init,
 * s_final and the checkpoints are fp32 in memory.
 * Arithmetic. At N = 64 with checkpoints every multiple of 16 steps (or none)
 * the chunked tensor-core form runs: every product is a tensor-core product
 * with bfloat16 operands (the inputs' own precision) and fp32 accumulation.
 * The scaled operands and the carried state (held and decayed in fp32) are
 * rounded to bfloat16 where they enter a product, except that the state
 * update takes its two scaled operands (k and b times the decay products) as
 * bfloat16 pairs hi + lo, about 16 bits, so that the carried state keeps
 * them at that precision. The element-wise work (decay products, the
 * triangular solve) is fp32. The bfloat16 y is rounded once from the fp32
 * result. Other N or checkpoint intervals run fp32 FMA throughout. */
int wkv7_forward_bf16(const wkv7_bf16* r, const wkv7_bf16* w, const wkv7_bf16* k, const wkv7_bf16* v,
                      const wkv7_bf16* a, const wkv7_bf16* b, const float* s_init, wkv7_bf16* y,
                      float* s_final, float* ckpt, int ckpt_every, int B, int T, int H, int N,
                      void* stream);

/*
 * Backward-through-time, fp32 inputs.
 *   r, w, k, v, a, b, dy  [B][T][H][N] (required; dy = dL/dy).
 *   s_init         [B][H][N][N] initial state or NULL for zeros; read only
 *                  when ckpt is NULL.
 *   ckpt           the checkpoints wkv7_forward wrote with the same
 *                  ckpt_every, or NULL: the library then runs its own
 *                  checkpointing forward into a workspace taken with
 *                  cudaMallocAsync on `stream` and freed on it after the
 *                  backward (WKV7_ERR_ALLOC if that fails). With ckpt NULL,
 *                  ckpt_every <= 0 lets the library pick the interval.
 *   dr, dw, dk, dv, da, db  [B][T][H][N] gradients (required).
 *   dS_init        [B][H][N][N] gradient of the initial state, or NULL.
 * Arithmetic. At N = 64 with 16-step checkpoints the chunked form runs in
 * two passes: the carried
 * gradient at every chunk boundary first (one sequential pass per (b, h), the
 * carry held and stored in fp32, in a workspace of B*H*ceil(T/16)*N*N floats
 * taken with cudaMallocAsync on `stream`, so WKV7_ERR_ALLOC can also be
 * returned when ckpt is given), then every chunk's gradients at once; every
 * product in split bfloat16, as in wkv7_forward. (Measured against an fp64
 * reference: every gradient element within 3e-5 (1 + |ref|) over the GPU
 * tests, within 1.7e-5 on the 8 x 4096 x 12 and 1 x 65536 x 40 workloads.)
 * Other N or checkpoint intervals run fp32 FMA throughout.
 * Returns WKV7_OK, WKV7_ERR_INVALID, WKV7_ERR_ALLOC or WKV7_ERR_CUDA.
 */
int wkv7_backward(const float* r, const float* w, const float* k, const float* v, const float* a,
                  const float* b, const float* dy, const float* s_init, const float* ckpt,
                  int ckpt_every, float* dr, float* dw, float* dk, float* dv, float* da, float* db,
                  float* dS_init, int B, int T, int H, int N, void* stream);

/* Backward with bfloat16 r, w, k, v, a, b and dy; checkpoints, s_init and every
 * gradient are fp32 in memory.
 * At N = 64 with 16-step checkpoints the chunked tensor-core form runs, split
 * in two passes. The carried gradient G at every chunk boundary is computed
 * first (one sequential pass per (b, h): bfloat16 operands, fp32
 * accumulation, G carried in fp32 and rounded to bfloat16 where it enters a
 * product) and stored as bfloat16 in a workspace of
 * B*H*ceil(T/16)*N*N values. Then every chunk's gradients are formed
 * independently with bfloat16 operands and fp32 accumulation: the chunk's
 * inputs, its stored bfloat16 carry and its fp32 checkpoint rounded once to
 * bfloat16; the decay scaling, the triangular solve and the dw sums are fp32.
 * (Measured relative L2 error against an fp64 reference at 4 x 4096 x 32
 * heads: the gradients 2e-3 to 5e-3, dS_init 1.7e-3.) The workspace is taken with
 * cudaMallocAsync on `stream` and freed on it after the call (together with
 * the checkpoint workspace when ckpt is NULL), so WKV7_ERR_ALLOC can also be
 * returned when ckpt is given. wkv7_backward_fused_bf16 runs the other form.
 * Other N or checkpoint intervals run fp32 FMA throughout. */
int wkv7_backward_bf16(const wkv7_bf16* r, const wkv7_bf16* w, const wkv7_bf16* k, const wkv7_bf16* v,
                       const wkv7_bf16* a, const wkv7_bf16* b, const wkv7_bf16* dy, const float* s_init,
                       const float* ckpt, int ckpt_every, float* dr, float* dw, float* dk, float* dv,
                       float* da, float* db, float* dS_init, int B, int T, int H, int N, void* stream);

/*
 * Backward of one segment of a longer sequence: as wkv7_backward (and
 * wkv7_backward_bf16), with the gradient of the loss w.r.t. the segment's
 * final state entering the reverse scan (the scan of "rx_pretrain.c" starts
 * its carry at zero; the Mamba-3 page's "serial_recalculated/backward.rs"
 * takes this final-state gradient as an input). Cutting a sequence at T1, the
 * segment [T1, T) is run first with the whole sequence's dS_final and
 * s_init = the state the forward reached at T1; its dS_init is then the
 * dS_final of the segment [0, T1).
 *   dS_final   [B][H][N][N] fp32 gradient entering through the final state, or
 *              NULL for zeros (then identical to wkv7_backward). An input: it
 *              must not overlap an output.
 * With T = 0, dS_init = dS_final. Other arguments, layouts, workspaces and
 * status codes as wkv7_backward / wkv7_backward_bf16.
 */
int wkv7_backward_segment(const float* r, const float* w, const float* k, const float* v, const float* a,
                          const float* b, const float* dy, const float* s_init, const float* dS_final,
                          const float* ckpt, int ckpt_every, float* dr, float* dw, float* dk, float* dv,
                          float* da, float* db, float* dS_init, int B, int T, int H, int N, void* stream);
int wkv7_backward_segment_bf16(const wkv7_bf16* r, const wkv7_bf16* w, const wkv7_bf16* k, const wkv7_bf16* v,
                               const wkv7_bf16* a, const wkv7_bf16* b, const wkv7_bf16* dy, const float* s_init,
                               const float* dS_final, const float* ckpt, int ckpt_every, float* dr, float* dw,
                               float* dk, float* dv, float* da, float* db, float* dS_init, int B, int T, int H,
                               int N, void* stream);

/*
 * The fused chunked backward (bfloat16 inputs, N = 64, 16-step checkpoints or
 * ckpt NULL): one pass per (b, h) over the chunks in reverse, with tf32
 * operands and fp32 accumulation in every product and the carried gradient
 * kept in fp32 (relative L2 error of the gradients about 5e-4, against 2e-3
 * to 5e-3 for the split form), and no carry workspace; slower than the split
 * form when B*H is below a few times the SM count. Arguments, layouts and
 * status codes as wkv7_backward_segment_bf16; N other than 64 or an interval
 * other than 16 return WKV7_ERR_INVALID.
 */
int wkv7_backward_fused_bf16(const wkv7_bf16* r, const wkv7_bf16* w, const wkv7_bf16* k, const wkv7_bf16* v,
                             const wkv7_bf16* a, const wkv7_bf16* b, const wkv7_bf16* dy, const float* s_init,
                             const float* dS_final, const float* ckpt, int ckpt_every, float* dr, float* dw,
                             float* dk, float* dv, float* da, float* db, float* dS_init, int B, int T, int H, int N,
                             void* stream);

/*
 * The decay given as logits (bfloat16 inputs, N = 64, 16-step checkpoints).
 * The RWKV-7 time-mix ("rx_pretrain.c", tm_pre_forward) forms the decay from a
 * logit z as w = exp(-0.606531 sigmoid(z)) (RX_WDECAY_COEFF); these calls take
 * z [B][T][H][N] in the place of w and form w in fp32 inside the scan kernels
 * where the decay tile is read, so w never exists in memory. The backward
 * returns dz = dL/dz (its backward's chain dw w (-0.606531) sigmoid(z)
 * (1 - sigmoid(z))) in the place of dw, and runs the split chunked form, with
 * the arithmetic of wkv7_backward_bf16. Other arguments, layouts, workspaces and
 * status codes as wkv7_forward_bf16 and wkv7_backward_segment_bf16; N other
 * than 64, or checkpoints with an interval other than 16, return
 * WKV7_ERR_INVALID.
 */
int wkv7_forward_logit_bf16(const wkv7_bf16* r, const wkv7_bf16* z, const wkv7_bf16* k, const wkv7_bf16* v,
                            const wkv7_bf16* a, const wkv7_bf16* b, const float* s_init, wkv7_bf16* y,
                            float* s_final, float* ckpt, int ckpt_every, int B, int T, int H, int N, void* stream);
int wkv7_backward_logit_bf16(const wkv7_bf16* r, const wkv7_bf16* z, const wkv7_bf16* k, const wkv7_bf16* v,
                             const wkv7_bf16* a, const wkv7_bf16* b, const wkv7_bf16* dy, const float* s_init,
                             const float* dS_final, const float* ckpt, int ckpt_every, float* dr, float* dz,
                             float* dk, float* dv, float* da, float* db, float* dS_init, int B, int T, int H, int N,
                             void* stream);

/*
 * Forward with the time-mix epilogue fused into the scan ("rx_pretrain.c":
 * gn_forward after rx_wkv7_forward_seq, and the bonus term): for every step
 * and head, with y the scan's output row of N channels,
 *     mean, var over the N channels;  rstd = 1 / sqrt(var + 64e-5)
 *     bonus = sum_j r_j k_j r_k[j]
 *     out = (y - mean) rstd ln_w + ln_b + bonus v
 * bfloat16 inputs at N = 64 (16-step checkpoints if ckpt is given);
 * decay_is_logit != 0 takes logits z in the place of w, as
 * wkv7_forward_logit_bf16. ln_w, ln_b, r_k: [H][N] fp32 (required).
 *   out    [B][T][H][N] bf16 (required; y itself is not written).
 *   nv     [B][T][H][N] bf16 normalized y, (y - mean) rstd, or NULL.
 *   stats  [B][T][H][2] fp32 (rstd, bonus) per row, or NULL.
 * s_final and ckpt as wkv7_forward_bf16 (the scan's state, unchanged by the
 * epilogue). N other than 64 returns WKV7_ERR_INVALID.
 */
int wkv7_forward_epilogue_bf16(const wkv7_bf16* r, const wkv7_bf16* w, const wkv7_bf16* k, const wkv7_bf16* v,
                               const wkv7_bf16* a, const wkv7_bf16* b, const float* s_init, const float* ln_w,
                               const float* ln_b, const float* r_k, wkv7_bf16* out, wkv7_bf16* nv, float* stats,
                               float* s_final, float* ckpt, int ckpt_every, int decay_is_logit, int B, int T, int H,
                               int N, void* stream);

/*
 * Backward of wkv7_forward_epilogue_bf16: the gradients of sum <dout, out>.
 *   dout        [B][T][H][N] bf16, the gradient of the epilogue's output.
 *   nv, stats   the normalized y and (rstd, bonus) rows the forward wrote.
 *   ln_w, r_k   [H][N] fp32, the forward's parameters (ln_b does not enter).
 *   dr, dw (dz with decay_is_logit), dk, dv, da, db, dS_init: as
 *               wkv7_backward_segment_bf16, with the bonus term's parts of
 *               dr, dk, dv included.
 *   dln_w, dln_b, dr_k  [H][N] fp32, summed over b and t (required).
 * The group-norm gradient that is the scan's upstream gradient,
 *     dy = rstd (dout ln_w - mean(dout ln_w) - nv mean(dout ln_w nv)),
 * is formed inside the scan's split backward where its kernels read dy (rounded
 * to bf16, as the scan's dy is), and the output pass adds the bonus terms to
 * dr, dk, dv as it stores them; each chunk's parameter terms go to a workspace
 * of B*H*ceil(T/16)*3*N floats (cudaMallocAsync on `stream`, WKV7_ERR_ALLOC)
 * that a last small kernel sums in a fixed order. N other than 64, or
 * checkpoints with an interval other than 16, return WKV7_ERR_INVALID.
 */
int wkv7_backward_epilogue_bf16(const wkv7_bf16* r, const wkv7_bf16* w, const wkv7_bf16* k, const wkv7_bf16* v,
                                const wkv7_bf16* a, const wkv7_bf16* b, const wkv7_bf16* dout, const wkv7_bf16* nv,
                                const float* stats, const float* ln_w, const float* r_k, const float* s_init,
                                const float* dS_final, const float* ckpt, int ckpt_every, int decay_is_logit,
                                float* dr, float* dw, float* dk, float* dv, float* da, float* db, float* dS_init,
                                float* dln_w, float* dln_b, float* dr_k, int B, int T, int H, int N, void* stream);

/* Bytes of the checkpoint buffer: B*H*ceil(T/ckpt_every)*N*N*4, or 0 for an
 * invalid size. */
size_t wkv7_ckpt_bytes(int B, int T, int H, int N, int ckpt_every);

/* The checkpoint interval the library picks for N and the input type
 * (bf16 != 0 for bfloat16 inputs): the backward replays whole chunks of this
 * length from shared memory. 0 for an unsupported N. */
int wkv7_default_ckpt_every(int N, int bf16);

/* Waits for `stream`, then reports (and clears) what the kernels flagged on
 * the current device: WKV7_OK, WKV7_ERR_TIMEOUT when a bounded wait inside a
 * kernel gave up, WKV7_ERR_BOUNDS when (in the debug build, which checks every
 * plain global load and store of the scan kernels against the buffer it
 * belongs to) a kernel found an index outside its buffer and skipped that
 * access, or WKV7_ERR_CUDA for a CUDA error. */
int wkv7_status(void* stream);

/* Message of the calling thread's last failed call ("" if none). */
const char* wkv7_last_error(void);

/*
 * Backward-through-time, fp32 inputs, with no device allocation. This entry
 * point has no counterpart on the pages; it serves callers that cannot
 * allocate device memory (a stream being captured into a graph that must not
 * contain allocation nodes, or a framework that owns every device byte through
 * its own allocator). It behaves like wkv7_backward with ckpt = NULL and the
 * default interval (16 steps), but its own forward writes the checkpoints into
 * a fixed 64 MiB scratch array of the library, held on every GPU that loads the
 * library until the process exits, instead of a cudaMallocAsync workspace.
 *   Limit: B*H*ceil(T/16)*N*N*4 bytes of checkpoints must fit in 64 MiB
 *   (e.g. B*H = 16 heads of T = 4096, N = 64); a larger problem returns
 *   WKV7_ERR_INVALID before anything is enqueued.
 *   The first call on a device looks the scratch array up
 *   (cudaGetSymbolAddress); make that first call before any stream capture.
 *   All calls share the one array and it keeps the last call's contents:
 *   every checkpoint a call reads is written by that call first, so nothing
 *   needs clearing, but calls whose work overlaps on the GPU (other streams,
 *   other threads) race on it; serialize them.
 * Arguments, layouts and status codes as wkv7_backward; no cudaMalloc,
 * cudaFree or allocating library call is made.
 */
int wkv7_backward_noalloc(const float* r, const float* w, const float* k, const float* v, const float* a,
                          const float* b, const float* dy, const float* s_init, float* dr, float* dw, float* dk,
                          float* dv, float* da, float* db, float* dS_init, int B, int T, int H, int N,
                          void* stream);

#ifdef __cplusplus
}
#endif

#endif /* WKV7_H */
