// WKV7 forward scan (RWKV-7 matrix-state recurrence), sm_103a.
//
// Computes, per (batch b, head h), for t = 0 .. T-1 ("rx_pretrain.c",
// rx_wkv7_forward_seq):
//   sa = S a_t ;  S <- S diag(w_t) + v_t k_t^T + sa b_t^T ;  y_t = S r_t
// with S the N x N fp32 state (row i = value index, column j = key index),
// and writes S every C steps to the checkpoint buffer for the backward.
//
// Work decomposition. Rows of S evolve independently: row i needs only the
// shared vectors a, w, k, b, r and its own v_i, and sa_i, y_i are sums over
// the row. A CTA owns ROWS rows of one head; G consecutive lanes share a row,
// each holding E = N / G columns in registers as E / 4 column quads
// (quad q = m * G + g, so the G lanes of a row read adjacent 16-byte pieces
// of every shared vector and the loads are free of bank conflicts). sa and y
// are xor-shuffle sums over the G lanes. The per-step input rows (strided by
// H*N in memory) arrive K steps at a time through 4-D TMA tensor loads into a
// two-stage shared-memory ring, completion tracked by mbarriers with bounded
// waits.
#include "wkv7_common.cuh"
#include "wkv7_launch.h"

namespace wkv7 {

template <typename TIn, int N, int G, int ROWS, int K>
struct FwdCfg {
  static constexpr int E = N / G;
  static constexpr int Q = E / 4;
  static constexpr int THREADS = ROWS * G;
  static constexpr int NSTAGE = 2;
  static constexpr int NVEC = 6;  // r, w, k, v, a, b
  static constexpr int VEC_ELEMS = K * N;
  static constexpr int STAGE_BYTES = NVEC * VEC_ELEMS * Elem<TIn>::bytes;
  static constexpr int SMEM_BYTES = NSTAGE * STAGE_BYTES + 64;
  static_assert(E % 4 == 0 && N % ROWS == 0 && 32 % G == 0, "bad forward tiling");
  static_assert(THREADS % 32 == 0, "forward CTA must be whole warps");
};

template <typename TIn, int N, int G, int ROWS, int K>
__global__ void __launch_bounds__(ROWS* G) wkv7_fwd_kernel(const __grid_constant__ FwdArgs args) {
  using Cfg = FwdCfg<TIn, N, G, ROWS, K>;
  constexpr int E = Cfg::E, Q = Cfg::Q;
  extern __shared__ __align__(128) unsigned char smem[];
  TIn* stage = reinterpret_cast<TIn*>(smem);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::NSTAGE * Cfg::STAGE_BYTES);

  const int T = args.T, H = args.H;
  constexpr int slabs = N / ROWS;
  const int slab = blockIdx.x % slabs;
  const int head = blockIdx.x / slabs;  // b * H + h
  const int bi = head / H, hi = head % H;
  const int tid = threadIdx.x;
  const int g = tid % G;
  const int row = slab * ROWS + tid / G;

  // ---- state in registers: S[m*4 + e] is column 4*(m*G + g) + e of `row`
  float S[E];
  if (args.s_init) {
    const float* src = args.s_init + ((size_t)head * N + row) * N;
#pragma unroll
    for (int m = 0; m < Q; ++m) {
      const float4 s4 = *reinterpret_cast<const float4*>(src + 4 * (m * G + g));
      S[4 * m] = s4.x; S[4 * m + 1] = s4.y; S[4 * m + 2] = s4.z; S[4 * m + 3] = s4.w;
    }
  } else {
#pragma unroll
    for (int e = 0; e < E; ++e) S[e] = 0.f;
  }

  const int nchunks = (T + K - 1) / K;
  if (tid == 0) {
    for (int s = 0; s < Cfg::NSTAGE; ++s) mbar_init(&full[s], 1);
    fence_mbar_init();
    for (int v = 0; v < Cfg::NVEC; ++v) prefetch_tensormap(&args.map[v]);
  }
  __syncthreads();

  auto issue = [&](int chunk, int st) {
    mbar_arrive_expect_tx(&full[st], Cfg::STAGE_BYTES);
    TIn* dst = stage + st * Cfg::NVEC * Cfg::VEC_ELEMS;
    for (int v = 0; v < Cfg::NVEC; ++v)
      tma_load_4d(dst + v * Cfg::VEC_ELEMS, &args.map[v], &full[st], 0, hi, chunk * K, bi);
  };
  if (tid == 0)
    for (int s = 0; s < Cfg::NSTAGE && s < nchunks; ++s) issue(s, s);

  TIn* y = static_cast<TIn*>(args.y);
  const size_t y_step = (size_t)H * N;
  TIn* y_ptr = y ? y + ((size_t)bi * T * H + hi) * N + row : nullptr;
  float* ck_ptr = args.ckpt ? args.ckpt + ((size_t)head * args.nck * N + row) * N : nullptr;
  int to_ckpt = 0;  // steps until the next checkpoint

  for (int c = 0; c < nchunks; ++c) {
    const int st = c % Cfg::NSTAGE;
    {
      const uint32_t par = (c / Cfg::NSTAGE) & 1;
      const bool ok = mbar_wait_bounded(args.status, &full[st], par);
      // Gave up (status word set): wait once more, bounded, for the copy in
      // flight into this CTA's shared memory, then leave together.
      if (!ok) mbar_wait_bounded(args.status, &full[st], par);
      if (!__syncthreads_and(ok)) return;
    }
    const TIn* base = stage + st * Cfg::NVEC * Cfg::VEC_ELEMS;
    const int nk = min(K, T - c * K);
    for (int kk = 0; kk < nk; ++kk) {
      if (to_ckpt == 0) {
        if (ck_ptr) {
#pragma unroll
          for (int m = 0; m < Q; ++m)
            *reinterpret_cast<float4*>(ck_ptr + 4 * (m * G + g)) =
                make_float4(S[4 * m], S[4 * m + 1], S[4 * m + 2], S[4 * m + 3]);
          ck_ptr += (size_t)N * N;
        }
        to_ckpt = args.C;
      }
      --to_ckpt;
      const TIn* r_ = base + 0 * Cfg::VEC_ELEMS + kk * N;
      const TIn* w_ = base + 1 * Cfg::VEC_ELEMS + kk * N;
      const TIn* k_ = base + 2 * Cfg::VEC_ELEMS + kk * N;
      const TIn* v_ = base + 3 * Cfg::VEC_ELEMS + kk * N;
      const TIn* a_ = base + 4 * Cfg::VEC_ELEMS + kk * N;
      const TIn* b_ = base + 5 * Cfg::VEC_ELEMS + kk * N;
      const float vi = ld1(v_ + row);

      // sa over the pre-update row; u = S w + k v_i does not need sa.
      float sa_part[Q];
      float u[E];
#pragma unroll
      for (int m = 0; m < Q; ++m) {
        const int col = 4 * (m * G + g);
        const float4 a4 = lds4(a_ + col), w4 = lds4(w_ + col), k4 = lds4(k_ + col);
        float s = S[4 * m] * a4.x;
        s = fmaf(S[4 * m + 1], a4.y, s);
        s = fmaf(S[4 * m + 2], a4.z, s);
        s = fmaf(S[4 * m + 3], a4.w, s);
        sa_part[m] = s;
        u[4 * m] = fmaf(S[4 * m], w4.x, k4.x * vi);
        u[4 * m + 1] = fmaf(S[4 * m + 1], w4.y, k4.y * vi);
        u[4 * m + 2] = fmaf(S[4 * m + 2], w4.z, k4.z * vi);
        u[4 * m + 3] = fmaf(S[4 * m + 3], w4.w, k4.w * vi);
      }
      float sa = 0.f;
#pragma unroll
      for (int m = 0; m < Q; ++m) sa += sa_part[m];
      sa = group_allreduce<G>(sa);

      float y_part[Q];
#pragma unroll
      for (int m = 0; m < Q; ++m) {
        const int col = 4 * (m * G + g);
        const float4 b4 = lds4(b_ + col), r4 = lds4(r_ + col);
        S[4 * m] = fmaf(sa, b4.x, u[4 * m]);
        S[4 * m + 1] = fmaf(sa, b4.y, u[4 * m + 1]);
        S[4 * m + 2] = fmaf(sa, b4.z, u[4 * m + 2]);
        S[4 * m + 3] = fmaf(sa, b4.w, u[4 * m + 3]);
        float s = S[4 * m] * r4.x;
        s = fmaf(S[4 * m + 1], r4.y, s);
        s = fmaf(S[4 * m + 2], r4.z, s);
        s = fmaf(S[4 * m + 3], r4.w, s);
        y_part[m] = s;
      }
      float yy = 0.f;
#pragma unroll
      for (int m = 0; m < Q; ++m) yy += y_part[m];
      yy = group_allreduce<G>(yy);
      if (y_ptr) {
        if (g == 0) st1(y_ptr, yy);
        y_ptr += y_step;
      }
    }
    __syncthreads();  // every thread is done with this stage
    if (tid == 0 && c + Cfg::NSTAGE < nchunks) issue(c + Cfg::NSTAGE, st);
  }

  if (args.s_final) {
    float* dst = args.s_final + ((size_t)head * N + row) * N;
#pragma unroll
    for (int m = 0; m < Q; ++m)
      *reinterpret_cast<float4*>(dst + 4 * (m * G + g)) =
          make_float4(S[4 * m], S[4 * m + 1], S[4 * m + 2], S[4 * m + 3]);
  }
}

// ------------------------------------------------------------ launcher ---

template <typename TIn, int N, int G, int ROWS, int K>
static cudaError_t launch_fwd_impl(const FwdArgs& args, cudaStream_t stream) {
  using Cfg = FwdCfg<TIn, N, G, ROWS, K>;
  auto kern = wkv7_fwd_kernel<TIn, N, G, ROWS, K>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)((N / ROWS) * args.B * args.H);
  kern<<<grid, Cfg::THREADS, Cfg::SMEM_BYTES, stream>>>(args);
  return cudaGetLastError();
}

int fwd_steps_per_stage(int N, bool bf16) {
  (void)N;
  (void)bf16;
  return 16;
}

cudaError_t launch_fwd(const FwdArgs& args, bool bf16, int N, cudaStream_t stream) {
  if (bf16) {
    switch (N) {
      case 16: return launch_fwd_impl<__nv_bfloat16, 16, 4, 16, 16>(args, stream);
      case 32: return launch_fwd_impl<__nv_bfloat16, 32, 4, 16, 16>(args, stream);
      case 64: return launch_fwd_impl<__nv_bfloat16, 64, 4, 16, 16>(args, stream);
    }
  } else {
    switch (N) {
      case 16: return launch_fwd_impl<float, 16, 4, 16, 16>(args, stream);
      case 32: return launch_fwd_impl<float, 32, 4, 16, 16>(args, stream);
      case 64: return launch_fwd_impl<float, 64, 4, 16, 16>(args, stream);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace wkv7
