// WKV7 backward-through-time (reverse scan), sm_103a.
//
// Per (batch b, head h), with G = dL/dS carried from t = T-1 down to 0 and
// starting at zero ("rx_pretrain.c", rx_wkv7_backward, equations (1)-(3)):
//   (1) dr_j = sum_i S_t[i][j] dy_i ;  G += dy r^T
//   (2) dk_j = sum_i G_ij v_i ;  db_j = sum_i G_ij sa_i ;  dw_j = sum_i G_ij S_prev_ij
//       dv_i = sum_j G_ij k_j ;  dsa_i = sum_j G_ij b_j
//   (3) da_j = sum_i dsa_i S_prev_ij ;  G <- G diag(w) + dsa a^T
// and dS_init = G after step 0.
//
// Recompute instead of store: the forward saved S every C steps. For each
// chunk, from the last to the first, the kernel reloads the chunk's
// checkpoint, replays the forward over the chunk (at most KS steps at a time)
// keeping each pre-step state S_prev and each sa in shared memory, and then
// walks the chunk backwards. dr only needs S_t and dy, so it is produced
// during the replay; the reverse walk produces the other six outputs and the
// carry in one pass.
//
// Work decomposition. One CTA per head. Thread (rg, cg) holds an R x E tile
// of S (replay) and of G (reverse): rows rg*R .. rg*R+R-1 and the E/4 column
// quads q = m*G + cg. Row sums (sa, dsa, dv) are xor-shuffle sums over the
// G lanes of a row group; column sums (dr, dk, db, dw, da) are per-thread
// partials over R rows, reduced across the row groups through shared memory
// once per step. Inputs arrive through 4-D TMA tensor loads (KS steps of
// r, w, k, v, a, b, dy per load) completed on an mbarrier with a bounded wait.
#include "wkv7_common.cuh"
#include "wkv7_launch.h"

namespace wkv7 {

template <typename TIn, int N, int R, int E, int KS>
struct BwdCfg {
  static constexpr int G = N / E;  // lanes per row group
  static constexpr int P = N / R;  // row groups
  static constexpr int Q = E / 4;
  static constexpr int THREADS = G * P;
  static constexpr int NVEC = 7;  // r, w, k, v, a, b, dy
  static constexpr int VEC_ELEMS = KS * N;
  static constexpr int STAGE_BYTES = NVEC * VEC_ELEMS * Elem<TIn>::bytes;
  static constexpr int NSUM = 4;  // dk, db, dw, da (dr reuses slot 0 in the replay)
  static constexpr size_t SBUF_BYTES = (size_t)KS * N * N * 4;
  static constexpr size_t SAB_BYTES = (size_t)KS * N * 4;
  static constexpr size_t COL_BYTES = (size_t)2 * NSUM * P * N * 4;
  static constexpr size_t OFF_SAB = SBUF_BYTES;
  static constexpr size_t OFF_STAGE = OFF_SAB + SAB_BYTES;
  static constexpr size_t OFF_COL = (OFF_STAGE + STAGE_BYTES + 127) / 128 * 128;
  static constexpr size_t OFF_BAR = OFF_COL + COL_BYTES;
  static constexpr size_t SMEM_BYTES = OFF_BAR + 64;
  static_assert(E % 4 == 0 && 32 % G == 0 && N % R == 0, "bad backward tiling");
  static_assert(THREADS % 32 == 0, "backward CTA must be whole warps");
  static_assert(SMEM_BYTES <= 227 * 1024, "backward shared memory over budget");
};

template <int R, typename TIn>
__device__ __forceinline__ void load_rows(const TIn* p, float (&out)[R]) {
#pragma unroll
  for (int i = 0; i < R; ++i) out[i] = ld1(p + i);
}

template <typename TIn, int N, int R, int E, int KS>
__global__ void __launch_bounds__(BwdCfg<TIn, N, R, E, KS>::THREADS)
    wkv7_bwd_kernel(const __grid_constant__ BwdArgs args) {
  using Cfg = BwdCfg<TIn, N, R, E, KS>;
  constexpr int G = Cfg::G, P = Cfg::P, Q = Cfg::Q, VE = Cfg::VEC_ELEMS;
  extern __shared__ __align__(128) unsigned char smem[];
  float* sbuf = reinterpret_cast<float*>(smem);                    // [KS][N][N]
  float* sab = reinterpret_cast<float*>(smem + Cfg::OFF_SAB);      // [KS][N]
  TIn* stage = reinterpret_cast<TIn*>(smem + Cfg::OFF_STAGE);      // [7][KS][N]
  float* colbuf = reinterpret_cast<float*>(smem + Cfg::OFF_COL);   // [2][NSUM][P][N]
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);

  const int T = args.T, H = args.H, C = args.C;
  const int head = blockIdx.x;
  const int bi = head / H, hi = head % H;
  const int tid = threadIdx.x;
  const int cg = tid % G, rg = tid / G;
  const int row0 = rg * R;
  const size_t vstep = (size_t)H * N;
  const size_t vbase = ((size_t)bi * T * H + hi) * N;

  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
    for (int v = 0; v < Cfg::NVEC; ++v) prefetch_tensormap(&args.map[v]);
  }
  __syncthreads();
  uint32_t phase = 0;

  // Stage KS steps of all seven input vectors starting at step t_begin.
  // Returns false (uniformly over the CTA) if the copy did not complete.
  auto stage_load = [&](int t_begin) -> bool {
    __syncthreads();  // previous readers of the stage are done
    if (tid == 0) {
      mbar_arrive_expect_tx(bar, Cfg::STAGE_BYTES);
      for (int v = 0; v < Cfg::NVEC; ++v) tma_load_4d(stage + v * VE, &args.map[v], bar, 0, hi, t_begin, bi);
    }
    bool ok = mbar_wait_bounded(args.status, bar, phase);
    if (!ok) mbar_wait_bounded(args.status, bar, phase);  // drain the copy in flight
    phase ^= 1u;
    return __syncthreads_and(ok) != 0;
  };
  auto col = [&](int m) { return 4 * (m * G + cg); };

  float dS[R][E];
#pragma unroll
  for (int i = 0; i < R; ++i)
#pragma unroll
    for (int e = 0; e < E; ++e) dS[i][e] = 0.f;

  for (int c = args.nck - 1; c >= 0; --c) {
    const int t0 = c * C, t1 = min(T, t0 + C);
    for (int s1 = t1; s1 > t0;) {
      const int s0 = max(t0, s1 - KS);
      const int L = s1 - s0;

      // ---- state before step t0, from the checkpoint
      float S[R][E];
      {
        const float* ck = args.ckpt + (((size_t)head * args.nck + c) * N + row0) * N;
#pragma unroll
        for (int i = 0; i < R; ++i)
#pragma unroll
          for (int m = 0; m < Q; ++m) {
            const float4 s4 = *reinterpret_cast<const float4*>(ck + (size_t)i * N + col(m));
            S[i][4 * m] = s4.x; S[i][4 * m + 1] = s4.y; S[i][4 * m + 2] = s4.z; S[i][4 * m + 3] = s4.w;
          }
      }

      // One forward step on the register tile, optionally recording sa.
      auto fwd_step = [&](int l, bool record) {
        const TIn* w_ = stage + 1 * VE + l * N;
        const TIn* k_ = stage + 2 * VE + l * N;
        const TIn* v_ = stage + 3 * VE + l * N;
        const TIn* a_ = stage + 4 * VE + l * N;
        const TIn* b_ = stage + 5 * VE + l * N;
        float vr[R];
        load_rows<R>(v_ + row0, vr);
        float sa[R];
#pragma unroll
        for (int i = 0; i < R; ++i) sa[i] = 0.f;
#pragma unroll
        for (int m = 0; m < Q; ++m) {
          const float4 a4 = lds4(a_ + col(m));
#pragma unroll
          for (int i = 0; i < R; ++i) {
            float s = S[i][4 * m] * a4.x;
            s = fmaf(S[i][4 * m + 1], a4.y, s);
            s = fmaf(S[i][4 * m + 2], a4.z, s);
            s = fmaf(S[i][4 * m + 3], a4.w, s);
            sa[i] += s;
          }
        }
#pragma unroll
        for (int i = 0; i < R; ++i) sa[i] = group_allreduce<G>(sa[i]);
        if (record && cg == 0) {
#pragma unroll
          for (int i = 0; i < R; ++i) sab[l * N + row0 + i] = sa[i];
        }
#pragma unroll
        for (int m = 0; m < Q; ++m) {
          const float4 w4 = lds4(w_ + col(m)), k4 = lds4(k_ + col(m)), b4 = lds4(b_ + col(m));
#pragma unroll
          for (int i = 0; i < R; ++i) {
            S[i][4 * m] = fmaf(sa[i], b4.x, fmaf(S[i][4 * m], w4.x, k4.x * vr[i]));
            S[i][4 * m + 1] = fmaf(sa[i], b4.y, fmaf(S[i][4 * m + 1], w4.y, k4.y * vr[i]));
            S[i][4 * m + 2] = fmaf(sa[i], b4.z, fmaf(S[i][4 * m + 2], w4.z, k4.z * vr[i]));
            S[i][4 * m + 3] = fmaf(sa[i], b4.w, fmaf(S[i][4 * m + 3], w4.w, k4.w * vr[i]));
          }
        }
      };

      // ---- advance from t0 to s0 without recording (only when C > KS)
      for (int a0 = t0; a0 < s0; a0 += KS) {
        if (!stage_load(a0)) return;
        const int na = min(KS, s0 - a0);
        for (int l = 0; l < na; ++l) fwd_step(l, false);
      }

      // ---- replay [s0, s1): record S_prev and sa, emit dr
      if (!stage_load(s0)) return;
      for (int l = 0; l < L; ++l) {
        float* sp = sbuf + (size_t)l * N * N + (size_t)row0 * N;
#pragma unroll
        for (int i = 0; i < R; ++i)
#pragma unroll
          for (int m = 0; m < Q; ++m)
            *reinterpret_cast<float4*>(sp + i * N + col(m)) =
                make_float4(S[i][4 * m], S[i][4 * m + 1], S[i][4 * m + 2], S[i][4 * m + 3]);
        fwd_step(l, true);
        float dyr[R];
        load_rows<R>(stage + 6 * VE + l * N + row0, dyr);
        float* cb = colbuf + (size_t)(l & 1) * Cfg::NSUM * P * N + (size_t)rg * N;
#pragma unroll
        for (int m = 0; m < Q; ++m) {
          float4 p4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int i = 0; i < R; ++i) {
            p4.x = fmaf(S[i][4 * m], dyr[i], p4.x);
            p4.y = fmaf(S[i][4 * m + 1], dyr[i], p4.y);
            p4.z = fmaf(S[i][4 * m + 2], dyr[i], p4.z);
            p4.w = fmaf(S[i][4 * m + 3], dyr[i], p4.w);
          }
          *reinterpret_cast<float4*>(cb + col(m)) = p4;
        }
        __syncthreads();
        const float* cr = colbuf + (size_t)(l & 1) * Cfg::NSUM * P * N;
        for (int o = tid; o < N; o += Cfg::THREADS) {
          float s = 0.f;
#pragma unroll
          for (int p = 0; p < P; ++p) s += cr[p * N + o];
          args.dr[vbase + (size_t)(s0 + l) * vstep + o] = s;
        }
      }
      __syncthreads();  // S_prev and sa of the whole sub-chunk are in shared memory

      // ---- reverse walk over [s0, s1)
      for (int l = L - 1; l >= 0; --l) {
        const size_t t = (size_t)(s0 + l);
        const TIn* r_ = stage + 0 * VE + l * N;
        const TIn* w_ = stage + 1 * VE + l * N;
        const TIn* k_ = stage + 2 * VE + l * N;
        const TIn* a_ = stage + 4 * VE + l * N;
        const TIn* b_ = stage + 5 * VE + l * N;
        float dyr[R], vr[R], sar[R];
        load_rows<R>(stage + 6 * VE + l * N + row0, dyr);
        load_rows<R>(stage + 3 * VE + l * N + row0, vr);
#pragma unroll
        for (int i = 0; i < R; ++i) sar[i] = sab[l * N + row0 + i];
        const float* sp = sbuf + (size_t)l * N * N + (size_t)row0 * N;

        float pk[E], pb[E], pw[E], dvp[R], dsp[R];
#pragma unroll
        for (int i = 0; i < R; ++i) { dvp[i] = 0.f; dsp[i] = 0.f; }
        float Sp[R][E];
#pragma unroll
        for (int m = 0; m < Q; ++m) {
          const float4 r4 = lds4(r_ + col(m)), k4 = lds4(k_ + col(m)), b4 = lds4(b_ + col(m));
          const float rc[4] = {r4.x, r4.y, r4.z, r4.w};
          const float kc[4] = {k4.x, k4.y, k4.z, k4.w};
          const float bc[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
          for (int i = 0; i < R; ++i) {
            const float4 s4 = *reinterpret_cast<const float4*>(sp + i * N + col(m));
            Sp[i][4 * m] = s4.x; Sp[i][4 * m + 1] = s4.y; Sp[i][4 * m + 2] = s4.z; Sp[i][4 * m + 3] = s4.w;
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j = 4 * m + e;
            float ak = 0.f, ab = 0.f, aw = 0.f;
#pragma unroll
            for (int i = 0; i < R; ++i) {
              dS[i][j] = fmaf(dyr[i], rc[e], dS[i][j]);
              ak = fmaf(dS[i][j], vr[i], ak);
              ab = fmaf(dS[i][j], sar[i], ab);
              aw = fmaf(dS[i][j], Sp[i][j], aw);
              dvp[i] = fmaf(dS[i][j], kc[e], dvp[i]);
              dsp[i] = fmaf(dS[i][j], bc[e], dsp[i]);
            }
            pk[j] = ak; pb[j] = ab; pw[j] = aw;
          }
        }
        float dsa[R];
#pragma unroll
        for (int i = 0; i < R; ++i) {
          dsa[i] = group_allreduce<G>(dsp[i]);
          dvp[i] = group_allreduce<G>(dvp[i]);
        }
        if (cg == 0) {
#pragma unroll
          for (int i = 0; i < R; ++i) args.dv[vbase + t * vstep + row0 + i] = dvp[i];
        }
        float pa[E];
#pragma unroll
        for (int m = 0; m < Q; ++m) {
          const float4 w4 = lds4(w_ + col(m)), a4 = lds4(a_ + col(m));
          const float wc[4] = {w4.x, w4.y, w4.z, w4.w};
          const float ac[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j = 4 * m + e;
            float s = 0.f;
#pragma unroll
            for (int i = 0; i < R; ++i) {
              s = fmaf(dsa[i], Sp[i][j], s);
              dS[i][j] = fmaf(dS[i][j], wc[e], dsa[i] * ac[e]);
            }
            pa[j] = s;
          }
        }
        float* cb = colbuf + (size_t)(l & 1) * Cfg::NSUM * P * N + (size_t)rg * N;
#pragma unroll
        for (int m = 0; m < Q; ++m) {
          const int j = 4 * m;
          *reinterpret_cast<float4*>(cb + 0 * P * N + col(m)) = make_float4(pk[j], pk[j + 1], pk[j + 2], pk[j + 3]);
          *reinterpret_cast<float4*>(cb + 1 * P * N + col(m)) = make_float4(pb[j], pb[j + 1], pb[j + 2], pb[j + 3]);
          *reinterpret_cast<float4*>(cb + 2 * P * N + col(m)) = make_float4(pw[j], pw[j + 1], pw[j + 2], pw[j + 3]);
          *reinterpret_cast<float4*>(cb + 3 * P * N + col(m)) = make_float4(pa[j], pa[j + 1], pa[j + 2], pa[j + 3]);
        }
        __syncthreads();
        const float* cr = colbuf + (size_t)(l & 1) * Cfg::NSUM * P * N;
        for (int o = tid; o < Cfg::NSUM * N; o += Cfg::THREADS) {
          const int which = o / N, j = o % N;
          float s = 0.f;
#pragma unroll
          for (int p = 0; p < P; ++p) s += cr[(which * P + p) * N + j];
          float* out = which == 0 ? args.dk : which == 1 ? args.db : which == 2 ? args.dw : args.da;
          out[vbase + t * vstep + j] = s;
        }
      }
      s1 = s0;
    }
  }

  if (args.dS_init) {
    float* dst = args.dS_init + ((size_t)head * N + row0) * N;
#pragma unroll
    for (int i = 0; i < R; ++i)
#pragma unroll
      for (int m = 0; m < Q; ++m)
        *reinterpret_cast<float4*>(dst + (size_t)i * N + col(m)) =
            make_float4(dS[i][4 * m], dS[i][4 * m + 1], dS[i][4 * m + 2], dS[i][4 * m + 3]);
  }
}

// ------------------------------------------------------------ launcher ---

template <typename TIn, int N, int R, int E, int KS>
static cudaError_t launch_bwd_impl(const BwdArgs& args, cudaStream_t stream) {
  using Cfg = BwdCfg<TIn, N, R, E, KS>;
  auto kern = wkv7_bwd_kernel<TIn, N, R, E, KS>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)(args.B * args.H), Cfg::THREADS, Cfg::SMEM_BYTES, stream>>>(args);
  return cudaGetLastError();
}

// Shared-memory capacity in recorded steps per sub-chunk.
int bwd_steps_per_stage(int N, bool bf16) {
  (void)bf16;
  return N == 64 ? 8 : 16;
}

cudaError_t launch_bwd(const BwdArgs& args, bool bf16, int N, cudaStream_t stream) {
  if (bf16) {
    switch (N) {
      case 16: return launch_bwd_impl<__nv_bfloat16, 16, 2, 4, 16>(args, stream);
      case 32: return launch_bwd_impl<__nv_bfloat16, 32, 2, 8, 16>(args, stream);
      case 64: return launch_bwd_impl<__nv_bfloat16, 64, 4, 8, 8>(args, stream);
    }
  } else {
    switch (N) {
      case 16: return launch_bwd_impl<float, 16, 2, 4, 16>(args, stream);
      case 32: return launch_bwd_impl<float, 32, 2, 8, 16>(args, stream);
      case 64: return launch_bwd_impl<float, 64, 4, 8, 8>(args, stream);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace wkv7
