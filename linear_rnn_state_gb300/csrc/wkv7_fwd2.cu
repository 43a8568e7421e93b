// WKV7 forward scan (sm_103a): column-scaled fast path with a direct-form
// path for chunks whose decays leave the safe range.
//
// Same result as "rx_pretrain.c", rx_wkv7_forward_seq:
//   sa = S a ;  S <- S diag(w) + v k^T + sa b^T ;  y = S r.
// Fast path (wkv7_scaled.cuh): per step
//   u~ = S~ + v k~^T ;  X = u~ a^(t+1) ;  S~ = u~ + sa b~^T ;  y = S~ r^ ;
//   sa(t+1) = X + sa(t) beta(t)
// four packed-fp32 multiply-adds per state element. sa is recomputed directly
// at every chunk start, so the look-ahead never spans chunks.
//
// One CTA per (b, h). Thread (rg, cg) owns rows rg*R .. rg*R+R-1 and the E/4
// column quads q = m*G + cg of the state in registers, as float2 pairs for
// the packed FMA. Row sums are xor-shuffle sums over the G lanes of a row
// group. Per chunk of K steps a TMA tensor load brings r, w, k, v, a, b into
// a two-stage ring; a prologue turns them into fp32 per-step vectors (scaled,
// or plain for a direct-form chunk), then the K steps run from shared memory.
#include "wkv7_launch.h"
#include "wkv7_scaled.cuh"

namespace wkv7 {

constexpr size_t align128(size_t x) { return (x + 127) / 128 * 128; }

template <typename TIn, int N, int R, int E, int K>
struct Fwd2Cfg {
  static constexpr int G = N / E;  // lanes per row group
  static constexpr int P = N / R;  // row groups
  static constexpr int THREADS = G * P;
  static constexpr int NWARPS = THREADS / 32;
  static constexpr int Q = E / 4;   // column quads per thread
  static constexpr int NP = E / 2;  // column pairs per thread
  static constexpr int NVEC = 6;    // r, w, k, v, a, b
  static constexpr int RAW_VEC = K * N;
  static constexpr int RAW_STAGE = NVEC * RAW_VEC;
  static constexpr int RAW_STAGE_BYTES = RAW_STAGE * Elem<TIn>::bytes;
  static constexpr int NSTAGE = 2;
  static constexpr int DV = K * N;  // floats per derived vector
  static constexpr size_t OFF_DER = align128((size_t)NSTAGE * RAW_STAGE_BYTES);
  static constexpr size_t DER_BYTES = (size_t)6 * DV * 4 + (size_t)K * 4;
  static constexpr size_t OFF_BAR = align128(OFF_DER + DER_BYTES);
  static constexpr size_t SMEM_BYTES = OFF_BAR + 64;
  static_assert(E % 4 == 0 && 32 % G == 0 && N % R == 0 && (R == 2 || R == 4), "bad tiling");
  static_assert(THREADS % 32 == 0, "whole warps");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory over budget");
};

enum { V_R = 0, V_W = 1, V_K = 2, V_V = 3, V_A = 4, V_B = 5 };

template <int R>
__device__ __forceinline__ void ld_rows(const float* p, float (&out)[R]) {
  if constexpr (R == 4) {
    const float4 v = ld_f4(p);
    out[0] = v.x; out[1] = v.y; out[2] = v.z; out[3] = v.w;
  } else {
    const float2 v = *reinterpret_cast<const float2*>(p);
    out[0] = v.x; out[1] = v.y;
  }
}

template <typename TIn, int N, int R, int E, int K>
__global__ void __launch_bounds__(Fwd2Cfg<TIn, N, R, E, K>::THREADS)
    wkv7_fwd2_kernel(const __grid_constant__ FwdArgs args) {
  using Cfg = Fwd2Cfg<TIn, N, R, E, K>;
  constexpr int G = Cfg::G, Q = Cfg::Q, NP = Cfg::NP, DV = Cfg::DV, RV = Cfg::RAW_VEC;
  extern __shared__ __align__(128) unsigned char smem[];
  TIn* raw = reinterpret_cast<TIn*>(smem);
  // Per-step fp32 vectors [K][N]. Scaled chunk: k~, b~, a^(t+1), r^, c, v.
  // Direct chunk: k, b, a(t), r, w, v.
  float* d_k = reinterpret_cast<float*>(smem + Cfg::OFF_DER);
  float* d_b = d_k + DV;
  float* d_a = d_b + DV;
  float* d_r = d_a + DV;
  float* d_c = d_r + DV;
  float* d_v = d_c + DV;
  float* beta = d_v + DV;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);

  const int T = args.T, H = args.H;
  const int head = blockIdx.x;
  const int bi = head / H, hi = head % H;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cg = tid % G, rg = tid / G;
  const int row0 = rg * R;
  auto colq = [&](int m) { return 4 * (m * G + cg); };

  // ---- state tile: S[i][2m + h] holds columns colq(m) + 2h, +1 of row row0 + i
  float2 S[R][NP];
#pragma unroll
  for (int i = 0; i < R; ++i)
#pragma unroll
    for (int m = 0; m < Q; ++m) {
      float4 s4 = make_float4(0.f, 0.f, 0.f, 0.f);
      if (args.s_init) s4 = ld_f4(args.s_init + ((size_t)head * N + row0 + i) * N + colq(m));
      S[i][2 * m] = make_float2(s4.x, s4.y);
      S[i][2 * m + 1] = make_float2(s4.z, s4.w);
    }

  const int nchunks = (T + K - 1) / K;
  if (tid == 0) {
    for (int s = 0; s < Cfg::NSTAGE; ++s) mbar_init(&full[s], 1);
    fence_mbar_init();
    for (int v = 0; v < Cfg::NVEC; ++v) prefetch_tensormap(&args.map[v]);
  }
  __syncthreads();
  auto issue = [&](int chunk, int st) {
    mbar_arrive_expect_tx(&full[st], Cfg::RAW_STAGE_BYTES);
    TIn* dst = raw + st * Cfg::RAW_STAGE;
    for (int v = 0; v < Cfg::NVEC; ++v) tma_load_4d(dst + v * RV, &args.map[v], &full[st], 0, hi, chunk * K, bi);
  };
  if (tid == 0)
    for (int s = 0; s < Cfg::NSTAGE && s < nchunks; ++s) issue(s, s);

  TIn* y = static_cast<TIn*>(args.y);
  const size_t vstep = (size_t)H * N;
  const size_t vbase = ((size_t)bi * T * H + hi) * N;
  float* ck_base = args.ckpt ? args.ckpt + ((size_t)head * args.nck * N + row0) * N : nullptr;
  int ck_left = 0;  // steps until the next checkpoint

  for (int c = 0; c < nchunks; ++c) {
    const int st = c % Cfg::NSTAGE;
    const int t0 = c * K;
    {
      const bool ok = mbar_wait_bounded(args.status, &full[st], (c / Cfg::NSTAGE) & 1);
      if (!ok) mbar_wait_bounded(args.status, &full[st], (c / Cfg::NSTAGE) & 1);  // drain
      // (also: every thread has finished the previous chunk's steps)
      if (!__syncthreads_and(ok)) return;
    }
    const TIn* rs = raw + st * Cfg::RAW_STAGE;

    // ---- is every decay of this chunk in the scaled form's safe range?
    bool unsafe = false;
    for (int o = tid; o < K * N; o += Cfg::THREADS)
      if (t0 + o / N < T && !decay_is_safe(raw1(rs + V_W * RV + o))) unsafe = true;
    const bool direct = __syncthreads_or(unsafe) != 0;

    // ---- prologue: per-step fp32 vectors for this chunk
    for (int j = tid; j < N; j += Cfg::THREADS) {
      float cv = 1.f;
      for (int l = 0; l < K; ++l) {
        const int o = l * N + j;
        const bool valid = t0 + l < T;
        const float w = valid ? raw1(rs + V_W * RV + o) : 1.f;
        const float k = valid ? raw1(rs + V_K * RV + o) : 0.f;
        const float b = valid ? raw1(rs + V_B * RV + o) : 0.f;
        const float r = valid ? raw1(rs + V_R * RV + o) : 0.f;
        d_v[o] = valid ? raw1(rs + V_V * RV + o) : 0.f;
        if (direct) {
          d_k[o] = k; d_b[o] = b; d_r[o] = r; d_c[o] = w;
          d_a[o] = valid ? raw1(rs + V_A * RV + o) : 0.f;
        } else {
          cv = cv * w;
          const float ic = __frcp_rn(cv);
          d_k[o] = k * ic; d_b[o] = b * ic; d_r[o] = r * cv; d_c[o] = cv;
          d_a[o] = (l + 1 < K && t0 + l + 1 < T) ? raw1(rs + V_A * RV + o + N) * cv : 0.f;
        }
      }
    }
    if (!direct) {  // beta(l) = b(l) . a(l+1) inside the chunk
      for (int l = warp; l < K; l += Cfg::NWARPS) {
        float s = 0.f;
        if (l + 1 < K && t0 + l + 1 < T)
          for (int j = lane; j < N; j += 32)
            s = fmaf(raw1(rs + V_B * RV + l * N + j), raw1(rs + V_A * RV + (l + 1) * N + j), s);
        s = group_allreduce<32>(s);
        if (lane == 0) beta[l] = s;
      }
    }
    // ---- sa at the chunk's first step, directly: S(t0-1) a(t0)
    float sa[R];
#pragma unroll
    for (int i = 0; i < R; ++i) sa[i] = 0.f;
#pragma unroll
    for (int m = 0; m < Q; ++m) {
      float a4[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) a4[e] = raw1(rs + V_A * RV + colq(m) + e);
#pragma unroll
      for (int i = 0; i < R; ++i) {
        sa[i] = fmaf(S[i][2 * m].x, a4[0], sa[i]);
        sa[i] = fmaf(S[i][2 * m].y, a4[1], sa[i]);
        sa[i] = fmaf(S[i][2 * m + 1].x, a4[2], sa[i]);
        sa[i] = fmaf(S[i][2 * m + 1].y, a4[3], sa[i]);
      }
    }
#pragma unroll
    for (int i = 0; i < R; ++i) sa[i] = group_allreduce<G>(sa[i]);
    __syncthreads();  // the per-step vectors are complete; the raw stage is free
    if (tid == 0 && c + Cfg::NSTAGE < nchunks) issue(c + Cfg::NSTAGE, st);

    if (!direct) {
      // ---- K scaled steps
#pragma unroll
      for (int l = 0; l < K; ++l) {
        const int t = t0 + l;
        if (ck_base && t < T) {
          if (ck_left == 0) {
            float* dst = ck_base + (size_t)(t / args.C) * N * N;
#pragma unroll
            for (int m = 0; m < Q; ++m) {
              float4 c4 = make_float4(1.f, 1.f, 1.f, 1.f);
              if (l > 0) c4 = ld_f4(d_c + (l - 1) * N + colq(m));
#pragma unroll
              for (int i = 0; i < R; ++i)
                *reinterpret_cast<float4*>(dst + (size_t)i * N + colq(m)) =
                    make_float4(S[i][2 * m].x * c4.x, S[i][2 * m].y * c4.y, S[i][2 * m + 1].x * c4.z,
                                S[i][2 * m + 1].y * c4.w);
            }
            ck_left = args.C;
          }
          --ck_left;
        }
        float vr[R];
        ld_rows<R>(d_v + l * N + row0, vr);
        float2 kv[NP], av[NP], bv[NP], rv[NP];
#pragma unroll
        for (int m = 0; m < Q; ++m) {
          const float4 k4 = ld_f4(d_k + l * N + colq(m));
          const float4 a4 = ld_f4(d_a + l * N + colq(m));
          const float4 b4 = ld_f4(d_b + l * N + colq(m));
          const float4 r4 = ld_f4(d_r + l * N + colq(m));
          kv[2 * m] = make_float2(k4.x, k4.y); kv[2 * m + 1] = make_float2(k4.z, k4.w);
          av[2 * m] = make_float2(a4.x, a4.y); av[2 * m + 1] = make_float2(a4.z, a4.w);
          bv[2 * m] = make_float2(b4.x, b4.y); bv[2 * m + 1] = make_float2(b4.z, b4.w);
          rv[2 * m] = make_float2(r4.x, r4.y); rv[2 * m + 1] = make_float2(r4.z, r4.w);
        }
        float X[R], Y[R];
#pragma unroll
        for (int i = 0; i < R; ++i) {
          const float2 vi = f2(vr[i]), si = f2(sa[i]);
          float2 xa = make_float2(0.f, 0.f), ya = make_float2(0.f, 0.f);
#pragma unroll
          for (int p = 0; p < NP; ++p) {
            const float2 u = ffma2(vi, kv[p], S[i][p]);
            xa = ffma2(u, av[p], xa);
            S[i][p] = ffma2(si, bv[p], u);
            ya = ffma2(S[i][p], rv[p], ya);
          }
          X[i] = xa.x + xa.y;
          Y[i] = ya.x + ya.y;
        }
        const float bl = beta[l];
#pragma unroll
        for (int i = 0; i < R; ++i) {
          X[i] = group_allreduce<G>(X[i]);
          Y[i] = group_allreduce<G>(Y[i]);
          sa[i] = fmaf(sa[i], bl, X[i]);
        }
        if (y && cg == 0 && t < T) {
#pragma unroll
          for (int i = 0; i < R; ++i) st1(y + vbase + (size_t)t * vstep + row0 + i, Y[i]);
        }
      }
      // ---- renormalise: S = S~ diag(c(last step))
#pragma unroll
      for (int m = 0; m < Q; ++m) {
        const float4 c4 = ld_f4(d_c + (K - 1) * N + colq(m));
#pragma unroll
        for (int i = 0; i < R; ++i) {
          S[i][2 * m] = fmul2(S[i][2 * m], make_float2(c4.x, c4.y));
          S[i][2 * m + 1] = fmul2(S[i][2 * m + 1], make_float2(c4.z, c4.w));
        }
      }
    } else {
      // ---- K direct-form steps (any decay): sa = S a; S = S w + v k + sa b; y = S r
      for (int l = 0; l < K; ++l) {
        const int t = t0 + l;
        if (ck_base && t < T) {
          if (ck_left == 0) {
            float* dst = ck_base + (size_t)(t / args.C) * N * N;
#pragma unroll
            for (int m = 0; m < Q; ++m)
#pragma unroll
              for (int i = 0; i < R; ++i)
                *reinterpret_cast<float4*>(dst + (size_t)i * N + colq(m)) =
                    make_float4(S[i][2 * m].x, S[i][2 * m].y, S[i][2 * m + 1].x, S[i][2 * m + 1].y);
            ck_left = args.C;
          }
          --ck_left;
        }
        float vr[R];
        ld_rows<R>(d_v + l * N + row0, vr);
        if (l > 0) {
#pragma unroll
          for (int i = 0; i < R; ++i) sa[i] = 0.f;
#pragma unroll
          for (int m = 0; m < Q; ++m) {
            const float4 a4 = ld_f4(d_a + l * N + colq(m));
#pragma unroll
            for (int i = 0; i < R; ++i) {
              float2 p = fmul2(S[i][2 * m], make_float2(a4.x, a4.y));
              p = ffma2(S[i][2 * m + 1], make_float2(a4.z, a4.w), p);
              sa[i] += p.x + p.y;
            }
          }
#pragma unroll
          for (int i = 0; i < R; ++i) sa[i] = group_allreduce<G>(sa[i]);
        }
        float Y[R];
#pragma unroll
        for (int i = 0; i < R; ++i) Y[i] = 0.f;
#pragma unroll
        for (int m = 0; m < Q; ++m) {
          const float4 w4 = ld_f4(d_c + l * N + colq(m));
          const float4 k4 = ld_f4(d_k + l * N + colq(m));
          const float4 b4 = ld_f4(d_b + l * N + colq(m));
          const float4 r4 = ld_f4(d_r + l * N + colq(m));
#pragma unroll
          for (int i = 0; i < R; ++i) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const float2 w2 = h ? make_float2(w4.z, w4.w) : make_float2(w4.x, w4.y);
              const float2 k2 = h ? make_float2(k4.z, k4.w) : make_float2(k4.x, k4.y);
              const float2 b2 = h ? make_float2(b4.z, b4.w) : make_float2(b4.x, b4.y);
              const float2 r2 = h ? make_float2(r4.z, r4.w) : make_float2(r4.x, r4.y);
              float2& s2 = S[i][2 * m + h];
              s2 = ffma2(f2(sa[i]), b2, ffma2(s2, w2, fmul2(k2, f2(vr[i]))));
              const float2 yr = fmul2(s2, r2);
              Y[i] += yr.x + yr.y;
            }
          }
        }
#pragma unroll
        for (int i = 0; i < R; ++i) Y[i] = group_allreduce<G>(Y[i]);
        if (y && cg == 0 && t < T) {
#pragma unroll
          for (int i = 0; i < R; ++i) st1(y + vbase + (size_t)t * vstep + row0 + i, Y[i]);
        }
      }
    }
  }

  if (args.s_final) {
#pragma unroll
    for (int i = 0; i < R; ++i)
#pragma unroll
      for (int m = 0; m < Q; ++m)
        *reinterpret_cast<float4*>(args.s_final + ((size_t)head * N + row0 + i) * N + colq(m)) =
            make_float4(S[i][2 * m].x, S[i][2 * m].y, S[i][2 * m + 1].x, S[i][2 * m + 1].y);
  }
}

// ------------------------------------------------------------ launcher ---

template <typename TIn, int N, int R, int E, int K>
static cudaError_t launch_fwd2_impl(const FwdArgs& args, cudaStream_t stream) {
  using Cfg = Fwd2Cfg<TIn, N, R, E, K>;
  auto kern = wkv7_fwd2_kernel<TIn, N, R, E, K>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)(args.B * args.H), Cfg::THREADS, Cfg::SMEM_BYTES, stream>>>(args);
  return cudaGetLastError();
}

int fwd2_box_steps(int N, bool bf16) {
  (void)N;
  (void)bf16;
  return 16;
}

cudaError_t launch_fwd2(const FwdArgs& args, bool bf16, int N, cudaStream_t stream) {
  if (bf16) {
    switch (N) {
      case 16: return launch_fwd2_impl<__nv_bfloat16, 16, 2, 4, 16>(args, stream);
      case 32: return launch_fwd2_impl<__nv_bfloat16, 32, 4, 8, 16>(args, stream);
      case 64: return launch_fwd2_impl<__nv_bfloat16, 64, 4, 8, 16>(args, stream);
    }
  } else {
    switch (N) {
      case 16: return launch_fwd2_impl<float, 16, 2, 4, 16>(args, stream);
      case 32: return launch_fwd2_impl<float, 32, 4, 8, 16>(args, stream);
      case 64: return launch_fwd2_impl<float, 64, 4, 8, 16>(args, stream);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace wkv7
