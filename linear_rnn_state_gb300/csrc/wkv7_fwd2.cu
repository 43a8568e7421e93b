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
  static constexpr size_t DER_BYTES = (size_t)6 * DV * 4 + (size_t)K * 4;  // + beta
  static constexpr size_t OFF_BAR = align128(OFF_DER + DER_BYTES);
  static constexpr size_t SMEM_BYTES = OFF_BAR + 64;
  static_assert(E % 4 == 0 && 32 % G == 0 && N % R == 0 && (R == 2 || R % 4 == 0) && R <= G, "bad tiling");
  static_assert(THREADS % 32 == 0, "whole warps");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory over budget");
};

enum { V_R = 0, V_W = 1, V_K = 2, V_V = 3, V_A = 4, V_B = 5 };

template <int R>
__device__ __forceinline__ void ld_rows(const float* p, float (&out)[R]) {
  if constexpr (R % 4 == 0) {
#pragma unroll
    for (int q = 0; q < R / 4; ++q) {
      const float4 v = ld_f4(p + 4 * q);
      out[4 * q] = v.x; out[4 * q + 1] = v.y; out[4 * q + 2] = v.z; out[4 * q + 3] = v.w;
    }
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
      const float* src = args.s_init + ((size_t)head * N + row0 + i) * N + colq(m);
      if (args.s_init && in_extent(args.status, args.ext.s_init, reinterpret_cast<const float4*>(src))) s4 = ld_f4(src);
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
#ifdef WKV7_DEBUG
    // The timeout test's hook: no load for the last chunk. Every earlier
    // chunk has been waited for by then, so nothing is in flight when that
    // wait gives up and the CTA leaves.
    if (args.debug_skip_last_load && chunk == nchunks - 1) return;
#endif
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

  // Prologue mapping: thread = (column quad pq, step group pg); each thread
  // forms the scaled vectors of 4 columns for SG consecutive steps.
  constexpr int NQ = N / 4;
  constexpr int SG = K * NQ / Cfg::THREADS;
  static_assert(SG >= 1 && K % SG == 0 && NQ <= 32 && Cfg::THREADS % NQ == 0, "prologue mapping");
  const int pq = tid % NQ, pg = tid / NQ;

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

    // ---- prologue, scaled form: c(l) = w(0)...w(l) of this chunk; k~ = k/c,
    // b~ = b/c, a^(l+1) = c(l) a(l+1), r^ = c r; beta(l) = b(l) . a(l+1).
    // Also checks the decays.
    bool unsafe = false;
    {
      const int col = 4 * pq;
      float4 cp = make_float4(1.f, 1.f, 1.f, 1.f);  // running product before step l
#pragma unroll
      for (int l = 0; l < K - SG; ++l) {
        if (l < pg * SG && t0 + l < T) {
          const float4 w4 = lds4(rs + V_W * RV + l * N + col);
          cp = make_float4(cp.x * w4.x, cp.y * w4.y, cp.z * w4.z, cp.w * w4.w);
        }
      }
#pragma unroll
      for (int g = 0; g < SG; ++g) {
        const int l = pg * SG + g;
        const int o = l * N + col;
        const bool valid = t0 + l < T;
        const bool next = l + 1 < K && t0 + l + 1 < T;
        const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 w4 = valid ? lds4(rs + V_W * RV + o) : make_float4(1.f, 1.f, 1.f, 1.f);
        const float4 k4 = valid ? lds4(rs + V_K * RV + o) : z;
        const float4 b4 = valid ? lds4(rs + V_B * RV + o) : z;
        const float4 r4 = valid ? lds4(rs + V_R * RV + o) : z;
        const float4 v4 = valid ? lds4(rs + V_V * RV + o) : z;
        const float4 a4 = next ? lds4(rs + V_A * RV + o + N) : z;
        if (!decay_is_safe(w4.x) || !decay_is_safe(w4.y) || !decay_is_safe(w4.z) || !decay_is_safe(w4.w))
          unsafe = true;
        const float4 c4 = make_float4(cp.x * w4.x, cp.y * w4.y, cp.z * w4.z, cp.w * w4.w);
        const float4 i4 = make_float4(rcp_approx(c4.x), rcp_approx(c4.y), rcp_approx(c4.z), rcp_approx(c4.w));
        *reinterpret_cast<float4*>(d_k + o) = make_float4(k4.x * i4.x, k4.y * i4.y, k4.z * i4.z, k4.w * i4.w);
        *reinterpret_cast<float4*>(d_b + o) = make_float4(b4.x * i4.x, b4.y * i4.y, b4.z * i4.z, b4.w * i4.w);
        *reinterpret_cast<float4*>(d_r + o) = make_float4(r4.x * c4.x, r4.y * c4.y, r4.z * c4.z, r4.w * c4.w);
        *reinterpret_cast<float4*>(d_a + o) = make_float4(a4.x * c4.x, a4.y * c4.y, a4.z * c4.z, a4.w * c4.w);
        *reinterpret_cast<float4*>(d_c + o) = c4;
        *reinterpret_cast<float4*>(d_v + o) = v4;
        float pb = b4.x * a4.x + b4.y * a4.y + b4.z * a4.z + b4.w * a4.w;
#pragma unroll
        for (int mask = 1; mask < NQ; mask <<= 1) pb += __shfl_xor_sync(0xffffffffu, pb, mask);
        if (pq == 0) beta[l] = pb;
        cp = c4;
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
        const float2 p = ffma2(S[i][2 * m + 1], make_float2(a4[2], a4[3]), fmul2(S[i][2 * m], make_float2(a4[0], a4[1])));
        sa[i] += hsum(p);
      }
    }
#pragma unroll
    for (int i = 0; i < R; ++i) sa[i] = group_allreduce<G>(sa[i]);
    const bool direct = __syncthreads_or(unsafe) != 0;
    if (direct) {
      // ---- rare: some decay outside the safe range; plain vectors instead
      for (int o = tid; o < K * N; o += Cfg::THREADS) {
        const bool valid = t0 + o / N < T;
        d_k[o] = valid ? raw1(rs + V_K * RV + o) : 0.f;
        d_b[o] = valid ? raw1(rs + V_B * RV + o) : 0.f;
        d_r[o] = valid ? raw1(rs + V_R * RV + o) : 0.f;
        d_a[o] = valid ? raw1(rs + V_A * RV + o) : 0.f;
        d_c[o] = valid ? raw1(rs + V_W * RV + o) : 1.f;
      }
      __syncthreads();
    }
    if (tid == 0 && c + Cfg::NSTAGE < nchunks) issue(c + Cfg::NSTAGE, st);

    // steps of this chunk that start with a checkpoint
    unsigned ckmask = 0;
    if (ck_base) {
      for (int l = 0; l < K && t0 + l < T; ++l) {
        if (ck_left == 0) {
          ckmask |= 1u << l;
          ck_left = args.C;
        }
        --ck_left;
      }
    }

    if (!direct) {
      // ---- K scaled steps, software-pipelined: the cross-lane sum X(l) that
      // feeds sa(l+1) is started before the rest of step l and the loads of
      // step l+1, and consumed last.
      float vr[R];
      float2 kv[NP], av[NP], bv[NP], rv[NP];
      auto load_step = [&](int l) {
#pragma unroll
        for (int i = 0; i < R; ++i) vr[i] = lds32(d_v + l * N + row0 + i);
#pragma unroll
        for (int m = 0; m < Q; ++m) {
          const float4 k4 = lds32x4(d_k + l * N + colq(m));
          const float4 a4 = lds32x4(d_a + l * N + colq(m));
          const float4 b4 = lds32x4(d_b + l * N + colq(m));
          const float4 r4 = lds32x4(d_r + l * N + colq(m));
          kv[2 * m] = make_float2(k4.x, k4.y); kv[2 * m + 1] = make_float2(k4.z, k4.w);
          av[2 * m] = make_float2(a4.x, a4.y); av[2 * m + 1] = make_float2(a4.z, a4.w);
          bv[2 * m] = make_float2(b4.x, b4.y); bv[2 * m + 1] = make_float2(b4.z, b4.w);
          rv[2 * m] = make_float2(r4.x, r4.y); rv[2 * m + 1] = make_float2(r4.z, r4.w);
        }
      };
      load_step(0);
#pragma unroll 4
      for (int l = 0; l < K; ++l) {
        const int t = t0 + l;
        if (ckmask & (1u << l)) {
          float* dst = ck_base + (size_t)(t / args.C) * N * N;
#pragma unroll
          for (int m = 0; m < Q; ++m) {
            const float4 c4 = l > 0 ? ld_f4(d_c + (l - 1) * N + colq(m)) : make_float4(1.f, 1.f, 1.f, 1.f);
#pragma unroll
            for (int i = 0; i < R; ++i) {
              float4* p = reinterpret_cast<float4*>(dst + (size_t)i * N + colq(m));
              if (in_extent(args.status, args.ext.ckpt, p))
                *p = make_float4(S[i][2 * m].x * c4.x, S[i][2 * m].y * c4.y, S[i][2 * m + 1].x * c4.z,
                                 S[i][2 * m + 1].y * c4.w);
            }
          }
        }
        const float bl = beta[l];
        // u~ = S~ + v k~ and the partial of X = u~ a^(l+1)
        float X[R];
#pragma unroll
        for (int i = 0; i < R; ++i) {
#pragma unroll
          for (int p = 0; p < NP; ++p) S[i][p] = ffma2(f2(vr[i]), kv[p], S[i][p]);
          float2 x0 = fmul2(S[i][0], av[0]);
          float2 x1 = fmul2(S[i][1], av[1]);
#pragma unroll
          for (int p = 2; p < NP; p += 2) {
            x0 = ffma2(S[i][p], av[p], x0);
            x1 = ffma2(S[i][p + 1], av[p + 1], x1);
          }
          X[i] = hsum(fadd2(x0, x1));
        }
        // start the cross-lane sums of X (needed only at the end of the step)
#pragma unroll
        for (int o = 1; o < G; o <<= 1)
#pragma unroll
          for (int i = 0; i < R; ++i) X[i] += __shfl_xor_sync(0xffffffffu, X[i], o);
        // S~ = u~ + sa b~ and y partials
        float Y[R];
#pragma unroll
        for (int i = 0; i < R; ++i) {
#pragma unroll
          for (int p = 0; p < NP; ++p) S[i][p] = ffma2(f2(sa[i]), bv[p], S[i][p]);
          float2 y0 = fmul2(S[i][0], rv[0]);
          float2 y1 = fmul2(S[i][1], rv[1]);
#pragma unroll
          for (int p = 2; p < NP; p += 2) {
            y0 = ffma2(S[i][p], rv[p], y0);
            y1 = ffma2(S[i][p + 1], rv[p + 1], y1);
          }
          Y[i] = hsum(fadd2(y0, y1));
        }
        if (l + 1 < K) load_step(l + 1);
        const float yv = rowsum_scatter<G, R>(Y, cg);
        if (y && t < T && row_writer<G, R>(cg)) {
          TIn* p = y + vbase + (size_t)t * vstep + row0 + row_of_lane<G, R>(cg);
          if (in_extent(args.status, args.ext.y, p)) st1(p, yv);
        }
#pragma unroll
        for (int i = 0; i < R; ++i) sa[i] = fmaf(sa[i], bl, X[i]);
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
        if (ckmask & (1u << l)) {
          float* dst = ck_base + (size_t)(t / args.C) * N * N;
#pragma unroll
          for (int m = 0; m < Q; ++m)
#pragma unroll
            for (int i = 0; i < R; ++i) {
              float4* p = reinterpret_cast<float4*>(dst + (size_t)i * N + colq(m));
              if (in_extent(args.status, args.ext.ckpt, p))
                *p = make_float4(S[i][2 * m].x, S[i][2 * m].y, S[i][2 * m + 1].x, S[i][2 * m + 1].y);
            }
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
            for (int i = 0; i < R; ++i)
              sa[i] += hsum(ffma2(S[i][2 * m + 1], make_float2(a4.z, a4.w), fmul2(S[i][2 * m], make_float2(a4.x, a4.y))));
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
              Y[i] += hsum(fmul2(s2, r2));
            }
          }
        }
        const float yv = rowsum_scatter<G, R>(Y, cg);
        if (y && t < T && row_writer<G, R>(cg)) {
          TIn* p = y + vbase + (size_t)t * vstep + row0 + row_of_lane<G, R>(cg);
          if (in_extent(args.status, args.ext.y, p)) st1(p, yv);
        }
      }
    }
  }

  if (args.s_final) {
#pragma unroll
    for (int i = 0; i < R; ++i)
#pragma unroll
      for (int m = 0; m < Q; ++m) {
        float4* p = reinterpret_cast<float4*>(args.s_final + ((size_t)head * N + row0 + i) * N + colq(m));
        if (in_extent(args.status, args.ext.s_final, p))
          *p = make_float4(S[i][2 * m].x, S[i][2 * m].y, S[i][2 * m + 1].x, S[i][2 * m + 1].y);
      }
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

// Steps per TMA box of the forward kernels' input rows (both forms stage 16).
int fwd_steps_per_stage(int N, bool bf16) {
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
