// WKV7 backward-through-time (sm_103a): column-scaled fast path, a direct
// form for windows whose decays leave the safe range, and a TMEM state stash.
//
// The reverse scan of "rx_pretrain.c", rx_wkv7_backward (equations (1)-(3)):
// with G = dL/dS carried from t = T-1 down to 0 (starting at zero),
//   dr = S_t^T dy ;  G += dy r^T ;  dk = G^T v ;  db = G^T sa ;
//   dw = colsum(G o S_prev) ;  dv = G k ;  dsa = G b ;  da = S_prev^T dsa ;
//   G <- G diag(w) + dsa a^T ;  dS_init = G after step 0.
//
// Work per head (one CTA). Steps are processed in windows of at most KS
// steps: windows tile each checkpoint chunk from its end, and the last
// window of the sequence is padded with identity steps. A window is (1)
// staged by TMA together with its chunk's checkpoint, (2) turned into fp32
// per-step vectors by a prologue, (3) replayed forward from the checkpoint,
// each thread storing its R x E tile of the pre-step state into its own TMEM
// lane (tcgen05.st) and emitting dr, then (4) walked backwards, reloading
// the tiles with tcgen05.ld, with all other outputs and the carry fused.
//
// Scaled form (wkv7_scaled.cuh), with c(t) the running product of w since
// the window start and G~ = G diag(c(t)) carried in the window's scale:
//   replay:  u~ = S~ + v k~^T ; S~ = u~ + sa b~^T ; sa(t+1) = u~ a^(t+1) + sa beta(t)
//   reverse: G~ += dy r^^T ; dk = (G~^T v)/c ; db = (G~^T sa)/c ;
//            dw = colsum(G~ o S~_prev) c(t-1)/c(t) ; dv = G~ k~ ;
//            dsa(t) = G~(t+1) b~(t) + dsa(t+1) beta(t) + dy rho(t) ;
//            da = (S~_prev^T dsa) c(t-1) ; G~ += dsa a^^T
// with beta(t) = b(t) . a(t+1) and rho(t) = r(t) . b(t): the row sum that
// feeds dsa(t) starts one step early. At window entry G~ = G diag(c(last));
// at window exit c = 1, so the carry leaves in true scale.
//
// Column sums (dr, dk, db, dw, da) are per-thread partials over R rows,
// reduce-scattered across the row groups of a warp with shuffles, and summed
// across warps through shared memory once per window; row sums (sa, dsa, dv)
// are xor-shuffle sums over the G lanes of a row group.
#include "wkv7_launch.h"
#include "wkv7_scaled.cuh"
#include "wkv7_tmem.cuh"

namespace wkv7 {
namespace {

__host__ __device__ constexpr size_t a128(size_t x) { return (x + 127) / 128 * 128; }
__host__ __device__ constexpr int pow2ceil32(int x) { return x <= 32 ? 32 : 2 * pow2ceil32((x + 1) / 2); }
__host__ __device__ constexpr int ilog2c(int x) { return x <= 1 ? 0 : 1 + ilog2c(x / 2); }

template <typename TIn, int N, int R, int E, int KS>
struct Bwd2Cfg {
  static constexpr int G = N / E;  // lanes per row group
  static constexpr int P = N / R;  // row groups
  static constexpr int THREADS = G * P;
  static constexpr int NWARPS = THREADS / 32;
  static constexpr int Q = E / 4, NP = E / 2, TILE = R * E;
  static constexpr int RG_ROUNDS = ilog2c(32 / G);  // shuffle rounds across row groups
  static constexpr int RGN = 1 << RG_ROUNDS;
  static constexpr int NVEC = 7;  // r, w, k, v, a, b, dy
  static constexpr int RAW_VEC = KS * N;
  static constexpr size_t RAW_BYTES = (size_t)NVEC * RAW_VEC * Elem<TIn>::bytes;
  static constexpr size_t CK_OFF = a128(RAW_BYTES);
  static constexpr size_t STAGE_BYTES = a128(CK_OFF + (size_t)N * N * 4);
  static constexpr int NSTAGE = 2;
  static constexpr int DV = KS * N;
  static constexpr int NDER = 10;  // k, b, a, r, c, ic, w, v, dy, sa
  static constexpr size_t OFF_DER = NSTAGE * STAGE_BYTES;
  static constexpr size_t OFF_SC = OFF_DER + (size_t)NDER * DV * 4;  // beta, rho partials
  static constexpr int NSUM = 5;                                       // dr, dk, db, dw, da
  static constexpr size_t OFF_COL = a128(OFF_SC + (size_t)2 * KS * 4);
  static constexpr size_t COL_BYTES = (size_t)KS * NWARPS * NSUM * N * 4;
  static constexpr size_t OFF_BAR = OFF_COL + COL_BYTES;
  static constexpr size_t SMEM_BYTES = OFF_BAR + 64;
  static constexpr int TMEM_COLS = pow2ceil32(KS * TILE);
  static_assert(E % 4 == 0 && 32 % G == 0 && N % R == 0 && (R == 2 || R == 4), "bad tiling");
  static_assert(THREADS % 32 == 0 && NWARPS <= 4, "one TMEM lane quarter per warp");
  static_assert(TILE == 8 || TILE == 32, "TMEM tile width");
  static_assert(KS * TILE <= 512, "TMEM capacity");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory over budget");
};

enum { V_R = 0, V_W = 1, V_K = 2, V_V = 3, V_A = 4, V_B = 5, V_DY = 6 };

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

__device__ __forceinline__ float2 lo2(float4 v) { return make_float2(v.x, v.y); }
__device__ __forceinline__ float2 hi2(float4 v) { return make_float2(v.z, v.w); }

// Reduce NV per-lane partial column sums across the row groups of a warp
// (lane bits log2(G) .. 4), halving the set each round (reduce-scatter). On
// return vals[0 .. NV / RGN) hold warp-complete sums of the original entries
// base + v; the return value is base.
template <int G, int NV>
__device__ __forceinline__ int colreduce(float (&vals)[NV], int lane) {
  constexpr int ROUNDS = ilog2c(32 / G);
  static_assert(NV % (1 << ROUNDS) == 0, "pad the partials");
  int base = 0;
#pragma unroll
  for (int r = 0; r < ROUNDS; ++r) {
    const int mask = 16 >> r;
    const bool upper = (lane & mask) != 0;
    const int h = (NV >> r) / 2;
#pragma unroll
    for (int v = 0; v < h; ++v) {
      const float send = upper ? vals[v] : vals[h + v];
      const float keep = upper ? vals[h + v] : vals[v];
      vals[v] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
    }
    if (upper) base += h;
  }
  return base;
}

template <typename TIn, int N, int R, int E, int KS>
__global__ void __launch_bounds__(Bwd2Cfg<TIn, N, R, E, KS>::THREADS, 1)
    wkv7_bwd2_kernel(const __grid_constant__ BwdArgs args) {
  using Cfg = Bwd2Cfg<TIn, N, R, E, KS>;
  constexpr int G = Cfg::G, Q = Cfg::Q, NP = Cfg::NP, DV = Cfg::DV, RV = Cfg::RAW_VEC;
  constexpr int TILE = Cfg::TILE, NWARPS = Cfg::NWARPS, NSUM = Cfg::NSUM, RGN = Cfg::RGN;
  extern __shared__ __align__(128) unsigned char smem[];
  float* d_k = reinterpret_cast<float*>(smem + Cfg::OFF_DER);
  float* d_b = d_k + DV;
  float* d_a = d_b + DV;
  float* d_r = d_a + DV;
  float* d_c = d_r + DV;
  float* d_ic = d_c + DV;
  float* d_w = d_ic + DV;
  float* d_v = d_w + DV;
  float* d_dy = d_v + DV;
  float* d_sa = d_dy + DV;
  float* beta = reinterpret_cast<float*>(smem + Cfg::OFF_SC);
  float* rho = beta + KS;
  float* colbuf = reinterpret_cast<float*>(smem + Cfg::OFF_COL);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_BAR + 32);

  const int T = args.T, H = args.H, C = args.C, nck = args.nck;
  const int head = blockIdx.x;
  const int bi = head / H, hi = head % H;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cg = tid % G, rg = tid / G;
  const int row0 = rg * R;
  const size_t vstep = (size_t)H * N;
  const size_t vbase = ((size_t)bi * T * H + hi) * N;
  auto colq = [&](int m) { return 4 * (m * G + cg); };

  if (warp == 0) tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
  if (tid == 0) {
    for (int s = 0; s < Cfg::NSTAGE; ++s) mbar_init(&full[s], 1);
    fence_mbar_init();
    for (int v = 0; v < Cfg::NVEC; ++v) prefetch_tensormap(&args.map[v]);
    prefetch_tensormap(&args.ckmap);
  }
  tmem_fence_before_sync();
  __syncthreads();
  tmem_fence_after_sync();
  const uint32_t tlane = *tmem_slot + ((uint32_t)((warp & 3) * 32) << 16);

  // ---- windows: chunk c (steps [c*C, min(T, c*C+C))) is covered from its end
  // by windows [s0, s1) of at most KS steps; a window that does not start at
  // the chunk start is preceded by "advance" pieces that replay from the
  // checkpoint without recording. Order: chunks from last to first.
  struct Win {
    int c, s1, p;
  };
  auto w_s0 = [&](const Win& w) { return max(w.c * C, w.s1 - KS); };
  auto w_np = [&](const Win& w) { return (w_s0(w) - w.c * C + KS - 1) / KS; };
  auto w_start = [&](const Win& w) { return w.p < w_np(w) ? w.c * C + w.p * KS : w_s0(w); };
  auto w_len = [&](const Win& w) {
    return w.p < w_np(w) ? min(KS, w_s0(w) - (w.c * C + w.p * KS)) : w.s1 - w_s0(w);
  };
  auto w_next = [&](Win& w) -> bool {
    if (w.p < w_np(w)) {
      ++w.p;
      return true;
    }
    const int s0 = w_s0(w);
    if (s0 > w.c * C) {
      w.s1 = s0;
      w.p = 0;
      return true;
    }
    if (w.c == 0) return false;
    --w.c;
    w.s1 = w.c * C + C;
    w.p = 0;
    return true;
  };
  auto issue = [&](const Win& w, int st) {
    unsigned char* base = smem + (size_t)st * Cfg::STAGE_BYTES;
    mbar_arrive_expect_tx(&full[st], (uint32_t)(Cfg::RAW_BYTES + (size_t)N * N * 4));
    const int t_begin = w_start(w);
    for (int v = 0; v < Cfg::NVEC; ++v)
      tma_load_4d(base + (size_t)v * RV * Elem<TIn>::bytes, &args.map[v], &full[st], 0, hi, t_begin, bi);
    tma_load_3d(base + Cfg::CK_OFF, &args.ckmap, &full[st], 0, 0, head * nck + w.c);
  };
  Win cur{nck - 1, T, 0};
  Win pre = cur;
  bool pre_valid = true;
  if (tid == 0)
    for (int s = 0; s < Cfg::NSTAGE && pre_valid; ++s) {
      issue(pre, s);
      pre_valid = w_next(pre);
    }

  // Prologue mapping: thread = (column quad pq, step group pg); each thread
  // forms the per-step vectors of 4 columns for SG consecutive steps.
  constexpr int NQ = N / 4;
  constexpr int SG = KS * NQ / Cfg::THREADS;
  static_assert(SG >= 1 && KS % SG == 0 && NQ <= 32 && Cfg::THREADS % NQ == 0, "prologue mapping");
  const int pq = tid % NQ, pg = tid / NQ;

  // the carry after the last step: the gradient entering through the final state (or zero)
  float2 Gt[R][NP];
#pragma unroll
  for (int i = 0; i < R; ++i)
#pragma unroll
    for (int m = 0; m < Q; ++m) {
      const float* src = args.dS_final + ((size_t)head * N + row0 + i) * N + colq(m);
      const float4 g4 = args.dS_final && in_extent(args.status, args.ext.dS_final, reinterpret_cast<const float4*>(src))
                            ? ld_f4(src)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
      Gt[i][2 * m] = make_float2(g4.x, g4.y);
      Gt[i][2 * m + 1] = make_float2(g4.z, g4.w);
    }
  float2 S[R][NP];
  bool completed = true;

  for (int widx = 0;; ++widx) {
    const int st = widx & 1;
    {
      const bool ok = mbar_wait_bounded(args.status, &full[st], (widx >> 1) & 1);
      if (!__syncthreads_and(ok)) {
        if (tid == 0)  // drain the copies that may still be in flight
          for (int k = 0; k < Cfg::NSTAGE; ++k)
            mbar_wait_bounded(args.status, &full[(widx + k) & 1], ((widx + k) >> 1) & 1);
        completed = false;
        break;
      }
    }
    const TIn* rs = reinterpret_cast<const TIn*>(smem + (size_t)st * Cfg::STAGE_BYTES);
    const float* cks = reinterpret_cast<const float*>(smem + (size_t)st * Cfg::STAGE_BYTES + Cfg::CK_OFF);
    const int start = w_start(cur), len = w_len(cur);
    const bool is_main = cur.p == w_np(cur);
    if (cur.p == 0) {  // the chunk's checkpoint: state before step c*C
#pragma unroll
      for (int i = 0; i < R; ++i)
#pragma unroll
        for (int m = 0; m < Q; ++m) {
          const float4 s4 = ld_f4(cks + (row0 + i) * N + colq(m));
          S[i][2 * m] = lo2(s4);
          S[i][2 * m + 1] = hi2(s4);
        }
    }

    // ---- prologue, scaled form (identity steps beyond len): c(l) = w(0)..w(l)
    // of this window; k~ = k/c, b~ = b/c, a^ = c(l-1) a, r^ = c r, 1/c;
    // beta(l) = b(l) . a(l+1) and rho(l) = r(l) . b(l). Also checks the decays.
    bool unsafe = false;
    {
      const int col = 4 * pq;
      const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
      float4 cp = make_float4(1.f, 1.f, 1.f, 1.f);  // running product before step l
#pragma unroll
      for (int l = 0; l < KS - SG; ++l) {
        if (l < pg * SG && l < len) {
          const float4 w4 = lds4(rs + V_W * RV + l * N + col);
          cp = make_float4(cp.x * w4.x, cp.y * w4.y, cp.z * w4.z, cp.w * w4.w);
        }
      }
#pragma unroll
      for (int g = 0; g < SG; ++g) {
        const int l = pg * SG + g;
        const int o = l * N + col;
        const bool valid = l < len;
        const bool next = l + 1 < len;
        const float4 w4 = valid ? lds4(rs + V_W * RV + o) : make_float4(1.f, 1.f, 1.f, 1.f);
        const float4 k4 = valid ? lds4(rs + V_K * RV + o) : z;
        const float4 b4 = valid ? lds4(rs + V_B * RV + o) : z;
        const float4 r4 = valid ? lds4(rs + V_R * RV + o) : z;
        const float4 a4 = valid ? lds4(rs + V_A * RV + o) : z;
        const float4 v4 = valid ? lds4(rs + V_V * RV + o) : z;
        const float4 y4 = valid ? lds4(rs + V_DY * RV + o) : z;
        const float4 an = next ? lds4(rs + V_A * RV + o + N) : z;
        if (!decay_is_safe(w4.x) || !decay_is_safe(w4.y) || !decay_is_safe(w4.z) || !decay_is_safe(w4.w))
          unsafe = true;
        const float4 c4 = make_float4(cp.x * w4.x, cp.y * w4.y, cp.z * w4.z, cp.w * w4.w);
        const float4 i4 = make_float4(rcp_approx(c4.x), rcp_approx(c4.y), rcp_approx(c4.z), rcp_approx(c4.w));
        *reinterpret_cast<float4*>(d_k + o) = make_float4(k4.x * i4.x, k4.y * i4.y, k4.z * i4.z, k4.w * i4.w);
        *reinterpret_cast<float4*>(d_b + o) = make_float4(b4.x * i4.x, b4.y * i4.y, b4.z * i4.z, b4.w * i4.w);
        *reinterpret_cast<float4*>(d_a + o) = make_float4(a4.x * cp.x, a4.y * cp.y, a4.z * cp.z, a4.w * cp.w);
        *reinterpret_cast<float4*>(d_r + o) = make_float4(r4.x * c4.x, r4.y * c4.y, r4.z * c4.z, r4.w * c4.w);
        *reinterpret_cast<float4*>(d_c + o) = c4;
        *reinterpret_cast<float4*>(d_ic + o) = i4;
        *reinterpret_cast<float4*>(d_w + o) = w4;
        *reinterpret_cast<float4*>(d_v + o) = v4;
        *reinterpret_cast<float4*>(d_dy + o) = y4;
        float pb = b4.x * an.x + b4.y * an.y + b4.z * an.z + b4.w * an.w;
        float pr = r4.x * b4.x + r4.y * b4.y + r4.z * b4.z + r4.w * b4.w;
#pragma unroll
        for (int mask = 1; mask < NQ; mask <<= 1) {
          pb += __shfl_xor_sync(0xffffffffu, pb, mask);
          pr += __shfl_xor_sync(0xffffffffu, pr, mask);
        }
        if (pq == 0) {
          beta[l] = pb;
          rho[l] = pr;
        }
        cp = c4;
      }
    }
    // sa at the window's first step, directly
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
        float2 p = fmul2(S[i][2 * m], make_float2(a4[0], a4[1]));
        p = ffma2(S[i][2 * m + 1], make_float2(a4[2], a4[3]), p);
        sa[i] += p.x + p.y;
      }
    }
#pragma unroll
    for (int i = 0; i < R; ++i) sa[i] = group_allreduce<G>(sa[i]);
    const bool direct = __syncthreads_or(unsafe) != 0;  // per-step vectors complete
    if (direct) {
      // ---- rare: some decay outside the safe range; plain vectors instead
      for (int o = tid; o < KS * N; o += Cfg::THREADS) {
        const bool valid = o / N < len;
        d_k[o] = valid ? raw1(rs + V_K * RV + o) : 0.f;
        d_b[o] = valid ? raw1(rs + V_B * RV + o) : 0.f;
        d_a[o] = valid ? raw1(rs + V_A * RV + o) : 0.f;
        d_r[o] = valid ? raw1(rs + V_R * RV + o) : 0.f;
        d_c[o] = 1.f;
        d_ic[o] = 1.f;
      }
      __syncthreads();
    }
    if (tid == 0 && pre_valid) {
      issue(pre, st);
      pre_valid = w_next(pre);
    }

    // ================================================== replay (forward)
    const bool record = is_main;
#pragma unroll 1
    for (int l = 0; l < KS; ++l) {
      if (!record && l >= len) break;
      if (record) {
        float tile[TILE];
#pragma unroll
        for (int i = 0; i < R; ++i)
#pragma unroll
          for (int p = 0; p < NP; ++p) {
            tile[i * E + 2 * p] = S[i][p].x;
            tile[i * E + 2 * p + 1] = S[i][p].y;
          }
        tmem_st<TILE>(tlane + (uint32_t)(l * TILE), tile);
      }
      float vr[R], dyr[R];
      ld_rows<R>(d_v + l * N + row0, vr);
      ld_rows<R>(d_dy + l * N + row0, dyr);
      float pdr[E];
      if (!direct) {
        if (record && cg == 0)
#pragma unroll
          for (int i = 0; i < R; ++i) d_sa[l * N + row0 + i] = sa[i];
        const bool ahead = l + 1 < KS;
        float2 kv[NP], bv[NP], av[NP];
#pragma unroll
        for (int m = 0; m < Q; ++m) {
          const float4 k4 = ld_f4(d_k + l * N + colq(m));
          const float4 b4 = ld_f4(d_b + l * N + colq(m));
          const float4 a4 = ahead ? ld_f4(d_a + (l + 1) * N + colq(m)) : make_float4(0.f, 0.f, 0.f, 0.f);
          kv[2 * m] = lo2(k4); kv[2 * m + 1] = hi2(k4);
          bv[2 * m] = lo2(b4); bv[2 * m + 1] = hi2(b4);
          av[2 * m] = lo2(a4); av[2 * m + 1] = hi2(a4);
        }
        const float bl = beta[l];
        // u~ = S~ + v k~
#pragma unroll
        for (int i = 0; i < R; ++i)
#pragma unroll
          for (int p = 0; p < NP; ++p) S[i][p] = ffma2(f2(vr[i]), kv[p], S[i][p]);
        float X[R];
#pragma unroll
        for (int i = 0; i < R; ++i) {
          float2 x0 = fmul2(S[i][0], av[0]);
          float2 x1 = fmul2(S[i][1], av[1]);
#pragma unroll
          for (int p = 2; p < NP; p += 2) {
            x0 = ffma2(S[i][p], av[p], x0);
            x1 = ffma2(S[i][p + 1], av[p + 1], x1);
          }
          X[i] = hsum(fadd2(x0, x1));
        }
        // S~ = u~ + sa b~, and dr partials over this thread's rows
#pragma unroll
        for (int i = 0; i < R; ++i)
#pragma unroll
          for (int p = 0; p < NP; ++p) S[i][p] = ffma2(f2(sa[i]), bv[p], S[i][p]);
#pragma unroll
        for (int p = 0; p < NP; ++p) {
          float2 d2 = fmul2(S[0][p], f2(dyr[0]));
#pragma unroll
          for (int i = 1; i < R; ++i) d2 = ffma2(S[i][p], f2(dyr[i]), d2);
          pdr[2 * p] = d2.x;
          pdr[2 * p + 1] = d2.y;
        }
#pragma unroll
        for (int i = 0; i < R; ++i) sa[i] = fmaf(sa[i], bl, group_allreduce<G>(X[i]));
      } else {
        if (l > 0) {
#pragma unroll
          for (int i = 0; i < R; ++i) sa[i] = 0.f;
#pragma unroll
          for (int m = 0; m < Q; ++m) {
            const float4 a4 = ld_f4(d_a + l * N + colq(m));
#pragma unroll
            for (int i = 0; i < R; ++i) {
              float2 p = fmul2(S[i][2 * m], lo2(a4));
              p = ffma2(S[i][2 * m + 1], hi2(a4), p);
              sa[i] += p.x + p.y;
            }
          }
#pragma unroll
          for (int i = 0; i < R; ++i) sa[i] = group_allreduce<G>(sa[i]);
        }
        if (record && cg == 0)
#pragma unroll
          for (int i = 0; i < R; ++i) d_sa[l * N + row0 + i] = sa[i];
#pragma unroll
        for (int m = 0; m < Q; ++m) {
          const float4 k4 = ld_f4(d_k + l * N + colq(m));
          const float4 b4 = ld_f4(d_b + l * N + colq(m));
          const float4 w4 = ld_f4(d_w + l * N + colq(m));
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int p = 2 * m + h;
            const float2 k2 = h ? hi2(k4) : lo2(k4), b2 = h ? hi2(b4) : lo2(b4), w2 = h ? hi2(w4) : lo2(w4);
            float2 dr2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int i = 0; i < R; ++i) {
              S[i][p] = ffma2(f2(sa[i]), b2, ffma2(S[i][p], w2, fmul2(k2, f2(vr[i]))));
              dr2 = ffma2(S[i][p], f2(dyr[i]), dr2);
            }
            pdr[2 * p] = dr2.x;
            pdr[2 * p + 1] = dr2.y;
          }
        }
      }
      if (record) {
        constexpr int NV = (E + RGN - 1) / RGN * RGN;
        float vals[NV];
#pragma unroll
        for (int v = 0; v < NV; ++v) vals[v] = v < E ? pdr[v] : 0.f;
        const int base = colreduce<G, NV>(vals, lane);
        float* cb = colbuf + ((size_t)(l * NWARPS + warp) * NSUM + 0) * N;
#pragma unroll
        for (int v = 0; v < NV / RGN; ++v) {
          const int e = base + v;
          if (e < E) cb[colq(e >> 2) + (e & 3)] = vals[v];
        }
      }
    }
    if (!record) {  // advance piece done: back to true scale
      if (!direct) {
#pragma unroll
        for (int m = 0; m < Q; ++m) {
          const float4 c4 = ld_f4(d_c + (KS - 1) * N + colq(m));
#pragma unroll
          for (int i = 0; i < R; ++i) {
            S[i][2 * m] = fmul2(S[i][2 * m], lo2(c4));
            S[i][2 * m + 1] = fmul2(S[i][2 * m + 1], hi2(c4));
          }
        }
      }
    } else {
      tmem_wait_st();
      __syncwarp();  // d_sa rows written by the row group's lane 0

      // ================================================ reverse walk
      // enter the window's scale: G~ = G diag(c(last step))
#pragma unroll
      for (int m = 0; m < Q; ++m) {
        const float4 c4 = ld_f4(d_c + (KS - 1) * N + colq(m));
#pragma unroll
        for (int i = 0; i < R; ++i) {
          Gt[i][2 * m] = fmul2(Gt[i][2 * m], lo2(c4));
          Gt[i][2 * m + 1] = fmul2(Gt[i][2 * m + 1], hi2(c4));
        }
      }
      float dsa_next[R], zc[R];
#pragma unroll
      for (int i = 0; i < R; ++i) {
        dsa_next[i] = 0.f;
        zc[i] = 0.f;
      }
      float spv[TILE];  // S~_prev tile of the step, loaded one step ahead
      tmem_ld<TILE>(tlane + (uint32_t)((KS - 1) * TILE), spv);
#pragma unroll 1
      for (int l = KS - 1; l >= 0; --l) {
        tmem_wait_ld();
        float dyr[R], vr[R], sar[R];
        ld_rows<R>(d_dy + l * N + row0, dyr);
        ld_rows<R>(d_v + l * N + row0, vr);
        ld_rows<R>(d_sa + l * N + row0, sar);
        const bool first = l == KS - 1;           // dsa from the full row sum
        const bool use_z = !direct && l > 0;      // row sum feeding dsa(t-1)
        const bool use_d = direct || first;
        float2 r2[NP], k2[NP], bz[NP], bd[NP];
#pragma unroll
        for (int m = 0; m < Q; ++m) {
          const float4 r4 = ld_f4(d_r + l * N + colq(m));
          const float4 k4 = ld_f4(d_k + l * N + colq(m));
          const float4 z4 = use_z ? ld_f4(d_b + (l - 1) * N + colq(m)) : make_float4(0.f, 0.f, 0.f, 0.f);
          const float4 d4 = use_d ? ld_f4(d_b + l * N + colq(m)) : make_float4(0.f, 0.f, 0.f, 0.f);
          r2[2 * m] = lo2(r4); r2[2 * m + 1] = hi2(r4);
          k2[2 * m] = lo2(k4); k2[2 * m + 1] = hi2(k4);
          bz[2 * m] = lo2(z4); bz[2 * m + 1] = hi2(z4);
          bd[2 * m] = lo2(d4); bd[2 * m + 1] = hi2(d4);
        }
        // G~ += dy r^
#pragma unroll
        for (int i = 0; i < R; ++i)
#pragma unroll
          for (int p = 0; p < NP; ++p) Gt[i][p] = ffma2(f2(dyr[i]), r2[p], Gt[i][p]);
        // column partials: dk (G~^T v), db (G~^T sa), dw (colsum G~ o S~_prev)
        constexpr int NV1 = (3 * E + RGN - 1) / RGN * RGN;
        float p1[NV1];
#pragma unroll
        for (int p = 0; p < NP; ++p) {
          const float2 s0 = make_float2(spv[2 * p], spv[2 * p + 1]);
          float2 ak = fmul2(Gt[0][p], f2(vr[0]));
          float2 ab = fmul2(Gt[0][p], f2(sar[0]));
          float2 aw = fmul2(Gt[0][p], s0);
#pragma unroll
          for (int i = 1; i < R; ++i) {
            ak = ffma2(Gt[i][p], f2(vr[i]), ak);
            ab = ffma2(Gt[i][p], f2(sar[i]), ab);
            aw = ffma2(Gt[i][p], make_float2(spv[i * E + 2 * p], spv[i * E + 2 * p + 1]), aw);
          }
          p1[2 * p] = ak.x; p1[2 * p + 1] = ak.y;
          p1[E + 2 * p] = ab.x; p1[E + 2 * p + 1] = ab.y;
          p1[2 * E + 2 * p] = aw.x; p1[2 * E + 2 * p + 1] = aw.y;
        }
#pragma unroll
        for (int v = 3 * E; v < NV1; ++v) p1[v] = 0.f;
        // row partials: dv (G~ k~), z (G~ b~(t-1)) and, first / direct, dsa (G~ b~(t))
        float pdv[R], pz[R], pds[R];
#pragma unroll
        for (int i = 0; i < R; ++i) {
          float2 d0 = fmul2(Gt[i][0], k2[0]), d1 = fmul2(Gt[i][1], k2[1]);
          float2 z0 = fmul2(Gt[i][0], bz[0]), z1 = fmul2(Gt[i][1], bz[1]);
#pragma unroll
          for (int p = 2; p < NP; p += 2) {
            d0 = ffma2(Gt[i][p], k2[p], d0); d1 = ffma2(Gt[i][p + 1], k2[p + 1], d1);
            z0 = ffma2(Gt[i][p], bz[p], z0); z1 = ffma2(Gt[i][p + 1], bz[p + 1], z1);
          }
          pdv[i] = hsum(fadd2(d0, d1));
          pz[i] = hsum(fadd2(z0, z1));
          pds[i] = 0.f;
          if (use_d) {
            float2 e0 = fmul2(Gt[i][0], bd[0]), e1 = fmul2(Gt[i][1], bd[1]);
#pragma unroll
            for (int p = 2; p < NP; p += 2) {
              e0 = ffma2(Gt[i][p], bd[p], e0);
              e1 = ffma2(Gt[i][p + 1], bd[p + 1], e1);
            }
            pds[i] = hsum(fadd2(e0, e1));
          }
        }
        const float bl = beta[l], rl = rho[l];
        float dsa[R];
#pragma unroll
        for (int i = 0; i < R; ++i) {
          dsa[i] = use_d ? group_allreduce<G>(pds[i]) : zc[i] + dsa_next[i] * bl + dyr[i] * rl;
          zc[i] = use_z ? group_allreduce<G>(pz[i]) : 0.f;
        }
        {
          const float dvv = rowsum_scatter<G, R>(pdv, cg);
          float* p = args.dv + vbase + (size_t)(start + l) * vstep + row0 + row_of_lane<G, R>(cg);
          if (l < len && row_writer<G, R>(cg) && in_extent(args.status, args.ext.dv, p)) *p = dvv;
        }
        // da partials (S~_prev^T dsa) and the carry G~ += dsa a^ (direct: G = G w + dsa a)
        constexpr int NV2 = (E + RGN - 1) / RGN * RGN;
        float p2[NV2];
        float2 a2[NP], w2[NP];
#pragma unroll
        for (int m = 0; m < Q; ++m) {
          const float4 a4 = ld_f4(d_a + l * N + colq(m));
          const float4 w4 = direct ? ld_f4(d_w + l * N + colq(m)) : make_float4(1.f, 1.f, 1.f, 1.f);
          a2[2 * m] = lo2(a4); a2[2 * m + 1] = hi2(a4);
          w2[2 * m] = lo2(w4); w2[2 * m + 1] = hi2(w4);
        }
#pragma unroll
        for (int p = 0; p < NP; ++p) {
          float2 aa = fmul2(f2(dsa[0]), make_float2(spv[2 * p], spv[2 * p + 1]));
#pragma unroll
          for (int i = 1; i < R; ++i) aa = ffma2(f2(dsa[i]), make_float2(spv[i * E + 2 * p], spv[i * E + 2 * p + 1]), aa);
          p2[2 * p] = aa.x;
          p2[2 * p + 1] = aa.y;
        }
#pragma unroll
        for (int v = E; v < NV2; ++v) p2[v] = 0.f;
        if (!direct) {
#pragma unroll
          for (int i = 0; i < R; ++i)
#pragma unroll
            for (int p = 0; p < NP; ++p) Gt[i][p] = ffma2(f2(dsa[i]), a2[p], Gt[i][p]);
        } else {
#pragma unroll
          for (int i = 0; i < R; ++i)
#pragma unroll
            for (int p = 0; p < NP; ++p) Gt[i][p] = ffma2(Gt[i][p], w2[p], fmul2(f2(dsa[i]), a2[p]));
        }
        if (l > 0) tmem_ld<TILE>(tlane + (uint32_t)((l - 1) * TILE), spv);  // next step's tile
#pragma unroll
        for (int i = 0; i < R; ++i) dsa_next[i] = dsa[i];

        float* cb = colbuf + (size_t)(l * NWARPS + warp) * NSUM * N;
        {
          const int base = colreduce<G, NV1>(p1, lane);
#pragma unroll
          for (int v = 0; v < NV1 / RGN; ++v) {
            const int o = base + v;
            if (o < 3 * E) {
              const int s = o / E, e = o % E;
              cb[(1 + s) * N + colq(e >> 2) + (e & 3)] = p1[v];
            }
          }
        }
        {
          const int base = colreduce<G, NV2>(p2, lane);
#pragma unroll
          for (int v = 0; v < NV2 / RGN; ++v) {
            const int e = base + v;
            if (e < E) cb[4 * N + colq(e >> 2) + (e & 3)] = p2[v];
          }
        }
      }
      __syncthreads();  // column partials of every warp are in shared memory

      // ---- cross-warp sums, scaled to true values, written out: one item is
      // a (step, column quad) with all five sums
      for (int idx = tid; idx < len * (N / 4); idx += Cfg::THREADS) {
        const int l = idx / (N / 4), col = 4 * (idx % (N / 4));
        const float4 cl = ld_f4(d_c + l * N + col);
        const float4 il = ld_f4(d_ic + l * N + col);
        const float4 cp = l > 0 ? ld_f4(d_c + (l - 1) * N + col) : make_float4(1.f, 1.f, 1.f, 1.f);
        float4 acc[NSUM];
#pragma unroll
        for (int s = 0; s < NSUM; ++s) acc[s] = ld_f4(colbuf + ((size_t)(l * NWARPS + 0) * NSUM + s) * N + col);
#pragma unroll
        for (int wv = 1; wv < NWARPS; ++wv)
#pragma unroll
          for (int s = 0; s < NSUM; ++s) {
            const float4 x = ld_f4(colbuf + ((size_t)(l * NWARPS + wv) * NSUM + s) * N + col);
            acc[s].x += x.x; acc[s].y += x.y; acc[s].z += x.z; acc[s].w += x.w;
          }
        const size_t go = vbase + (size_t)(start + l) * vstep + col;
        const float4 cw = make_float4(cp.x * il.x, cp.y * il.y, cp.z * il.z, cp.w * il.w);
        auto put = [&](float* out, const Extent& x, const float4& a, const float4& sc) {
          float4* p = reinterpret_cast<float4*>(out + go);
          if (in_extent(args.status, x, p)) *p = make_float4(a.x * sc.x, a.y * sc.y, a.z * sc.z, a.w * sc.w);
        };
        put(args.dr, args.ext.dr, acc[0], cl);
        put(args.dk, args.ext.dk, acc[1], il);
        put(args.db, args.ext.db, acc[2], il);
        put(args.dw, args.ext.dw, acc[3], cw);
        put(args.da, args.ext.da, acc[4], cp);
      }
    }
    if (!w_next(cur)) break;
  }

  if (completed && args.dS_init) {
#pragma unroll
    for (int i = 0; i < R; ++i)
#pragma unroll
      for (int m = 0; m < Q; ++m) {
        float4* p = reinterpret_cast<float4*>(args.dS_init + ((size_t)head * N + row0 + i) * N + colq(m));
        if (in_extent(args.status, args.ext.dS_init, p))
          *p = make_float4(Gt[i][2 * m].x, Gt[i][2 * m].y, Gt[i][2 * m + 1].x, Gt[i][2 * m + 1].y);
      }
  }
  tmem_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tmem_fence_after_sync();
    tmem_dealloc(*tmem_slot, Cfg::TMEM_COLS);
  }
}

template <typename TIn, int N, int R, int E, int KS>
cudaError_t launch_bwd2_impl(const BwdArgs& args, cudaStream_t stream) {
  using Cfg = Bwd2Cfg<TIn, N, R, E, KS>;
  auto kern = wkv7_bwd2_kernel<TIn, N, R, E, KS>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)(args.B * args.H), Cfg::THREADS, Cfg::SMEM_BYTES, stream>>>(args);
  return cudaGetLastError();
}

}  // namespace

int bwd2_steps_per_window(int N, bool bf16) {
  (void)N;
  (void)bf16;
  return 16;
}

cudaError_t launch_bwd2(const BwdArgs& args, bool bf16, int N, cudaStream_t stream) {
  if (bf16) {
    switch (N) {
      case 16: return launch_bwd2_impl<__nv_bfloat16, 16, 2, 4, 16>(args, stream);
      case 32: return launch_bwd2_impl<__nv_bfloat16, 32, 4, 8, 16>(args, stream);
      case 64: return launch_bwd2_impl<__nv_bfloat16, 64, 4, 8, 16>(args, stream);
    }
  } else {
    switch (N) {
      case 16: return launch_bwd2_impl<float, 16, 2, 4, 16>(args, stream);
      case 32: return launch_bwd2_impl<float, 32, 4, 8, 16>(args, stream);
      case 64: return launch_bwd2_impl<float, 64, 4, 8, 16>(args, stream);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace wkv7
