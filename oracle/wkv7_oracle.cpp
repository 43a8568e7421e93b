// WKV7 oracle: a plain, slow CPU implementation of the RWKV-7 matrix-state
// recurrence and its backward-through-time.
//
// TEST INFRASTRUCTURE ONLY. The tests, the smoke check and the benchmark's
// CPU-baseline leg may call it; the library's compute path never does. It
// shares no code, header or table with the CUDA kernels.
//
// Source of the method: "Foundry/rwkvx/rx_pretrain.c" (page "rx_pretrain.c",
// functions rx_wkv7_forward_seq and rx_wkv7_backward, with the reverse-scan
// equations (1)-(3) stated in the comment above rx_wkv7_backward). Per
// (batch b, head h), with an N x N state S (row i = value index, column j =
// key index) and per-step vectors r, w, k, v, a, b of length N:
//
//   forward, t = 0 .. T-1:
//     sa_i = sum_j S_ij a_j                       (pre-update state)
//     S_ij <- S_ij w_j + v_i k_j + sa_i b_j
//     y_i  = sum_j S_ij r_j                       (post-update state)
//
//   backward, G = dL/dS starts at the gradient of the final state: zero in
//   the C file (no loss term reads s_final), or a given dS_final when the
//   sequence is one segment of a longer one (the Mamba-3 page's
//   "serial_recalculated/backward.rs" takes that final-state gradient as an
//   input in the same way); t = T-1 .. 0, with S_prev the state before step t
//   and S_t after it:
//     (1) dr_j = sum_i S_t_ij dy_i ;  G_ij += dy_i r_j
//     (2) dk_j = sum_i G_ij v_i ;  db_j = sum_i G_ij sa_i ;
//         dw_j = sum_i G_ij S_prev_ij   (w is the effective decay itself)
//         dv_i = sum_j G_ij k_j ;  dsa_i = sum_j G_ij b_j
//     (3) da_j = sum_i dsa_i S_prev_ij ;  G_ij <- G_ij w_j + dsa_i a_j
//   after t = 0, G is the gradient of the initial state.
//
// Layout (rx_pretrain.c helpers "vx" and "sx"): vectors are [B][T][H][N],
// states are [B][H][N][N] with S_ij at ((b*H + h)*N + i)*N + j.
//
// The forward keeps the state of every step of a head (like the C file's
// backward, which caches every pre-step state and sa) so the backward reads
// S_prev and S_t instead of recomputing them. Heads run on std::thread
// workers; the caller chooses how many so the per-head caches fit in RAM.
// The scalar type is a template: double is the parity reference, float is
// kept for debugging only.

#include <cstddef>
#include <cstdint>
#include <cstring>
#include <exception>
#include <new>
#include <thread>
#include <vector>

namespace {

template <typename F>
struct HeadView {
  // Vectors of one (b, h): element (t, n) at base[t * stride + n].
  const F* r; const F* w; const F* k; const F* v; const F* a; const F* b;
  const F* dy;
  std::size_t stride;
};

template <typename F>
HeadView<F> head_view(const F* r, const F* w, const F* k, const F* v, const F* a,
                      const F* b, const F* dy, int bi, int hi, int T, int H, int N) {
  const std::size_t off = (static_cast<std::size_t>(bi) * T * H + hi) * N;
  HeadView<F> hv;
  hv.r = r + off; hv.w = w + off; hv.k = k + off; hv.v = v + off;
  hv.a = a + off; hv.b = b + off; hv.dy = dy ? dy + off : nullptr;
  hv.stride = static_cast<std::size_t>(H) * N;
  return hv;
}

// One forward step on state S (N x N, row-major): writes sa (pre-update
// product S a) and updates S in place. Returns nothing; y is read separately.
template <typename F>
void step(F* S, F* sa, const F* w, const F* k, const F* v, const F* a, const F* b, int N) {
  for (int i = 0; i < N; ++i) {
    F acc = 0;
    for (int j = 0; j < N; ++j) acc += S[i * N + j] * a[j];
    sa[i] = acc;
  }
  for (int i = 0; i < N; ++i)
    for (int j = 0; j < N; ++j)
      S[i * N + j] = S[i * N + j] * w[j] + v[i] * k[j] + sa[i] * b[j];
}

// Forward of one head. S holds the initial state on entry, the final on exit.
template <typename F>
void forward_head(const HeadView<F>& hv, F* S, F* y, std::size_t y_stride, int T, int N) {
  std::vector<F> sa(N);
  for (int t = 0; t < T; ++t) {
    const std::size_t o = t * hv.stride;
    step(S, sa.data(), hv.w + o, hv.k + o, hv.v + o, hv.a + o, hv.b + o, N);
    if (y) {
      const F* r = hv.r + o;
      for (int i = 0; i < N; ++i) {
        F acc = 0;
        for (int j = 0; j < N; ++j) acc += S[i * N + j] * r[j];
        y[t * y_stride + i] = acc;
      }
    }
  }
}

// Gradient outputs of one head, same strides as the inputs.
template <typename F>
struct HeadGrads { F* dr; F* dw; F* dk; F* dv; F* da; F* db; };

template <typename F>
void backward_head(const HeadView<F>& hv, const F* s_init, const F* dS_final, const HeadGrads<F>& g,
                   F* dS_init, int T, int N) {
  const std::size_t NN = static_cast<std::size_t>(N) * N;
  // states[t] = state before step t (t = 0..T-1); states[T] = final state.
  std::vector<F> states((static_cast<std::size_t>(T) + 1) * NN);
  std::vector<F> sa_all(static_cast<std::size_t>(T) * N);
  F* S = states.data();
  if (s_init) std::memcpy(S, s_init, NN * sizeof(F));
  else std::memset(S, 0, NN * sizeof(F));
  for (int t = 0; t < T; ++t) {
    const std::size_t o = t * hv.stride;
    F* next = states.data() + (t + 1) * NN;
    std::memcpy(next, states.data() + t * NN, NN * sizeof(F));
    step(next, sa_all.data() + static_cast<std::size_t>(t) * N, hv.w + o, hv.k + o, hv.v + o,
         hv.a + o, hv.b + o, N);
  }

  std::vector<F> G(NN, F(0)), dsa(N);
  if (dS_final) std::memcpy(G.data(), dS_final, NN * sizeof(F));
  for (int t = T - 1; t >= 0; --t) {
    const std::size_t o = t * hv.stride;
    const F* r = hv.r + o; const F* w = hv.w + o; const F* k = hv.k + o;
    const F* v = hv.v + o; const F* a = hv.a + o; const F* b = hv.b + o;
    const F* dy = hv.dy + o;
    const F* sa = sa_all.data() + static_cast<std::size_t>(t) * N;
    const F* Sp = states.data() + t * NN;        // S_prev
    const F* St = states.data() + (t + 1) * NN;  // S_t

    // (1) read-out
    for (int j = 0; j < N; ++j) {
      F acc = 0;
      for (int i = 0; i < N; ++i) acc += St[i * N + j] * dy[i];
      g.dr[o + j] = acc;
    }
    for (int i = 0; i < N; ++i)
      for (int j = 0; j < N; ++j) G[i * N + j] += dy[i] * r[j];

    // (2) state-update gradients
    for (int j = 0; j < N; ++j) {
      F ak = 0, ab = 0, aw = 0;
      for (int i = 0; i < N; ++i) {
        ak += G[i * N + j] * v[i];
        ab += G[i * N + j] * sa[i];
        aw += G[i * N + j] * Sp[i * N + j];
      }
      g.dk[o + j] = ak; g.db[o + j] = ab; g.dw[o + j] = aw;
    }
    for (int i = 0; i < N; ++i) {
      F av = 0, as = 0;
      for (int j = 0; j < N; ++j) {
        av += G[i * N + j] * k[j];
        as += G[i * N + j] * b[j];
      }
      g.dv[o + i] = av; dsa[i] = as;
    }

    // (3) in-context term and the carry to t-1
    for (int j = 0; j < N; ++j) {
      F acc = 0;
      for (int i = 0; i < N; ++i) acc += dsa[i] * Sp[i * N + j];
      g.da[o + j] = acc;
    }
    for (int i = 0; i < N; ++i)
      for (int j = 0; j < N; ++j) G[i * N + j] = G[i * N + j] * w[j] + dsa[i] * a[j];
  }
  if (dS_init) std::memcpy(dS_init, G.data(), NN * sizeof(F));
}

// Runs fn(head) for head = 0..BH-1 on up to nthreads workers.
template <typename Fn>
int for_heads(int BH, int nthreads, Fn fn) {
  if (nthreads <= 0) nthreads = static_cast<int>(std::thread::hardware_concurrency());
  if (nthreads <= 0) nthreads = 1;
  if (nthreads > BH) nthreads = BH;
  std::vector<int> status(nthreads, 0);
  auto worker = [&](int tid) {
    try {
      for (int hd = tid; hd < BH; hd += nthreads) fn(hd);
    } catch (const std::bad_alloc&) {
      status[tid] = -1;
    } catch (...) {
      status[tid] = -3;
    }
  };
  std::vector<std::thread> pool;
  try {
    for (int t = 1; t < nthreads; ++t) pool.emplace_back(worker, t);
  } catch (...) {
    for (auto& th : pool) th.join();
    return -1;
  }
  worker(0);
  for (auto& th : pool) th.join();
  for (int s : status)
    if (s) return s;
  return 0;
}

template <typename F>
int forward_all(const F* r, const F* w, const F* k, const F* v, const F* a, const F* b,
                const F* s_init, F* y, F* s_final, int B, int T, int H, int N, int nthreads) {
  if (!r || !w || !k || !v || !a || !b) return -2;
  if (B <= 0 || T <= 0 || H <= 0 || N <= 0) return -2;
  const std::size_t NN = static_cast<std::size_t>(N) * N;
  return for_heads(B * H, nthreads, [&](int hd) {
    const int bi = hd / H, hi = hd % H;
    HeadView<F> hv = head_view<F>(r, w, k, v, a, b, nullptr, bi, hi, T, H, N);
    std::vector<F> S(NN, F(0));
    if (s_init) std::memcpy(S.data(), s_init + hd * NN, NN * sizeof(F));
    F* yh = y ? y + (static_cast<std::size_t>(bi) * T * H + hi) * N : nullptr;
    forward_head(hv, S.data(), yh, hv.stride, T, N);
    if (s_final) std::memcpy(s_final + hd * NN, S.data(), NN * sizeof(F));
  });
}

template <typename F>
int backward_all(const F* r, const F* w, const F* k, const F* v, const F* a, const F* b,
                 const F* dy, const F* s_init, const F* dS_final, F* dr, F* dw, F* dk, F* dv,
                 F* da, F* db, F* dS_init, int B, int T, int H, int N, int nthreads) {
  if (!r || !w || !k || !v || !a || !b || !dy) return -2;
  if (!dr || !dw || !dk || !dv || !da || !db) return -2;
  if (B <= 0 || T <= 0 || H <= 0 || N <= 0) return -2;
  const std::size_t NN = static_cast<std::size_t>(N) * N;
  return for_heads(B * H, nthreads, [&](int hd) {
    const int bi = hd / H, hi = hd % H;
    HeadView<F> hv = head_view<F>(r, w, k, v, a, b, dy, bi, hi, T, H, N);
    const std::size_t off = (static_cast<std::size_t>(bi) * T * H + hi) * N;
    HeadGrads<F> g{dr + off, dw + off, dk + off, dv + off, da + off, db + off};
    backward_head(hv, s_init ? s_init + hd * NN : nullptr, dS_final ? dS_final + hd * NN : nullptr, g,
                  dS_init ? dS_init + hd * NN : nullptr, T, N);
  });
}

}  // namespace

extern "C" {

// All pointers are host memory. s_init may be NULL (zero initial state),
// dS_final may be NULL (no gradient into the final state); y, s_final and
// dS_init may be NULL (not written). Returns 0, -1 when a
// cache cannot be allocated, -2 on an invalid argument. nthreads <= 0 uses
// every hardware thread.
int oracle_wkv7_forward_f64(const double* r, const double* w, const double* k,
                            const double* v, const double* a, const double* b,
                            const double* s_init, double* y, double* s_final,
                            int B, int T, int H, int N, int nthreads) {
  return forward_all(r, w, k, v, a, b, s_init, y, s_final, B, T, H, N, nthreads);
}

int oracle_wkv7_backward_f64(const double* r, const double* w, const double* k,
                             const double* v, const double* a, const double* b,
                             const double* dy, const double* s_init, const double* dS_final,
                             double* dr, double* dw, double* dk, double* dv, double* da,
                             double* db, double* dS_init, int B, int T, int H, int N,
                             int nthreads) {
  return backward_all(r, w, k, v, a, b, dy, s_init, dS_final, dr, dw, dk, dv, da, db, dS_init,
                      B, T, H, N, nthreads);
}

int oracle_wkv7_forward_f32(const float* r, const float* w, const float* k, const float* v,
                            const float* a, const float* b, const float* s_init, float* y,
                            float* s_final, int B, int T, int H, int N, int nthreads) {
  return forward_all(r, w, k, v, a, b, s_init, y, s_final, B, T, H, N, nthreads);
}

int oracle_wkv7_backward_f32(const float* r, const float* w, const float* k, const float* v,
                             const float* a, const float* b, const float* dy,
                             const float* s_init, const float* dS_final, float* dr, float* dw,
                             float* dk, float* dv, float* da, float* db, float* dS_init, int B,
                             int T, int H, int N, int nthreads) {
  return backward_all(r, w, k, v, a, b, dy, s_init, dS_final, dr, dw, dk, dv, da, db, dS_init,
                      B, T, H, N, nthreads);
}

}  // extern "C"
