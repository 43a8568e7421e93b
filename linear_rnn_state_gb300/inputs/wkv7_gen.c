/*
 * Seeded synthetic inputs for the WKV7 scan (r, w, k, v, a, b, dy, s_init)
 * and, at the end of the file, for the RWKV-8 normalized recurrence.
 *
 * This module draws random numbers and shapes them into the six recurrence
 * inputs, the upstream gradient dy and the optional initial state. It holds
 * none of the recurrence's arithmetic; the CUDA path and the CPU oracle both
 * consume the buffers it fills, and neither shares any other code.
 *
 * Random source: splitmix64 (Steele, Lea and Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014; the 64-bit mixing function
 * with the 0x9E3779B97F4A7C15 increment). Output m (m = 0, 1, ...) of a
 * generator seeded with s is mix(s + (m + 1) * 0x9E3779B97F4A7C15), so any
 * draw can be computed on its own and the fill runs on many threads.
 *
 * Value semantics (the RWKV-7 time-mix, rx_pretrain.c "tm_pre_forward"):
 *   r, k, v = n / sqrt(N)
 *   w       = exp(-0.606531 * sigmoid(z))         (decay coefficient e^-0.5)
 *   kk      = x / (||x||_2 + 1e-12) per (b, t, h) row of N
 *   a       = -kk,  b = kk * sigmoid(u)
 *   dy      = n,    s_init = std * n  (optional)
 * with n, z, x, u standard normals from Box-Muller (cosine branch; normal
 * number q uses uniforms 2q and 2q + 1, u = ((x >> 11) + 1) * 2^-53 in (0, 1]).
 * Streams, each M = B*T*H*N normals long, in this order: r, k, v, z, x, u,
 * dy; s_init follows with B*H*N*N normals. Everything is computed in double
 * and rounded once (round to nearest even) to the requested storage type.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define GOLDEN_GAMMA 0x9E3779B97F4A7C15ULL
#define WDECAY_COEFF 0.606531

enum { OUT_F64 = 0, OUT_F32 = 1, OUT_BF16 = 2 };

static inline uint64_t sm64_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

/* Output number m of splitmix64 seeded with `seed`. */
uint64_t wkv7_gen_splitmix64_at(uint64_t seed, uint64_t m) {
  return sm64_mix(seed + (m + 1) * GOLDEN_GAMMA);
}

/* Uniform in (0, 1]: the top 53 bits plus one, scaled by 2^-53. */
double wkv7_gen_uniform_at(uint64_t seed, uint64_t m) {
  return (double)((wkv7_gen_splitmix64_at(seed, m) >> 11) + 1) * (1.0 / 9007199254740992.0);
}

/* Standard normal number q (Box-Muller, cosine branch). */
double wkv7_gen_normal_at(uint64_t seed, uint64_t q) {
  const double u1 = wkv7_gen_uniform_at(seed, 2 * q);
  const double u2 = wkv7_gen_uniform_at(seed, 2 * q + 1);
  return sqrt(-2.0 * log(u1)) * cos(6.283185307179586476925286766559 * u2);
}

/* Round a double to bfloat16 (1-8-7) with round-to-nearest-even, directly
 * from the double (no intermediate float, so no double rounding). Values
 * beyond the bf16 range become +-inf; NaN stays NaN. Subnormal results are
 * not produced by this generator's value ranges and are flushed to zero. */
uint16_t wkv7_gen_bf16_rne(double x) {
  uint64_t bits;
  memcpy(&bits, &x, sizeof bits);
  const uint16_t sign = (uint16_t)((bits >> 48) & 0x8000u);
  const int exp = (int)((bits >> 52) & 0x7FF);
  uint64_t man = bits & ((1ULL << 52) - 1);
  if (exp == 0x7FF) return (uint16_t)(sign | 0x7F80u | (man ? 0x40u : 0u));
  int e = exp - 1023 + 127; /* bf16 / fp32 biased exponent */
  if (exp == 0 || e <= 0) return sign;
  /* keep 7 mantissa bits, round the remaining 45 to nearest even */
  uint64_t keep = man >> 45;
  const uint64_t rest = man & ((1ULL << 45) - 1);
  const uint64_t half = 1ULL << 44;
  if (rest > half || (rest == half && (keep & 1))) {
    keep += 1;
    if (keep == 128) { keep = 0; e += 1; }
  }
  if (e >= 255) return (uint16_t)(sign | 0x7F80u);
  return (uint16_t)(sign | (uint16_t)(e << 7) | (uint16_t)keep);
}

static inline void store(void *dst, int kind, size_t idx, double x) {
  if (kind == OUT_F64) ((double *)dst)[idx] = x;
  else if (kind == OUT_F32) ((float *)dst)[idx] = (float)x;
  else ((uint16_t *)dst)[idx] = wkv7_gen_bf16_rne(x);
}

static inline double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

typedef struct {
  uint64_t seed;
  int B, T, H, N, kind;
  double s_init_std;
  void *r, *w, *k, *v, *a, *b, *dy, *s_init;
  size_t row_begin, row_end;   /* (b, t, h) rows */
  size_t srow_begin, srow_end; /* (b, h, i) state rows */
} fill_job;

static void *fill_worker(void *arg) {
  fill_job *J = (fill_job *)arg;
  const size_t N = (size_t)J->N;
  const uint64_t M = (uint64_t)J->B * J->T * J->H * N;
  const double inv_sqrt_n = 1.0 / sqrt((double)N);
  double x[256];
  for (size_t row = J->row_begin; row < J->row_end; ++row) {
    const size_t base = row * N;
    for (size_t n = 0; n < N; ++n) {
      const uint64_t f = base + n;
      store(J->r, J->kind, f, wkv7_gen_normal_at(J->seed, 0 * M + f) * inv_sqrt_n);
      store(J->k, J->kind, f, wkv7_gen_normal_at(J->seed, 1 * M + f) * inv_sqrt_n);
      store(J->v, J->kind, f, wkv7_gen_normal_at(J->seed, 2 * M + f) * inv_sqrt_n);
      const double z = wkv7_gen_normal_at(J->seed, 3 * M + f);
      store(J->w, J->kind, f, exp(-WDECAY_COEFF * sigmoid(z)));
      x[n] = wkv7_gen_normal_at(J->seed, 4 * M + f);
      store(J->dy, J->kind, f, wkv7_gen_normal_at(J->seed, 6 * M + f));
    }
    double ss = 0.0;
    for (size_t n = 0; n < N; ++n) ss += x[n] * x[n];
    const double inv = 1.0 / (sqrt(ss) + 1e-12);
    for (size_t n = 0; n < N; ++n) {
      const uint64_t f = base + n;
      const double kk = x[n] * inv;
      const double u = wkv7_gen_normal_at(J->seed, 5 * M + f);
      store(J->a, J->kind, f, -kk);
      store(J->b, J->kind, f, kk * sigmoid(u));
    }
  }
  if (J->s_init) {
    for (size_t srow = J->srow_begin; srow < J->srow_end; ++srow) {
      for (size_t j = 0; j < N; ++j) {
        const uint64_t f = srow * N + j;
        ((double *)J->s_init)[f] = J->s_init_std * wkv7_gen_normal_at(J->seed, 7 * M + f);
      }
    }
  }
  return NULL;
}

/*
 * Fill the inputs of one workload.
 *   kind: 0 = double, 1 = float, 2 = bfloat16 (uint16 bit patterns) for
 *         r, w, k, v, a, b, dy, each [B][T][H][N] row-major.
 *   s_init: NULL to skip, else a double [B][H][N][N] buffer filled with
 *         s_init_std * normal (callers round it to their state type).
 *   nthreads <= 0 uses every online core.
 * Returns 0, or -2 on an invalid argument, -1 if a thread cannot start.
 */
int wkv7_gen_inputs(uint64_t seed, int B, int T, int H, int N, int kind,
                    void *r, void *w, void *k, void *v, void *a, void *b, void *dy,
                    double *s_init, double s_init_std, int nthreads) {
  if (B <= 0 || T <= 0 || H <= 0 || N <= 0 || N > 256) return -2;
  if (kind < 0 || kind > 2) return -2;
  if (!r || !w || !k || !v || !a || !b || !dy) return -2;
  if (nthreads <= 0) {
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    nthreads = n > 0 ? (int)n : 1;
  }
  if (nthreads > 256) nthreads = 256;
  const size_t rows = (size_t)B * T * H;
  const size_t srows = (size_t)B * H * N;
  if ((size_t)nthreads > rows) nthreads = (int)rows;
  fill_job jobs[256];
  pthread_t tids[256];
  int started = 0, rc = 0;
  for (int i = 0; i < nthreads; ++i) {
    fill_job *J = &jobs[i];
    J->seed = seed; J->B = B; J->T = T; J->H = H; J->N = N; J->kind = kind;
    J->s_init_std = s_init_std;
    J->r = r; J->w = w; J->k = k; J->v = v; J->a = a; J->b = b; J->dy = dy;
    J->s_init = s_init;
    J->row_begin = rows * i / nthreads;
    J->row_end = rows * (i + 1) / nthreads;
    J->srow_begin = srows * i / nthreads;
    J->srow_end = srows * (i + 1) / nthreads;
  }
  for (int i = 1; i < nthreads; ++i) {
    if (pthread_create(&tids[i], NULL, fill_worker, &jobs[i]) != 0) { rc = -1; break; }
    started = i;
  }
  fill_worker(&jobs[0]);
  for (int i = 1; i <= started; ++i) pthread_join(tids[i], NULL);
  return rc;
}

/*
 * Seeded synthetic inputs for the RWKV-8 normalized recurrence (the
 * burn_dragon_kernel page "src/sequence/rwkv8/backward.rs"), in double.
 *
 * Value semantics (the page gives no value ranges; these are readings):
 *   q      = max(n, 0)                        non-negative query weights
 *   v      = n / sqrt(E)
 *   decay  = exp(-0.606531 * sigmoid(z))       the RWKV-7 decay range (0.545, 1)
 *   dy     = n
 *   rho_init      = std * n        (optional)
 *   rho_norm_init = std * |n|      (optional; a running sum of q is >= 0)
 *   d_rho_final   = n, d_rho_norm_final = n   (optional)
 * Streams, in this order, each as long as its array: q [B][H][T][L],
 * v [B][Hv][T][E], z [H][L], dy [B][H][T][E], rho_init [B][H][L][E],
 * rho_norm_init [B][H][L], d_rho_final [B][H][L][E], d_rho_norm_final
 * [B][H][L]; stream s starts at normal number (sum of the earlier lengths),
 * so every array is the same whichever optional arrays are asked for.
 */
typedef struct {
  uint64_t seed, base;
  double *out;
  size_t begin, end;
  int kind; /* 0 plain normal, 1 max(n, 0), 2 n * scale, 3 |n| * scale, 4 decay */
  double scale;
} rwkv8_job;

static void *rwkv8_worker(void *arg) {
  rwkv8_job *J = (rwkv8_job *)arg;
  for (size_t f = J->begin; f < J->end; ++f) {
    const double n = wkv7_gen_normal_at(J->seed, J->base + f);
    double x;
    switch (J->kind) {
      case 1: x = n > 0.0 ? n : 0.0; break;
      case 2: x = n * J->scale; break;
      case 3: x = fabs(n) * J->scale; break;
      case 4: x = exp(-WDECAY_COEFF * sigmoid(n)); break;
      default: x = n; break;
    }
    J->out[f] = x;
  }
  return NULL;
}

static int rwkv8_fill(uint64_t seed, uint64_t base, double *out, size_t count, int kind, double scale,
                      int nthreads) {
  if (!out || count == 0) return 0;
  rwkv8_job jobs[256];
  pthread_t tids[256];
  if ((size_t)nthreads > count) nthreads = (int)count;
  for (int i = 0; i < nthreads; ++i) {
    jobs[i].seed = seed; jobs[i].base = base; jobs[i].out = out;
    jobs[i].begin = count * i / nthreads; jobs[i].end = count * (i + 1) / nthreads;
    jobs[i].kind = kind; jobs[i].scale = scale;
  }
  int started = 0, rc = 0;
  for (int i = 1; i < nthreads; ++i) {
    if (pthread_create(&tids[i], NULL, rwkv8_worker, &jobs[i]) != 0) { rc = -1; break; }
    started = i;
  }
  rwkv8_worker(&jobs[0]);
  for (int i = 1; i <= started; ++i) pthread_join(tids[i], NULL);
  return rc;
}

/*
 * Fill the RWKV-8 inputs. q, v, decay and dy are required; the four state
 * arrays may be NULL (not drawn). Returns 0, -2 on an invalid argument or -1
 * if a thread cannot start. nthreads <= 0 uses every online core.
 */
int rwkv8_gen_inputs(uint64_t seed, int B, int T, int H, int Hv, int L, int E, double *q, double *v,
                     double *decay, double *dy, double *rho_init, double *rho_norm_init, double state_std,
                     double *d_rho_final, double *d_rho_norm_final, int nthreads) {
  if (B <= 0 || T <= 0 || H <= 0 || L <= 0 || E <= 0 || (Hv != 1 && Hv != H)) return -2;
  if (!q || !v || !decay || !dy) return -2;
  if (nthreads <= 0) {
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    nthreads = n > 0 ? (int)n : 1;
  }
  if (nthreads > 256) nthreads = 256;
  const uint64_t nq = (uint64_t)B * H * T * L, nv = (uint64_t)B * Hv * T * E, nz = (uint64_t)H * L;
  const uint64_t ny = (uint64_t)B * H * T * E, ns = (uint64_t)B * H * L * E, nn = (uint64_t)B * H * L;
  uint64_t base = 0;
  int rc = 0;
  rc |= rwkv8_fill(seed, base, q, nq, 1, 1.0, nthreads); base += nq;
  rc |= rwkv8_fill(seed, base, v, nv, 2, 1.0 / sqrt((double)E), nthreads); base += nv;
  rc |= rwkv8_fill(seed, base, decay, nz, 4, 1.0, nthreads); base += nz;
  rc |= rwkv8_fill(seed, base, dy, ny, 0, 1.0, nthreads); base += ny;
  rc |= rwkv8_fill(seed, base, rho_init, ns, 2, state_std, nthreads); base += ns;
  rc |= rwkv8_fill(seed, base, rho_norm_init, nn, 3, state_std, nthreads); base += nn;
  rc |= rwkv8_fill(seed, base, d_rho_final, ns, 0, 1.0, nthreads); base += ns;
  rc |= rwkv8_fill(seed, base, d_rho_norm_final, nn, 0, 1.0, nthreads);
  return rc ? -1 : 0;
}

/*
 * The decay logits z [B][T][H][N] behind the w that wkv7_gen_inputs draws
 * (stream 3 of the same seed: w = exp(-0.606531 sigmoid(z)) there), rounded
 * once to the requested storage kind, for callers that pass the decay as
 * logits. Returns 0, or -2 on an invalid argument.
 */
int wkv7_gen_logits(uint64_t seed, int B, int T, int H, int N, int kind, void *z) {
  if (B <= 0 || T <= 0 || H <= 0 || N <= 0 || N > 256 || kind < 0 || kind > 2 || !z) return -2;
  const uint64_t M = (uint64_t)B * T * H * N;
  for (uint64_t f = 0; f < M; ++f) store(z, kind, (size_t)f, wkv7_gen_normal_at(seed, 3 * M + f));
  return 0;
}
