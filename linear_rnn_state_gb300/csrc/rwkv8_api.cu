// C ABI of the RWKV-8 normalized recurrence (rwkv8.h): argument validation,
// the backward's workspaces (checkpoints when none are given, the per-(b, h)
// decay terms, the per-head value terms of a shared value row) and launches.
#include <cstdarg>
#include <cstdio>
#include <cstdlib>

#include "rwkv8.h"
#include "rwkv8_launch.h"
#include "wkv7_launch.h"

namespace rwkv8 {
namespace {

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  return wkv7::api_fail(code, buf);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_dims(int B, int T, int H, int Hv, int L, int E) {
  if (B < 0 || T < 0 || H < 0) return fail(WKV7_ERR_INVALID, "B, T and H must be >= 0 (got %d, %d, %d)", B, T, H);
  if (L != kL || E != kE) return fail(WKV7_ERR_INVALID, "L and E must be 64 (got %d, %d)", L, E);
  if (Hv != 1 && Hv != H) return fail(WKV7_ERR_INVALID, "value heads must be 1 or H (got %d, H = %d)", Hv, H);
  const unsigned long long heads = (unsigned long long)B * H;
  if (heads >= (1ull << 28)) return fail(WKV7_ERR_INVALID, "B*H too large");
  if (heads * (unsigned long long)T * kL * 4ull >= (1ull << 46)) return fail(WKV7_ERR_INVALID, "B*H*T too large");
  return WKV7_OK;
}

struct Span {
  const void* p;
  size_t bytes;
  const char* name;
};

bool overlaps(const Span& x, const Span& y) {
  if (!x.p || !y.p || !x.bytes || !y.bytes) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(x.p), a1 = a0 + x.bytes;
  const uintptr_t b0 = reinterpret_cast<uintptr_t>(y.p), b1 = b0 + y.bytes;
  return a0 < b1 && b0 < a1;
}

int check_spans(const Span* ins, int nin, const Span* outs, int nout, int required_in, int required_out) {
  for (int i = 0; i < nin; ++i) {
    if (i < required_in && !ins[i].p && ins[i].bytes) return fail(WKV7_ERR_INVALID, "%s must not be NULL", ins[i].name);
    if (ins[i].p && !aligned16(ins[i].p)) return fail(WKV7_ERR_INVALID, "%s is not 16-byte aligned", ins[i].name);
  }
  for (int o = 0; o < nout; ++o) {
    if (o < required_out && !outs[o].p && outs[o].bytes)
      return fail(WKV7_ERR_INVALID, "%s must not be NULL", outs[o].name);
    if (outs[o].p && !aligned16(outs[o].p)) return fail(WKV7_ERR_INVALID, "%s is not 16-byte aligned", outs[o].name);
    for (int i = 0; i < nin; ++i)
      if (overlaps(outs[o], ins[i])) return fail(WKV7_ERR_INVALID, "%s overlaps input %s", outs[o].name, ins[i].name);
    for (int q = 0; q < o; ++q)
      if (overlaps(outs[o], outs[q])) return fail(WKV7_ERR_INVALID, "%s overlaps output %s", outs[o].name, outs[q].name);
  }
  return WKV7_OK;
}

// RWKV8_SEQUENTIAL=1 selects the kernels that walk each (b, h) through its
// chunks in one CTA; by default the forward's chain runs alone and its
// per-chunk work runs for every chunk at once. The backward walks each (b, h)
// through its chunks in one CTA unless RWKV8_SPLIT_BACKWARD=1 selects its
// split form (the carried gradients alone, then every chunk at once), which
// measured slower.
bool sequential() {
  const char* s = std::getenv("RWKV8_SEQUENTIAL");
  return s && s[0] == '1';
}
bool split_backward() {
  const char* s = std::getenv("RWKV8_SPLIT_BACKWARD");
  return s && s[0] == '1' && !sequential();
}

// A stream-ordered workspace (WKV7_FAIL_ALLOC=1 makes the allocation fail, for tests).
int take_workspace(unsigned char** ws, size_t bytes, cudaStream_t stream) {
  const char* inject = std::getenv("WKV7_FAIL_ALLOC");
  if (inject && inject[0] == '1')
    return fail(WKV7_ERR_ALLOC, "workspace allocation failed (injected by WKV7_FAIL_ALLOC)");
  cudaError_t e = cudaMallocAsync(reinterpret_cast<void**>(ws), bytes, stream);
  if (e != cudaSuccess) {
    cudaGetLastError();
    *ws = nullptr;
    return fail(WKV7_ERR_ALLOC, "workspace of %zu bytes: %s", bytes, cudaGetErrorString(e));
  }
  return WKV7_OK;
}

// Frees a workspace (if any) after the launches that use it, reporting the
// first launch error `e` or the free's own.
int release_workspace(unsigned char* ws, cudaError_t e, const char* what, cudaStream_t stream) {
  const cudaError_t e2 = ws ? cudaFreeAsync(ws, stream) : cudaSuccess;
  if (e != cudaSuccess) return fail(WKV7_ERR_CUDA, "%s launch: %s", what, cudaGetErrorString(e));
  if (e2 != cudaSuccess) return fail(WKV7_ERR_CUDA, "cudaFreeAsync(workspace): %s", cudaGetErrorString(e2));
  return WKV7_OK;
}

size_t ckpt_bytes(int B, int T, int H) {
  return ((size_t)B * H * nchunks(T) * kL * kE + (size_t)B * H * nchunks(T) * kL) * sizeof(float);
}

// Copies (or zeroes) an initial state into a final one for T = 0.
int pass_state(const float* src, float* dst, size_t bytes, cudaStream_t s) {
  if (!dst || !bytes) return WKV7_OK;
  cudaError_t e = src ? cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, s) : cudaMemsetAsync(dst, 0, bytes, s);
  if (e != cudaSuccess) return fail(WKV7_ERR_CUDA, "state copy: %s", cudaGetErrorString(e));
  return WKV7_OK;
}

int forward_impl(const float* q, const float* v, const float* decay, const float* rho_init, const float* rho_norm_init,
                 float* y, float* rho_final, float* rho_norm_final, float* ckpt, int B, int T, int H, int Hv, int L,
                 int E, cudaStream_t stream) {
  int rc = check_dims(B, T, H, Hv, L, E);
  if (rc) return rc;
  const size_t seq = (size_t)B * H * T * kL * 4, vseq = (size_t)B * Hv * T * kE * 4;
  const size_t st = (size_t)B * H * kL * kE * 4, nst = (size_t)B * H * kL * 4;
  const Span ins[] = {{q, seq, "q"},
                      {v, vseq, "v"},
                      {decay, (size_t)H * kL * 4, "decay"},
                      {rho_init, st, "rho_init"},
                      {rho_norm_init, nst, "rho_norm_init"}};
  const Span outs[] = {{y, (size_t)B * H * T * kE * 4, "y"},
                       {rho_final, st, "rho_final"},
                       {rho_norm_final, nst, "rho_norm_final"},
                       {ckpt, ckpt_bytes(B, T, H), "ckpt"}};
  if ((size_t)B * H == 0) return WKV7_OK;  // nothing to read or write
  if ((rc = check_spans(ins, 5, outs, 4, 3, 1))) return rc;
  if (T == 0) {
    if ((rc = pass_state(rho_init, rho_final, st, stream))) return rc;
    return pass_state(rho_norm_init, rho_norm_final, nst, stream);
  }
  Args a{};
  a.q = q, a.v = v, a.decay = decay, a.rho_init = rho_init, a.rho_norm_init = rho_norm_init;
  a.y = y, a.rho_final = rho_final, a.rho_norm_final = rho_norm_final, a.ckpt = ckpt;
  a.B = B, a.T = T, a.H = H, a.Hv = Hv;
  if (sequential()) {
    cudaError_t e = launch_forward(a, stream);
    if (e != cudaSuccess) return fail(WKV7_ERR_CUDA, "forward launch: %s", cudaGetErrorString(e));
    return WKV7_OK;
  }
  // The per-chunk readout starts from the checkpoints: without a buffer from
  // the caller they go to a workspace.
  unsigned char* ws = nullptr;
  if (y && !ckpt) {
    if ((rc = take_workspace(&ws, ckpt_bytes(B, T, H), stream))) return rc;
    a.ckpt = reinterpret_cast<float*>(ws);
  }
  cudaError_t e = launch_state(a, stream);
  if (e == cudaSuccess && y) e = launch_forward_chunks(a, stream);
  return release_workspace(ws, e, "forward", stream);
}

int backward_impl(const float* q, const float* v, const float* decay, const float* dy, const float* rho_init,
                  const float* rho_norm_init, const float* d_rho_final, const float* d_rho_norm_final,
                  const float* ckpt, float* dq, float* dv, float* ddecay, float* d_rho_init, float* d_rho_norm_init,
                  int B, int T, int H, int Hv, int L, int E, cudaStream_t stream) {
  int rc = check_dims(B, T, H, Hv, L, E);
  if (rc) return rc;
  const size_t seq = (size_t)B * H * T * kL * 4, vseq = (size_t)B * Hv * T * kE * 4;
  const size_t st = (size_t)B * H * kL * kE * 4, nst = (size_t)B * H * kL * 4;
  const Span ins[] = {{q, seq, "q"},
                      {v, vseq, "v"},
                      {decay, (size_t)H * kL * 4, "decay"},
                      {dy, (size_t)B * H * T * kE * 4, "dy"},
                      {rho_init, st, "rho_init"},
                      {rho_norm_init, nst, "rho_norm_init"},
                      {d_rho_final, st, "d_rho_final"},
                      {d_rho_norm_final, nst, "d_rho_norm_final"},
                      {ckpt, ckpt_bytes(B, T, H), "ckpt"}};
  const Span outs[] = {{dq, seq, "dq"},
                       {dv, vseq, "dv"},
                       {ddecay, (size_t)H * kL * 4, "ddecay"},
                       {d_rho_init, st, "d_rho_init"},
                       {d_rho_norm_init, nst, "d_rho_norm_init"}};
  if ((rc = check_spans(ins, 9, outs, 5, 4, 3))) return rc;
  if ((size_t)H == 0) return WKV7_OK;
  if ((size_t)B == 0 || T == 0) {
    // No step: ddecay is an empty sum, the initial-state gradients are the
    // final-state ones.
    cudaError_t e = cudaMemsetAsync(ddecay, 0, (size_t)H * kL * 4, stream);
    if (e != cudaSuccess) return fail(WKV7_ERR_CUDA, "ddecay clear: %s", cudaGetErrorString(e));
    if ((rc = pass_state(d_rho_final, d_rho_init, st, stream))) return rc;
    return pass_state(d_rho_norm_final, d_rho_norm_init, nst, stream);
  }

  // Workspace: [checkpoints if none given][ddecay terms per (b, h)][dv terms per head if Hv = 1]
  // and, for the split form, [G15][R0][Gn15][<G15, rho0>][ddecay terms per chunk], per (b, h) and chunk.
  auto pad = [](size_t x) { return (x + 255) / 256 * 256; };
  const bool split = split_backward();
  const size_t tasks = (size_t)B * H * nchunks(T);
  const size_t ck_ws = ckpt ? 0 : pad(ckpt_bytes(B, T, H));
  const size_t dd_ws = pad((size_t)B * H * kL * 4);
  const size_t dv_ws = Hv == 1 && H > 1 ? pad((size_t)B * H * T * kE * 4) : 0;
  const size_t g15_ws = split ? pad(tasks * kL * kE * 4) : 0;
  const size_t r0_ws = split ? pad(tasks * kC * kL * 4) : 0;
  const size_t vec_ws = split ? pad(tasks * kL * 4) : 0;  // each of Gn15, <G15, rho0>, ddecay terms
  const size_t ws_bytes = ck_ws + dd_ws + dv_ws + g15_ws + r0_ws + 3 * vec_ws;
  const char* inject = std::getenv("WKV7_FAIL_ALLOC");
  if (inject && inject[0] == '1')
    return fail(WKV7_ERR_ALLOC, "workspace allocation failed (injected by WKV7_FAIL_ALLOC)");
  unsigned char* ws = nullptr;
  cudaError_t e = cudaMallocAsync(reinterpret_cast<void**>(&ws), ws_bytes, stream);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(WKV7_ERR_ALLOC, "backward workspace of %zu bytes: %s", ws_bytes, cudaGetErrorString(e));
  }
  Args a{};
  a.q = q, a.v = v, a.decay = decay, a.dy = dy;
  a.B = B, a.T = T, a.H = H, a.Hv = Hv;
  if (!ckpt) {
    Args f = a;
    f.rho_init = rho_init, f.rho_norm_init = rho_norm_init;
    f.ckpt = reinterpret_cast<float*>(ws);
    f.y = nullptr;  // checkpoints only
    e = sequential() ? launch_forward(f, stream) : launch_state(f, stream);
    if (e != cudaSuccess) {
      cudaFreeAsync(ws, stream);
      return fail(WKV7_ERR_CUDA, "checkpointing forward launch: %s", cudaGetErrorString(e));
    }
  }
  a.ckpt = ckpt ? const_cast<float*>(ckpt) : reinterpret_cast<float*>(ws);
  a.d_rho_final = d_rho_final, a.d_rho_norm_final = d_rho_norm_final;
  a.dq = dq;
  unsigned char* p = ws + ck_ws;
  a.ddecay_bh = reinterpret_cast<float*>(p);
  p += dd_ws;
  a.dv = dv_ws ? reinterpret_cast<float*>(p) : dv;
  p += dv_ws;
  a.d_rho_init = d_rho_init, a.d_rho_norm_init = d_rho_norm_init;
  if (split) {
    a.g15 = reinterpret_cast<float*>(p);
    p += g15_ws;
    a.r0 = reinterpret_cast<float*>(p);
    p += r0_ws;
    a.gn15 = reinterpret_cast<float*>(p);
    a.gdot = reinterpret_cast<float*>(p + vec_ws);
    a.ddecay_part = reinterpret_cast<float*>(p + 2 * vec_ws);
    e = launch_backward_chain(a, stream);
    if (e == cudaSuccess) e = launch_backward_chunks(a, stream);
    if (e == cudaSuccess) e = launch_chunk_sum(a, stream);
  } else {
    e = launch_backward(a, stream);
  }
  if (e == cudaSuccess) e = launch_group_sum(a.ddecay_bh, ddecay, (size_t)H * kL, (size_t)H * kL, B, stream);
  if (e == cudaSuccess && dv_ws) e = launch_head_sum(a.dv, dv, B, H, T, stream);
  cudaError_t e2 = cudaFreeAsync(ws, stream);
  if (e != cudaSuccess) return fail(WKV7_ERR_CUDA, "backward launch: %s", cudaGetErrorString(e));
  if (e2 != cudaSuccess) return fail(WKV7_ERR_CUDA, "cudaFreeAsync(workspace): %s", cudaGetErrorString(e2));
  return WKV7_OK;
}

}  // namespace
}  // namespace rwkv8

extern "C" {

size_t rwkv8_ckpt_bytes(int B, int T, int H, int L, int E) {
  if (B < 0 || T < 0 || H < 0 || L != rwkv8::kL || E != rwkv8::kE) return 0;
  return rwkv8::ckpt_bytes(B, T, H);
}

int rwkv8_forward(const float* q, const float* v, const float* decay, const float* rho_init,
                  const float* rho_norm_init, float* y, float* rho_final, float* rho_norm_final, float* ckpt,
                  int B, int T, int H, int Hv, int L, int E, void* stream) {
  return rwkv8::forward_impl(q, v, decay, rho_init, rho_norm_init, y, rho_final, rho_norm_final, ckpt, B, T, H, Hv,
                             L, E, static_cast<cudaStream_t>(stream));
}

int rwkv8_backward(const float* q, const float* v, const float* decay, const float* dy, const float* rho_init,
                   const float* rho_norm_init, const float* d_rho_final, const float* d_rho_norm_final,
                   const float* ckpt, float* dq, float* dv, float* ddecay, float* d_rho_init,
                   float* d_rho_norm_init, int B, int T, int H, int Hv, int L, int E, void* stream) {
  return rwkv8::backward_impl(q, v, decay, dy, rho_init, rho_norm_init, d_rho_final, d_rho_norm_final, ckpt, dq, dv,
                              ddecay, d_rho_init, d_rho_norm_init, B, T, H, Hv, L, E,
                              static_cast<cudaStream_t>(stream));
}

}  // extern "C"
