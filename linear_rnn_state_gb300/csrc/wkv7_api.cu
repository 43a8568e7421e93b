// C ABI of the WKV7 library: argument validation, TMA tensor-map encoding,
// the backward's optional checkpoint workspace, and the device status word.
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <mutex>
#include <string>

#include "wkv7.h"
#ifdef WKV7_DEBUG
#include "wkv7_debug.h"
#endif
#include "wkv7_common.cuh"
#include "wkv7_launch.h"

namespace wkv7 {
namespace {

__device__ unsigned g_status_word;

thread_local std::string t_last_error;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return code;
}

int fail_cuda(cudaError_t e, const char* what) {
  return fail(WKV7_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// ---------------------------------------------------------- validation ---

constexpr int kMaxDevices = 64;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_dims(int B, int T, int H, int N) {
  if (B < 0 || T < 0 || H < 0) return fail(WKV7_ERR_INVALID, "B, T and H must be >= 0 (got %d, %d, %d)", B, T, H);
  if (N != 16 && N != 32 && N != 64) return fail(WKV7_ERR_INVALID, "N must be 16, 32 or 64 (got %d)", N);
  // Grid sizes stay below 2^31 and tensor-map strides below 2^40 bytes.
  const unsigned long long heads = (unsigned long long)B * H;
  if (heads * (N / 16) >= (1ull << 31)) return fail(WKV7_ERR_INVALID, "B*H too large");
  const unsigned long long elems = heads * (unsigned long long)T * N;
  if (elems * 4ull >= (1ull << 40)) return fail(WKV7_ERR_INVALID, "B*T*H*N too large");
  return WKV7_OK;
}

struct Span {
  const void* p;
  size_t bytes;
  const char* name;
};

bool overlaps(const Span& x, const Span& y) {
  if (!x.p || !y.p) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(x.p), a1 = a0 + x.bytes;
  const uintptr_t b0 = reinterpret_cast<uintptr_t>(y.p), b1 = b0 + y.bytes;
  return a0 < b1 && b0 < a1;
}

// Required pointers non-null, every pointer 16-byte aligned, no output
// overlapping an input or another output.
int check_spans(const Span* ins, int nin, const Span* outs, int nout, int required_in, int required_out) {
  for (int i = 0; i < nin; ++i) {
    if (i < required_in && !ins[i].p) return fail(WKV7_ERR_INVALID, "%s must not be NULL", ins[i].name);
    if (ins[i].p && !aligned16(ins[i].p)) return fail(WKV7_ERR_INVALID, "%s is not 16-byte aligned", ins[i].name);
  }
  for (int o = 0; o < nout; ++o) {
    if (o < required_out && !outs[o].p) return fail(WKV7_ERR_INVALID, "%s must not be NULL", outs[o].name);
    if (outs[o].p && !aligned16(outs[o].p)) return fail(WKV7_ERR_INVALID, "%s is not 16-byte aligned", outs[o].name);
    for (int i = 0; i < nin; ++i)
      if (overlaps(outs[o], ins[i])) return fail(WKV7_ERR_INVALID, "%s overlaps input %s", outs[o].name, ins[i].name);
    for (int q = 0; q < o; ++q)
      if (overlaps(outs[o], outs[q])) return fail(WKV7_ERR_INVALID, "%s overlaps output %s", outs[o].name, outs[q].name);
  }
  return WKV7_OK;
}

size_t ckpt_bytes(int B, int T, int H, int N, int C) {
  const size_t nck = (size_t)(((long long)T + C - 1) / C);
  return (size_t)B * H * nck * N * N * sizeof(float);
}

// ------------------------------------------------------ device helpers ---

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// [B][T][H][N] tensor as a 4-D map (N, H, T, B) with a box of `steps` rows of
// one head; `swizzle128` lays the box out in shared memory with 128-byte
// swizzling (rows of N = 64 bf16 elements, as the tensor cores read them).
int make_map(CUtensorMap* map, const void* base, bool bf16, int B, int T, int H, int N, int steps,
             bool swizzle128 = false) {
  auto enc = encode_fn();
  if (!enc) return fail(WKV7_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  const cuuint64_t es = bf16 ? 2 : 4;
  cuuint64_t dims[4] = {(cuuint64_t)N, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
  cuuint64_t strides[3] = {N * es, (cuuint64_t)H * N * es, (cuuint64_t)T * H * N * es};
  cuuint32_t box[4] = {(cuuint32_t)N, 1, (cuuint32_t)steps, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4,
                   const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(WKV7_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return WKV7_OK;
}

// The split backward's carry workspace [B*H*nchunks][64][64] bf16 as a 3-D map
// (64, 64, B*H*nchunks), one carry per box, 128-byte swizzled.
int make_carry_map(CUtensorMap* map, const void* carry, size_t nblocks) {
  auto enc = encode_fn();
  if (!enc) return fail(WKV7_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  cuuint64_t dims[3] = {64, 64, (cuuint64_t)nblocks};
  cuuint64_t strides[2] = {64 * 2, 64 * 64 * 2};
  cuuint32_t box[3] = {64, 64, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(carry), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(WKV7_ERR_CUDA, "cuTensorMapEncodeTiled (carry) failed (%d)", (int)r);
  return WKV7_OK;
}

// Checkpoints [B*H*nck][N][N] fp32 as a 3-D map (N, N, B*H*nck), one state per box.
int make_ckpt_map(CUtensorMap* map, const float* ckpt, int B, int H, int N, int nck) {
  auto enc = encode_fn();
  if (!enc) return fail(WKV7_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  cuuint64_t dims[3] = {(cuuint64_t)N, (cuuint64_t)N, (cuuint64_t)B * H * nck};
  cuuint64_t strides[2] = {(cuuint64_t)N * 4, (cuuint64_t)N * N * 4};
  cuuint32_t box[3] = {(cuuint32_t)N, (cuuint32_t)N, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(ckpt), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(WKV7_ERR_CUDA, "cuTensorMapEncodeTiled (checkpoints) failed (%d)", (int)r);
  return WKV7_OK;
}

std::mutex g_status_mu;
unsigned* g_status_ptr[kMaxDevices];

// Device address of this library's status word on the current device.
int status_word(unsigned** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(WKV7_ERR_CUDA, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_status_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_status_word);
    if (e != cudaSuccess) return fail_cuda(e, "cudaGetSymbolAddress(status)");
    g_status_ptr[dev] = static_cast<unsigned*>(p);
  }
  *out = g_status_ptr[dev];
  return WKV7_OK;
}

#ifdef WKV7_DEBUG
// Debug build: set by the hooks of include/wkv7_debug.h.
std::atomic<int> g_debug_skip_last_load{0};
std::atomic<int> g_debug_out_kernel{0};
std::atomic<size_t> g_debug_extent_cut{0};
#endif

// The extent of a buffer as the kernels check it in the debug build: its size,
// less the bytes wkv7_debug_cut_extents asked to cut off its end.
Extent extent(const void* p, size_t bytes) {
#ifdef WKV7_DEBUG
  const size_t cut = g_debug_extent_cut.load();
  bytes = bytes > cut ? bytes - cut : 0;
#endif
  return Extent{p, p ? bytes : 0};
}

// The buffers of a forward launch, as the api validated them; the checkpoint
// buffer holds ck_bytes.
void set_extents(FwdArgs& a, int N, bool bf16, size_t ck_bytes) {
  const size_t vec = (size_t)a.B * a.T * a.H * N, st = (size_t)a.B * a.H * N * N * 4, par = (size_t)a.H * N * 4;
  for (int v = 0; v < 6; ++v) a.ext.in[v] = extent(a.in[v], vec * (bf16 ? 2 : 4));
  a.ext.y = extent(a.y, vec * (bf16 ? 2 : 4));
  a.ext.nv = extent(a.nv, vec * 2);
  a.ext.stats = extent(a.stats, (size_t)a.B * a.T * a.H * 2 * 4);
  a.ext.s_init = extent(a.s_init, st);
  a.ext.s_final = extent(a.s_final, st);
  a.ext.ckpt = extent(a.ckpt, ck_bytes);
  a.ext.ln_w = extent(a.ln_w, par);
  a.ext.ln_b = extent(a.ln_b, par);
  a.ext.r_k = extent(a.r_k, par);
}

// The buffers of a backward launch; the checkpoints take ck_bytes.
void set_extents(BwdArgs& a, int N, bool bf16, size_t ck_bytes) {
  const size_t vec = (size_t)a.B * a.T * a.H * N, st = (size_t)a.B * a.H * N * N * 4, par = (size_t)a.H * N * 4;
  const size_t nchunks = ((size_t)a.T + kChunk - 1) / kChunk;
  for (int v = 0; v < 7; ++v) a.ext.in[v] = extent(a.in[v], vec * (bf16 ? 2 : 4));
  a.ext.in[7] = extent(a.epi_nv, vec * 2);
  a.ext.ckpt = extent(a.ckpt, ck_bytes);
  a.ext.carry = extent(a.carry, a.carry ? bwd4_workspace_bytes(a.B, a.T, a.H, bf16) : 0);
  float* const g[6] = {a.dr, a.dw, a.dk, a.dv, a.da, a.db};
  Extent* const x[6] = {&a.ext.dr, &a.ext.dw, &a.ext.dk, &a.ext.dv, &a.ext.da, &a.ext.db};
  for (int q = 0; q < 6; ++q) *x[q] = extent(g[q], vec * 4);
  a.ext.dS_init = extent(a.dS_init, st);
  a.ext.dS_final = extent(a.dS_final, st);
  a.ext.stats = extent(a.epi_stats, (size_t)a.B * a.T * a.H * 2 * 4);
  a.ext.ln_w = extent(a.epi_ln_w, par);
  a.ext.r_k = extent(a.epi_r_k, par);
  a.ext.part = extent(a.epi_part, (size_t)a.B * a.H * nchunks * 3 * N * 4);
}

// ------------------------------------------------------------ forward ---

// The epilogue of wkv7_forward_epilogue_bf16 (null for the plain forward).
struct Epilogue {
  const float *ln_w, *ln_b, *r_k;
  void* nv;
  float* stats;
};

int forward_impl(bool bf16, const void* const in[6], const float* s_init, void* y, float* s_final,
                 float* ckpt, int C, int B, int T, int H, int N, cudaStream_t stream, bool logit = false,
                 const Epilogue* epi = nullptr) {
  int rc = check_dims(B, T, H, N);
  if (rc) return rc;
  if (ckpt && C < 1) return fail(WKV7_ERR_INVALID, "ckpt_every must be >= 1 (got %d)", C);
  if (logit && (N != 64 || (ckpt && C != kChunk)))
    return fail(WKV7_ERR_INVALID, "decay logits need N = 64 and ckpt_every = %d (got N = %d, %d)", kChunk, N, C);
  if (epi && (N != 64 || (ckpt && C != kChunk)))
    return fail(WKV7_ERR_INVALID, "the epilogue needs N = 64 and ckpt_every = %d (got N = %d, %d)", kChunk, N, C);
  const size_t es = bf16 ? 2 : 4;
  const size_t vec = (size_t)B * T * H * N * es;
  const size_t st = (size_t)B * H * N * N * 4;
  const Span ins[7] = {{in[0], vec, "r"}, {in[1], vec, "w"}, {in[2], vec, "k"}, {in[3], vec, "v"},
                       {in[4], vec, "a"}, {in[5], vec, "b"}, {s_init, st, "s_init"}};
  const Span outs[3] = {{y, vec, "y"}, {s_final, st, "s_final"},
                        {ckpt, ckpt ? ckpt_bytes(B, T, H, N, C) : 0, "ckpt"}};
  // Empty problems: nothing to scan. With T = 0 the final state is the
  // initial one; zero-sized vector buffers may be NULL.
  if ((size_t)B * H == 0) return WKV7_OK;
  if (T == 0) {
    rc = check_spans(ins + 6, 1, outs + 1, 1, 0, 0);
    if (rc) return rc;
    if (!s_final) return WKV7_OK;
    cudaError_t e = s_init ? cudaMemcpyAsync(s_final, s_init, st, cudaMemcpyDeviceToDevice, stream)
                           : cudaMemsetAsync(s_final, 0, st, stream);
    return e == cudaSuccess ? WKV7_OK : fail_cuda(e, "empty forward");
  }
  rc = check_spans(ins, 7, outs, 3, 6, 0);
  if (rc) return rc;
  if (epi) {
    const size_t par = (size_t)H * N * 4;
    const Span eins[10] = {ins[0], ins[1], ins[2], ins[3], ins[4], ins[5], ins[6],
                           {epi->ln_w, par, "ln_w"}, {epi->ln_b, par, "ln_b"}, {epi->r_k, par, "r_k"}};
    const Span eouts[5] = {outs[0], outs[1], outs[2], {epi->nv, vec, "nv"},
                           {epi->stats, (size_t)B * T * H * 2 * 4, "stats"}};
    if ((rc = check_spans(eins, 10, eouts, 5, 6, 1))) return rc;
    if (!epi->ln_w || !epi->ln_b || !epi->r_k) return fail(WKV7_ERR_INVALID, "ln_w, ln_b and r_k are required");
  }

  FwdArgs args;
  const int K = fwd_steps_per_stage(N, bf16);
  for (int v = 0; v < 6; ++v) {
    if ((rc = make_map(&args.map[v], in[v], bf16, B, T, H, N, K))) return rc;
    args.in[v] = in[v];
  }
  if ((rc = status_word(&args.status))) return rc;
  args.s_init = s_init;
  args.y = y;
  args.s_final = s_final;
  args.ckpt = ckpt;
  args.w_logit = logit ? 1 : 0;
  if (epi) {
    args.epilogue = 1;
    args.ln_w = epi->ln_w;
    args.ln_b = epi->ln_b;
    args.r_k = epi->r_k;
    args.nv = epi->nv;
    args.stats = epi->stats;
  }
#ifdef WKV7_DEBUG
  args.debug_skip_last_load = g_debug_skip_last_load.load();
#endif
  args.C = ckpt ? C : 1;
  args.nck = ckpt ? (T + C - 1) / C : 0;
  args.B = B;
  args.T = T;
  args.H = H;
  set_extents(args, N, bf16, ckpt ? ckpt_bytes(B, T, H, N, C) : 0);
  cudaError_t e = use_chunked_fwd(N, ckpt ? C : kChunk) ? launch_fwd3(args, bf16, stream) : launch_fwd2(args, bf16, N, stream);
  if (e != cudaSuccess) return fail_cuda(e, "forward launch");
  return WKV7_OK;
}

// ----------------------------------------------------------- backward ---

// Which chunked backward runs for bf16 inputs at N = 64 with 16-step
// checkpoints: the split pair (default) or the fused one-pass kernel.
enum class BwdForm { kAuto, kFused };

// The epilogue's backward fused into the split backward (wkv7_backward_epilogue_bf16):
// in[6] is then dout, and these are the epilogue's other inputs and the per-chunk
// parameter terms' workspace.
struct EpiBwd {
  const void* nv;
  const float *stats, *ln_w, *r_k;
  float* part;
};

int backward_impl(bool bf16, const void* const in[7], const float* s_init, const float* dS_final, const float* ckpt,
                  int C, float* const grads[6], float* dS_init, int B, int T, int H, int N, cudaStream_t stream,
                  bool logit = false, BwdForm form = BwdForm::kAuto, const EpiBwd* eb = nullptr) {
  int rc = check_dims(B, T, H, N);
  if (rc) return rc;
  if (ckpt && C < 1) return fail(WKV7_ERR_INVALID, "ckpt_every must be >= 1 (got %d)", C);
  const int C_eff = ckpt ? C : (C >= 1 ? C : bwd2_steps_per_window(N, bf16));
  if (logit && (N != 64 || C_eff != kChunk))
    return fail(WKV7_ERR_INVALID, "decay logits need N = 64 and ckpt_every = %d (got N = %d, %d)", kChunk, N, C_eff);
  if (form == BwdForm::kFused && (N != 64 || C_eff != kChunk))
    return fail(WKV7_ERR_INVALID, "the fused backward needs N = 64 and ckpt_every = %d (got N = %d, %d)", kChunk, N,
                C_eff);
  const size_t es = bf16 ? 2 : 4;
  const size_t vec = (size_t)B * T * H * N * es;
  const size_t gvec = (size_t)B * T * H * N * 4;
  const size_t st = (size_t)B * H * N * N * 4;
  const Span ins[10] = {{in[0], vec, "r"},  {in[1], vec, "w"},     {in[2], vec, "k"},
                       {in[3], vec, "v"},  {in[4], vec, "a"},     {in[5], vec, "b"},
                       {in[6], vec, "dy"}, {s_init, st, "s_init"}, {ckpt, ckpt ? ckpt_bytes(B, T, H, N, C) : 0, "ckpt"},
                       {dS_final, st, "dS_final"}};
  const Span outs[7] = {{grads[0], gvec, "dr"}, {grads[1], gvec, "dw"}, {grads[2], gvec, "dk"},
                        {grads[3], gvec, "dv"}, {grads[4], gvec, "da"}, {grads[5], gvec, "db"},
                        {dS_init, st, "dS_init"}};
  // Empty problems: no step runs, so the carried gradient stays zero.
  if ((size_t)B * H == 0) return WKV7_OK;
  if (T == 0) {  // no step: the gradient of the initial state is the one entering the final state
    const Span states[2] = {ins[7], ins[9]};
    rc = check_spans(states, 2, outs + 6, 1, 0, 0);
    if (rc) return rc;
    if (!dS_init) return WKV7_OK;
    cudaError_t e = dS_final ? cudaMemcpyAsync(dS_init, dS_final, st, cudaMemcpyDeviceToDevice, stream)
                             : cudaMemsetAsync(dS_init, 0, st, stream);
    return e == cudaSuccess ? WKV7_OK : fail_cuda(e, "empty backward");
  }
  rc = check_spans(ins, 10, outs, 7, 7, 6);
  if (rc) return rc;

  // bf16 inputs at N = 64 with 16-step checkpoints take a chunked tensor-core
  // backward: the split one (carry chain + parallel output pass), which keeps
  // the carry of every chunk in the workspace too, or, when the caller asks
  // for it (wkv7_backward_fused_bf16), the fused one (one CTA per head). fp32
  // inputs there take the split one in split bf16 (fp32 carries in the
  // workspace).
  const bool chunked = bf16 && N == 64 && C_eff == kChunk;
  const bool split = chunked && form != BwdForm::kFused;
  const bool split32 = !bf16 && N == 64 && C_eff == kChunk;
  const size_t ck_ws = ckpt ? 0 : (ckpt_bytes(B, T, H, N, C_eff) + 255) / 256 * 256;
  const size_t ws_bytes = ck_ws + (split || split32 ? bwd4_workspace_bytes(B, T, H, bf16) : 0);
  if (ws_bytes) {
    // Fault injection for tests: make the workspace allocation fail.
    const char* inject = std::getenv("WKV7_FAIL_ALLOC");
    if (inject && inject[0] == '1')
      return fail(WKV7_ERR_ALLOC, "workspace allocation failed (injected by WKV7_FAIL_ALLOC)");
  }

  BwdArgs args;
  const int KS = bwd2_steps_per_window(N, bf16);
  for (int v = 0; v < 7; ++v)
    if ((rc = make_map(&args.map[v], in[v], bf16, B, T, H, N, KS))) return rc;

  float* ws = nullptr;
  if (ws_bytes) {
    cudaError_t e = cudaMallocAsync(reinterpret_cast<void**>(&ws), ws_bytes, stream);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return fail(WKV7_ERR_ALLOC, "backward workspace of %zu bytes: %s", ws_bytes, cudaGetErrorString(e));
    }
  }
  if (!ckpt) {
    FwdArgs fa;
    const int K = fwd_steps_per_stage(N, bf16);
    for (int v = 0; v < 6; ++v) {
      if ((rc = make_map(&fa.map[v], in[v], bf16, B, T, H, N, K))) {
        cudaFreeAsync(ws, stream);
        return rc;
      }
      fa.in[v] = in[v];
    }
    if ((rc = status_word(&fa.status))) {
      cudaFreeAsync(ws, stream);
      return rc;
    }
    fa.s_init = s_init;
    fa.y = nullptr;
    fa.s_final = nullptr;
    fa.ckpt = ws;
    fa.w_logit = logit ? 1 : 0;
    fa.C = C_eff;
    fa.nck = (T + C_eff - 1) / C_eff;
    fa.B = B;
    fa.T = T;
    fa.H = H;
    set_extents(fa, N, bf16, ckpt_bytes(B, T, H, N, C_eff));
    cudaError_t e = use_chunked_fwd(N, C_eff) ? launch_fwd3(fa, bf16, stream) : launch_fwd2(fa, bf16, N, stream);
    if (e != cudaSuccess) {
      cudaFreeAsync(ws, stream);
      return fail_cuda(e, "checkpointing forward launch");
    }
  }
  if ((rc = status_word(&args.status))) {
    if (ws) cudaFreeAsync(ws, stream);
    return rc;
  }
  args.ckpt = ckpt ? ckpt : ws;
  if ((rc = make_ckpt_map(&args.ckmap, args.ckpt, B, H, N, (T + C_eff - 1) / C_eff))) {
    if (ws) cudaFreeAsync(ws, stream);
    return rc;
  }
  args.dr = grads[0];
  args.dw = grads[1];
  args.dk = grads[2];
  args.dv = grads[3];
  args.da = grads[4];
  args.db = grads[5];
  args.dS_init = dS_init;
  args.dS_final = dS_final;
  args.w_logit = logit ? 1 : 0;
  args.carry = split || split32 ? ws + ck_ws / sizeof(float) : nullptr;
#ifdef WKV7_DEBUG
  args.out_kernel = g_debug_out_kernel.load();
#endif
  if (eb) {
    if (!split) {
      if (ws) cudaFreeAsync(ws, stream);
      return fail(WKV7_ERR_INVALID, "the epilogue's backward runs in the split chunked form only");
    }
    args.epilogue = 1;
    args.epi_nv = eb->nv;
    args.epi_stats = eb->stats;
    args.epi_ln_w = eb->ln_w;
    args.epi_r_k = eb->r_k;
    args.epi_part = eb->part;
    rc = make_map(&args.map_nv, eb->nv, true, B, T, H, N, KS);
  }
  if (split) {
    for (int v = 0; v < 7 && rc == WKV7_OK; ++v) rc = make_map(&args.swmap[v], in[v], true, B, T, H, N, kChunk, true);
    if (rc == WKV7_OK) rc = make_carry_map(&args.gcmap, args.carry, (size_t)B * H * ((T + kChunk - 1) / kChunk));
    if (rc) {
      cudaFreeAsync(ws, stream);
      return rc;
    }
  }
  for (int v = 0; v < 7; ++v) args.in[v] = in[v];
  args.C = C_eff;
  args.nck = (T + C_eff - 1) / C_eff;
  args.B = B;
  args.T = T;
  args.H = H;
  set_extents(args, N, bf16, ckpt_bytes(B, T, H, N, C_eff));
  cudaError_t e;
  if (split32) {
    e = launch_bwd4_carry_f32(args, stream);
    if (e == cudaSuccess) e = launch_bwd4_out_f32(args, stream);
  } else {
    e = split ? launch_bwd4(args, stream) : chunked ? launch_bwd3(args, stream) : launch_bwd2(args, bf16, N, stream);
  }
  if (ws) {
    cudaError_t e2 = cudaFreeAsync(ws, stream);
    if (e == cudaSuccess && e2 != cudaSuccess) return fail_cuda(e2, "cudaFreeAsync(workspace)");
  }
  if (e != cudaSuccess) return fail_cuda(e, "backward launch");
  return WKV7_OK;
}

}  // namespace

// Error hook for the other entry points of the library (rwkv8_api.cu): the
// message goes to the same thread-local slot wkv7_last_error() reads.
int api_fail(int code, const char* msg) { return fail(code, "%s", msg); }

// ======================================== backward without allocation ===
//
// For callers that cannot allocate device memory: code running inside a
// CUDA graph being captured or replayed where allocation nodes are not
// allowed, or a host framework that owns all device memory through its own
// allocator and forbids library calls to cudaMalloc. The checkpoints of the
// backward's own forward pass go to a fixed scratch array of this library
// instead of a stream-ordered workspace.

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;  // 64 MiB

// Every GPU that loads the library holds this array until the process exits.
// Host code must not pass the name itself to a kernel: in host code it is a
// stand-in, not a device address. The device address comes from
// cudaGetSymbolAddress, once per device (noalloc_scratch below).
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
float* g_noalloc_ptr[kMaxDevices];

// Device address of the scratch array on the current device; looked up on
// the first call on each device.
int noalloc_scratch(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(WKV7_ERR_CUDA, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return fail_cuda(e, "cudaGetSymbolAddress(no-allocation scratch)");
    g_noalloc_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_noalloc_ptr[dev];
  return WKV7_OK;
}

int backward_noalloc_impl(const float* const in[7], const float* s_init, float* const grads[6], float* dS_init,
                          int B, int T, int H, int N, cudaStream_t stream) {
  int rc = check_dims(B, T, H, N);
  if (rc) return rc;
  const size_t vec = (size_t)B * T * H * N * 4;
  const size_t st = (size_t)B * H * N * N * 4;
  const Span ins[8] = {{in[0], vec, "r"}, {in[1], vec, "w"}, {in[2], vec, "k"}, {in[3], vec, "v"},
                       {in[4], vec, "a"}, {in[5], vec, "b"}, {in[6], vec, "dy"}, {s_init, st, "s_init"}};
  const Span outs[7] = {{grads[0], vec, "dr"}, {grads[1], vec, "dw"}, {grads[2], vec, "dk"},
                        {grads[3], vec, "dv"}, {grads[4], vec, "da"}, {grads[5], vec, "db"},
                        {dS_init, st, "dS_init"}};
  if ((size_t)B * H == 0) return WKV7_OK;
  if (T == 0) {
    rc = check_spans(ins + 7, 1, outs + 6, 1, 0, 0);
    if (rc) return rc;
    if (!dS_init) return WKV7_OK;
    cudaError_t e = cudaMemsetAsync(dS_init, 0, st, stream);
    return e == cudaSuccess ? WKV7_OK : fail_cuda(e, "empty backward");
  }
  rc = check_spans(ins, 8, outs, 7, 7, 6);
  if (rc) return rc;
  const int C = bwd2_steps_per_window(N, false);
  const size_t bytes = ckpt_bytes(B, T, H, N, C);
  if (bytes > kNoAllocScratchBytes)
    return fail(WKV7_ERR_INVALID,
                "wkv7_backward_noalloc: this problem needs %zu bytes of checkpoints "
                "(B*H*ceil(T/%d)*N*N*4), the fixed scratch holds %zu",
                bytes, C, kNoAllocScratchBytes);

  float* scratch = nullptr;
  if ((rc = noalloc_scratch(&scratch))) return rc;
  FwdArgs fa;
  for (int v = 0; v < 6; ++v) {
    if ((rc = make_map(&fa.map[v], in[v], false, B, T, H, N, fwd_steps_per_stage(N, false)))) return rc;
    fa.in[v] = in[v];
  }
  if ((rc = status_word(&fa.status))) return rc;
  fa.s_init = s_init;
  fa.y = nullptr;
  fa.s_final = nullptr;
  fa.ckpt = scratch;  // every checkpoint the backward reads is written first
  fa.C = C;
  fa.nck = (T + C - 1) / C;
  fa.B = B;
  fa.T = T;
  fa.H = H;
  BwdArgs ba;
  ba.dS_final = nullptr;
  for (int v = 0; v < 7; ++v)
    if ((rc = make_map(&ba.map[v], in[v], false, B, T, H, N, bwd2_steps_per_window(N, false)))) return rc;
  if ((rc = make_ckpt_map(&ba.ckmap, scratch, B, H, N, fa.nck))) return rc;
  if ((rc = status_word(&ba.status))) return rc;
  ba.ckpt = scratch;
  ba.dr = grads[0];
  ba.dw = grads[1];
  ba.dk = grads[2];
  ba.dv = grads[3];
  ba.da = grads[4];
  ba.db = grads[5];
  ba.dS_init = dS_init;
  ba.C = C;
  ba.nck = fa.nck;
  ba.B = B;
  ba.T = T;
  ba.H = H;
  for (int v = 0; v < 7; ++v) ba.in[v] = in[v];
  set_extents(fa, N, false, bytes);
  set_extents(ba, N, false, bytes);
  cudaError_t e = use_chunked_fwd(N, C) ? launch_fwd3(fa, false, stream) : launch_fwd2(fa, false, N, stream);
  if (e != cudaSuccess) return fail_cuda(e, "checkpointing forward launch");
  e = launch_bwd2(ba, false, N, stream);
  if (e != cudaSuccess) return fail_cuda(e, "backward launch");
  return WKV7_OK;
}

}  // namespace
}  // namespace wkv7

// ============================================================== C ABI ===

using namespace wkv7;

extern "C" {

int wkv7_forward(const float* r, const float* w, const float* k, const float* v, const float* a,
                 const float* b, const float* s_init, float* y, float* s_final, float* ckpt,
                 int ckpt_every, int B, int T, int H, int N, void* stream) {
  const void* in[6] = {r, w, k, v, a, b};
  return forward_impl(false, in, s_init, y, s_final, ckpt, ckpt_every, B, T, H, N,
                      static_cast<cudaStream_t>(stream));
}

int wkv7_forward_bf16(const wkv7_bf16* r, const wkv7_bf16* w, const wkv7_bf16* k, const wkv7_bf16* v,
                      const wkv7_bf16* a, const wkv7_bf16* b, const float* s_init, wkv7_bf16* y,
                      float* s_final, float* ckpt, int ckpt_every, int B, int T, int H, int N,
                      void* stream) {
  const void* in[6] = {r, w, k, v, a, b};
  return forward_impl(true, in, s_init, y, s_final, ckpt, ckpt_every, B, T, H, N,
                      static_cast<cudaStream_t>(stream));
}

int wkv7_backward(const float* r, const float* w, const float* k, const float* v, const float* a,
                  const float* b, const float* dy, const float* s_init, const float* ckpt,
                  int ckpt_every, float* dr, float* dw, float* dk, float* dv, float* da, float* db,
                  float* dS_init, int B, int T, int H, int N, void* stream) {
  const void* in[7] = {r, w, k, v, a, b, dy};
  float* const grads[6] = {dr, dw, dk, dv, da, db};
  return backward_impl(false, in, s_init, nullptr, ckpt, ckpt_every, grads, dS_init, B, T, H, N,
                       static_cast<cudaStream_t>(stream));
}

int wkv7_backward_segment(const float* r, const float* w, const float* k, const float* v, const float* a,
                          const float* b, const float* dy, const float* s_init, const float* dS_final,
                          const float* ckpt, int ckpt_every, float* dr, float* dw, float* dk, float* dv, float* da,
                          float* db, float* dS_init, int B, int T, int H, int N, void* stream) {
  const void* in[7] = {r, w, k, v, a, b, dy};
  float* const grads[6] = {dr, dw, dk, dv, da, db};
  return backward_impl(false, in, s_init, dS_final, ckpt, ckpt_every, grads, dS_init, B, T, H, N,
                       static_cast<cudaStream_t>(stream));
}

int wkv7_backward_segment_bf16(const wkv7_bf16* r, const wkv7_bf16* w, const wkv7_bf16* k, const wkv7_bf16* v,
                               const wkv7_bf16* a, const wkv7_bf16* b, const wkv7_bf16* dy, const float* s_init,
                               const float* dS_final, const float* ckpt, int ckpt_every, float* dr, float* dw,
                               float* dk, float* dv, float* da, float* db, float* dS_init, int B, int T, int H,
                               int N, void* stream) {
  const void* in[7] = {r, w, k, v, a, b, dy};
  float* const grads[6] = {dr, dw, dk, dv, da, db};
  return backward_impl(true, in, s_init, dS_final, ckpt, ckpt_every, grads, dS_init, B, T, H, N,
                       static_cast<cudaStream_t>(stream));
}

int wkv7_backward_bf16(const wkv7_bf16* r, const wkv7_bf16* w, const wkv7_bf16* k, const wkv7_bf16* v,
                       const wkv7_bf16* a, const wkv7_bf16* b, const wkv7_bf16* dy, const float* s_init,
                       const float* ckpt, int ckpt_every, float* dr, float* dw, float* dk, float* dv,
                       float* da, float* db, float* dS_init, int B, int T, int H, int N, void* stream) {
  const void* in[7] = {r, w, k, v, a, b, dy};
  float* const grads[6] = {dr, dw, dk, dv, da, db};
  return backward_impl(true, in, s_init, nullptr, ckpt, ckpt_every, grads, dS_init, B, T, H, N,
                       static_cast<cudaStream_t>(stream));
}

int wkv7_backward_fused_bf16(const wkv7_bf16* r, const wkv7_bf16* w, const wkv7_bf16* k, const wkv7_bf16* v,
                             const wkv7_bf16* a, const wkv7_bf16* b, const wkv7_bf16* dy, const float* s_init,
                             const float* dS_final, const float* ckpt, int ckpt_every, float* dr, float* dw,
                             float* dk, float* dv, float* da, float* db, float* dS_init, int B, int T, int H, int N,
                             void* stream) {
  const void* in[7] = {r, w, k, v, a, b, dy};
  float* const grads[6] = {dr, dw, dk, dv, da, db};
  return backward_impl(true, in, s_init, dS_final, ckpt, ckpt_every, grads, dS_init, B, T, H, N,
                       static_cast<cudaStream_t>(stream), false, BwdForm::kFused);
}

int wkv7_forward_logit_bf16(const wkv7_bf16* r, const wkv7_bf16* z, const wkv7_bf16* k, const wkv7_bf16* v,
                            const wkv7_bf16* a, const wkv7_bf16* b, const float* s_init, wkv7_bf16* y,
                            float* s_final, float* ckpt, int ckpt_every, int B, int T, int H, int N, void* stream) {
  const void* in[6] = {r, z, k, v, a, b};
  return forward_impl(true, in, s_init, y, s_final, ckpt, ckpt_every, B, T, H, N,
                      static_cast<cudaStream_t>(stream), true);
}

int wkv7_forward_epilogue_bf16(const wkv7_bf16* r, const wkv7_bf16* w, const wkv7_bf16* k, const wkv7_bf16* v,
                               const wkv7_bf16* a, const wkv7_bf16* b, const float* s_init, const float* ln_w,
                               const float* ln_b, const float* r_k, wkv7_bf16* out, wkv7_bf16* nv, float* stats,
                               float* s_final, float* ckpt, int ckpt_every, int decay_is_logit, int B, int T, int H,
                               int N, void* stream) {
  const void* in[6] = {r, w, k, v, a, b};
  const Epilogue epi{ln_w, ln_b, r_k, nv, stats};
  return forward_impl(true, in, s_init, out, s_final, ckpt, ckpt_every, B, T, H, N,
                      static_cast<cudaStream_t>(stream), decay_is_logit != 0, &epi);
}

int wkv7_backward_epilogue_bf16(const wkv7_bf16* r, const wkv7_bf16* w, const wkv7_bf16* k, const wkv7_bf16* v,
                                const wkv7_bf16* a, const wkv7_bf16* b, const wkv7_bf16* dout, const wkv7_bf16* nv,
                                const float* stats, const float* ln_w, const float* r_k, const float* s_init,
                                const float* dS_final, const float* ckpt, int ckpt_every, int decay_is_logit,
                                float* dr, float* dw, float* dk, float* dv, float* da, float* db, float* dS_init,
                                float* dln_w, float* dln_b, float* dr_k, int B, int T, int H, int N, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int rc = check_dims(B, T, H, N);
  if (rc) return rc;
  if (N != 64 || (ckpt && ckpt_every != kChunk))
    return fail(WKV7_ERR_INVALID, "the epilogue needs N = 64 and ckpt_every = %d (got N = %d, %d)", kChunk, N,
                ckpt_every);
  const size_t vec = (size_t)B * T * H * N * 2, rows = (size_t)B * T * H, par = (size_t)H * N * 4;
  const Span ins[6] = {{dout, vec, "dout"}, {nv, vec, "nv"}, {stats, rows * 8, "stats"},
                       {ln_w, par, "ln_w"}, {r_k, par, "r_k"}, {r, vec, "r"}};
  const Span outs[3] = {{dln_w, par, "dln_w"}, {dln_b, par, "dln_b"}, {dr_k, par, "dr_k"}};
  if ((size_t)H == 0) return WKV7_OK;
  if ((rc = check_spans(ins, 6, outs, 3, (size_t)B * T ? 6 : 0, 3))) return rc;
  const void* in[7] = {r, w, k, v, a, b, dout};
  float* const grads[6] = {dr, dw, dk, dv, da, db};
  if ((size_t)B * T == 0) {  // no row: the parameters' gradients are empty sums
    for (float* p : {dln_w, dln_b, dr_k}) {
      cudaError_t e = cudaMemsetAsync(p, 0, par, s);
      if (e != cudaSuccess) return fail_cuda(e, "epilogue clear");
    }
    return backward_impl(true, in, s_init, dS_final, ckpt, ckpt_every, grads, dS_init, B, T, H, N, s,
                         decay_is_logit != 0);
  }
  // every chunk's parameter terms: [B][H][nchunks][3][N] fp32
  const int nchunks = (T + kChunk - 1) / kChunk;
  const size_t ws_bytes = (size_t)B * H * nchunks * 3 * N * 4;
  const char* inject = std::getenv("WKV7_FAIL_ALLOC");
  if (inject && inject[0] == '1') return fail(WKV7_ERR_ALLOC, "workspace allocation failed (injected by WKV7_FAIL_ALLOC)");
  float* part = nullptr;
  cudaError_t e = cudaMallocAsync(reinterpret_cast<void**>(&part), ws_bytes, s);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(WKV7_ERR_ALLOC, "epilogue workspace of %zu bytes: %s", ws_bytes, cudaGetErrorString(e));
  }
  const EpiBwd eb{nv, stats, ln_w, r_k, part};
  rc = backward_impl(true, in, s_init, dS_final, ckpt, ckpt_every, grads, dS_init, B, T, H, N, s, decay_is_logit != 0,
                     BwdForm::kAuto, &eb);
  if (rc == WKV7_OK) {
    e = launch_epi_params(part, dln_w, dln_b, dr_k, B, H, nchunks, s);
    if (e != cudaSuccess) rc = fail_cuda(e, "epilogue parameter sums");
  }
  cudaError_t e2 = cudaFreeAsync(part, s);
  if (rc == WKV7_OK && e2 != cudaSuccess) return fail_cuda(e2, "cudaFreeAsync(epilogue workspace)");
  return rc;
}

int wkv7_backward_logit_bf16(const wkv7_bf16* r, const wkv7_bf16* z, const wkv7_bf16* k, const wkv7_bf16* v,
                             const wkv7_bf16* a, const wkv7_bf16* b, const wkv7_bf16* dy, const float* s_init,
                             const float* dS_final, const float* ckpt, int ckpt_every, float* dr, float* dz,
                             float* dk, float* dv, float* da, float* db, float* dS_init, int B, int T, int H, int N,
                             void* stream) {
  const void* in[7] = {r, z, k, v, a, b, dy};
  float* const grads[6] = {dr, dz, dk, dv, da, db};
  return backward_impl(true, in, s_init, dS_final, ckpt, ckpt_every, grads, dS_init, B, T, H, N,
                       static_cast<cudaStream_t>(stream), true);
}

size_t wkv7_ckpt_bytes(int B, int T, int H, int N, int ckpt_every) {
  if (ckpt_every < 1 || check_dims(B, T, H, N) != WKV7_OK) return 0;
  return ckpt_bytes(B, T, H, N, ckpt_every);
}

int wkv7_default_ckpt_every(int N, int bf16) {
  if (N != 16 && N != 32 && N != 64) return 0;
  return bwd2_steps_per_window(N, bf16 != 0);
}

int wkv7_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e, "stream synchronize");
  unsigned* word = nullptr;
  int rc = status_word(&word);
  if (rc) return rc;
  unsigned host = 0;
  e = cudaMemcpy(&host, word, sizeof host, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail_cuda(e, "reading the status word");
  if (host) {
    const unsigned zero = 0;
    e = cudaMemcpy(word, &zero, sizeof zero, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return fail_cuda(e, "clearing the status word");
    if (host & STATUS_TIMEOUT) return fail(WKV7_ERR_TIMEOUT, "a kernel gave up a bounded wait");
    if (host & STATUS_BOUNDS) return fail(WKV7_ERR_BOUNDS, "a kernel skipped an access outside its buffer");
  }
  return WKV7_OK;
}

const char* wkv7_last_error(void) { return t_last_error.c_str(); }

#ifdef WKV7_DEBUG
int wkv7_debug_skip_last_load(int on) {
  g_debug_skip_last_load.store(on ? 1 : 0);
  return WKV7_OK;
}

int wkv7_debug_out_kernel(int which) {
  g_debug_out_kernel.store(which == 1 ? 1 : 0);
  return WKV7_OK;
}

int wkv7_debug_cut_extents(size_t bytes) {
  g_debug_extent_cut.store(bytes);
  return WKV7_OK;
}
#endif

int wkv7_backward_noalloc(const float* r, const float* w, const float* k, const float* v, const float* a,
                          const float* b, const float* dy, const float* s_init, float* dr, float* dw, float* dk,
                          float* dv, float* da, float* db, float* dS_init, int B, int T, int H, int N,
                          void* stream) {
  const float* in[7] = {r, w, k, v, a, b, dy};
  float* const grads[6] = {dr, dw, dk, dv, da, db};
  return backward_noalloc_impl(in, s_init, grads, dS_init, B, T, H, N, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
