"""Python binding of the WKV7 C ABI (include/wkv7.h).

Argument marshalling only: every step of the scan runs in the CUDA kernels of
libwkv7.so. The raw functions carry the C names and take integer device
addresses; ``forward`` and ``backward`` take torch tensors, allocate the
outputs with torch and call the raw functions on torch's current stream.
There is no CPU path: if the library is missing, the call fails.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libwkv7.so")

OK, ERR_ALLOC, ERR_INVALID, ERR_CUDA, ERR_TIMEOUT, ERR_BOUNDS = 0, -1, -2, -3, -4, -5

# C functions declared in include/wkv7.h, with their argument counts.
EXPORTS = {
    "wkv7_forward": 16,
    "wkv7_forward_bf16": 16,
    "wkv7_backward": 22,
    "wkv7_backward_bf16": 22,
    "wkv7_backward_segment": 23,
    "wkv7_backward_segment_bf16": 23,
    "wkv7_ckpt_bytes": 5,
    "wkv7_default_ckpt_every": 2,
    "wkv7_status": 1,
    "wkv7_last_error": 0,
    "wkv7_backward_noalloc": 20,
    "wkv7_forward_logit_bf16": 16,
    "wkv7_backward_logit_bf16": 23,
    "wkv7_backward_fused_bf16": 23,
    "wkv7_forward_epilogue_bf16": 22,
    "wkv7_backward_epilogue_bf16": 31,
}


class Wkv7Error(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"WKV7 error {code}: {message}")
        self.code = code


_lib = None


def load(path: str | None = None):
    """Load libwkv7.so (built by ``__graft_entry__.build()``)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"the WKV7 CUDA library is not built ({p} missing); run __graft_entry__.build()")
    lib = ctypes.CDLL(p)
    vp, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.wkv7_forward.argtypes = [vp] * 10 + [i] * 5 + [vp]
    lib.wkv7_forward_bf16.argtypes = [vp] * 10 + [i] * 5 + [vp]
    lib.wkv7_backward.argtypes = [vp] * 9 + [i] + [vp] * 7 + [i] * 4 + [vp]
    lib.wkv7_backward_bf16.argtypes = [vp] * 9 + [i] + [vp] * 7 + [i] * 4 + [vp]
    lib.wkv7_backward_segment.argtypes = [vp] * 10 + [i] + [vp] * 7 + [i] * 4 + [vp]
    lib.wkv7_backward_segment_bf16.argtypes = [vp] * 10 + [i] + [vp] * 7 + [i] * 4 + [vp]
    for f in ("wkv7_forward", "wkv7_forward_bf16", "wkv7_backward", "wkv7_backward_bf16", "wkv7_backward_segment",
              "wkv7_backward_segment_bf16"):
        getattr(lib, f).restype = i
    lib.wkv7_ckpt_bytes.argtypes = [i] * 5
    lib.wkv7_ckpt_bytes.restype = sz
    lib.wkv7_default_ckpt_every.argtypes = [i, i]
    lib.wkv7_default_ckpt_every.restype = i
    lib.wkv7_status.argtypes = [vp]
    lib.wkv7_status.restype = i
    lib.wkv7_last_error.argtypes = []
    lib.wkv7_last_error.restype = ctypes.c_char_p
    lib.wkv7_backward_noalloc.argtypes = [vp] * 15 + [i] * 4 + [vp]
    lib.wkv7_backward_noalloc.restype = i
    lib.wkv7_forward_logit_bf16.argtypes = [vp] * 10 + [i] * 5 + [vp]
    lib.wkv7_forward_logit_bf16.restype = i
    lib.wkv7_backward_logit_bf16.argtypes = [vp] * 10 + [i] + [vp] * 7 + [i] * 4 + [vp]
    lib.wkv7_backward_logit_bf16.restype = i
    lib.wkv7_backward_fused_bf16.argtypes = [vp] * 10 + [i] + [vp] * 7 + [i] * 4 + [vp]
    lib.wkv7_backward_fused_bf16.restype = i
    lib.wkv7_forward_epilogue_bf16.argtypes = [vp] * 15 + [i] * 6 + [vp]
    lib.wkv7_forward_epilogue_bf16.restype = i
    lib.wkv7_backward_epilogue_bf16.argtypes = [vp] * 14 + [i, i] + [vp] * 10 + [i] * 4 + [vp]
    lib.wkv7_backward_epilogue_bf16.restype = i
    if path is None:
        _lib = lib
    return lib


def last_error() -> str:
    return load().wkv7_last_error().decode()


def _check(rc: int):
    if rc != OK:
        raise Wkv7Error(rc, last_error())
    return rc


# ------------------------------------------------------------ raw C ABI ---

def wkv7_forward(r, w, k, v, a, b, s_init, y, s_final, ckpt, ckpt_every, B, T, H, N, stream):
    return load().wkv7_forward(r, w, k, v, a, b, s_init, y, s_final, ckpt, ckpt_every, B, T, H, N, stream)


def wkv7_forward_bf16(r, w, k, v, a, b, s_init, y, s_final, ckpt, ckpt_every, B, T, H, N, stream):
    return load().wkv7_forward_bf16(r, w, k, v, a, b, s_init, y, s_final, ckpt, ckpt_every, B, T, H, N, stream)


def wkv7_backward(r, w, k, v, a, b, dy, s_init, ckpt, ckpt_every, dr, dw, dk, dv, da, db, dS_init,
                  B, T, H, N, stream):
    return load().wkv7_backward(r, w, k, v, a, b, dy, s_init, ckpt, ckpt_every, dr, dw, dk, dv, da, db,
                                dS_init, B, T, H, N, stream)


def wkv7_backward_bf16(r, w, k, v, a, b, dy, s_init, ckpt, ckpt_every, dr, dw, dk, dv, da, db, dS_init,
                       B, T, H, N, stream):
    return load().wkv7_backward_bf16(r, w, k, v, a, b, dy, s_init, ckpt, ckpt_every, dr, dw, dk, dv, da, db,
                                     dS_init, B, T, H, N, stream)


def wkv7_backward_segment(r, w, k, v, a, b, dy, s_init, dS_final, ckpt, ckpt_every, dr, dw, dk, dv, da, db,
                          dS_init, B, T, H, N, stream):
    """wkv7_backward_segment (include/wkv7.h): pointers as ints."""
    return load().wkv7_backward_segment(r, w, k, v, a, b, dy, s_init, dS_final, ckpt, ckpt_every, dr, dw, dk, dv,
                                        da, db, dS_init, B, T, H, N, stream)


def wkv7_backward_segment_bf16(r, w, k, v, a, b, dy, s_init, dS_final, ckpt, ckpt_every, dr, dw, dk, dv, da, db,
                               dS_init, B, T, H, N, stream):
    """wkv7_backward_segment_bf16 (include/wkv7.h): pointers as ints."""
    return load().wkv7_backward_segment_bf16(r, w, k, v, a, b, dy, s_init, dS_final, ckpt, ckpt_every, dr, dw, dk,
                                             dv, da, db, dS_init, B, T, H, N, stream)


def wkv7_backward_fused_bf16(r, w, k, v, a, b, dy, s_init, dS_final, ckpt, ckpt_every, dr, dw, dk, dv, da, db,
                             dS_init, B, T, H, N, stream):
    """wkv7_backward_fused_bf16 (include/wkv7.h): the one-pass chunked backward."""
    return load().wkv7_backward_fused_bf16(r, w, k, v, a, b, dy, s_init, dS_final, ckpt, ckpt_every, dr, dw, dk, dv,
                                           da, db, dS_init, B, T, H, N, stream)


def wkv7_backward_noalloc(r, w, k, v, a, b, dy, s_init, dr, dw, dk, dv, da, db, dS_init, B, T, H, N, stream):
    """Backward without any device allocation (fp32 inputs): checkpoints go to
    the library's fixed 64 MiB scratch array. For callers that cannot allocate;
    calls that overlap on the GPU race on the shared scratch."""
    return load().wkv7_backward_noalloc(r, w, k, v, a, b, dy, s_init, dr, dw, dk, dv, da, db, dS_init,
                                        B, T, H, N, stream)


def wkv7_forward_logit_bf16(r, z, k, v, a, b, s_init, y, s_final, ckpt, ckpt_every, B, T, H, N, stream):
    """wkv7_forward_logit_bf16 (include/wkv7.h): the decay given as logits z."""
    return load().wkv7_forward_logit_bf16(r, z, k, v, a, b, s_init, y, s_final, ckpt, ckpt_every, B, T, H, N, stream)


def wkv7_backward_logit_bf16(r, z, k, v, a, b, dy, s_init, dS_final, ckpt, ckpt_every, dr, dz, dk, dv, da, db,
                             dS_init, B, T, H, N, stream):
    """wkv7_backward_logit_bf16 (include/wkv7.h): returns dz in the place of dw."""
    return load().wkv7_backward_logit_bf16(r, z, k, v, a, b, dy, s_init, dS_final, ckpt, ckpt_every, dr, dz, dk, dv,
                                           da, db, dS_init, B, T, H, N, stream)


def wkv7_ckpt_bytes(B, T, H, N, ckpt_every) -> int:
    return load().wkv7_ckpt_bytes(B, T, H, N, ckpt_every)


def wkv7_default_ckpt_every(N, bf16) -> int:
    return load().wkv7_default_ckpt_every(N, int(bool(bf16)))


def wkv7_status(stream) -> int:
    return load().wkv7_status(stream)


# ------------------------------------------------------- torch helpers ---

def _addr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    import torch

    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _inputs_dtype(r):
    import torch

    if r.dtype == torch.bfloat16:
        return True
    if r.dtype == torch.float32:
        return False
    raise TypeError(f"inputs must be float32 or bfloat16, got {r.dtype}")


def forward(r, w, k, v, a, b, s_init=None, *, ckpt_every: int | None = None, want_y: bool = True,
            want_s_final: bool = True, want_ckpt: bool = True, stream=None):
    """Run the forward scan on CUDA tensors [B][T][H][N] (all float32 or all
    bfloat16). Returns (y, s_final, ckpt, ckpt_every); skipped outputs are None."""
    import torch

    bf16 = _inputs_dtype(r)
    B, T, H, N = r.shape
    C = ckpt_every or wkv7_default_ckpt_every(N, bf16)
    dev = r.device
    y = torch.empty_like(r) if want_y else None
    s_final = torch.empty((B, H, N, N), dtype=torch.float32, device=dev) if want_s_final else None
    ckpt = None
    if want_ckpt:
        nck = (T + C - 1) // C
        ckpt = torch.empty((B, H, nck, N, N), dtype=torch.float32, device=dev)
    fn = wkv7_forward_bf16 if bf16 else wkv7_forward
    _check(fn(*(_addr(x) for x in (r, w, k, v, a, b, s_init, y, s_final, ckpt)), C, B, T, H, N, _stream(stream)))
    return y, s_final, ckpt, C


def backward(r, w, k, v, a, b, dy, s_init=None, ckpt=None, ckpt_every: int = 0, *, want_dS_init: bool = True,
             dS_final=None, fused: bool = False, stream=None):
    """Backward-through-time. Returns dict dr, dw, dk, dv, da, db (float32
    [B][T][H][N]) and dS_init (float32 [B][H][N][N] or None). dS_final
    (float32 [B][H][N][N]) is the gradient entering through the final state
    (None: zero). fused=True runs wkv7_backward_fused_bf16 (bfloat16 inputs,
    N = 64, 16-step checkpoints)."""
    import torch

    bf16 = _inputs_dtype(r)
    B, T, H, N = r.shape
    dev = r.device
    g = {n: torch.empty((B, T, H, N), dtype=torch.float32, device=dev) for n in ("dr", "dw", "dk", "dv", "da", "db")}
    g["dS_init"] = torch.empty((B, H, N, N), dtype=torch.float32, device=dev) if want_dS_init else None
    fn = wkv7_backward_segment_bf16 if bf16 else wkv7_backward_segment
    if fused:
        fn = wkv7_backward_fused_bf16
    _check(fn(*(_addr(x) for x in (r, w, k, v, a, b, dy, s_init, dS_final, ckpt)), ckpt_every,
              *(_addr(g[n]) for n in ("dr", "dw", "dk", "dv", "da", "db", "dS_init")), B, T, H, N, _stream(stream)))
    return g


def forward_logit(r, z, k, v, a, b, s_init=None, *, want_ckpt: bool = True, stream=None):
    """forward() with the decay given as logits z (bfloat16 tensors, N = 64):
    w = exp(-0.606531 sigmoid(z)) is formed inside the kernels. Returns
    (y, s_final, ckpt, 16)."""
    import torch

    B, T, H, N = r.shape
    dev = r.device
    y = torch.empty_like(r)
    s_final = torch.empty((B, H, N, N), dtype=torch.float32, device=dev)
    ckpt = torch.empty((B, H, (T + 15) // 16, N, N), dtype=torch.float32, device=dev) if want_ckpt else None
    _check(wkv7_forward_logit_bf16(*(_addr(x) for x in (r, z, k, v, a, b, s_init, y, s_final, ckpt)), 16, B, T, H, N,
                                   _stream(stream)))
    return y, s_final, ckpt, 16


def backward_logit(r, z, k, v, a, b, dy, s_init=None, ckpt=None, *, dS_final=None, stream=None):
    """backward() with the decay given as logits z: returns dict dr, dz, dk,
    dv, da, db and dS_init."""
    import torch

    B, T, H, N = r.shape
    dev = r.device
    g = {n: torch.empty((B, T, H, N), dtype=torch.float32, device=dev) for n in ("dr", "dz", "dk", "dv", "da", "db")}
    g["dS_init"] = torch.empty((B, H, N, N), dtype=torch.float32, device=dev)
    _check(wkv7_backward_logit_bf16(*(_addr(x) for x in (r, z, k, v, a, b, dy, s_init, dS_final, ckpt)), 16,
                                    *(_addr(g[n]) for n in ("dr", "dz", "dk", "dv", "da", "db", "dS_init")), B, T, H,
                                    N, _stream(stream)))
    return g


def wkv7_forward_epilogue_bf16(r, w, k, v, a, b, s_init, ln_w, ln_b, r_k, out, nv, stats, s_final, ckpt,
                               ckpt_every, decay_is_logit, B, T, H, N, stream):
    """wkv7_forward_epilogue_bf16 (include/wkv7.h): pointers as ints."""
    return load().wkv7_forward_epilogue_bf16(r, w, k, v, a, b, s_init, ln_w, ln_b, r_k, out, nv, stats, s_final, ckpt,
                                             ckpt_every, decay_is_logit, B, T, H, N, stream)


def forward_epilogue(r, w, k, v, a, b, ln_w, ln_b, r_k, s_init=None, *, decay_is_logit: bool = False,
                     want_ckpt: bool = True, stream=None):
    """Forward with the group-norm + bonus epilogue fused (bfloat16 tensors,
    N = 64). Returns (out, nv, stats, s_final, ckpt)."""
    import torch

    B, T, H, N = r.shape
    dev = r.device
    out = torch.empty_like(r)
    nv = torch.empty_like(r)
    stats = torch.empty((B, T, H, 2), dtype=torch.float32, device=dev)
    s_final = torch.empty((B, H, N, N), dtype=torch.float32, device=dev)
    ckpt = torch.empty((B, H, (T + 15) // 16, N, N), dtype=torch.float32, device=dev) if want_ckpt else None
    _check(wkv7_forward_epilogue_bf16(*(_addr(x) for x in (r, w, k, v, a, b, s_init, ln_w, ln_b, r_k, out, nv, stats,
                                                           s_final, ckpt)), 16, int(decay_is_logit), B, T, H, N,
                                      _stream(stream)))
    return out, nv, stats, s_final, ckpt


def wkv7_backward_epilogue_bf16(r, w, k, v, a, b, dout, nv, stats, ln_w, r_k, s_init, dS_final, ckpt, ckpt_every,
                                decay_is_logit, dr, dw, dk, dv, da, db, dS_init, dln_w, dln_b, dr_k, B, T, H, N,
                                stream):
    """wkv7_backward_epilogue_bf16 (include/wkv7.h): pointers as ints."""
    return load().wkv7_backward_epilogue_bf16(r, w, k, v, a, b, dout, nv, stats, ln_w, r_k, s_init, dS_final, ckpt,
                                              ckpt_every, decay_is_logit, dr, dw, dk, dv, da, db, dS_init, dln_w,
                                              dln_b, dr_k, B, T, H, N, stream)


def backward_epilogue(r, w, k, v, a, b, dout, nv, stats, ln_w, r_k, s_init=None, ckpt=None, *,
                      decay_is_logit: bool = False, dS_final=None, stream=None):
    """Backward of forward_epilogue. Returns dict dr, dw (or dz), dk, dv, da,
    db, dS_init, dln_w, dln_b, dr_k."""
    import torch

    B, T, H, N = r.shape
    dev = r.device
    dwn = "dz" if decay_is_logit else "dw"
    g = {n: torch.empty((B, T, H, N), dtype=torch.float32, device=dev) for n in ("dr", dwn, "dk", "dv", "da", "db")}
    g["dS_init"] = torch.empty((B, H, N, N), dtype=torch.float32, device=dev)
    for n in ("dln_w", "dln_b", "dr_k"):
        g[n] = torch.empty((H, N), dtype=torch.float32, device=dev)
    _check(wkv7_backward_epilogue_bf16(
        *(_addr(x) for x in (r, w, k, v, a, b, dout, nv, stats, ln_w, r_k, s_init, dS_final, ckpt)), 16,
        int(decay_is_logit), *(_addr(g[n]) for n in ("dr", dwn, "dk", "dv", "da", "db", "dS_init", "dln_w", "dln_b",
                                                    "dr_k")), B, T, H, N, _stream(stream)))
    return g


def status(stream=None) -> None:
    """Wait for the stream and raise if a kernel reported a timeout (or, in
    the debug build, an access outside a buffer)."""
    _check(wkv7_status(_stream(stream)))
