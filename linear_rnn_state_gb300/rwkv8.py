"""Python binding of the RWKV-8 C ABI (include/rwkv8.h).

Argument marshalling only: every step of the recurrence runs in the CUDA
kernels of libwkv7.so (the same library as the WKV7 scan). The raw functions
carry the C names and take integer device addresses; ``forward`` and
``backward`` take torch tensors, allocate the outputs with torch and call the
raw functions on torch's current stream. There is no CPU path.
"""
from __future__ import annotations

import ctypes

from . import wkv7

CHUNK = 16  # RWKV8_CHUNK

# C functions declared in include/rwkv8.h, with their argument counts.
EXPORTS = {
    "rwkv8_ckpt_bytes": 5,
    "rwkv8_forward": 16,
    "rwkv8_backward": 21,
}

_typed = set()


def load(path: str | None = None):
    """The loaded library with the rwkv8_* signatures set."""
    lib = wkv7.load(path)
    if id(lib) not in _typed:
        vp, i = ctypes.c_void_p, ctypes.c_int
        lib.rwkv8_ckpt_bytes.argtypes = [i] * 5
        lib.rwkv8_ckpt_bytes.restype = ctypes.c_size_t
        lib.rwkv8_forward.argtypes = [vp] * 9 + [i] * 6 + [vp]
        lib.rwkv8_forward.restype = i
        lib.rwkv8_backward.argtypes = [vp] * 14 + [i] * 6 + [vp]
        lib.rwkv8_backward.restype = i
        _typed.add(id(lib))
    return lib


# ------------------------------------------------------------ raw C ABI ---

def rwkv8_ckpt_bytes(B, T, H, L, E) -> int:
    return load().rwkv8_ckpt_bytes(B, T, H, L, E)


def rwkv8_forward(q, v, decay, rho_init, rho_norm_init, y, rho_final, rho_norm_final, ckpt, B, T, H, Hv, L, E, stream):
    return load().rwkv8_forward(q, v, decay, rho_init, rho_norm_init, y, rho_final, rho_norm_final, ckpt,
                                B, T, H, Hv, L, E, stream)


def rwkv8_backward(q, v, decay, dy, rho_init, rho_norm_init, d_rho_final, d_rho_norm_final, ckpt, dq, dv, ddecay,
                   d_rho_init, d_rho_norm_init, B, T, H, Hv, L, E, stream):
    return load().rwkv8_backward(q, v, decay, dy, rho_init, rho_norm_init, d_rho_final, d_rho_norm_final, ckpt,
                                 dq, dv, ddecay, d_rho_init, d_rho_norm_init, B, T, H, Hv, L, E, stream)


# ------------------------------------------------------- torch helpers ---

def _addr(t):
    return None if t is None else t.data_ptr()


def _shapes(q, v):
    B, H, T, L = q.shape
    Hv, E = v.shape[1], v.shape[3]
    return B, T, H, Hv, L, E


def forward(q, v, decay, rho_init=None, rho_norm_init=None, *, want_ckpt: bool = True, stream=None):
    """Forward on CUDA float32 tensors q [B][H][T][L], v [B][Hv][T][E],
    decay [H][L]. Returns (y, rho_final, rho_norm_final, ckpt)."""
    import torch

    B, T, H, Hv, L, E = _shapes(q, v)
    dev = q.device
    y = torch.empty((B, H, T, E), dtype=torch.float32, device=dev)
    rho_final = torch.empty((B, H, L, E), dtype=torch.float32, device=dev)
    rho_norm_final = torch.empty((B, H, L), dtype=torch.float32, device=dev)
    ckpt = None
    if want_ckpt:
        ckpt = torch.empty(max(rwkv8_ckpt_bytes(B, T, H, L, E) // 4, 1), dtype=torch.float32, device=dev)
    rc = rwkv8_forward(*(_addr(x) for x in (q, v, decay, rho_init, rho_norm_init, y, rho_final, rho_norm_final,
                                            ckpt)), B, T, H, Hv, L, E, wkv7._stream(stream))
    wkv7._check(rc)
    return y, rho_final, rho_norm_final, ckpt


def backward(q, v, decay, dy, rho_init=None, rho_norm_init=None, ckpt=None, *, d_rho_final=None,
             d_rho_norm_final=None, stream=None):
    """Backward. Returns dict dq, dv, ddecay, d_rho_init, d_rho_norm_init
    (float32, the shapes of q, v, decay and the states)."""
    import torch

    B, T, H, Hv, L, E = _shapes(q, v)
    dev = q.device
    g = {
        "dq": torch.empty_like(q, dtype=torch.float32),
        "dv": torch.empty_like(v, dtype=torch.float32),
        "ddecay": torch.empty((H, L), dtype=torch.float32, device=dev),
        "d_rho_init": torch.empty((B, H, L, E), dtype=torch.float32, device=dev),
        "d_rho_norm_init": torch.empty((B, H, L), dtype=torch.float32, device=dev),
    }
    rc = rwkv8_backward(*(_addr(x) for x in (q, v, decay, dy, rho_init, rho_norm_init, d_rho_final, d_rho_norm_final,
                                             ckpt, g["dq"], g["dv"], g["ddecay"], g["d_rho_init"],
                                             g["d_rho_norm_init"])), B, T, H, Hv, L, E, wkv7._stream(stream))
    wkv7._check(rc)
    return g
