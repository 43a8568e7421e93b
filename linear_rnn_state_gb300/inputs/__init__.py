"""Seeded synthetic inputs for the WKV7 scan and the RWKV-8 recurrence.

A module of its own: it draws random numbers and shapes them into the scan's
inputs, and holds none of the recurrence's arithmetic. The CUDA path and the
oracle both consume what it returns. The C source (``wkv7_gen.c``) documents
the draw order and the value semantics.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "wkv7_gen.c")
_LIB = os.path.join(_HERE, "libwkv7_gen.so")

CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off"]

KIND = {"f64": 0, "f32": 1, "bf16": 2}
NP_STORAGE = {"f64": np.float64, "f32": np.float32, "bf16": np.uint16}
NAMES = ("r", "w", "k", "v", "a", "b", "dy")


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        vp, i = ctypes.c_void_p, ctypes.c_int
        lib.wkv7_gen_inputs.argtypes = [ctypes.c_uint64, i, i, i, i, i] + [vp] * 7 + [
            ctypes.POINTER(ctypes.c_double), ctypes.c_double, i]
        lib.wkv7_gen_inputs.restype = i
        lib.wkv7_gen_splitmix64_at.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
        lib.wkv7_gen_splitmix64_at.restype = ctypes.c_uint64
        lib.wkv7_gen_uniform_at.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
        lib.wkv7_gen_uniform_at.restype = ctypes.c_double
        lib.wkv7_gen_normal_at.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
        lib.wkv7_gen_normal_at.restype = ctypes.c_double
        lib.wkv7_gen_bf16_rne.argtypes = [ctypes.c_double]
        lib.wkv7_gen_bf16_rne.restype = ctypes.c_uint16
        dp = ctypes.POINTER(ctypes.c_double)
        lib.rwkv8_gen_inputs.argtypes = [ctypes.c_uint64] + [i] * 6 + [dp] * 6 + [ctypes.c_double] + [dp] * 2 + [i]
        lib.rwkv8_gen_inputs.restype = i
        lib.wkv7_gen_logits.argtypes = [ctypes.c_uint64, i, i, i, i, i, vp]
        lib.wkv7_gen_logits.restype = i
        _lib = lib
    return _lib


def generate(B: int, T: int, H: int, N: int, storage: str = "f64", s_init_std: float | None = None,
             seed: int = 0, nthreads: int = 0) -> dict:
    """Fill r, w, k, v, a, b, dy ([B][T][H][N]) and, if ``s_init_std`` is
    given, s_init ([B][H][N][N], float64; callers round it to the state type).

    ``storage`` is "f64", "f32" or "bf16" (bf16 arrays hold uint16 bit patterns).
    """
    lib = _load()
    shape = (B, T, H, N)
    out = {n: np.empty(shape, dtype=NP_STORAGE[storage]) for n in NAMES}
    s_init = np.empty((B, H, N, N), dtype=np.float64) if s_init_std is not None else None
    rc = lib.wkv7_gen_inputs(
        ctypes.c_uint64(seed), B, T, H, N, KIND[storage],
        *(out[n].ctypes.data_as(ctypes.c_void_p) for n in NAMES),
        None if s_init is None else s_init.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
        float(s_init_std or 0.0), nthreads)
    if rc != 0:
        raise RuntimeError(f"wkv7_gen_inputs failed with status {rc}")
    out["s_init"] = s_init
    return out


def generate_logits(B: int, T: int, H: int, N: int, storage: str = "f64", seed: int = 0) -> np.ndarray:
    """The decay logits z [B][T][H][N] behind generate()'s w (same seed):
    w = exp(-0.606531 sigmoid(z)). bf16 storage returns uint16 bit patterns."""
    lib = _load()
    z = np.empty((B, T, H, N), dtype=NP_STORAGE[storage])
    rc = lib.wkv7_gen_logits(ctypes.c_uint64(seed), B, T, H, N, KIND[storage], z.ctypes.data_as(ctypes.c_void_p))
    if rc != 0:
        raise RuntimeError(f"wkv7_gen_logits failed with status {rc}")
    return z


def bf16_bits_to_f64(u16: np.ndarray) -> np.ndarray:
    """Exact upcast of bfloat16 bit patterns (uint16) to float64."""
    return (u16.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def as_f64(x: np.ndarray, storage: str) -> np.ndarray:
    """The exact values a buffer of the given storage holds, as float64."""
    if storage == "bf16":
        return bf16_bits_to_f64(x)
    return np.asarray(x, dtype=np.float64)


def generate_rwkv8(B: int, T: int, H: int, Hv: int, L: int, E: int, storage: str = "f32",
                   state_std: float | None = None, boundary: bool = False, seed: int = 0,
                   nthreads: int = 0) -> dict:
    """Inputs of the RWKV-8 normalized recurrence (value semantics and draw
    order in ``wkv7_gen.c``, rwkv8_gen_inputs): q [B][H][T][L], v [B][Hv][T][E],
    decay [H][L], dy [B][H][T][E]; with ``state_std`` also rho_init and
    rho_norm_init, with ``boundary`` also d_rho_final and d_rho_norm_final
    (else those keys hold None). Drawn in double and rounded once to
    ``storage`` ("f64" or "f32")."""
    if storage not in ("f64", "f32"):
        raise ValueError("storage must be f64 or f32")
    lib = _load()
    dp = ctypes.POINTER(ctypes.c_double)
    arr = {
        "q": np.empty((B, H, T, L)), "v": np.empty((B, Hv, T, E)), "decay": np.empty((H, L)),
        "dy": np.empty((B, H, T, E)),
        "rho_init": np.empty((B, H, L, E)) if state_std is not None else None,
        "rho_norm_init": np.empty((B, H, L)) if state_std is not None else None,
        "d_rho_final": np.empty((B, H, L, E)) if boundary else None,
        "d_rho_norm_final": np.empty((B, H, L)) if boundary else None,
    }

    def ptr(x):
        return None if x is None else x.ctypes.data_as(dp)

    rc = lib.rwkv8_gen_inputs(
        ctypes.c_uint64(seed), B, T, H, Hv, L, E, ptr(arr["q"]), ptr(arr["v"]), ptr(arr["decay"]),
        ptr(arr["dy"]), ptr(arr["rho_init"]), ptr(arr["rho_norm_init"]), float(state_std or 0.0),
        ptr(arr["d_rho_final"]), ptr(arr["d_rho_norm_final"]), nthreads)
    if rc != 0:
        raise RuntimeError(f"rwkv8_gen_inputs failed with status {rc}")
    if storage == "f32":
        arr = {k: None if x is None else x.astype(np.float32) for k, x in arr.items()}
    return arr
