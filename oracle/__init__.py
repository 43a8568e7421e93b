"""WKV7 oracle: plain CPU reference of the RWKV-7 scan and its backward.

TEST INFRASTRUCTURE ONLY. The tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg use it; the library's compute path never does.
It shares no code with the CUDA kernels: the arithmetic lives in
``wkv7_oracle.cpp`` (written from the recurrence in "rx_pretrain.c",
rx_wkv7_forward_seq / rx_wkv7_backward), this module only marshals numpy
arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "wkv7_oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle_wkv7.so")

# -ffp-contract=off keeps a*b+c as two roundings on every host (aarch64 gcc
# would otherwise fuse them), so the oracle rounds the same way everywhere.
CXXFLAGS = ["-O2", "-std=c++17", "-fPIC", "-shared", "-pthread", "-ffp-contract=off"]


def compile_library(src: str, out: str) -> str:
    """Compile an oracle source file into a shared library."""
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["g++", *CXXFLAGS, "-o", tmp, src], check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the oracle into a shared library next to its source."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        compile_library(_SRC, _LIB)
    return _LIB


class Oracle:
    """ctypes handle on one build of the oracle library."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        fp = ctypes.POINTER(ctypes.c_float)
        i = ctypes.c_int
        for suffix, p in (("f64", dp), ("f32", fp)):
            fwd = getattr(lib, f"oracle_wkv7_forward_{suffix}")
            fwd.argtypes = [p] * 9 + [i] * 5
            fwd.restype = i
            bwd = getattr(lib, f"oracle_wkv7_backward_{suffix}")
            bwd.argtypes = [p] * 16 + [i] * 5
            bwd.restype = i
        self.lib = lib

    def forward(self, r, w, k, v, a, b, s_init=None, *, nthreads: int = 0, dtype=np.float64):
        """Forward scan. Inputs [B][T][H][N]; s_init [B][H][N][N] or None (zeros).

        Returns (y [B][T][H][N], s_final [B][H][N][N]) in ``dtype``.
        """
        r, w, k, v, a, b = (_prep(x, dtype) for x in (r, w, k, v, a, b))
        s_init = _prep(s_init, dtype)
        B, T, H, N = r.shape
        y = np.empty_like(r)
        s_final = np.empty((B, H, N, N), dtype=dtype)
        fn = self.lib.oracle_wkv7_forward_f64 if dtype == np.float64 else self.lib.oracle_wkv7_forward_f32
        rc = fn(*(_ptr(x, dtype) for x in (r, w, k, v, a, b, s_init, y, s_final)), B, T, H, N, nthreads)
        if rc != 0:
            raise RuntimeError(f"oracle forward failed with status {rc}")
        return y, s_final

    def backward(self, r, w, k, v, a, b, dy, s_init=None, dS_final=None, *, nthreads: int = 0,
                 dtype=np.float64):
        """Backward-through-time. Returns dict dr, dw, dk, dv, da, db ([B][T][H][N])
        and dS_init ([B][H][N][N]) in ``dtype``. dS_final ([B][H][N][N]) is the
        gradient entering through s_final; None means none (zeros).
        """
        r, w, k, v, a, b, dy = (_prep(x, dtype) for x in (r, w, k, v, a, b, dy))
        s_init = _prep(s_init, dtype)
        dS_final = _prep(dS_final, dtype)
        B, T, H, N = r.shape
        out = {n: np.empty_like(r) for n in ("dr", "dw", "dk", "dv", "da", "db")}
        out["dS_init"] = np.empty((B, H, N, N), dtype=dtype)
        fn = self.lib.oracle_wkv7_backward_f64 if dtype == np.float64 else self.lib.oracle_wkv7_backward_f32
        args = [_ptr(x, dtype) for x in (r, w, k, v, a, b, dy, s_init, dS_final)]
        args += [_ptr(out[n], dtype) for n in ("dr", "dw", "dk", "dv", "da", "db", "dS_init")]
        rc = fn(*args, B, T, H, N, nthreads)
        if rc != 0:
            raise RuntimeError(f"oracle backward failed with status {rc}")
        return out

    def backward_heads(self, r, w, k, v, a, b, dy, s_init, heads, *, nthreads: int = 0):
        """Oracle forward + backward for selected (b, h) pairs of a large workload.

        Each input is [B][T][H][N] (any float dtype, upcast to float64); s_init is
        [B][H][N][N] or None. Returns (y, s_final, grads) with a leading axis over
        ``heads``: y and the six input grads as [P][T][N], s_final and dS_init as
        [P][N][N].
        """
        sel = lambda x: np.stack([np.asarray(x[bi, :, hi, :], dtype=np.float64)
                                  for bi, hi in heads])[:, :, None, :]
        ins = [sel(x) for x in (r, w, k, v, a, b, dy)]
        si = None if s_init is None else np.stack(
            [np.asarray(s_init[bi, hi], dtype=np.float64) for bi, hi in heads])[:, None]
        y, s_final = self.forward(*ins[:6], si, nthreads=nthreads)
        g = self.backward(*ins, si, nthreads=nthreads)
        grads = {n: g[n][:, :, 0, :] for n in ("dr", "dw", "dk", "dv", "da", "db")}
        grads["dS_init"] = g["dS_init"][:, 0]
        return y[:, :, 0, :], s_final[:, 0], grads


def _ptr(x, dtype):
    if x is None:
        return None
    assert x.dtype == dtype and x.flags["C_CONTIGUOUS"], (x.dtype, x.flags)
    ctype = ctypes.c_double if dtype == np.float64 else ctypes.c_float
    return x.ctypes.data_as(ctypes.POINTER(ctype))


def _prep(x, dtype):
    return None if x is None else np.ascontiguousarray(x, dtype=dtype)


_default = None


def _get() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default


def forward(*args, **kw):
    return _get().forward(*args, **kw)


def backward(*args, **kw):
    return _get().backward(*args, **kw)


def backward_heads(*args, **kw):
    return _get().backward_heads(*args, **kw)


# ----------------------------------------------- decay given as logits ---
# The RWKV-7 time-mix ("rx_pretrain.c", tm_pre_forward) forms the decay from a
# logit z (its w0 + tanh(shw w1) w2) as w = exp(-RX_WDECAY_COEFF * sigmoid(z)),
# and its backward turns dw into the logit's gradient through
# dsig = dw * w * (-RX_WDECAY_COEFF), dz = dsig * sigmoid(z) * (1 - sigmoid(z)).
# These two functions are that chain around the scan, in float64.

WDECAY_COEFF = 0.606531  # RX_WDECAY_COEFF of "rx_pretrain.c"


def decay_from_logit(z):
    """w = exp(-0.606531 * sigmoid(z)), elementwise, float64."""
    z = np.asarray(z, dtype=np.float64)
    return np.exp(-WDECAY_COEFF / (1.0 + np.exp(-z)))


def forward_logit(r, z, k, v, a, b, s_init=None, **kw):
    """forward() with the decay given as logits z."""
    return forward(r, decay_from_logit(z), k, v, a, b, s_init, **kw)


def backward_logit(r, z, k, v, a, b, dy, s_init=None, dS_final=None, **kw):
    """backward() with the decay given as logits z: returns dz in place of dw."""
    z = np.asarray(z, dtype=np.float64)
    w = decay_from_logit(z)
    g = backward(r, w, k, v, a, b, dy, s_init, dS_final, **kw)
    sig = 1.0 / (1.0 + np.exp(-z))
    g["dz"] = g.pop("dw") * w * (-WDECAY_COEFF) * sig * (1.0 - sig)
    return g
