"""Parity bars shared by the GPU tests of bf16-input paths.

The stated bar for bf16 inputs is a relative L2 error of at most 2e-2 against
the fp64 oracle. A whole-tensor norm hides a single wrong element or one
wrong step of a chunk, so every bf16 output is held to the bar three ways:

* whole tensor:       ||gpu - ref||_2 / ||ref||_2 <= 2e-2;
* per chunk:          the same ratio over every (b, h, 16-step chunk) of a
                      per-step output [B][T][H][X] (the ragged tail chunk
                      included) and over every (b, h) of a state [B][H][N][N];
* element by element: |gpu - ref| <= TAU * (|ref| + rms), rms the root mean
                      square of the reference over the element's chunk.

Floor. A chunk's own norm can be far below the tensor's typical chunk for a
reason that has nothing to do with the kernel: cancellation. A one-step tail
chunk of dv is dy (r . k), a single dot product times a vector, and when
r . k nearly cancels its rounding error is large against the result, though
small against the terms it sums. So every chunk's norm (and rms) is floored at
FLOOR = 0.1 of the tensor's typical chunk norm (rms over the tensor times the
square root of the chunk's element count). A wrong element of the tensor's
typical size still fails the chunk bar in any chunk (an error of one rms
against a floor of 0.1 * rms * 32 for a 16 x 64 chunk is 0.3), and the element
guard fails an element that is off by 0.1 of the tensor's rms even where its
chunk is near zero.

TAU comes from the rounding model of the chunked kernels: operands rounded to
bf16 (unit roundoff 2^-8) enter a chain of a few tensor-core products with
fp32 accumulation; an fp64 model of those roundings gives an element error of
RMS about 4.5e-3 of the element's scale (|ref| + its chunk's rms). The error is
not spread evenly: the worst chunk's relative error runs about twice the
tensor's (measured: 8e-3 against 4.3e-3 on the whole 4 x 4096 x 32 workload),
so sigma = 9e-3 there. A test compares at most about 2e8 elements, whose
largest Gaussian deviate is about sqrt(2 ln 2e8) = 6.2 standard deviations:
6.2 * 9e-3 = 5.6e-2, rounded up to TAU = 0.1. dw (and dz, its chain to the
logit) is formed from the identity w dw = anchor - sum x - a da, whose up to
eight terms x = r dr - k dk - b db + a da are each several times w dw itself,
so its errors are larger against its own scale: TAU_IDENTITY = 0.2. Largest
values seen over the GPU suite and every element of the whole workload:
0.057 (da) and 0.107 (dw). Either bar still fails an element that is wrong by
its own size (a sign flip scores 2 |ref| / (|ref| + rms), near 1).

Near-zero tensors: a reference that is exactly zero (dw at T = 1 from a zero
state) requires the GPU value to be zero as well.

PARITY_STATS (a file path) makes every check append its three figures as one
JSON line, for the record of how close each output comes to its bar.
"""
from __future__ import annotations

import json
import os

import numpy as np

REL_L2 = 2e-2
TAU = 0.1
TAU_IDENTITY = 0.2  # dw and dz
FLOOR = 0.1
CHUNK = 16


def _as4(x, kind):
    x = np.asarray(x, dtype=np.float64)
    if kind == "seq":
        if x.ndim == 2:  # one head: [T][X]
            x = x[None, :, None, :]
        elif x.ndim == 3:  # [B][T][H] scalars per row
            x = x[..., None]
    elif kind == "state":
        if x.ndim == 2:
            x = x[None, None]
    else:
        raise ValueError(kind)
    return x


def _blocks(x, kind):
    """Return (blocks [nblk][m] zero-padded, counts [nblk]) of the chunks."""
    if kind == "state":
        B, H = x.shape[:2]
        blk = x.reshape(B * H, -1)
        return blk, np.full(B * H, blk.shape[1])
    B, T, H = x.shape[:3]
    X = int(np.prod(x.shape[3:]))
    nck = max(1, -(-T // CHUNK))
    pad = np.zeros((B, nck * CHUNK, H, X))
    pad[:, :T] = x.reshape(B, T, H, X)
    blk = pad.reshape(B, nck, CHUNK, H, X).transpose(0, 1, 3, 2, 4).reshape(B * nck * H, CHUNK * X)
    steps = np.minimum(CHUNK, T - CHUNK * np.arange(nck))
    counts = np.broadcast_to((steps * X)[None, :, None], (B, nck, H)).reshape(-1)
    return blk, counts


def stats(got, ref, kind="seq"):
    """(whole-tensor rel L2, worst per-chunk rel L2, worst scaled element
    error) of got against ref; kind "seq" for [B][T][H][X] (or one head
    [T][X]) and "state" for [B][H][N][N]."""
    g = _as4(got, kind)
    r = _as4(ref, kind)
    assert g.shape == r.shape, (g.shape, r.shape)
    if r.size == 0:
        return 0.0, 0.0, 0.0
    rms_all = float(np.sqrt(np.mean(r * r)))
    whole = float(np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-300))
    gb, cnt = _blocks(g, kind)
    rb, _ = _blocks(r, kind)
    floor = max(FLOOR * rms_all, 1e-300)
    rms = np.maximum(np.sqrt((rb * rb).sum(1) / np.maximum(cnt, 1)), floor)
    err = np.abs(gb - rb)
    chunk = np.sqrt((err * err).sum(1)) / (rms * np.sqrt(np.maximum(cnt, 1)))
    elem = err / (np.abs(rb) + rms[:, None])
    return whole, float(chunk.max()), float(elem.max())


def _record(name, kind, s):
    path = os.environ.get("PARITY_STATS")
    if not path:
        return
    test = os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0]
    with open(path, "a") as f:
        f.write(json.dumps({"test": test, "name": name, "kind": kind, "whole": s[0], "chunk": s[1], "elem": s[2]}) + "\n")


def record_f32(name, scaled_max):
    """Record, under PARITY_STATS, an fp32 check's largest |gpu - ref| / (1 + |ref|)."""
    _record(name, "fp32", (float(scaled_max), float(scaled_max), float(scaled_max)))


def check_bf16(name, got, ref, kind="seq", tau=None):
    """Assert the bf16 bar on got against ref: whole tensor, every chunk, and
    every element (see the module docstring). The element guard takes
    TAU_IDENTITY for dw and dz (names starting so), TAU otherwise."""
    if tau is None:
        tau = TAU_IDENTITY if name.startswith(("dw", "dz")) else TAU
    g = np.asarray(got, dtype=np.float64)
    assert np.all(np.isfinite(g)), f"{name}: non-finite values"
    s = stats(g, ref, kind)
    _record(name, kind, s)
    whole, chunk, elem = s
    assert whole <= REL_L2, f"{name}: relative L2 error {whole:.3e} over the tensor"
    assert chunk <= REL_L2, f"{name}: relative L2 error {chunk:.3e} in its worst chunk (bar {REL_L2})"
    assert elem <= tau, f"{name}: scaled element error {elem:.3e} (bar {tau})"
