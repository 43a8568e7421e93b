"""Oracle of the scan's epilogue in the RWKV-7 time-mix: group norm per head
plus the "bonus" term, and its backward, in float64.

TEST INFRASTRUCTURE ONLY (the tests use it; the library's compute path never
does). Written from "rx_pretrain.c": gn_forward (mean and variance over the N
channels of each head, rstd = 1 / sqrt(var + 64e-5), then the per-channel
scale ln_x_w and shift ln_x_b), the post-scan loop of rx_timemix_forward_seq
(bonus_h = sum_j r_j k_j r_k[j] over the head's channels, added as
bonus_h * v), and the matching part of the time-mix backward (the bonus
backward and the group-norm backward that yields the scan's upstream
gradient dy). The gate g and the output projection that follow on the page
are outside the epilogue.

Layouts: y, r, k, v and the output [B][T][H][N]; ln_w, ln_b, r_k [H][N].
Every function is a plain loop over (b, t) vectorised over heads.
"""
from __future__ import annotations

import numpy as np

GN_EPS = 64e-5  # the variance guard of gn_forward


def forward(y, r, k, v, ln_w, ln_b, r_k):
    """out = group_norm(y) * ln_w + ln_b + bonus * v. Returns (out, stats)
    with stats = dict(mean, rstd, bonus), each [B][T][H]."""
    y, r, k, v = (np.asarray(x, dtype=np.float64) for x in (y, r, k, v))
    ln_w, ln_b, r_k = (np.asarray(x, dtype=np.float64) for x in (ln_w, ln_b, r_k))
    B, T, H, N = y.shape
    out = np.empty_like(y)
    mean = np.empty((B, T, H))
    rstd = np.empty((B, T, H))
    bonus = np.empty((B, T, H))
    for b in range(B):
        for t in range(T):
            yt = y[b, t]                                   # [H][N]
            m = yt.mean(axis=-1)
            var = ((yt - m[:, None]) ** 2).mean(axis=-1)
            rs = 1.0 / np.sqrt(var + GN_EPS)
            s = (r[b, t] * k[b, t] * r_k).sum(axis=-1)
            out[b, t] = (yt - m[:, None]) * rs[:, None] * ln_w + ln_b + s[:, None] * v[b, t]
            mean[b, t], rstd[b, t], bonus[b, t] = m, rs, s
    return out, {"mean": mean, "rstd": rstd, "bonus": bonus}


def backward(dout, y, r, k, v, ln_w, ln_b, r_k):
    """Gradients of sum <dout, out>: dy (the scan's upstream gradient), the
    bonus path's parts of dr, dk, dv, and the parameters' dln_w, dln_b, dr_k
    (summed over b and t)."""
    dout, y, r, k, v = (np.asarray(x, dtype=np.float64) for x in (dout, y, r, k, v))
    ln_w, r_k = np.asarray(ln_w, dtype=np.float64), np.asarray(r_k, dtype=np.float64)
    B, T, H, N = y.shape
    g = {n: np.empty_like(y) for n in ("dy", "dr", "dk", "dv")}
    g.update({n: np.zeros((H, N)) for n in ("dln_w", "dln_b", "dr_k")})
    for b in range(B):
        for t in range(T):
            yt, do = y[b, t], dout[b, t]
            m = yt.mean(axis=-1)
            var = ((yt - m[:, None]) ** 2).mean(axis=-1)
            rs = 1.0 / np.sqrt(var + GN_EPS)
            nv = (yt - m[:, None]) * rs[:, None]
            s = (r[b, t] * k[b, t] * r_k).sum(axis=-1)
            # bonus: out += s v with s = sum_j r_j k_j r_k[j]
            db = (do * v[b, t]).sum(axis=-1)
            g["dv"][b, t] = do * s[:, None]
            g["dr"][b, t] = db[:, None] * k[b, t] * r_k
            g["dk"][b, t] = db[:, None] * r[b, t] * r_k
            g["dr_k"] += db[:, None] * r[b, t] * k[b, t]
            # group norm: out += nv * ln_w + ln_b
            g["dln_w"] += do * nv
            g["dln_b"] += do
            dn = do * ln_w
            mdn = dn.mean(axis=-1)
            mdnn = (dn * nv).mean(axis=-1)
            g["dy"][b, t] = rs[:, None] * (dn - mdn[:, None] - nv * mdnn[:, None])
    return g
