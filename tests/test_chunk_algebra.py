"""The chunk algebra the tensor-core kernels implement, written out in fp64
numpy and checked against the oracle (CPU only).

WKV7 ("rx_pretrain.c", rx_wkv7_forward_seq and the reverse scan of
rx_wkv7_backward, equations (1)-(3)): over a chunk of len steps with start
state S0 and running decay products c(t) = w_0 ... w_t (c(-1) = 1), the state
is S_t = S~_t diag(c(t)) and every step is a rank-2 update of S~. With
    A^ = a c(t-1), R^ = r c(t), K~ = k / c(t), B~ = b / c(t),
    Kb = k c_L / c(t), Bb = b c_L / c(t)           (c_L = c(len-1))
    Mka = A^ K~^T, Mba = A^ B~^T (strictly lower), Mkr = R^ K~^T, Mbr = R^ B~^T
    (lower with the diagonal), T = (I - Mba)^-1,
the forward is
    SA = T (A^ S0^T + Mka V),  Y = R^ S0^T + Mkr V + Mbr SA,
    S_end = S0 diag(c_L) + V^T Kb + SA^T Bb,
and the backward, with Gc the gradient of the state after the chunk,
    DSA = T^T (Bb Gc^T + Mbr^T DY),  DV = Kb Gc^T + Mkr^T DY + Mka^T DSA,
    DK~ = (V Gc) diag(c_L) + triu(V DY^T) R^ + triu(V DSA^T, 1) A^,    dk = DK~ / c
    DB~ = (SA Gc) diag(c_L) + triu(SA DY^T) R^ + triu(SA DSA^T, 1) A^, db = DB~ / c
    DR^ = DY S0 + tril(DY V^T) K~ + tril(DY SA^T) B~,                  dr = DR^ c
    DA^ = DSA S0 + tril(DSA V^T, -1) K~ + tril(DSA SA^T, -1) B~,        da = DA^ c(t-1)
    Gc' = Gc diag(c_L) + DY^T R^ + DSA^T A^                     (the carry)
    w dw = colsum(Gc' o S0) - sum_{u<t} x(u) - a da,  x = r dr - k dk - b db + a da
         = sum_{u>=t} x(u) - a da + colsum(Gc o S_end)          (both anchors),
with the anchors from the chunk's own column products
    colsum(Gc o S_end) = c_L colsum(Gc o S0) + sum_t (Kb o V Gc + Bb o SA Gc)
    colsum(Gc' o S0)   = c_L colsum(Gc o S0) + sum_t (R^ o DY S0 + A^ o DSA S0).

RWKV-8 ("src/sequence/rwkv8/backward.rs", burn_dragon_kernel): the chunk
closed forms with non-negative powers of the fixed decay d only
    n_tau = d^tau n0 + sum_{s<tau} d^(tau-1-s) q_s,  U = qw / (n + EPS)
    y_tau = (U[tau] d^tau)^T rho0 + sum_{s<tau} A[tau][s] v_s,
    A[tau][s] = sum_l U[tau][l] q_s[l] d_l^(tau-1-s)
    rho_end = d^len rho0 + sum_s (q_s d^(len-1-s)) v_s^T
and the backward of the chunk: R, Gv, dv, Gn and the four closed-form decay
terms (with the norm term sum_tau Gn_tau n_tau).

Inputs: seeded normal draws (numpy), decays in the RWKV-7 range, lengths
that leave a ragged last chunk; every output of the oracle is matched to
1e-11 relative.
"""
import importlib.util
import os

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rel(name, got, ref, tol=1e-11):
    err = np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-300)
    assert err <= tol, f"{name}: max relative error {err:.3e}"


# ------------------------------------------------------------------ WKV7 ---

def wkv7_chunk_forward(S0, r, w, k, v, a, b):
    """One chunk (rows t = 0 .. len-1, columns j of the key side, i of the
    value side). Returns (Y, SA, S_end, the chunk's operands)."""
    L = r.shape[0]
    c = np.cumprod(w, axis=0)
    cprev = np.vstack([np.ones((1, w.shape[1])), c[:-1]])
    cL = c[-1]
    Ah, Rh, Kt, Bt = a * cprev, r * c, k / c, b / c
    Kb, Bb = k * cL / c, b * cL / c
    Mka, Mba = np.tril(Ah @ Kt.T, -1), np.tril(Ah @ Bt.T, -1)
    Mkr, Mbr = np.tril(Rh @ Kt.T), np.tril(Rh @ Bt.T)
    Tm = np.linalg.inv(np.eye(L) - Mba)
    SA = Tm @ (Ah @ S0.T + Mka @ v)
    Y = Rh @ S0.T + Mkr @ v + Mbr @ SA
    S_end = S0 * cL[None, :] + v.T @ Kb + SA.T @ Bb
    ops = dict(c=c, cprev=cprev, cL=cL, Ah=Ah, Rh=Rh, Kt=Kt, Bt=Bt, Kb=Kb, Bb=Bb, Mka=Mka, Mkr=Mkr, Mbr=Mbr, Tm=Tm)
    return Y, SA, S_end, ops


def wkv7_chunk_backward(S0, r, w, k, v, a, b, dy, Gc):
    """Gradients of one chunk given the gradient Gc of the state after it.
    Returns (dr, dw, dk, dv, da, db, Gc' = gradient of S0), dw by both anchors."""
    Y, SA, S_end, o = wkv7_chunk_forward(S0, r, w, k, v, a, b)
    Ah, Rh, Kt, Bt, Kb, Bb = (o[n] for n in ("Ah", "Rh", "Kt", "Bt", "Kb", "Bb"))
    c, cprev, cL = o["c"], o["cprev"], o["cL"]
    DSA = o["Tm"].T @ (Bb @ Gc.T + o["Mbr"].T @ dy)
    DV = Kb @ Gc.T + o["Mkr"].T @ dy + o["Mka"].T @ DSA
    DKt = (v @ Gc) * cL[None, :] + np.triu(v @ dy.T) @ Rh + np.triu(v @ DSA.T, 1) @ Ah
    DBt = (SA @ Gc) * cL[None, :] + np.triu(SA @ dy.T) @ Rh + np.triu(SA @ DSA.T, 1) @ Ah
    DRh = dy @ S0 + np.tril(dy @ v.T) @ Kt + np.tril(dy @ SA.T) @ Bt
    DAh = DSA @ S0 + np.tril(DSA @ v.T, -1) @ Kt + np.tril(DSA @ SA.T, -1) @ Bt
    dk, db, dr, da = DKt / c, DBt / c, DRh * c, DAh * cprev
    Gc_prev = Gc * cL[None, :] + dy.T @ Rh + DSA.T @ Ah
    x = r * dr - k * dk - b * db + a * da
    # the output kernel takes both anchors from the chunk's own column products
    base = cL * (Gc * S0).sum(axis=0)
    _rel("colsum(Gc o S_end)", base + (Kb * (v @ Gc) + Bb * (SA @ Gc)).sum(axis=0), (Gc * S_end).sum(axis=0), 1e-10)
    _rel("colsum(Gc' o S0)", base + (Rh * (dy @ S0) + Ah * (DSA @ S0)).sum(axis=0), (Gc_prev * S0).sum(axis=0), 1e-10)
    start = (Gc_prev * S0).sum(axis=0) - np.vstack([np.zeros((1, x.shape[1])), np.cumsum(x, axis=0)[:-1]]) - a * da
    end = np.cumsum(x[::-1], axis=0)[::-1] - a * da + (Gc * S_end).sum(axis=0)
    return dr, start / w, end / w, dk, DV, da, db, Gc_prev


def _wkv7_inputs(T, N, seed):
    rng = np.random.default_rng(seed)
    f = lambda *s: rng.standard_normal(s)  # noqa: E731
    w = np.exp(-0.606531 / (1 + np.exp(-f(T, N))))  # the RWKV-7 decay range
    kk = f(T, N)
    kk /= np.linalg.norm(kk, axis=1, keepdims=True)
    # a = -kappa, b = kappa * alpha: the stable in-context form of the update
    alpha = rng.uniform(0.2, 1.0, (T, N))
    return dict(r=f(T, N) / np.sqrt(N), w=w, k=f(T, N) / np.sqrt(N), v=f(T, N), a=-kk, b=kk * alpha,
                dy=f(T, N), s0=0.3 * f(N, N), dsf=f(N, N))


@pytest.mark.parametrize("T,L", [(11, 4), (16, 16), (37, 16), (5, 8)])
def test_wkv7_chunk_algebra_matches_the_oracle(T, L):
    import __graft_entry__  # noqa: F401
    import oracle

    N = 4
    d = _wkv7_inputs(T, N, seed=T * 100 + L)
    shape = lambda x: x[None, :, None, :]  # noqa: E731  [B=1][T][H=1][N]
    y_ref, sf_ref = oracle.forward(*(shape(d[n]) for n in "rwkvab"), d["s0"][None, None])
    g_ref = oracle.backward(*(shape(d[n]) for n in "rwkvab"), shape(d["dy"]), d["s0"][None, None],
                            d["dsf"][None, None])
    # forward chunk by chunk
    S, ys, starts = d["s0"], [], []
    for t0 in range(0, T, L):
        sl = slice(t0, min(T, t0 + L))
        starts.append(S)
        Y, _, S, _ = wkv7_chunk_forward(S, *(d[n][sl] for n in "rwkvab"))
        ys.append(Y)
    _rel("y", np.vstack(ys), y_ref[0, :, 0])
    _rel("s_final", S, sf_ref[0, 0])
    # backward chunk by chunk in reverse, the carry entering as Gc
    Gc, out = d["dsf"], {n: [] for n in ("dr", "dw_start", "dw_end", "dk", "dv", "da", "db")}
    for ci, t0 in reversed(list(enumerate(range(0, T, L)))):
        sl = slice(t0, min(T, t0 + L))
        *g, Gc = wkv7_chunk_backward(starts[ci], *(d[n][sl] for n in "rwkvab"), d["dy"][sl], Gc)
        for n, x in zip(out, g):
            out[n].insert(0, x)
    for n in ("dr", "dk", "dv", "da", "db"):
        _rel(n, np.vstack(out[n]), g_ref[n][0, :, 0])
    _rel("dw (start anchor)", np.vstack(out["dw_start"]), g_ref["dw"][0, :, 0], 1e-9)
    _rel("dw (end anchor)", np.vstack(out["dw_end"]), g_ref["dw"][0, :, 0], 1e-9)
    _rel("dS_init", Gc, g_ref["dS_init"][0, 0])


# ---------------------------------------------------------------- RWKV-8 ---

EPS = 1e-6


def _pw(d, upto):
    return d[None, :] ** np.arange(upto + 1)[:, None]  # pw[k][l] = d_l^k


def _norm_before(n0, q, pw):
    ln = q.shape[0]
    return np.array([pw[tau] * n0 + sum(pw[tau - 1 - s] * q[s] for s in range(tau)) for tau in range(ln)])


def rwkv8_chunk_forward(rho0, n0, q, v, d):
    """One chunk of the normalized recurrence from its start state:
    returns (y, rho_end, n_end)."""
    ln = q.shape[0]
    pw = _pw(d, ln)
    n = _norm_before(n0, q, pw)
    U = q / (q.sum(axis=1, keepdims=True) + EPS) / (n + EPS)
    A = np.zeros((ln, ln))
    for tau in range(ln):
        for s in range(tau):
            A[tau, s] = (U[tau] * q[s] * pw[tau - 1 - s]).sum()
    y = (U * pw[:ln]) @ rho0 + A @ v
    qt = q * pw[ln - 1 - np.arange(ln)]
    return y, pw[ln][:, None] * rho0 + qt.T @ v, pw[ln] * n0 + qt.sum(axis=0)


def rwkv8_chunk_backward(rho0, n0, q, v, d, dy, G15, Gn15):
    """Gradients of one chunk given G15, Gn15 (the gradients of the state
    after its last step): returns (dq, dv, ddecay, G_start, Gn_start)."""
    ln = q.shape[0]
    pw = _pw(d, ln)
    n = _norm_before(n0, q, pw)
    sq = q.sum(axis=1) + EPS
    qw = q / sq[:, None]
    U = qw / (n + EPS)
    M, R0, W = dy @ v.T, dy @ rho0.T, v @ G15.T
    R = np.array([pw[tau] * R0[tau] + sum(pw[tau - 1 - s] * q[s] * M[tau, s] for s in range(tau))
                  for tau in range(ln)])
    g_qw = R / (n + EPS)
    g_n = -U * g_qw
    Gv = np.array([pw[ln - 1 - tau] * W[tau] + sum(pw[s - 1 - tau] * U[s] * M[s, tau] for s in range(tau + 1, ln))
                   for tau in range(ln)])
    Gn = np.array([pw[ln - 1 - tau] * Gn15 + sum(pw[s - 1 - tau] * g_n[s] for s in range(tau + 1, ln))
                   for tau in range(ln)])
    dq = (g_qw - (g_qw * qw).sum(axis=1, keepdims=True)) / sq[:, None] + Gv + Gn
    A = np.zeros((ln, ln))  # A[s][tau] = sum_l U[s] q_tau d^(s-1-tau), s > tau
    for s in range(ln):
        for tau in range(s):
            A[s, tau] = (U[s] * q[tau] * pw[s - 1 - tau]).sum()
    dv = (q * pw[ln - 1 - np.arange(ln)]) @ G15 + A.T @ dy
    G_start = pw[ln][:, None] * G15 + (U * pw[:ln]).T @ dy
    Gn_start = pw[ln] * Gn15 + (pw[:ln] * g_n).sum(axis=0)
    dd = ln * pw[ln - 1] * (G15 * rho0).sum(axis=1)
    for s in range(1, ln):
        dd = dd + s * pw[s - 1] * U[s] * R0[s]
    for s in range(ln - 1):
        dd = dd + (ln - 1 - s) * pw[ln - 2 - s] * q[s] * W[s]
    for s in range(ln):
        for s2 in range(s - 1):
            dd = dd + (s - 1 - s2) * pw[s - 2 - s2] * q[s2] * U[s] * M[s, s2]
    dd = dd + (Gn * n).sum(axis=0)
    return dq, dv, dd, G_start, Gn_start


def _load_rwkv8_oracle():
    spec = importlib.util.spec_from_file_location("rwkv8_oracle", os.path.join(ROOT, "oracle", "rwkv8_oracle.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.parametrize("T,C", [(11, 4), (16, 16), (37, 16), (3, 8)])
def test_rwkv8_chunk_algebra_matches_the_oracle(T, C):
    orc = _load_rwkv8_oracle()
    L, E = 5, 3
    rng = np.random.default_rng(T * 10 + C)
    q = np.maximum(rng.standard_normal((T, L)), 0.0)
    v = rng.standard_normal((T, E))
    d = np.exp(-0.606531 / (1 + np.exp(-rng.standard_normal(L))))
    dy = rng.standard_normal((T, E))
    rho_init, n_init = 0.1 * rng.standard_normal((L, E)), 0.1 * np.abs(rng.standard_normal(L))
    d_rho_final, d_n_final = rng.standard_normal((L, E)), rng.standard_normal(L)
    y_ref, rf_ref, nf_ref = orc.forward(q[None, None], v[None, None], d[None], rho_init[None, None], n_init[None, None])
    g_ref = orc.backward(q[None, None], v[None, None], d[None], dy[None, None], rho_init[None, None],
                         n_init[None, None], d_rho_final[None, None], d_n_final[None, None])
    rho, n, ys, starts = rho_init, n_init, [], []
    chunks = [slice(t0, min(T, t0 + C)) for t0 in range(0, T, C)]
    for sl in chunks:
        starts.append((rho, n))
        y, rho, n = rwkv8_chunk_forward(rho, n, q[sl], v[sl], d)
        ys.append(y)
    _rel("y", np.vstack(ys), y_ref[0, 0])
    _rel("rho_final", rho, rf_ref[0, 0])
    _rel("rho_norm_final", n, nf_ref[0, 0])
    G, Gn, dd = d_rho_final, d_n_final, np.zeros(L)
    dq, dv = [None] * len(chunks), [None] * len(chunks)
    for ci in reversed(range(len(chunks))):
        sl = chunks[ci]
        dq[ci], dv[ci], ddc, G, Gn = rwkv8_chunk_backward(*starts[ci], q[sl], v[sl], d, dy[sl], G, Gn)
        dd = dd + ddc
    _rel("dq", np.vstack(dq), g_ref["dq"][0, 0])
    _rel("dv", np.vstack(dv), g_ref["dv"][0, 0])
    _rel("ddecay", dd, g_ref["ddecay"][0], 1e-10)
    _rel("d_rho_init", G, g_ref["d_rho_init"][0, 0])
    _rel("d_rho_norm_init", Gn, g_ref["d_rho_norm_init"][0, 0])


def test_rwkv8_backward_splits_into_chains_and_chunks():
    """The backward split the way the forward is: the carried G of every column
    block alone (G_start = d^len G15 + (U d^s)^T DY over the block's columns),
    Gn as the sum over blocks of partial chains built from each block's part
    of R (g_n is linear in R), then every chunk's gradients from its (G15,
    Gn15) alone. Against the oracle; the algebra a split backward kernel rests on."""
    orc = _load_rwkv8_oracle()
    rng = np.random.default_rng(5)
    T, C, L, E, NB = 37, 8, 6, 8, 4
    W = E // NB
    q = np.maximum(rng.standard_normal((T, L)), 0.0)
    v, dy = rng.standard_normal((T, E)), rng.standard_normal((T, E))
    d = np.exp(-0.606531 / (1 + np.exp(-rng.standard_normal(L))))
    rho_i, n_i = 0.1 * rng.standard_normal((L, E)), 0.1 * np.abs(rng.standard_normal(L))
    dG, dGn = rng.standard_normal((L, E)), rng.standard_normal(L)
    g_ref = orc.backward(q[None, None], v[None, None], d[None], dy[None, None], rho_i[None, None],
                         n_i[None, None], dG[None, None], dGn[None, None])
    chunks = [slice(t0, min(T, t0 + C)) for t0 in range(0, T, C)]
    starts, rho, n = [], rho_i, n_i
    for sl in chunks:
        starts.append((rho, n))
        _, rho, n = rwkv8_chunk_forward(rho, n, q[sl], v[sl], d)
    # the chains alone, per column block
    G15, Gn15 = [None] * len(chunks), [None] * len(chunks)
    Gb = [dG[:, cb * W:(cb + 1) * W].copy() for cb in range(NB)]
    Gnp = [dGn.copy() if cb == 0 else np.zeros(L) for cb in range(NB)]
    for ci in reversed(range(len(chunks))):
        sl = chunks[ci]
        rho0, n0 = starts[ci]
        ln = sl.stop - sl.start
        G15[ci], Gn15[ci] = np.hstack(Gb), sum(Gnp)
        pw = _pw(d, ln)
        nb = _norm_before(n0, q[sl], pw)
        U = q[sl] / (q[sl].sum(axis=1, keepdims=True) + EPS) / (nb + EPS)
        for cb in range(NB):
            cs = slice(cb * W, (cb + 1) * W)
            Mp, R0p = dy[sl][:, cs] @ v[sl][:, cs].T, dy[sl][:, cs] @ rho0[:, cs].T
            Rp = np.array([pw[t] * R0p[t] + sum(pw[t - 1 - s] * q[sl][s] * Mp[t, s] for s in range(t))
                           for t in range(ln)])
            Gnp[cb] = pw[ln] * Gnp[cb] + (pw[:ln] * (-U * Rp / (nb + EPS))).sum(axis=0)
            Gb[cb] = pw[ln][:, None] * Gb[cb] + (U * pw[:ln]).T @ dy[sl][:, cs]
    _rel("d_rho_init", np.hstack(Gb), g_ref["d_rho_init"][0, 0])
    _rel("d_rho_norm_init", sum(Gnp), g_ref["d_rho_norm_init"][0, 0])
    # every chunk from its own (G15, Gn15)
    dq, dv, dd = [], [], np.zeros(L)
    for ci, sl in enumerate(chunks):
        a, b, c, _, _ = rwkv8_chunk_backward(*starts[ci], q[sl], v[sl], d, dy[sl], G15[ci], Gn15[ci])
        dq.append(a)
        dv.append(b)
        dd = dd + c
    _rel("dq", np.vstack(dq), g_ref["dq"][0, 0])
    _rel("dv", np.vstack(dv), g_ref["dv"][0, 0])
    _rel("ddecay", dd, g_ref["ddecay"][0], 1e-10)
