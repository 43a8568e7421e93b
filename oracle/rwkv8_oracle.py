"""RWKV-8 oracle: plain fp64 CPU reference of the normalized linear recurrence
with a time-invariant decay, and of its backward.

TEST INFRASTRUCTURE ONLY. The tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg use it; the library's compute path never does,
and it shares no code with the CUDA kernels.

Source: the burn_dragon_kernel page "src/sequence/rwkv8/backward.rs".
  * compute_chunk_traces: the state update is delta = q (x) v added to a
    decayed state, with a "before" trace (the state each step reads is the one
    before that step's update).
  * backward_chunk_impl: the readout and the formulas of its gradient:
    query weights qw = q / (sum_l q + EPS), normalized state
    rho / (rho_norm + EPS), y_t[e] = sum_l qw_t[l] rho_before_t[l, e] /
    (rho_norm_before_t[l] + EPS); the reverse carries of the state gradient and
    of the norm gradient; grad_value = sum_l G q, grad_query = the weights'
    gradient + sum_e G v + the norm carry, grad_decay = sum over batch and
    time of sum_e G rho_before + Gn rho_norm_before.
  * EPS = 1e-6 (the module constant).
The recurrence bodies themselves (rwkv8_forward_recurrence_before_*) are not
on the page. Their plainest reading, which the page's gradient formulas fix
(grad_decay multiplies the carry by rho_before, the carry runs as the same
"before" recurrence on reversed time):
    rho_before_0 = rho_init (zeros if absent), n_before_0 = rho_norm_init
    rho_after_t  = decay (.) rho_before_t + q_t (x) v_t   (decay per row l)
    n_after_t    = decay (.) n_before_t + q_t
    rho_before_{t+1} = rho_after_t
The backward carry G_t = dL/d rho_after_t starts at the gradient entering
through the final state (the page starts it at zero: boundary_grad_rho_after
is zeros in the sequential fallback) and runs
    G_{t-1} = decay (.) G_t + (gradient of y_t w.r.t. rho_before_t)
so that after t = 0 it is the gradient of rho_init.

Layouts follow the page: q [B][H][T][L], v [B][Hv][T][E] with Hv = 1 (one
value row shared by every head) or Hv = H, decay [H][L] (the page's
[1, H, L]), y and dy [B][H][T][E], states rho [B][H][L][E], rho_norm [B][H][L].
With Hv = 1 the value gradient is summed over heads (the page's value_heads
== 1 branch).

Every function loops over time in plain numpy, vectorised over (b, h) only.
"""
from __future__ import annotations

import numpy as np

EPS = 1.0e-6


def _value_per_head(v: np.ndarray, H: int) -> np.ndarray:
    Hv = v.shape[1]
    if Hv == H:
        return v
    if Hv != 1:
        raise ValueError(f"value heads {Hv} must be 1 or {H}")
    return np.broadcast_to(v, (v.shape[0], H) + v.shape[2:])


def _check(q, v, decay):
    if q.ndim != 4 or v.ndim != 4 or decay.ndim != 2:
        raise ValueError("q [B][H][T][L], v [B][Hv][T][E], decay [H][L]")
    B, H, T, L = q.shape
    if v.shape[0] != B or v.shape[2] != T or decay.shape != (H, L):
        raise ValueError("inconsistent shapes")
    return B, H, T, L, v.shape[3]


def forward(q, v, decay, rho_init=None, rho_norm_init=None, *, history=False):
    """Forward scan in float64.

    Returns (y, rho_final, rho_norm_final) and, with ``history``, also the
    states every step read: rho_before [B][H][T][L][E], n_before [B][H][T][L].
    """
    q = np.asarray(q, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    decay = np.asarray(decay, dtype=np.float64)
    B, H, T, L, E = _check(q, v, decay)
    vh = _value_per_head(v, H)
    rho = np.zeros((B, H, L, E)) if rho_init is None else np.array(rho_init, dtype=np.float64)
    n = np.zeros((B, H, L)) if rho_norm_init is None else np.array(rho_norm_init, dtype=np.float64)
    d = decay[None, :, :]
    y = np.empty((B, H, T, E))
    hist_rho = np.empty((B, H, T, L, E)) if history else None
    hist_n = np.empty((B, H, T, L)) if history else None
    for t in range(T):
        qt = q[:, :, t, :]
        if history:
            hist_rho[:, :, t] = rho
            hist_n[:, :, t] = n
        # readout of the state before this step's update
        qw = qt / (qt.sum(axis=-1, keepdims=True) + EPS)
        rho_hat = rho / (n[..., None] + EPS)
        y[:, :, t, :] = np.einsum("bhl,bhle->bhe", qw, rho_hat)
        # state update: decay each row l, add q (x) v
        rho = d[..., None] * rho + qt[..., None] * vh[:, :, t, None, :]
        n = d * n + qt
    if history:
        return y, rho, n, hist_rho, hist_n
    return y, rho, n


def backward(q, v, decay, dy, rho_init=None, rho_norm_init=None, d_rho_final=None, d_rho_norm_final=None):
    """Backward-through-time in float64 for the loss
    L = sum <dy, y> + <d_rho_final, rho_final> + <d_rho_norm_final, rho_norm_final>.

    Returns a dict with dq [B][H][T][L], dv (v's shape), ddecay [H][L],
    d_rho_init [B][H][L][E] and d_rho_norm_init [B][H][L].
    """
    q = np.asarray(q, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    dy = np.asarray(dy, dtype=np.float64)
    decay = np.asarray(decay, dtype=np.float64)
    B, H, T, L, E = _check(q, v, decay)
    Hv = v.shape[1]
    vh = _value_per_head(v, H)
    _, _, _, hist_rho, hist_n = forward(q, v, decay, rho_init, rho_norm_init, history=True)
    d = decay[None, :, :]
    G = np.zeros((B, H, L, E)) if d_rho_final is None else np.array(d_rho_final, dtype=np.float64)
    Gn = np.zeros((B, H, L)) if d_rho_norm_final is None else np.array(d_rho_norm_final, dtype=np.float64)
    dq = np.empty((B, H, T, L))
    dv_h = np.empty((B, H, T, E))
    ddecay = np.zeros((H, L))
    for t in range(T - 1, -1, -1):
        # here G = dL/d rho_after_t and Gn = dL/d n_after_t
        qt, vt, dyt = q[:, :, t, :], vh[:, :, t, :], dy[:, :, t, :]
        rb, nb = hist_rho[:, :, t], hist_n[:, :, t]
        # through the update rho_after = decay rho_before + q v, n_after = decay n_before + q
        dq_t = np.einsum("bhle,bhe->bhl", G, vt) + Gn
        dv_h[:, :, t, :] = np.einsum("bhle,bhl->bhe", G, qt)
        ddecay += (np.einsum("bhle,bhle->bhl", G, rb) + Gn * nb).sum(axis=0)
        # through the readout y_t = sum_l qw[l] rb[l, :] / (nb[l] + EPS)
        s = qt.sum(axis=-1, keepdims=True) + EPS
        qw = qt / s
        den = nb + EPS
        g_qw = np.einsum("bhe,bhle->bhl", dyt, rb / den[..., None])
        g_rhat = qw[..., None] * dyt[:, :, None, :]
        g_rb = g_rhat / den[..., None]
        g_nb = -np.einsum("bhle,bhle->bhl", g_rhat, rb) / den ** 2
        dq_t += (g_qw - (g_qw * qw).sum(axis=-1, keepdims=True)) / s
        dq[:, :, t, :] = dq_t
        # carry to the previous step's after-state
        G = d[..., None] * G + g_rb
        Gn = d * Gn + g_nb
    dv = dv_h if Hv == H else dv_h.sum(axis=1, keepdims=True)
    return {"dq": dq, "dv": dv, "ddecay": ddecay, "d_rho_init": G, "d_rho_norm_init": Gn}
