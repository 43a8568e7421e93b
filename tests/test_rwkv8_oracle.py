"""Pins of the RWKV-8 oracle (oracle/rwkv8_oracle.py) to what the page and the
mathematics fix, independently of the oracle's own loop:

* the forward against its closed form, the sums
      rho_before_t = decay^t rho_init + sum_{s<t} decay^(t-1-s) q_s v_s^T,
      n_before_t   = decay^t n_init   + sum_{s<t} decay^(t-1-s) q_s,
  evaluated term by term (O(T^2) brute force), with the readout of
  "sequence/rwkv8/backward.rs" (backward_chunk_impl: query weights
  q / (sum q + EPS), state / (norm + EPS));
* decay = 1 (exclusive prefix sums, numpy cumsum) and decay = 0 (only the
  previous token is seen);
* every gradient against fp64 central finite differences of
  L = sum <dy, y> + <D_rho, rho_final> + <D_n, rho_norm_final>;
* the Euler identity of the part of L that is linear in (v, rho_init);
* one value row shared by every head equals that row copied to every head,
  with the value gradient summed over heads;
* causality: y_t depends on q_s for s <= t and on v_s only for s < t.
A mistake planted in the oracle must fail at least one of these
(test_rwkv8_oracle_mutants.py).
"""
import importlib.util
import os

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ORACLE_PATH = os.path.join(ROOT, "oracle", "rwkv8_oracle.py")
EPS = 1.0e-6  # the page's module constant


def load_oracle(path=ORACLE_PATH, name="rwkv8_oracle_under_test"):
    spec = importlib.util.spec_from_file_location(name, path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _inputs(B, T, H, Hv, L, E, seed, state=True, boundary=True):
    rng = np.random.default_rng(seed)
    d = {
        "q": np.abs(rng.standard_normal((B, H, T, L))) + 0.05,
        "v": rng.standard_normal((B, Hv, T, E)),
        "decay": rng.uniform(0.3, 0.95, (H, L)),
        "dy": rng.standard_normal((B, H, T, E)),
        "rho_init": 0.3 * rng.standard_normal((B, H, L, E)) if state else None,
        "rho_norm_init": 0.3 * np.abs(rng.standard_normal((B, H, L))) if state else None,
        "d_rho_final": rng.standard_normal((B, H, L, E)) if boundary else None,
        "d_rho_norm_final": rng.standard_normal((B, H, L)) if boundary else None,
    }
    return d


def _brute_forward(q, v, decay, rho0, n0):
    """y from the closed-form sums, one output at a time."""
    B, H, T, L = q.shape
    Hv, E = v.shape[1], v.shape[3]
    y = np.zeros((B, H, T, E))
    for b in range(B):
        for h in range(H):
            hv = 0 if Hv == 1 else h
            for t in range(T):
                rho = np.zeros((L, E)) if rho0 is None else rho0[b, h] * (decay[h] ** t)[:, None]
                n = np.zeros(L) if n0 is None else n0[b, h] * decay[h] ** t
                for s in range(t):
                    f = decay[h] ** (t - 1 - s)
                    rho = rho + (f * q[b, h, s])[:, None] * v[b, hv, s][None, :]
                    n = n + f * q[b, h, s]
                weights = q[b, h, t] / (q[b, h, t].sum() + EPS)
                for e in range(E):
                    y[b, h, t, e] = sum(weights[l] * rho[l, e] / (n[l] + EPS) for l in range(L))
    return y


def _loss(orc, d, **over):
    x = dict(d)
    x.update(over)
    y, rho, n = orc.forward(x["q"], x["v"], x["decay"], x["rho_init"], x["rho_norm_init"])
    L = float(np.sum(x["dy"] * y))
    if x["d_rho_final"] is not None:
        L += float(np.sum(x["d_rho_final"] * rho))
    if x["d_rho_norm_final"] is not None:
        L += float(np.sum(x["d_rho_norm_final"] * n))
    return L


# ---------------------------------------------------------------- pins


def pin_closed_form(orc):
    for Hv in (1, 2):
        d = _inputs(2, 6, 2, Hv, 3, 4, seed=1 + Hv)
        y, rho, n = orc.forward(d["q"], d["v"], d["decay"], d["rho_init"], d["rho_norm_init"])
        ref = _brute_forward(d["q"], d["v"], d["decay"], d["rho_init"], d["rho_norm_init"])
        np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-13)
        # the final state is the before-state of a step T
        T = d["q"].shape[2]
        vv = d["v"] if Hv == 2 else np.repeat(d["v"], 2, axis=1)
        fr = d["rho_init"] * (d["decay"] ** T)[None, :, :, None]
        fn = d["rho_norm_init"] * (d["decay"] ** T)[None]
        for s in range(T):
            f = d["decay"] ** (T - 1 - s)
            fr = fr + (f[None] * d["q"][:, :, s])[..., None] * vv[:, :, s, None, :]
            fn = fn + f[None] * d["q"][:, :, s]
        np.testing.assert_allclose(rho, fr, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(n, fn, rtol=1e-12, atol=1e-13)


def pin_unit_decay_prefix_sums(orc):
    d = _inputs(1, 9, 2, 2, 4, 3, seed=7, state=False)
    decay = np.ones_like(d["decay"])
    y, rho, n = orc.forward(d["q"], d["v"], decay)
    qv = d["q"][..., :, None] * d["v"][..., None, :]  # [B][H][T][L][E]
    rho_b = np.cumsum(qv, axis=2) - qv
    n_b = np.cumsum(d["q"], axis=2) - d["q"]
    w = d["q"] / (d["q"].sum(-1, keepdims=True) + EPS)
    ref = np.einsum("bhtl,bhtle->bhte", w, rho_b / (n_b[..., None] + EPS))
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(rho, qv.sum(axis=2), rtol=1e-12)
    np.testing.assert_allclose(n, d["q"].sum(axis=2), rtol=1e-12)


def pin_zero_decay_previous_token(orc):
    d = _inputs(2, 7, 2, 1, 3, 5, seed=8, state=False)
    decay = np.zeros_like(d["decay"])
    y, _, _ = orc.forward(d["q"], d["v"], decay)
    q, v = d["q"], d["v"]
    w = q / (q.sum(-1, keepdims=True) + EPS)
    assert np.all(y[:, :, 0] == 0.0)
    frac = q[:, :, :-1] / (q[:, :, :-1] + EPS)  # rho / (n + EPS) for the previous token
    ref = np.einsum("bhtl,bhtl->bht", w[:, :, 1:], frac)[..., None] * v[:, :, :-1][:, :, :, :]
    np.testing.assert_allclose(y[:, :, 1:], ref, rtol=1e-12, atol=1e-14)


def pin_finite_differences(orc):
    """Every gradient against central differences (h = 1e-6) of the loss."""
    for Hv, state, boundary in ((2, True, True), (1, True, True), (2, False, False)):
        d = _inputs(2, 5, 2, Hv, 3, 2, seed=11 + Hv + 2 * state, state=state, boundary=boundary)
        g = orc.backward(d["q"], d["v"], d["decay"], d["dy"], d["rho_init"], d["rho_norm_init"], d["d_rho_final"],
                         d["d_rho_norm_final"])
        names = [("q", "dq"), ("v", "dv"), ("decay", "ddecay")]
        if state:
            names += [("rho_init", "d_rho_init"), ("rho_norm_init", "d_rho_norm_init")]
        h = 1e-6
        for x_name, g_name in names:
            x = d[x_name]
            fd = np.empty_like(x)
            for idx in np.ndindex(x.shape):
                xp, xm = x.copy(), x.copy()
                xp[idx] += h
                xm[idx] -= h
                fd[idx] = (_loss(orc, d, **{x_name: xp}) - _loss(orc, d, **{x_name: xm})) / (2 * h)
            got = g[g_name]
            assert got.shape == x.shape, g_name
            np.testing.assert_allclose(got, fd, rtol=2e-6, atol=2e-7, err_msg=f"{g_name} Hv={Hv}")
        if not state:  # zero initial states still get their gradient
            zr, zn = np.zeros((2, 2, 3, 2)), np.zeros((2, 2, 3))
            g2 = orc.backward(d["q"], d["v"], d["decay"], d["dy"], zr, zn)
            np.testing.assert_allclose(g2["d_rho_init"], g["d_rho_init"], rtol=1e-13, atol=1e-15)


def pin_euler_identity(orc):
    """y and rho_final are jointly linear in (v, rho_init); rho_norm_final does
    not depend on them, so sum <dv, v> + <d_rho_init, rho_init> equals the
    loss without its rho_norm_final term."""
    for Hv in (1, 2):
        d = _inputs(2, 8, 2, Hv, 4, 3, seed=21 + Hv)
        g = orc.backward(d["q"], d["v"], d["decay"], d["dy"], d["rho_init"], d["rho_norm_init"], d["d_rho_final"],
                         d["d_rho_norm_final"])
        lhs = float(np.sum(g["dv"] * d["v"]) + np.sum(g["d_rho_init"] * d["rho_init"]))
        rhs = _loss(orc, d, d_rho_norm_final=None)
        assert abs(lhs - rhs) <= 1e-11 * (1 + abs(rhs)), (lhs, rhs)


def pin_shared_value_row(orc):
    d = _inputs(2, 6, 3, 1, 4, 3, seed=31)
    v_full = np.repeat(d["v"], 3, axis=1)
    y1, r1, n1 = orc.forward(d["q"], d["v"], d["decay"], d["rho_init"], d["rho_norm_init"])
    y3, r3, n3 = orc.forward(d["q"], v_full, d["decay"], d["rho_init"], d["rho_norm_init"])
    np.testing.assert_array_equal(y1, y3)
    np.testing.assert_array_equal(r1, r3)
    args = (d["dy"], d["rho_init"], d["rho_norm_init"], d["d_rho_final"], d["d_rho_norm_final"])
    g1 = orc.backward(d["q"], d["v"], d["decay"], *args)
    g3 = orc.backward(d["q"], v_full, d["decay"], *args)
    assert g1["dv"].shape == d["v"].shape
    np.testing.assert_allclose(g1["dv"], g3["dv"].sum(axis=1, keepdims=True), rtol=1e-13, atol=1e-14)
    for k in ("dq", "ddecay", "d_rho_init", "d_rho_norm_init"):
        np.testing.assert_allclose(g1[k], g3[k], rtol=1e-13, atol=1e-14)


def pin_causality(orc):
    d = _inputs(1, 8, 2, 2, 3, 4, seed=41)
    y, _, _ = orc.forward(d["q"], d["v"], d["decay"], d["rho_init"], d["rho_norm_init"])
    t = 4
    v2 = d["v"].copy()
    v2[:, :, t:] += 1.0  # v_t reaches y only from step t + 1 on
    q2 = d["q"].copy()
    q2[:, :, t + 1:] += 1.0
    y2, _, _ = orc.forward(q2, v2, d["decay"], d["rho_init"], d["rho_norm_init"])
    np.testing.assert_array_equal(y[:, :, :t + 1], y2[:, :, :t + 1])
    assert np.abs(y[:, :, t + 1:] - y2[:, :, t + 1:]).min() > 0


PINS = [pin_zero_decay_previous_token, pin_unit_decay_prefix_sums, pin_closed_form, pin_causality,
        pin_shared_value_row, pin_euler_identity, pin_finite_differences]


@pytest.fixture(scope="module")
def orc():
    return load_oracle()


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_rwkv8_oracle_pin(orc, pin):
    pin(orc)
