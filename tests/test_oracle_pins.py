"""Pins for the oracle, independent of the oracle's own code.

Each test checks the oracle against something the mathematics fixes: closed
forms of special cases, an unrolled-product brute force, a textbook IIR
filter, exact rational arithmetic with symbolic derivatives, central finite
differences, and identities that follow from how each input enters the
recurrence ("rx_pretrain.c": rx_wkv7_forward_seq, and the reverse-scan
equations (1)-(3) above rx_wkv7_backward).
"""
import itertools

import numpy as np
import pytest


def _inputs(gen, B, T, H, N, seed=0, s_init_std=0.3):
    d = gen.generate(B, T, H, N, "f64", s_init_std, seed=seed)
    return [d[n] for n in ("r", "w", "k", "v", "a", "b")], d["dy"], d["s_init"]


def _loss(oracle, ins, s_init, dy):
    y, _ = oracle.forward(*ins, s_init)
    return float(np.sum(dy * y))


# ---------------------------------------------------------------- forward --

def test_pure_accumulation_closed_form(oracle_mod, gen_mod):
    """a = b = 0, w = 1: S_t = s_init + sum_{s<=t} v_s k_s^T, so
    y_t = s_init r_t + sum_{s<=t} (k_s . r_t) v_s."""
    (r, w, k, v, a, b), _, s0 = _inputs(gen_mod, 2, 20, 3, 8, seed=1, s_init_std=0.5)
    a = np.zeros_like(a); b = np.zeros_like(b); w = np.ones_like(w)
    y, sf = oracle_mod.forward(r, w, k, v, a, b, s0)
    T = r.shape[1]
    kr = np.einsum("bshn,bthn->bhts", k, r) * np.tril(np.ones((T, T)))
    y_ref = np.einsum("bhts,bshi->bthi", kr, v) + np.einsum("bhij,bthj->bthi", s0, r)
    sf_ref = s0 + np.einsum("bshi,bshj->bhij", v, k)
    np.testing.assert_allclose(y, y_ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(sf, sf_ref, rtol=1e-12, atol=1e-12)


def test_memoryless_closed_form(oracle_mod, gen_mod):
    """w = 0, a = b = 0: every step erases the state, y_t = (k_t . r_t) v_t,
    whatever the initial state."""
    (r, w, k, v, a, b), _, s0 = _inputs(gen_mod, 1, 17, 2, 16, seed=2)
    z = np.zeros_like(a)
    y, sf = oracle_mod.forward(r, np.zeros_like(w), k, v, z, z, s0)
    y_ref = np.einsum("bthn,bthn->bth", k, r)[..., None] * v
    np.testing.assert_allclose(y, y_ref, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(sf, np.einsum("bhi,bhj->bhij", v[:, -1], k[:, -1]), rtol=1e-13)


def _unrolled(r, w, k, v, a, b, s0):
    """y and s_final from the product form S_t = s0 A_0..A_t + sum_s v_s k_s^T
    A_{s+1}..A_t with A_t = diag(w_t) + a_t b_t^T (no recursion on S)."""
    B, T, H, N = r.shape
    y = np.zeros_like(r)
    sf = np.zeros((B, H, N, N))
    for bi, hi in itertools.product(range(B), range(H)):
        A = [np.diag(w[bi, t, hi]) + np.outer(a[bi, t, hi], b[bi, t, hi]) for t in range(T)]
        for t in range(T):
            St = s0[bi, hi].copy()
            for u in range(t + 1):
                St = St @ A[u]
            for s in range(t + 1):
                P = np.outer(v[bi, s, hi], k[bi, s, hi])
                for u in range(s + 1, t + 1):
                    P = P @ A[u]
                St = St + P
            y[bi, t, hi] = St @ r[bi, t, hi]
            if t == T - 1:
                sf[bi, hi] = St
    return y, sf


def test_unrolled_product_brute_force(oracle_mod, gen_mod):
    ins, _, s0 = _inputs(gen_mod, 2, 7, 2, 5, seed=3)
    y, sf = oracle_mod.forward(*ins, s0)
    y_ref, sf_ref = _unrolled(*ins, s0)
    np.testing.assert_allclose(y, y_ref, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(sf, sf_ref, rtol=1e-11, atol=1e-13)


def test_scalar_state_is_first_order_iir(oracle_mod):
    """N = 1 with time-invariant inputs: s_t = (w + a b) s_{t-1} + v k is a
    first-order IIR filter; scipy.signal.lfilter computes it."""
    signal = pytest.importorskip("scipy.signal")
    T = 50
    w0, a0, b0, k0, v0, r0, s00 = 0.9, -0.7, 0.4, 0.8, -1.3, 0.6, 0.25
    full = lambda c: np.full((1, T, 1, 1), c)
    y, sf = oracle_mod.forward(full(r0), full(w0), full(k0), full(v0), full(a0), full(b0),
                               np.full((1, 1, 1, 1), s00))
    lam = w0 + a0 * b0
    s, _ = signal.lfilter([1.0], [1.0, -lam], np.full(T, v0 * k0), zi=[lam * s00])
    np.testing.assert_allclose(y[0, :, 0, 0], s * r0, rtol=1e-13)
    np.testing.assert_allclose(sf[0, 0, 0, 0], s[-1], rtol=1e-13)


# --------------------------------------------------------------- exact -----

def test_exact_rational_forward_and_gradients(oracle_mod):
    """T = 3, N = 2 with dyadic inputs (exact in binary): forward from the
    product form and every gradient by symbolic differentiation of
    L = sum dy . y, all in exact rationals (sympy)."""
    sp = pytest.importorskip("sympy")
    T, N = 3, 2
    rng = np.random.default_rng(7)
    dy_ = lambda: rng.integers(-8, 9, size=(T, N)) / 8.0
    vals = {n: rng.integers(-8, 9, size=(T, N)) / 8.0 for n in ("r", "k", "v", "a", "b")}
    vals["w"] = rng.integers(1, 9, size=(T, N)) / 8.0
    s0v = rng.integers(-8, 9, size=(N, N)) / 8.0
    dyv = dy_()
    sym = {n: [[sp.Symbol(f"{n}{t}_{j}") for j in range(N)] for t in range(T)] for n in vals}
    s0s = sp.Matrix(N, N, lambda i, j: sp.Symbol(f"s{i}_{j}"))
    col = lambda n, t: sp.Matrix(N, 1, lambda i, _: sym[n][t][i])
    A = [sp.diag(*sym["w"][t]) + col("a", t) * col("b", t).T for t in range(T)]
    L = 0
    for t in range(T):
        St = s0s
        for u in range(t + 1):
            St = St * A[u]
        for s in range(t + 1):
            P = col("v", s) * col("k", s).T
            for u in range(s + 1, t + 1):
                P = P * A[u]
            St = St + P
        yt = St * col("r", t)
        L = L + sum(sp.Rational(int(dyv[t, i] * 8), 8) * yt[i] for i in range(N))
    subs = {sym[n][t][j]: sp.Rational(int(vals[n][t, j] * 8), 8)
            for n in vals for t in range(T) for j in range(N)}
    subs.update({s0s[i, j]: sp.Rational(int(s0v[i, j] * 8), 8) for i in range(N) for j in range(N)})

    shp = lambda x: np.asarray(x, dtype=np.float64).reshape(1, T, 1, N)
    ins = [shp(vals[n]) for n in ("r", "w", "k", "v", "a", "b")]
    s0 = s0v.reshape(1, 1, N, N)
    dy = shp(dyv)
    y, _ = oracle_mod.forward(*ins, s0)
    assert float(np.sum(dy * y)) == pytest.approx(float(L.subs(subs)), rel=1e-14)
    g = oracle_mod.backward(*ins, dy, s0)
    for n, gname in (("r", "dr"), ("w", "dw"), ("k", "dk"), ("v", "dv"), ("a", "da"), ("b", "db")):
        for t in range(T):
            for j in range(N):
                exact = float(sp.diff(L, sym[n][t][j]).subs(subs))
                assert g[gname][0, t, 0, j] == pytest.approx(exact, rel=1e-13, abs=1e-14), (gname, t, j)
    for i in range(N):
        for j in range(N):
            exact = float(sp.diff(L, s0s[i, j]).subs(subs))
            assert g["dS_init"][0, 0, i, j] == pytest.approx(exact, rel=1e-13, abs=1e-14)


# ------------------------------------------------------------ backward -----

GRAD_OF = {"r": "dr", "w": "dw", "k": "dk", "v": "dv", "a": "da", "b": "db"}
ORDER = ("r", "w", "k", "v", "a", "b")


def _fd_check(oracle, ins, dy, s0, coords, h=1e-5, tol=1e-7):
    """Central differences of L = <dy, y>: truncation error O(h^2), rounding
    O(eps |L| / h), both far below ``tol`` for inputs of order one."""
    g = oracle.backward(*ins, dy, s0)
    for name, idx in coords:
        if name == "s_init":
            base, gval = s0, g["dS_init"][idx]
        else:
            base, gval = ins[ORDER.index(name)], g[GRAD_OF[name]][idx]
        old = base[idx]
        base[idx] = old + h
        lp = _loss(oracle, ins, s0, dy)
        base[idx] = old - h
        lm = _loss(oracle, ins, s0, dy)
        base[idx] = old
        fd = (lp - lm) / (2 * h)
        assert abs(fd - gval) <= tol * max(1.0, abs(gval)), (name, idx, fd, gval)


def test_finite_differences_every_coordinate(oracle_mod, gen_mod):
    ins, dy, s0 = _inputs(gen_mod, 1, 6, 2, 3, seed=4, s_init_std=0.7)
    coords = [(n, idx) for n in ORDER for idx in np.ndindex(ins[0].shape)]
    coords += [("s_init", idx) for idx in np.ndindex(s0.shape)]
    _fd_check(oracle_mod, ins, dy, s0, coords)


def test_finite_differences_sampled_tiny_workload(oracle_mod, gen_mod):
    """The tiny workload's shape (B=1, T=64, H=2, N=16) with a carried-in
    state, 20 random coordinates per tensor."""
    ins, dy, s0 = _inputs(gen_mod, 1, 64, 2, 16, seed=5, s_init_std=0.1)
    rng = np.random.default_rng(0)
    coords = []
    for n in ORDER:
        for _ in range(20):
            coords.append((n, tuple(int(rng.integers(0, s)) for s in ins[0].shape)))
    for _ in range(20):
        coords.append(("s_init", tuple(int(rng.integers(0, s)) for s in s0.shape)))
    _fd_check(oracle_mod, ins, dy, s0, coords, h=1e-5, tol=1e-6)


def test_homogeneity_identities(oracle_mod, gen_mod):
    """y is linear in r_t (row by row), jointly linear in (v, s_init) and in
    (k, s_init); A_t depends on a_t, b_t only through a_t b_t^T and the input
    term on v_t k_t^T. Euler's theorem and these invariances give
      per row:  dr_t . r_t = dy_t . y_t,  da_t . a_t = db_t . b_t,
                dv_t . v_t = dk_t . k_t
      global:   <dy, y> = <dv, v> + <dS_init, s_init> = <dk, k> + <dS_init, s_init>."""
    ins, dy, s0 = _inputs(gen_mod, 2, 64, 3, 16, seed=6, s_init_std=0.4)
    r, w, k, v, a, b = ins
    y, _ = oracle_mod.forward(*ins, s0)
    g = oracle_mod.backward(*ins, dy, s0)
    row = lambda x, z: np.sum(x * z, axis=-1)
    np.testing.assert_allclose(row(g["dr"], r), row(dy, y), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(row(g["da"], a), row(g["db"], b), rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(row(g["dv"], v), row(g["dk"], k), rtol=1e-9, atol=1e-12)
    total = np.sum(dy * y)
    s_term = np.sum(g["dS_init"] * s0)
    assert np.sum(g["dv"] * v) + s_term == pytest.approx(total, rel=1e-10)
    assert np.sum(g["dk"] * k) + s_term == pytest.approx(total, rel=1e-10)


def test_structure_causality_linearity_zero_b(oracle_mod, gen_mod):
    ins, dy, s0 = _inputs(gen_mod, 1, 24, 2, 8, seed=8)
    y, _ = oracle_mod.forward(*ins, s0)
    g = oracle_mod.backward(*ins, dy, s0)
    t0 = 10
    # causality of the forward: inputs after t0 do not change y up to t0
    pert = [x.copy() for x in ins]
    for x in pert:
        x[:, t0 + 1:] += 0.37
    y2, _ = oracle_mod.forward(*pert, s0)
    np.testing.assert_array_equal(y2[:, : t0 + 1], y[:, : t0 + 1])
    # gradients at t >= t0 do not depend on dy before t0
    dy2 = dy.copy()
    dy2[:, :t0] = 5.0
    g2 = oracle_mod.backward(*ins, dy2, s0)
    for n in GRAD_OF.values():
        np.testing.assert_array_equal(g2[n][:, t0:], g[n][:, t0:])
    # every gradient is linear in dy
    g3 = oracle_mod.backward(*ins, 2.5 * dy, s0)
    for n in list(GRAD_OF.values()) + ["dS_init"]:
        np.testing.assert_allclose(g3[n], 2.5 * g[n], rtol=1e-12, atol=1e-14)
    # with b = 0 the in-context term vanishes: da = 0
    ins_b0 = list(ins)
    ins_b0[5] = np.zeros_like(ins[5])
    g4 = oracle_mod.backward(*ins_b0, dy, s0)
    assert np.all(g4["da"] == 0.0)


def test_row_permutation_equivariance(oracle_mod, gen_mod):
    """Permuting the value index i (rows of S) in v, s_init and dy permutes
    y, dv and the rows of dS_init and leaves every column gradient alone."""
    ins, dy, s0 = _inputs(gen_mod, 1, 20, 2, 8, seed=9)
    perm = np.random.default_rng(1).permutation(8)
    r, w, k, v, a, b = ins
    y, sf = oracle_mod.forward(*ins, s0)
    g = oracle_mod.backward(*ins, dy, s0)
    ins_p = [r, w, k, v[..., perm], a, b]
    y_p, sf_p = oracle_mod.forward(*ins_p, s0[:, :, perm, :])
    g_p = oracle_mod.backward(*ins_p, dy[..., perm], s0[:, :, perm, :])
    np.testing.assert_allclose(y_p, y[..., perm], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(sf_p, sf[:, :, perm, :], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(g_p["dv"], g["dv"][..., perm], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(g_p["dS_init"], g["dS_init"][:, :, perm, :], rtol=1e-12, atol=1e-14)
    for n in ("dr", "dw", "dk", "da", "db"):
        np.testing.assert_allclose(g_p[n], g[n], rtol=1e-11, atol=1e-13)


def test_float_template_tracks_double(oracle_mod, gen_mod):
    ins, dy, s0 = _inputs(gen_mod, 1, 64, 2, 16, seed=10, s_init_std=0.1)
    y64, sf64 = oracle_mod.forward(*ins, s0)
    y32, sf32 = oracle_mod.forward(*ins, s0, dtype=np.float32)
    np.testing.assert_allclose(y32, y64, rtol=1e-4, atol=1e-5)
    g64 = oracle_mod.backward(*ins, dy, s0)
    g32 = oracle_mod.backward(*ins, dy, s0, dtype=np.float32)
    for n in g64:
        np.testing.assert_allclose(g32[n], g64[n], rtol=1e-4, atol=1e-4)


def test_backward_heads_matches_whole_run(oracle_mod, gen_mod):
    """The per-head helper used for sampled parity equals the whole run."""
    ins, dy, s0 = _inputs(gen_mod, 2, 30, 3, 8, seed=11)
    y, sf = oracle_mod.forward(*ins, s0)
    g = oracle_mod.backward(*ins, dy, s0)
    heads = [(1, 2), (0, 0)]
    yh, sfh, gh = oracle_mod.backward_heads(*ins, dy, s0, heads)
    for p, (bi, hi) in enumerate(heads):
        np.testing.assert_array_equal(yh[p], y[bi, :, hi])
        np.testing.assert_array_equal(sfh[p], sf[bi, hi])
        for n in GRAD_OF.values():
            np.testing.assert_array_equal(gh[n][p], g[n][bi, :, hi])
        np.testing.assert_array_equal(gh["dS_init"][p], g["dS_init"][bi, hi])


# ------------------------------------- gradient entering through s_final ----
# A sequence cut into segments: the gradient of the loss w.r.t. a segment's
# final state (dS_final) is the next segment's dS_init. Pinned by finite
# differences of L = <dy, y> + <dS_final, s_final>, by composing two segments
# and by Euler's identity for (v, s_init).

def _loss_final(oracle, ins, s_init, dy, dsf):
    y, sf = oracle.forward(*ins, s_init)
    return float(np.sum(dy * y) + np.sum(dsf * sf))


def test_final_state_gradient_finite_differences(oracle_mod, gen_mod):
    ins, dy, s0 = _inputs(gen_mod, 1, 5, 2, 3, seed=21, s_init_std=0.6)
    dsf = np.random.default_rng(21).standard_normal(s0.shape)
    g = oracle_mod.backward(*ins, dy, s0, dsf)
    h = 1e-5
    coords = [(n, idx) for n in ORDER for idx in np.ndindex(ins[0].shape)]
    coords += [("s_init", idx) for idx in np.ndindex(s0.shape)]
    for name, idx in coords:
        if name == "s_init":
            base, gval = s0, g["dS_init"][idx]
        else:
            base, gval = ins[ORDER.index(name)], g[GRAD_OF[name]][idx]
        old = base[idx]
        base[idx] = old + h
        lp = _loss_final(oracle_mod, ins, s0, dy, dsf)
        base[idx] = old - h
        lm = _loss_final(oracle_mod, ins, s0, dy, dsf)
        base[idx] = old
        fd = (lp - lm) / (2 * h)
        assert abs(fd - gval) <= 1e-7 * max(1.0, abs(gval)), (name, idx, fd, gval)


def test_final_state_gradient_composes_segments(oracle_mod, gen_mod):
    """Backward over [0, T) with dS_final equals the backward of [T1, T) with
    dS_final followed by the backward of [0, T1) with the first one's dS_init
    as its dS_final (each segment starting from the state the forward reached)."""
    ins, dy, s0 = _inputs(gen_mod, 2, 23, 2, 5, seed=22, s_init_std=0.4)
    dsf = np.random.default_rng(22).standard_normal(s0.shape)
    full = oracle_mod.backward(*ins, dy, s0, dsf)
    T1 = 9
    first = [x[:, :T1].copy() for x in ins]
    second = [x[:, T1:].copy() for x in ins]
    _, s_mid = oracle_mod.forward(*first, s0)
    g2 = oracle_mod.backward(*second, dy[:, T1:].copy(), s_mid, dsf)
    g1 = oracle_mod.backward(*first, dy[:, :T1].copy(), s0, g2["dS_init"])
    for n in GRAD_OF.values():
        np.testing.assert_allclose(np.concatenate([g1[n], g2[n]], axis=1), full[n], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(g1["dS_init"], full["dS_init"], rtol=1e-12, atol=1e-13)


def test_final_state_gradient_euler_identity(oracle_mod, gen_mod):
    """y and s_final are jointly linear in (v, s_init), so
    sum <dv, v> + <dS_init, s_init> = <dy, y> + <dS_final, s_final>; with dy = 0
    nothing flows into r."""
    ins, dy, s0 = _inputs(gen_mod, 2, 12, 3, 6, seed=23, s_init_std=0.5)
    dsf = np.random.default_rng(23).standard_normal(s0.shape)
    g = oracle_mod.backward(*ins, dy, s0, dsf)
    lhs = np.sum(g["dv"] * ins[3]) + np.sum(g["dS_init"] * s0)
    assert lhs == pytest.approx(_loss_final(oracle_mod, ins, s0, dy, dsf), rel=1e-12)
    g0 = oracle_mod.backward(*ins, np.zeros_like(dy), s0, dsf)
    assert np.all(g0["dr"] == 0.0)
