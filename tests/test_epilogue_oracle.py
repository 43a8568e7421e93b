"""Pins of the epilogue oracle (oracle/epilogue_oracle.py: group norm per head
with "rx_pretrain.c"'s gn_forward, plus the bonus (sum_j r_j k_j r_k[j]) v):

* closed forms: with ln_w = 1, ln_b = 0 and r_k = 0 every head of the output
  has mean 0 and mean square var / (var + 64e-5); with ln_w = 0 the output is
  ln_b + bonus * v with the bonus summed term by term;
* every gradient (dy, dr, dk, dv, dln_w, dln_b, dr_k) against central
  differences of sum <dout, out>;
* invariance: adding a constant to a head's y leaves the output unchanged,
  so dy sums to zero over each head;
* planted mistakes fail a pin.
"""
import importlib.util
import os

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PATH = os.path.join(ROOT, "oracle", "epilogue_oracle.py")
EPS = 64e-5


def load(path=PATH, name="epilogue_oracle_under_test"):
    spec = importlib.util.spec_from_file_location(name, path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _inputs(seed, B=2, T=3, H=2, N=5):
    rng = np.random.default_rng(seed)
    d = {n: rng.standard_normal((B, T, H, N)) for n in ("y", "r", "k", "v", "dout")}
    d["ln_w"] = rng.uniform(0.5, 1.5, (H, N))
    d["ln_b"] = 0.1 * rng.standard_normal((H, N))
    d["r_k"] = rng.standard_normal((H, N))
    return d


def pin_closed_forms(orc):
    d = _inputs(1)
    H, N = d["ln_w"].shape
    out, st = orc.forward(d["y"], d["r"], d["k"], d["v"], np.ones((H, N)), np.zeros((H, N)), np.zeros((H, N)))
    var = d["y"].var(axis=-1)
    np.testing.assert_allclose(out.mean(axis=-1), 0.0, atol=1e-13)
    np.testing.assert_allclose((out ** 2).mean(axis=-1), var / (var + EPS), rtol=1e-12)
    out2, st2 = orc.forward(d["y"], d["r"], d["k"], d["v"], np.zeros((H, N)), d["ln_b"], d["r_k"])
    B, T = d["y"].shape[:2]
    for b in range(B):
        for t in range(T):
            for h in range(H):
                s = sum(d["r"][b, t, h, j] * d["k"][b, t, h, j] * d["r_k"][h, j] for j in range(N))
                np.testing.assert_allclose(out2[b, t, h], d["ln_b"][h] + s * d["v"][b, t, h], rtol=1e-12, atol=1e-14)


def pin_finite_differences(orc):
    d = _inputs(2)
    g = orc.backward(d["dout"], d["y"], d["r"], d["k"], d["v"], d["ln_w"], d["ln_b"], d["r_k"])
    names = ("y", "r", "k", "v", "ln_w", "ln_b", "r_k")

    def loss(**over):
        x = {n: over.get(n, d[n]) for n in names}
        out, _ = orc.forward(x["y"], x["r"], x["k"], x["v"], x["ln_w"], x["ln_b"], x["r_k"])
        return float(np.sum(d["dout"] * out))

    h = 1e-6
    for x_name, g_name in (("y", "dy"), ("r", "dr"), ("k", "dk"), ("v", "dv"), ("ln_w", "dln_w"), ("ln_b", "dln_b"),
                           ("r_k", "dr_k")):
        x = d[x_name]
        fd = np.empty_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            fd[idx] = (loss(**{x_name: xp}) - loss(**{x_name: xm})) / (2 * h)
        np.testing.assert_allclose(g[g_name], fd, rtol=1e-6, atol=1e-7, err_msg=g_name)


def pin_shift_invariance(orc):
    d = _inputs(3)
    out, _ = orc.forward(d["y"], d["r"], d["k"], d["v"], d["ln_w"], d["ln_b"], d["r_k"])
    shift = np.random.default_rng(4).standard_normal(d["y"].shape[:3])[..., None]
    out2, _ = orc.forward(d["y"] + shift, d["r"], d["k"], d["v"], d["ln_w"], d["ln_b"], d["r_k"])
    np.testing.assert_allclose(out2, out, rtol=1e-11, atol=1e-12)
    g = orc.backward(d["dout"], d["y"], d["r"], d["k"], d["v"], d["ln_w"], d["ln_b"], d["r_k"])
    np.testing.assert_allclose(g["dy"].sum(axis=-1), 0.0, atol=1e-12)


PINS = [pin_closed_forms, pin_shift_invariance, pin_finite_differences]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_epilogue_pin(pin):
    pin(load())


MUTANTS = {
    "eps_dropped": ("rs = 1.0 / np.sqrt(var + GN_EPS)\n            s = (r[b, t] * k[b, t] * r_k).sum(axis=-1)\n            out",
                    "rs = 1.0 / np.sqrt(var)\n            s = (r[b, t] * k[b, t] * r_k).sum(axis=-1)\n            out"),
    "bonus_without_r_k": ("s = (r[b, t] * k[b, t] * r_k).sum(axis=-1)\n            out",
                          "s = (r[b, t] * k[b, t]).sum(axis=-1)\n            out"),
    "shift_on_bonus": ("* ln_w + ln_b + s[:, None] * v[b, t]", "* ln_w + s[:, None] * (v[b, t] + ln_b)"),
    "gn_grad_drops_mean": ('g["dy"][b, t] = rs[:, None] * (dn - mdn[:, None] - nv * mdnn[:, None])',
                           'g["dy"][b, t] = rs[:, None] * (dn - nv * mdnn[:, None])'),
    "gn_grad_drops_projection": ('g["dy"][b, t] = rs[:, None] * (dn - mdn[:, None] - nv * mdnn[:, None])',
                                 'g["dy"][b, t] = rs[:, None] * (dn - mdn[:, None])'),
    "dr_uses_r": ('g["dr"][b, t] = db[:, None] * k[b, t] * r_k', 'g["dr"][b, t] = db[:, None] * r[b, t] * r_k'),
    "dv_drops_bonus": ('g["dv"][b, t] = do * s[:, None]', 'g["dv"][b, t] = do'),
    "dln_w_unnormalized": ('g["dln_w"] += do * nv', 'g["dln_w"] += do * yt'),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_epilogue_mutant_is_caught(name, tmp_path):
    src = open(PATH).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, name
    p = tmp_path / f"epi_{name}.py"
    p.write_text(src.replace(old, new))
    orc = load(str(p), f"epi_{name}")
    for pin in PINS:
        try:
            pin(orc)
        except AssertionError:
            return
    pytest.fail(f"no pin catches the mutant {name}")
