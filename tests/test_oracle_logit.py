"""Pins of the oracle's decay-from-logit chain (oracle.decay_from_logit,
forward_logit, backward_logit): the time-mix of "rx_pretrain.c"
(tm_pre_forward and its backward) forms w = exp(-0.606531 sigmoid(z)).

* closed forms of w at z -> -inf, z = 0 and z -> +inf;
* dz against fp64 central differences of L = sum <dy, y> + <dS_final, s_final>
  with respect to z, with and without an initial state and dS_final;
* planted mistakes in the chain (a dropped factor, a wrong sign) fail the
  finite-difference pin.
"""
import importlib.util
import os

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
COEFF = 0.606531  # RX_WDECAY_COEFF


def _inputs(B, T, H, N, seed, state):
    rng = np.random.default_rng(seed)
    d = {n: rng.standard_normal((B, T, H, N)) / np.sqrt(N) for n in ("r", "k", "v")}
    d["z"] = rng.standard_normal((B, T, H, N))
    kk = rng.standard_normal((B, T, H, N))
    kk /= np.linalg.norm(kk, axis=-1, keepdims=True)
    d["a"], d["b"] = -kk, kk * rng.uniform(0.2, 0.8, (B, T, H, N))
    d["dy"] = rng.standard_normal((B, T, H, N))
    d["s_init"] = 0.2 * rng.standard_normal((B, H, N, N)) if state else None
    d["dS_final"] = rng.standard_normal((B, H, N, N)) if state else None
    return d


def pin_closed_form(orc):
    w = orc.decay_from_logit(np.array([-60.0, 0.0, 60.0]))
    np.testing.assert_allclose(w, [1.0, np.exp(-COEFF / 2), np.exp(-COEFF)], rtol=1e-14)


def pin_finite_differences(orc):
    for state in (False, True):
        d = _inputs(1, 6, 2, 3, seed=5 + state, state=state)
        ins = [d[n] for n in ("r", "z", "k", "v", "a", "b")]
        g = orc.backward_logit(*ins, d["dy"], d["s_init"], d["dS_final"])

        def loss(z):
            y, sf = orc.forward_logit(d["r"], z, d["k"], d["v"], d["a"], d["b"], d["s_init"])
            val = float(np.sum(d["dy"] * y))
            if d["dS_final"] is not None:
                val += float(np.sum(d["dS_final"] * sf))
            return val

        h = 1e-6
        fd = np.empty_like(d["z"])
        for idx in np.ndindex(d["z"].shape):
            zp, zm = d["z"].copy(), d["z"].copy()
            zp[idx] += h
            zm[idx] -= h
            fd[idx] = (loss(zp) - loss(zm)) / (2 * h)
        np.testing.assert_allclose(g["dz"], fd, rtol=1e-6, atol=1e-8)


PINS = [pin_closed_form, pin_finite_differences]


@pytest.fixture(scope="module")
def orc(oracle_mod):
    return oracle_mod


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_logit_pin(orc, pin):
    pin(orc)


MUTANTS = {
    "drops_w": ('g.pop("dw") * w * (-WDECAY_COEFF)', 'g.pop("dw") * (-WDECAY_COEFF)'),
    "sign": ('g.pop("dw") * w * (-WDECAY_COEFF)', 'g.pop("dw") * w * WDECAY_COEFF'),
    "drops_one_minus_sigmoid": ("* sig * (1.0 - sig)", "* sig"),
    "decay_without_sigmoid": ("np.exp(-WDECAY_COEFF / (1.0 + np.exp(-z)))", "np.exp(-WDECAY_COEFF * z)"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_logit_mutant_is_caught(oracle_mod, name, tmp_path):
    src = open(os.path.join(ROOT, "oracle", "__init__.py")).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, name
    pkg = tmp_path / "oracle_mut"
    pkg.mkdir()
    (pkg / "__init__.py").write_text(src.replace(old, new).replace(
        '_HERE = os.path.dirname(os.path.abspath(__file__))', f'_HERE = {os.path.join(ROOT, "oracle")!r}'))
    spec = importlib.util.spec_from_file_location(f"oracle_mut_{name}", pkg / "__init__.py")
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    for pin in PINS:
        try:
            pin(mod)
        except AssertionError:
            return
    pytest.fail(f"no pin catches the mutant {name}")
