"""Writes oracle_tiny.json beside this script: the oracles' outputs on tiny
seeded inputs, kept as a regression fixture of the oracle itself.

Every value here comes from oracle/ (the WKV7 scan of "rx_pretrain.c", the
RWKV-8 recurrence of "src/sequence/rwkv8/backward.rs" and the time-mix
epilogue) applied to inputs of linear_rnn_state_gb300.inputs, the seeded
generator both sides share; nothing is computed any other way. The pages print
no worked example, so these fixtures pin nothing by themselves: the oracle is
pinned by the tests of test_oracle_pins.py and its siblings, and this file
only makes any later change to the oracle's arithmetic show up (regenerate it
on purpose, naming in the commit the passage or reading that justifies the
change).

Run from the repository root: python tests/golden/make_golden.py
"""
import importlib.util
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_tiny.json")


def _l(x):
    return None if x is None else np.asarray(x, dtype=np.float64).ravel().tolist()


def cases():
    import oracle
    from linear_rnn_state_gb300 import inputs

    def load(name):
        spec = importlib.util.spec_from_file_location(name, os.path.join(ROOT, "oracle", f"{name}.py"))
        m = importlib.util.module_from_spec(spec)
        spec.loader.exec_module(m)
        return m

    r8, epi = load("rwkv8_oracle"), load("epilogue_oracle")
    out = {}

    # WKV7 scan, fp64 inputs with an initial state
    shp = dict(B=1, T=5, H=2, N=4)
    d = inputs.generate(shp["B"], shp["T"], shp["H"], shp["N"], "f64", 0.1, seed=2024)
    names = ("r", "w", "k", "v", "a", "b")
    y, sf = oracle.forward(*(d[n] for n in names), d["s_init"])
    g = oracle.backward(*(d[n] for n in names), d["dy"], d["s_init"])
    out["wkv7"] = {"shape": shp, "seed": 2024, "s_init_std": 0.1,
                   "inputs": {n: _l(d[n]) for n in names + ("dy", "s_init")},
                   "y": _l(y), "s_final": _l(sf), **{k: _l(v) for k, v in g.items()}}

    # the decay given as logits
    z = inputs.generate_logits(shp["B"], shp["T"], shp["H"], shp["N"], "f64", seed=2025)
    yl, sfl = oracle.forward_logit(d["r"], z, d["k"], d["v"], d["a"], d["b"])
    gl = oracle.backward_logit(d["r"], z, d["k"], d["v"], d["a"], d["b"], d["dy"])
    out["wkv7_logit"] = {"seed_z": 2025, "z": _l(z), "y": _l(yl), "s_final": _l(sfl),
                         **{k: _l(v) for k, v in gl.items()}}

    # the epilogue on the scan's y
    rng = np.random.default_rng(7)
    H, N = shp["H"], shp["N"]
    ln_w, ln_b, r_k = rng.uniform(0.5, 1.5, (H, N)), 0.1 * rng.standard_normal((H, N)), rng.standard_normal((H, N))
    eo, st = epi.forward(y, d["r"], d["k"], d["v"], ln_w, ln_b, r_k)
    eg = epi.backward(d["dy"], y, d["r"], d["k"], d["v"], ln_w, ln_b, r_k)
    out["epilogue"] = {"params": {"ln_w": _l(ln_w), "ln_b": _l(ln_b), "r_k": _l(r_k)}, "out": _l(eo),
                       **{f"stats_{k}": _l(v) for k, v in st.items()}, **{k: _l(v) for k, v in eg.items()}}

    # RWKV-8 with initial states and final-state gradients, one shared value row
    s8 = dict(B=1, T=6, H=2, Hv=1, L=4, E=3)
    d8 = inputs.generate_rwkv8(s8["B"], s8["T"], s8["H"], s8["Hv"], s8["L"], s8["E"], "f32", state_std=0.1,
                               boundary=True, seed=2026)
    o8 = {k: None if x is None else x.astype(np.float64) for k, x in d8.items()}
    y8, rf8, nf8 = r8.forward(o8["q"], o8["v"], o8["decay"], o8["rho_init"], o8["rho_norm_init"])
    g8 = r8.backward(o8["q"], o8["v"], o8["decay"], o8["dy"], o8["rho_init"], o8["rho_norm_init"],
                     o8["d_rho_final"], o8["d_rho_norm_final"])
    out["rwkv8"] = {"shape": s8, "seed": 2026, "inputs": {k: _l(x) for k, x in o8.items()}, "y": _l(y8),
                    "rho_final": _l(rf8), "rho_norm_final": _l(nf8), **{k: _l(v) for k, v in g8.items()}}
    return out


if __name__ == "__main__":
    with open(OUT, "w") as f:
        json.dump(cases(), f, indent=0, sort_keys=True)
        f.write("\n")
    print(f"wrote {OUT} ({os.path.getsize(OUT)} bytes)")
