"""The RWKV-8 pins must catch plausible mistakes in the RWKV-8 oracle.

Each case plants one mistake into a temporary copy of oracle/rwkv8_oracle.py
and requires at least one pin of test_rwkv8_oracle.py to fail against it.
The committed oracle is untouched.
"""
import pytest

import test_rwkv8_oracle as pins

MUTANTS = {
    "weights_not_normalized": ("qw = qt / (qt.sum(axis=-1, keepdims=True) + EPS)\n        rho_hat",
                               "qw = qt\n        rho_hat"),
    "norm_eps_wrong": ("rho_hat = rho / (n[..., None] + EPS)", "rho_hat = rho / (n[..., None] + 1e-3)"),
    "state_not_normalized": ("rho_hat = rho / (n[..., None] + EPS)", "rho_hat = rho"),
    "update_drops_decay": ("rho = d[..., None] * rho + qt[..., None]", "rho = rho + qt[..., None]"),
    "norm_update_drops_decay": ("n = d * n + qt", "n = n + qt"),
    "readout_after_update": ("        y[:, :, t, :] = np.einsum(\"bhl,bhle->bhe\", qw, rho_hat)\n",
                             "        y[:, :, t, :] = np.einsum(\"bhl,bhle->bhe\", qw, (d[..., None] * rho + "
                             "qt[..., None] * vh[:, :, t, None, :]) / (n[..., None] + EPS))\n"),
    "forward_ignores_rho_init": (
        "rho = np.zeros((B, H, L, E)) if rho_init is None else np.array(rho_init, dtype=np.float64)",
        "rho = np.zeros((B, H, L, E))"),
    "dq_drops_norm_carry": ('dq_t = np.einsum("bhle,bhe->bhl", G, vt) + Gn', 'dq_t = np.einsum("bhle,bhe->bhl", G, vt)'),
    "ddecay_drops_norm_term": ("ddecay += (np.einsum(\"bhle,bhle->bhl\", G, rb) + Gn * nb).sum(axis=0)",
                               "ddecay += np.einsum(\"bhle,bhle->bhl\", G, rb).sum(axis=0)"),
    "ddecay_uses_after_state": ("ddecay += (np.einsum(\"bhle,bhle->bhl\", G, rb) + Gn * nb).sum(axis=0)",
                                "ddecay += (np.einsum(\"bhle,bhle->bhl\", G, d[..., None] * rb) + Gn * nb).sum(axis=0)"),
    "norm_grad_sign": ("g_nb = -np.einsum", "g_nb = np.einsum"),
    "norm_grad_power": ("/ den ** 2", "/ den"),
    "weights_grad_drops_projection": ("dq_t += (g_qw - (g_qw * qw).sum(axis=-1, keepdims=True)) / s",
                                      "dq_t += g_qw / s"),
    "carry_drops_decay": ("G = d[..., None] * G + g_rb", "G = G + g_rb"),
    "norm_carry_drops_decay": ("Gn = d * Gn + g_nb", "Gn = Gn + g_nb"),
    "dv_uses_v": ('dv_h[:, :, t, :] = np.einsum("bhle,bhl->bhe", G, qt)',
                  'dv_h[:, :, t, :] = np.einsum("bhle,bhl->bhe", G, qt * 0 + 1)'),
    "shared_value_grad_not_summed": ("dv_h.sum(axis=1, keepdims=True)", "dv_h[:, :1]"),
    "boundary_ignored": (
        "G = np.zeros((B, H, L, E)) if d_rho_final is None else np.array(d_rho_final, dtype=np.float64)",
        "G = np.zeros((B, H, L, E))"),
    "norm_boundary_ignored": (
        "Gn = np.zeros((B, H, L)) if d_rho_norm_final is None else np.array(d_rho_norm_final, dtype=np.float64)",
        "Gn = np.zeros((B, H, L))"),
    "backward_reads_next_state": ("rb, nb = hist_rho[:, :, t], hist_n[:, :, t]",
                                  "rb, nb = hist_rho[:, :, min(t + 1, T - 1)], hist_n[:, :, min(t + 1, T - 1)]"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_rwkv8_mutant_is_caught(name, tmp_path):
    src = open(pins.ORACLE_PATH).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation site of {name} not found exactly once"
    path = tmp_path / f"rwkv8_mutant_{name}.py"
    path.write_text(src.replace(old, new))
    orc = pins.load_oracle(str(path), name=f"rwkv8_mutant_{name}")
    for pin in pins.PINS:
        try:
            pin(orc)
        except (AssertionError, ValueError, FloatingPointError):
            return
    pytest.fail(f"no pin catches the mutant {name}")
